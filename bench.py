#!/usr/bin/env python
"""Benchmark of the KDA recurrence library on GB300.

Headline: chunked-prefill tokens/s on B=1, H=32, T=65536, d_k=d_v=128 (bf16
q/k/v/g, fp32 beta and state, initial state N(0, 0.01)), inputs resident in
HBM (2.1 GB of inputs per step, larger than the 129 MB L2, so no flush is
needed between steps).  One step = one kda_chunk_fwd call over the whole
workload.  Also reported on the same JSON line:

* ``roofline``: the dominant kernel's algorithmic bytes per launch over its
  mean launch time (CUDA events recorded by the library around each launch on
  its stream during the timed region), against the measured HBM copy peak;
* ``path_roofline``: the same for the whole step;
* ``e2e``: the same metric through the Python API with pinned host buffers
  (inputs copied in and o + final state copied out inside every timed step);
* ``decode``: 100 decode steps of 256 sequences x 96 heads (fp32 state
  128x128 per head), GB/s against the same peak;
* ``cpu_baseline``: the fp64 CPU oracle on a bounded sample of the workload;
* ``clocks``: nvidia-smi samples taken during the timed region.

``--impl reference`` times the CPU oracle instead (the only reference this
method has), on the same workload and metric.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

WORKLOAD = "prefill_b1_h32_t65536_d128"
PROFILE_WORKLOAD = "prefill_b1_h32_t8192_d128"   # same shape and recipe, 8192 tokens (268 MB of inputs)
METRIC = "KDA prefill tokens/s (H=32,d=128,T=64K); decode GB/s; % of GB300 roofline"
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["kda", "reference"], default="kda")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-snapshots", action="store_true")
    ap.add_argument("--no-gated", action="store_true")
    ap.add_argument("--no-ablation", action="store_true",
                    help="skip the decay-map ablation (diagonal tiles by position pairs, bounded and -Softplus maps)")
    ap.add_argument("--snapshot-interval", type=int, default=512)
    ap.add_argument("--decode-steps", type=int, default=100)
    ap.add_argument("--decode-only", action="store_true",
                    help="run only the decode legs (a short command for profiler captures of the decode kernels)")
    ap.add_argument("--workload", choices=[WORKLOAD, PROFILE_WORKLOAD, "prefill_b8_h96_t8192_d128",
                                           "varlen_12seq_1m_h32_d128"], default=WORKLOAD,
                    help="the headline workload (default), a T=8192 cut of it for profiler captures, "
                         "or one of the other prefill workloads")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# ----------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def _selector(self):
        import torch

        try:
            u = torch.cuda.get_device_properties(self.dev).uuid
            return ["-i", "GPU-" + str(u)]
        except Exception:
            return []

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits", "-lms", "50",
               *self._selector()]
        try:
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.2)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == len(self.FIELDS):
                rows.append(parts)
        os.unlink(self.path)
        sm = [float(r[1]) for r in rows if re.match(r"^[0-9.]+$", r[1])]
        smax = [float(r[2]) for r in rows if re.match(r"^[0-9.]+$", r[2])]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, val in zip(names, r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ------------------------------------------------------ library profiling hook
def _prof(lib, on: bool):
    lib.kda_profile_enable.argtypes = [ctypes.c_int32]
    lib.kda_profile_enable(1 if on else 0)


def _collect(lib, max_records=4096):
    lib.kda_profile_collect.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32]
    lib.kda_profile_collect.restype = ctypes.c_int32
    names = ctypes.create_string_buffer(64 * max_records)
    ms = (ctypes.c_float * max_records)()
    seen = lib.kda_profile_collect(names, ms, max_records)
    recs = []
    for i in range(min(seen, max_records)):
        nm = names.raw[64 * i: 64 * i + 64].split(b"\0", 1)[0].decode()
        recs.append((nm, float(ms[i])))
    return seen, recs


# Source text each kernel's machine code depends on: the shared headers, plus
# its own translation unit with the other kernels' sections cut out (marker
# lines of kda_chunk_tc.cu), so that a change elsewhere does not invalidate a
# committed ncu traffic figure.
_TC_SECTIONS = {"chunk_prep_tc": [("// -------------------------------------------------------------- chain kernel",
                                   "// --------------------------------------------------------------- host side")]}


def _kernel_src_sha(kernel: str = "", csrc: str = "") -> str:
    h = hashlib.sha256()
    d = csrc or os.path.join(ROOT, "linear_attention_recurrence_chunk_gb300", "csrc")
    if kernel in _TC_SECTIONS:
        for fn in ("kda_internal.cuh", "tc_ptx.cuh", "chain_common.cuh", "prep_split_body.cuh"):
            h.update(open(os.path.join(d, fn), "rb").read())
        text = open(os.path.join(d, "kda_chunk_tc.cu"), encoding="utf-8").read()
        for a, b in _TC_SECTIONS[kernel]:
            i, j = text.index(a), text.index(b)
            text = text[:i] + text[j:]
        h.update(text.encode("utf-8"))
        return h.hexdigest()[:16]
    for fn in sorted(os.listdir(d)):
        if fn.endswith((".cu", ".cuh")):
            h.update(open(os.path.join(d, fn), "rb").read())
    return h.hexdigest()[:16]


def _traffic_from_profiles(kernel: str, units_per_launch: float, pdir: str = "", csrc: str = ""):
    """DRAM bytes per launch of ``kernel`` from the committed ncu summaries, if
    they were taken on the current kernel sources (else None)."""
    pdir = pdir or os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    sha = _kernel_src_sha(kernel, csrc)
    pat = re.compile(r"^traffic:\s+kernel=(\S+)\s+dram_bytes_per_unit=([0-9.eE+-]+)\s+src_sha=(\S+)")
    for fn in sorted(os.listdir(pdir)):
        if not fn.endswith((".md", ".txt")):
            continue
        for line in open(os.path.join(pdir, fn)):
            m = pat.match(line.strip())
            if m and m.group(1) == kernel and m.group(3) == sha:
                return float(m.group(2)) * units_per_launch
    return None


# ---------------------------------------------------------------- workloads
def prefill_alg_bytes(w, kernel: str) -> float:
    """Algorithmic bytes the kernel must move per launch: the path's inputs
    (q, k, g, v, beta) belong to the kernel that reads them, its outputs (o,
    final state) and the initial state to the kernel that writes / reads them."""
    eb = 2 if w.dtype == "bf16" else 4
    ht = w.tokens * w.H
    inputs = ht * ((3 * w.d_k + w.d_v) * eb + 4)
    outputs = ht * w.d_v * eb
    states = w.num_seqs * w.H * w.d_k * w.d_v * 4 * (2 if w.s0_std is not None else 1)
    if "prep" in kernel:
        return float(inputs)
    if "chain" in kernel:
        return float(outputs + states)
    if "fused" in kernel or kernel == "path":
        return float(inputs + outputs + states)
    return 0.0


def get_workload(name):
    import kda_synth as ks

    if name == PROFILE_WORKLOAD:
        w = ks.workloads()[WORKLOAD]
        w.name, w.T = PROFILE_WORKLOAD, 8192
        return w
    return ks.workloads()[name]


def global_workload(w, ws: int):
    """The whole job at ``ws`` ranks under weak scaling: ``ws`` copies of the
    workload's shape as one batch of sequences (B x ws sequences, or the varlen
    length list repeated ws times), each with its own seeded values."""
    import dataclasses

    if ws == 1:
        return w
    if w.seq_lens is None:
        return dataclasses.replace(w, name=f"{w.name}_x{ws}", B=w.B * ws)
    lens = np.tile(np.asarray(w.seq_lens), ws)
    return dataclasses.replace(w, name=f"{w.name}_x{ws}", T=int(lens.sum()), seq_lens=lens)


def shard_sequences(num_seqs: int, ws: int):
    """(first sequence, count) of each rank: contiguous blocks, sizes differing
    by at most one, every sequence (with all its heads) on exactly one rank."""
    base, extra = divmod(num_seqs, ws)
    out, first = [], 0
    for r in range(ws):
        n = base + (1 if r < extra else 0)
        out.append((first, n))
        first += n
    return out


def rank_workload(w, rank: int, ws: int):
    """This rank's part of the whole job: its block of sequences, all heads."""
    if ws == 1:
        return w
    wg = global_workload(w, ws)
    first, n = shard_sequences(wg.num_seqs, ws)[rank]
    return wg.shard(first, n, name=f"{wg.name}[seqs {first}:{first + n}]")


def maybe_spawn(args) -> bool:
    """``--gpus N`` (N > 1) without a launcher: start N local ranks under
    torch.distributed.run on 127.0.0.1 with the same arguments and wait for
    them.  Returns True when it did (this process then only relays)."""
    if args.gpus <= 1 or "WORLD_SIZE" in os.environ:
        return False
    import socket

    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *sys.argv[1:]]
    rc = subprocess.call(cmd)
    if rc != 0:
        sys.exit(rc)
    return True


def dist_setup(args):
    import torch

    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    if ws > 1 and args.impl == "kda":
        import torch.distributed as dist

        # one process per GPU over NCCL; gloo where there is no GPU (host-side tests)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo", init_method="env://")
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def min_over_ranks(x: float, ws: int) -> float:
    return -max_over_ranks(-x, ws)


def job_throughput(units_per_rank: float, steps: int, max_ms: float, ws: int) -> float:
    """Whole-job units/s under weak scaling: every rank processes the same
    units per step; the job takes as long as its slowest rank."""
    return ws * units_per_rank * steps / (max_ms / 1e3)


def bench_prefill(args, ws_size, local):
    import torch

    import kda_synth as ks
    import linear_attention_recurrence_chunk_gb300 as kda
    from kda_synth.torchio import prefill_inputs

    ws_rank = int(os.environ.get("RANK", "0"))
    w = rank_workload(get_workload(args.workload), ws_rank, ws_size)
    t = prefill_inputs(w, "cuda")
    lib = kda.load_library()
    stream = torch.cuda.current_stream()
    o = torch.empty_like(t["v"])
    sf = torch.empty((w.num_seqs, w.H, w.d_k, w.d_v), dtype=torch.float32, device="cuda")
    ws_bytes = kda.kda_chunk_fwd_workspace_size(w.B, w.T, w.H, w.d_k, w.d_v, w.num_seqs, torch.bfloat16)
    wsp = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")

    def step():
        kda.kda_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], initial_state=t["s0"], cu_seqlens=t["cu"],
                          o=o, final_state=sf, workspace=wsp, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st, code = kda.kda_device_error()
    if st != 0:
        raise RuntimeError(f"device error {code} during warm-up")

    sampler = ClockSampler(local)
    barrier(ws_size)
    torch.cuda.synchronize()
    sampler.start()
    _prof(lib, True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    _prof(lib, False)
    barrier(ws_size)
    clocks = sampler.stop()
    elapsed_ms = e0.elapsed_time(e1)
    seen, recs = _collect(lib)
    max_ms = max_over_ranks(elapsed_ms, ws_size)

    per_kernel = {}
    for nm, ms in recs:
        per_kernel.setdefault(nm, []).append(ms)
    return {"w": w, "t": t, "elapsed_ms": elapsed_ms, "max_ms": max_ms, "launches": seen,
            "per_kernel": per_kernel, "clocks": clocks, "o": o, "sf": sf, "wsp": wsp}


def timed_steps(step, steps: int, stream):
    """Runs ``steps`` calls of ``step`` with a CUDA event before each and after
    the last, on the launch stream.  Returns (mean ms per step, spread) where
    spread holds the per-step min / median / max."""
    import torch

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record(stream)
    for i in range(steps):
        step()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    total = ev[0].elapsed_time(ev[steps])
    return total / steps, {"min_ms": min(per), "median_ms": statistics.median(per), "max_ms": max(per)}


def side_leg_steps(steps: int) -> int:
    """Timed steps of each side leg: at least 20."""
    return max(20, steps // 10)


def bench_snapshots(args, r, steps):
    """The same prefill with the state kept every ``--snapshot-interval`` tokens
    (the prefix-cache snapshots, 512 tokens on the pages), timed with CUDA
    events on the launch stream like the main leg."""
    import torch

    import linear_attention_recurrence_chunk_gb300 as kda

    w, t = r["w"], r["t"]
    every = args.snapshot_interval
    slots = (w.tokens // every) if t["cu"] is not None else w.B * (w.T // every)
    snaps = torch.empty((max(slots, 1), w.H, w.d_k, w.d_v), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        kda.kda_chunk_fwd_snapshots(t["q"], t["k"], t["v"], t["g"], t["beta"], every, initial_state=t["s0"],
                                    cu_seqlens=t["cu"], o=r["o"], final_state=r["sf"], snapshots=snaps,
                                    workspace=r["wsp"], stream=stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    st, code = kda.kda_device_error()
    if st != 0:
        raise RuntimeError(f"device error {code} in the snapshot leg")
    ms, spread = timed_steps(step, steps, stream)
    plain_ms = r["elapsed_ms"] / args.steps
    del snaps
    return {"interval_tokens": every, "snapshots_per_step": slots * w.H,
            "snapshot_bytes_per_step": slots * w.H * w.d_k * w.d_v * 4, "value": w.tokens / (ms / 1e3),
            "unit": "tokens/s", "ms_per_step": ms, "steps": steps, "spread": spread,
            "slowdown_vs_plain": ms / plain_ms}


def bench_gated(args, r, steps):
    """The same prefill with the output epilogue (Sigmoid gate times the per-head
    RMSNorm of o) fused before o is written; synthetic gate logits and norm
    weights of the workload's shape."""
    import torch

    import linear_attention_recurrence_chunk_gb300 as kda

    w, t = r["w"], r["t"]
    gen = torch.Generator(device="cuda").manual_seed(77)
    gate = torch.randn(t["v"].shape, generator=gen, device="cuda").to(torch.bfloat16)
    nw = 1 + 0.1 * torch.randn((w.H, w.d_v), generator=gen, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        kda.kda_chunk_fwd_gated(t["q"], t["k"], t["v"], t["g"], t["beta"], gate, norm_weight=nw,
                                initial_state=t["s0"], cu_seqlens=t["cu"], o=r["o"], final_state=r["sf"],
                                workspace=r["wsp"], stream=stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    st, code = kda.kda_device_error()
    if st != 0:
        raise RuntimeError(f"device error {code} in the gated leg")
    lib = kda.load_library()
    _prof(lib, True)
    ms, spread = timed_steps(step, steps, stream)
    _prof(lib, False)
    _, recs = _collect(lib)
    per = {}
    for nm, v in recs:
        per.setdefault(nm, []).append(v)
    kernels = {nm: round(statistics.mean(v), 4) for nm, v in per.items()}
    if "chunk_chain_tc_gated" in kernels:
        note = ("fused into the 32-column chain: the CTAs of a head form a cluster and exchange row sums of "
                "squares")
    else:
        note = "fused into the all-columns chain: the o warps of the CTA exchange row sums of squares"
    del gate, nw
    return {"value": w.tokens / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms, "steps": steps,
            "spread": spread, "slowdown_vs_plain": ms / (r["elapsed_ms"] / args.steps), "kernels_ms": kernels,
            "note": note}


def bench_decay_ablation(args, r, steps):
    """The ablation of the lower-bounded decay on the same workload: the
    diagonal 16x16 tiles of the intra-chunk matrices formed pair by pair on the
    CUDA cores (one exponential per position pair and key channel) instead of
    on the tensor cores, first under the bounded map itself (the cost of the
    slow path alone), then under the unbounded -Softplus map that needs it.
    Whole-call and per-kernel times with CUDA events on the launch stream."""
    import torch

    import linear_attention_recurrence_chunk_gb300 as kda

    lib = kda.load_library()
    w, t = r["w"], r["t"]
    stream = torch.cuda.current_stream()
    # The pair paths run the single-stream prep kernel and the chain as two
    # kernels, so the tensor-core diagonal is timed the same way here: the same
    # single-stream kernel structure (KDA_PREP_STREAMS=1, which also runs two
    # kernels), beside the plain call as it runs by default.
    plain_ms = r["elapsed_ms"] / args.steps
    default_ms = plain_ms
    default_prep = statistics.mean(r["per_kernel"]["chunk_prep_tc"]) if "chunk_prep_tc" in r["per_kernel"] else None
    os.environ["KDA_PREP_STREAMS"] = "1"
    try:
        def plain_step():
            kda.kda_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], initial_state=t["s0"],
                              cu_seqlens=t["cu"], o=r["o"], final_state=r["sf"], workspace=r["wsp"],
                              stream=stream)

        for _ in range(max(3, args.warmup)):
            plain_step()
        torch.cuda.synchronize()
        _prof(lib, True)
        plain_ms, _ = timed_steps(plain_step, steps, stream)
        _prof(lib, False)
        _, recs = _collect(lib)
        plain_prep = statistics.mean([v for nm, v in recs if nm == "chunk_prep_tc_single"])
    finally:
        del os.environ["KDA_PREP_STREAMS"]
    out = {"tensor_core_diagonal": {"ms_per_step": plain_ms, "prep_ms": plain_prep, "prep_kernel": "single-stream",
                                    "default_call_ms": default_ms, "default_prep_ms": default_prep}}
    for name, dmap in (("bounded_pairs", kda.DECAY_BOUNDED), ("softplus_pairs", kda.DECAY_SOFTPLUS)):
        def step():
            kda.kda_chunk_fwd_decay_variant(t["q"], t["k"], t["v"], t["g"], t["beta"], decay_map=dmap,
                                            diag_by_pairs=True, initial_state=t["s0"], cu_seqlens=t["cu"],
                                            o=r["o"], final_state=r["sf"], workspace=r["wsp"], stream=stream)

        for _ in range(max(3, args.warmup)):
            step()
        torch.cuda.synchronize()
        st, code = kda.kda_device_error()
        if st != 0:
            raise RuntimeError(f"device error {code} in the {name} leg")
        _prof(lib, True)
        ms, spread = timed_steps(step, steps, stream)
        _prof(lib, False)
        _, recs = _collect(lib)
        prep = [v for nm, v in recs if nm.startswith("chunk_prep_tc")]
        prep_ms = statistics.mean(prep) if prep else None
        out[name] = {"ms_per_step": ms, "prep_ms": prep_ms, "value": w.tokens / (ms / 1e3), "unit": "tokens/s",
                     "steps": steps, "spread": spread, "slowdown_vs_tensor_core": ms / plain_ms,
                     "prep_slowdown_vs_tensor_core": (prep_ms / plain_prep) if prep_ms else None}
    return out


def bench_e2e(args, w, wsp, steps):
    """Same metric through the Python API from pinned host buffers: every step
    copies its inputs host -> device, runs the call and copies o and the final
    state back.  Steps are pipelined the way a caller streaming requests would:
    two device buffer sets, the next step's inputs copied on one stream while
    the current step computes on another and its results return on a third
    (host -> device is the bound: ~210 GB/s measured on these boxes)."""
    import torch

    import linear_attention_recurrence_chunk_gb300 as kda
    from kda_synth.torchio import prefill_inputs

    host = {k: v for k, v in prefill_inputs(w, "cpu", pin=True).items() if k != "cu" and v is not None}
    dev = [{k: torch.empty(v.shape, dtype=v.dtype, device="cuda") for k, v in host.items()} for _ in range(2)]
    outs = [(torch.empty(dev[0]["v"].shape, dtype=dev[0]["v"].dtype, device="cuda"),
             torch.empty((w.num_seqs, w.H, w.d_k, w.d_v), dtype=torch.float32, device="cuda")) for _ in range(2)]
    o_host = [torch.empty(dev[0]["v"].shape, dtype=dev[0]["v"].dtype).pin_memory() for _ in range(2)]
    sf_host = [torch.empty((w.num_seqs, w.H, w.d_k, w.d_v), dtype=torch.float32).pin_memory() for _ in range(2)]
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = o_host[0].numel() * o_host[0].element_size() + sf_host[0].numel() * 4
    ev = lambda: torch.cuda.Event()
    copied, computed, returned = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    for b_ in range(2):   # the buffers start free
        computed[b_].record(s_run)
        returned[b_].record(s_out)

    def step(i):
        b_ = i % 2
        with torch.cuda.stream(s_in):   # inputs of step i, once step i-2 no longer reads the set
            s_in.wait_event(computed[b_])
            for k_ in host:
                dev[b_][k_].copy_(host[k_], non_blocking=True)
            copied[b_].record(s_in)
        with torch.cuda.stream(s_run):   # the call, once its inputs landed and step i-2's results left
            s_run.wait_event(copied[b_])
            s_run.wait_event(returned[b_])
            x = dev[b_]
            kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], initial_state=x["s0"], o=outs[b_][0],
                              final_state=outs[b_][1], workspace=wsp, stream=s_run)
            computed[b_].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(computed[b_])
            o_host[b_].copy_(outs[b_][0], non_blocking=True)
            sf_host[b_].copy_(outs[b_][1], non_blocking=True)
            returned[b_].record(s_out)

    for i in range(2):
        step(i)
    torch.cuda.synchronize()
    block = 5   # steps per spread sample
    e0 = torch.cuda.Event(enable_timing=True)
    marks = []
    t0 = time.perf_counter()
    e0.record(s_in)   # before the first timed copy in ...
    for i in range(steps):
        step(i)
        if (i + 1) % block == 0 or i + 1 == steps:   # ... after a copy out, which follows every earlier step
            e = torch.cuda.Event(enable_timing=True)
            e.record(s_out)
            marks.append((i + 1, e))
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    ms = e0.elapsed_time(marks[-1][1])
    per_block, prev_n, prev_t = [], 0, 0.0
    for n_, e in marks:
        t_ = e0.elapsed_time(e)
        per_block.append((t_ - prev_t) / (n_ - prev_n))
        prev_n, prev_t = n_, t_
    return {"value": w.tokens * steps / (ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": steps, "ms_per_step": ms / steps,
            "spread": {"blocks_of_steps": block, "min_ms": min(per_block), "median_ms": statistics.median(per_block),
                       "max_ms": max(per_block)},
            "wall_s": round(wall, 3), "pipelined": "next step's inputs copied while the current one computes"}


def bench_decode(args, peak_gbs):
    import torch

    import kda_synth as ks
    import linear_attention_recurrence_chunk_gb300 as kda

    d = ks.workloads()["decode_n256_h96_d128_x100"]
    steps = min(args.decode_steps, d.steps)
    heads = d.N * d.H
    lib = kda.load_library()
    state = torch.from_numpy(d.fill_state()).reshape(d.N, d.H, d.d_k, d.d_v).cuda()
    toks = []
    for s in range(steps):
        x = {}
        for name, width in (("q", d.d_k), ("k", d.d_k), ("v", d.d_v), ("g", d.d_k)):
            a = d.fill_step(s, name)
            x[name] = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).reshape(d.N, d.H, width).cuda()
        x["beta"] = torch.from_numpy(d.fill_step(s, "beta")).reshape(d.N, d.H).cuda()
        toks.append(x)
    o = torch.empty((d.N, d.H, d.d_v), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    # warm-up on a scratch copy of the state (the timed steps start from the seeded state)
    scratch = state.clone()
    for s in range(3):
        x = toks[s]
        kda.kda_decode_step(x["q"], x["k"], x["v"], x["g"], x["beta"], scratch, o=o, stream=stream)
    del scratch
    torch.cuda.synchronize()
    _prof(lib, True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s in range(steps):
        x = toks[s]
        kda.kda_decode_step(x["q"], x["k"], x["v"], x["g"], x["beta"], state, o=o, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    _prof(lib, False)
    seen, recs = _collect(lib)
    ms = e0.elapsed_time(e1)
    per_step_bytes = heads * (2 * d.d_k * d.d_v * 4 + (3 * d.d_k + d.d_v) * 2 + 4 + d.d_v * 2)
    kms = [m for n, m in recs if n == "decode_step"]
    kmean = statistics.mean(kms) if kms else ms / steps
    gbs = per_step_bytes / (kmean / 1e3) / 1e9
    res = {"workload": d.name, "steps": steps, "ms_per_step": ms / steps, "kernel_ms": kmean,
           "bytes_per_step": per_step_bytes, "GB/s": gbs, "frac": gbs / peak_gbs, "gpu_launches": seen}

    # The fused layer step on the same shapes: conv width 4, gated RMSNorm output.
    # Per head-step it moves the state (R+W), q/k/v/z/gate in, o out, beta logit
    # and the conv cache (R+W); the conv and norm weights are shared by all sequences.
    W, C = 4, 2 * d.d_k + d.d_v
    cache = torch.zeros((d.N, d.H, W - 1, C), dtype=torch.bfloat16, device="cuda")
    conv_w = torch.full((d.H, C, W), 0.25, dtype=torch.float32, device="cuda")
    A_log = torch.zeros(d.H, dtype=torch.float32, device="cuda")
    nw = torch.ones((d.H, d.d_v), dtype=torch.float32, device="cuda")

    def layer(x, st):
        kda.kda_decode_layer_step(x["q"], x["k"], x["v"], x["g"], A_log, x["beta"], cache, conv_w, st,
                                  out_gate=x["v"], norm_weight=nw, o=o, stream=stream)

    scratch = state.clone()
    for s in range(3):
        layer(toks[s], scratch)
    del scratch
    torch.cuda.synchronize()
    _prof(lib, True)
    e0.record(stream)
    for s in range(steps):
        layer(toks[s], state)
    e1.record(stream)
    torch.cuda.synchronize()
    _prof(lib, False)
    seen2, recs2 = _collect(lib)
    ms2 = e0.elapsed_time(e1)
    layer_bytes = heads * (2 * d.d_k * d.d_v * 4 + (3 * d.d_k + 2 * d.d_v) * 2 + 4 + d.d_v * 2 + 2 * (W - 1) * C * 2) \
        + d.H * (C * W + d.d_v + 1) * 4
    kms2 = [m for n, m in recs2 if n == "decode_layer"]
    kmean2 = statistics.mean(kms2) if kms2 else ms2 / steps
    gbs2 = layer_bytes / (kmean2 / 1e3) / 1e9
    res["layer_step"] = {"conv_width": W, "out_gate": True, "ms_per_step": ms2 / steps, "kernel_ms": kmean2,
                         "bytes_per_step": layer_bytes, "GB/s": gbs2, "frac": gbs2 / peak_gbs, "gpu_launches": seen2}
    return res


def oracle_sample(w, ntok):
    """The fp64 oracle, as it stands, on every head of sequence 0 over its
    first ``ntok`` tokens.  Returns (outputs, threads used)."""
    import oracle

    ins = [w.chain_inputs(0, h, ntok) for h in range(w.H)]
    n = [len(x["beta"]) for x in ins]
    cat = {k: np.concatenate([x[k] for x in ins]) for k in ("q", "k", "v", "g", "beta")}
    s0 = None if w.s0_std is None else np.stack([x["s0"] for x in ins]).astype(np.float64)
    row0 = np.concatenate([[0], np.cumsum(n)[:-1]])
    dt = oracle.BF16 if w.dtype == "bf16" else oracle.F32
    outs, _, threads = oracle.chains(cat["q"], cat["k"], cat["v"], cat["g"], cat["beta"], dt, w.d_k, w.d_v, 1,
                                     row0, n, s0)
    return outs, threads


def cpu_baseline(w, target_s=12.0):
    """The fp64 oracle as it stands, on all heads over the first n tokens
    (n picked from a short probe so that the run takes about ``target_s``)."""
    import oracle

    probe_tok = 512
    t0 = time.perf_counter()
    _, threads = oracle_sample(w, probe_tok)
    probe = time.perf_counter() - t0
    n = int(min(w.T, max(1024, probe_tok * target_s / max(probe, 1e-3))))
    n = max(1024, (n // 1024) * 1024)
    t0 = time.perf_counter()
    _, threads = oracle_sample(w, n)
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"all {w.H} heads x first {n} tokens of {w.name} (fp64 C oracle, OpenMP over heads)",
            "seconds": round(dt, 3), "max_threads": oracle.max_threads()}


def run_reference(args):
    """CPU oracle arm: each step runs the oracle on a bounded sample of the
    workload (all heads, n tokens), n sized so that warm-up + steps take about
    a minute."""
    import kda_synth as ks

    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = ks.workloads()[WORKLOAD]
    t0 = time.perf_counter()
    _, threads = oracle_sample(w, 256)
    probe = time.perf_counter() - t0
    budget = 60.0 / max(1, args.steps + args.warmup)
    n = int(max(16, min(w.T, 256 * budget / max(probe, 1e-4))))
    for _ in range(args.warmup):
        oracle_sample(w, n)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample(w, n)
    dt = time.perf_counter() - t0
    value = n * args.steps / dt
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "d_k": w.d_k, "d_v": w.d_v},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": f"per step: all {w.H} heads x first {n} tokens of {w.name}"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if maybe_spawn(args):
        return
    if args.impl == "reference":
        run_reference(args)
        return
    import torch

    ws_size, rank, local = dist_setup(args)
    peak, peak_kind = peaks()
    if args.decode_only:
        dec = bench_decode(args, peak)
        if rank == 0:
            print(json.dumps({"metric": "KDA decode GB/s (256 sequences x 96 heads, d=128)", "value": dec["GB/s"],
                              "unit": "GB/s", "n_gpus": ws_size, "decode": dec}), flush=True)
        return
    r = bench_prefill(args, ws_size, local)
    w = r["w"]
    steps = args.steps
    value = job_throughput(w.tokens, steps, r["max_ms"], ws_size)

    # dominant kernel = largest total time in the timed region
    totals = {k: sum(v) for k, v in r["per_kernel"].items()}
    dom = max(totals, key=totals.get) if totals else None
    roof = None
    if dom:
        mean_ms = statistics.mean(r["per_kernel"][dom])
        alg = prefill_alg_bytes(w, dom)
        ach = alg / (mean_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": dom, "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
                "peak_source": peak_kind, "alg_bytes_per_launch": alg, "mean_launch_ms": mean_ms,
                "traffic": _traffic_from_profiles(dom, w.tokens * w.H),
                "share": totals[dom] / max(sum(totals.values()), 1e-9)}
    path_alg = prefill_alg_bytes(w, "path")
    path_ach = path_alg / (r["max_ms"] / steps / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws_size, "steps": steps,
        "warmup": args.warmup, "ms_per_step": r["max_ms"] / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "head_tokens_per_s": value * w.H,   # a token is one position across all H heads
        "config": {"workload": args.workload, "B": w.B, "T": w.T, "H": w.H, "d_k": w.d_k, "d_v": w.d_v,
                   "state": "fp32, S0 ~ N(0, 0.01)", "chunk": 64,
                   "l2": "no flush: 2.1 GB of inputs per step, larger than L2",
                   "parallelism": ("single GPU" if ws_size == 1 else
                                   f"dp{ws_size}: the job is {ws_size} x the workload's sequences; each rank runs "
                                   f"its own block of sequences (all heads), no collective on the data path"),
                   "global_sequences": w.num_seqs * ws_size},
        "roofline": roof,
        "path_roofline": {"bound": "hbm", "achieved": path_ach, "peak": peak, "unit": "GB/s",
                          "frac": path_ach / peak, "alg_bytes_per_step": path_alg},
        "kernels": {k: {"launches": len(v), "mean_ms": statistics.mean(v), "share": totals[k] / sum(totals.values())}
                    for k, v in r["per_kernel"].items()},
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
    }
    if not args.no_snapshots:
        line["snapshots"] = bench_snapshots(args, r, side_leg_steps(steps))
    if not args.no_gated:
        line["gated"] = bench_gated(args, r, side_leg_steps(steps))
    if not args.no_ablation:
        line["decay_ablation"] = bench_decay_ablation(args, r, side_leg_steps(steps))
    if not args.no_e2e:
        line["e2e"] = bench_e2e(args, w, r["wsp"], side_leg_steps(steps))
        if ws_size > 1:
            line["e2e"]["value"] = min_over_ranks(line["e2e"]["value"], ws_size) * ws_size
    del r
    torch.cuda.empty_cache()
    if not args.no_decode:
        line["decode"] = bench_decode(args, peak)
    if rank == 0 and ws_size == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws_size > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
