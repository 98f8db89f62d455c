"""The benchmark's multi-rank logic on CPU: two ranks over gloo (as torchrun
would start them, rendezvous on 127.0.0.1) go through the same process-group
setup, barrier, max/min-over-ranks timing and weak-scaling aggregation that
bench.py uses with NCCL on GPUs, and the reference arm does no work on ranks
other than 0.  The job is sharded by sequence: every (sequence, head) unit of
the whole job is computed by exactly one rank, on exactly the values the
whole job's generator gives it."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import argparse, json, os, sys
sys.path.insert(0, os.environ["KDA_ROOT"])
import bench
args = argparse.Namespace(impl="kda", gpus=2, steps=3, warmup=1)
ws, rank, local = bench.dist_setup(args)
import torch.distributed as dist
assert dist.is_initialized() and dist.get_backend() == "gloo"
bench.barrier(ws)
elapsed = [12.5, 20.0][rank]           # each rank's own timed region, ms
tput = [4.0e6, 3.0e6][rank]            # each rank's own end-to-end throughput
wr = bench.rank_workload(bench.get_workload(bench.WORKLOAD), rank, ws)
res = {"rank": rank, "ws": ws, "seq_base": wr.seq_base, "num_seqs": wr.num_seqs, "tok_base": wr.tok_base,
       "max_ms": bench.max_over_ranks(elapsed, ws),
       "min_tput": bench.min_over_ranks(tput, ws),
       "value": bench.job_throughput(1000.0, 3, bench.max_over_ranks(elapsed, ws), ws)}
bench.barrier(ws)
dist.destroy_process_group()
ref = argparse.Namespace(impl="reference", gpus=2, steps=1, warmup=0)
if rank != 0:
    bench.run_reference(ref)           # must return at once, printing nothing
print("RESULT " + json.dumps(res), flush=True)
"""


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_time_and_aggregate_like_the_benchmark():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, KDA_ROOT=ROOT, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2",
                   RANK=str(rank), LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", CHILD], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=240)
        except subprocess.TimeoutExpired:
            for q in procs:
                q.kill()
            raise
        assert p.returncode == 0, err[-2000:]
        lines = [ln for ln in out.splitlines() if ln.startswith("RESULT ")]
        assert len(lines) == 1 and out.strip() == lines[0], out   # nothing else printed (no reference line)
        outs.append(json.loads(lines[0][len("RESULT "):]))
    assert sorted((r["seq_base"], r["num_seqs"]) for r in outs) == [(0, 1), (1, 1)]   # one sequence each
    assert sorted(r["tok_base"] for r in outs) == [0, 65536]
    for r in outs:
        assert r["ws"] == 2
        assert r["max_ms"] == 20.0                      # the job takes as long as its slowest rank
        assert r["min_tput"] == 3.0e6                   # end-to-end: the slowest rank, times the ranks
        assert abs(r["value"] - 2 * 1000.0 * 3 / 0.020) < 1e-6


def test_shards_cover_every_sequence_and_head_once():
    sys.path.insert(0, ROOT)
    import numpy as np

    import bench
    import kda_synth as ks

    for name in ("prefill_b1_h32_t65536_d128", "prefill_b8_h96_t8192_d128", "varlen_12seq_1m_h32_d128"):
        w = ks.workloads()[name]
        for ws in (1, 2, 3, 4, 8):
            wg = bench.global_workload(w, ws)
            assert wg.num_seqs == w.num_seqs * ws and wg.tokens == w.tokens * ws
            seen = {}
            for rank in range(ws):
                wr = bench.rank_workload(w, rank, ws)
                assert wr.num_seqs == w.num_seqs and wr.tokens == w.tokens   # weak scaling: same work per rank
                for s in range(wr.num_seqs):
                    for h in range(wr.H):
                        key = (wr.seq_base + s, h)
                        assert key not in seen, (name, ws, key)
                        seen[key] = rank
            assert set(seen) == {(s, h) for s in range(wg.num_seqs) for h in range(wg.H)}
            # a rank's values are the whole job's values of its sequences
            wr = bench.rank_workload(w, ws - 1, ws)
            s_loc = wr.num_seqs - 1
            a = wr.chain_inputs(s_loc, wr.H - 1, ntok=64)
            b = wg.chain_inputs(wr.seq_base + s_loc, wr.H - 1, ntok=64)
            for k in ("q", "k", "v", "g", "beta"):
                assert np.array_equal(a[k], b[k]), (name, ws, k)
            if w.s0_std is not None:
                assert np.array_equal(a["s0"], b["s0"])
