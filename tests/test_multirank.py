"""The benchmark's multi-rank logic on CPU: two ranks over gloo (as torchrun
would start them, rendezvous on 127.0.0.1) go through the same process-group
setup, barrier, max/min-over-ranks timing and weak-scaling aggregation that
bench.py uses with NCCL on GPUs, and the reference arm does no work on ranks
other than 0."""
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
res = {"rank": rank, "ws": ws,
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
    for r in outs:
        assert r["ws"] == 2
        assert r["max_ms"] == 20.0                      # the job takes as long as its slowest rank
        assert r["min_tput"] == 3.0e6                   # end-to-end: the slowest rank, times the ranks
        assert abs(r["value"] - 2 * 1000.0 * 3 / 0.020) < 1e-6
