"""The C-ABI library without a GPU: it loads, exports every entry point that
include/kda.h declares, sizes workspaces, and rejects bad arguments on the
host before any CUDA call."""
import ctypes
import os
import re

import pytest

import linear_attention_recurrence_chunk_gb300 as kda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"KDA_API\s+[\w\s\*]*?\b(kda_\w+)\s*\(", text))
    return names


def test_library_exports_every_declared_symbol():
    lib = kda.load_library()
    names = _declared()
    assert {"kda_chunk_fwd", "kda_decode_step", "kda_chunk_fwd_workspace_size", "kda_status_string",
            "kda_device_error"} <= names
    for n in names:
        assert hasattr(lib, n), f"{n} not exported by {kda.library_path()}"


def test_status_strings():
    lib = kda.load_library()
    for code, name in kda.STATUS.items():
        assert lib.kda_status_string(code).decode() == name
    assert lib.kda_status_string(77).decode() == "KDA_ERR_UNKNOWN"


def test_workspace_size():
    lib = kda.load_library()
    f = lib.kda_chunk_fwd_workspace_size
    a = f(1, 65536, 32, 128, 128, 1, 1)
    b = f(1, 65536 * 2, 32, 128, 128, 1, 1)
    assert 0 < a < b
    assert f(8, 8192, 96, 128, 128, 8, 1) > 0
    # varlen form: B = 1, many sequences
    assert f(1, 1 << 20, 32, 128, 128, 12, 1) >= f(1, 1 << 20, 32, 128, 128, 1, 1)
    SIZE_MAX = (1 << 64) - 1
    assert f(1, 100, 32, 96, 128, 1, 1) == SIZE_MAX      # unsupported head size
    assert f(2, 100, 32, 128, 128, 3, 1) == SIZE_MAX      # batched: num_seqs must be B... or varlen with B != 1
    assert f(1, -1, 32, 128, 128, 1, 1) == SIZE_MAX
    assert f(1, 100, 0, 128, 128, 1, 1) == SIZE_MAX
    assert f(1, 100, 2, 128, 128, 1, 7) == SIZE_MAX       # bad dtype


FAKE = 1 << 40   # never dereferenced: every case below fails validation first


def _chunk(lib, **kw):
    args = dict(q=FAKE, k=FAKE + (1 << 30), v=FAKE + (2 << 30), g=FAKE + (3 << 30), beta=FAKE + (4 << 30),
                s0=None, cu=None, num_seqs=1, B=1, T=64, H=2, dk=128, dv=128, dt=1, o=FAKE + (5 << 30),
                sf=None, ws=FAKE + (6 << 30), wsb=1 << 40)
    args.update(kw)
    return lib.kda_chunk_fwd(args["q"], args["k"], args["v"], args["g"], args["beta"], args["s0"], args["cu"],
                             args["num_seqs"], args["B"], args["T"], args["H"], args["dk"], args["dv"], args["dt"],
                             args["o"], args["sf"], args["ws"], args["wsb"], None)


def test_chunk_fwd_rejects_bad_arguments_on_host():
    lib = kda.load_library()
    assert _chunk(lib, q=None) == 1
    assert _chunk(lib, ws=None) == 1
    assert _chunk(lib, dk=96) == 2
    assert _chunk(lib, dv=32) == 2
    assert _chunk(lib, dt=5) == 1
    assert _chunk(lib, q=FAKE + 8) == 1                         # 16-byte alignment
    assert _chunk(lib, beta=FAKE + (4 << 30) + 2) == 1          # beta: 4-byte alignment
    assert _chunk(lib, ws=FAKE + (6 << 30) + 16) == 1          # 256-byte workspace alignment
    assert _chunk(lib, wsb=1024) == 1                           # workspace too small
    assert _chunk(lib, o=FAKE + 4096) == 1                      # o overlaps q
    assert _chunk(lib, B=2, num_seqs=2, cu=FAKE + (7 << 30)) == 1   # varlen needs B == 1
    assert _chunk(lib, B=2, num_seqs=1) == 1                    # batched needs num_seqs == B
    assert _chunk(lib, H=0) == 1
    assert _chunk(lib, T=-5) == 1
    # final state overlapping an input other than initial_state
    assert _chunk(lib, sf=FAKE + (2 << 30)) == 1
    # B = 0: nothing to do, no CUDA call
    assert _chunk(lib, B=0, num_seqs=0) == 0


def _snap(lib, **kw):
    args = dict(q=FAKE, k=FAKE + (1 << 30), v=FAKE + (2 << 30), g=FAKE + (3 << 30), beta=FAKE + (4 << 30),
                s0=None, cu=None, num_seqs=2, B=2, T=1024, H=2, dk=128, dv=128, dt=1, o=FAKE + (5 << 30),
                sf=None, snaps=FAKE + (8 << 30), interval=512, cap=4, ws=FAKE + (6 << 30), wsb=1 << 40)
    args.update(kw)
    return lib.kda_chunk_fwd_snapshots(args["q"], args["k"], args["v"], args["g"], args["beta"], args["s0"],
                                       args["cu"], args["num_seqs"], args["B"], args["T"], args["H"], args["dk"],
                                       args["dv"], args["dt"], args["o"], args["sf"], args["snaps"],
                                       args["interval"], args["cap"], args["ws"], args["wsb"], None)


def test_chunk_fwd_snapshots_rejects_bad_arguments_on_host():
    lib = kda.load_library()
    assert _snap(lib, interval=0) == 1                          # no interval
    assert _snap(lib, interval=-64) == 1
    assert _snap(lib, interval=100) == 1                        # not a multiple of the 64-token chunk
    assert _snap(lib, cap=3) == 1                               # B * floor(T / interval) = 4 slots needed
    assert _snap(lib, cap=-1) == 1
    assert _snap(lib, snaps=None) == 1                          # snapshots needed but no buffer
    assert _snap(lib, snaps=FAKE + (8 << 30) + 4) == 1          # 16-byte alignment
    assert _snap(lib, snaps=FAKE + (2 << 30) + 64) == 1         # overlaps v
    assert _snap(lib, snaps=FAKE + (5 << 30) + 64) == 1         # overlaps o
    # varlen: floor(T / interval) slots bound the total
    assert _snap(lib, B=1, num_seqs=3, cu=FAKE + (7 << 30), T=2048, cap=3) == 1
    assert _snap(lib, q=None) == 1                              # the kda_chunk_fwd checks still apply
    assert _snap(lib, dk=96) == 2
    assert _snap(lib, B=0, num_seqs=0, cap=0) == 0              # nothing to do, no CUDA call


def _gated(lib, **kw):
    args = dict(q=FAKE, k=FAKE + (1 << 30), v=FAKE + (2 << 30), g=FAKE + (3 << 30), beta=FAKE + (4 << 30),
                s0=None, cu=None, num_seqs=1, B=1, T=64, H=2, dk=128, dv=128, dt=1, o=FAKE + (5 << 30),
                sf=None, gate=FAKE + (8 << 30), nw=FAKE + (9 << 30), eps=1e-6, ws=FAKE + (6 << 30), wsb=1 << 40)
    args.update(kw)
    return lib.kda_chunk_fwd_gated(args["q"], args["k"], args["v"], args["g"], args["beta"], args["s0"], args["cu"],
                                   args["num_seqs"], args["B"], args["T"], args["H"], args["dk"], args["dv"],
                                   args["dt"], args["o"], args["sf"], args["gate"], args["nw"], args["eps"],
                                   args["ws"], args["wsb"], None)


def test_chunk_fwd_gated_rejects_bad_arguments_on_host():
    lib = kda.load_library()
    assert _gated(lib, gate=None) == 1                          # the gate is the point of the call
    assert _gated(lib, dt=0) == 2                               # fp32: not on the tensor-core path
    assert _gated(lib, dk=64) == 2
    assert _gated(lib, gate=FAKE + (8 << 30) + 2) == 1          # 16-byte alignment
    assert _gated(lib, nw=FAKE + (9 << 30) + 4) == 1
    assert _gated(lib, eps=-1.0) == 1
    assert _gated(lib, gate=FAKE + (5 << 30) + 64) == 1         # o overlaps the gate
    assert _gated(lib, q=None) == 1                             # the kda_chunk_fwd checks still apply
    assert _gated(lib, B=0, num_seqs=0) == 0                    # nothing to do, no CUDA call


def _variant(lib, **kw):
    args = dict(q=FAKE, k=FAKE + (1 << 30), v=FAKE + (2 << 30), g=FAKE + (3 << 30), beta=FAKE + (4 << 30),
                s0=None, cu=None, num_seqs=1, B=1, T=64, H=2, dk=128, dv=128, dt=1, o=FAKE + (5 << 30),
                sf=None, dmap=1, pairs=1, ws=FAKE + (6 << 30), wsb=1 << 40)
    args.update(kw)
    return lib.kda_chunk_fwd_decay_variant(args["q"], args["k"], args["v"], args["g"], args["beta"], args["s0"],
                                           args["cu"], args["num_seqs"], args["B"], args["T"], args["H"], args["dk"],
                                           args["dv"], args["dt"], args["o"], args["sf"], args["dmap"],
                                           args["pairs"], args["ws"], args["wsb"], None)


def test_chunk_fwd_decay_variant_rejects_bad_arguments_on_host():
    lib = kda.load_library()
    assert _variant(lib, dmap=2) == 1 and _variant(lib, dmap=-1) == 1   # no such decay map
    assert _variant(lib, pairs=2) == 1
    assert _variant(lib, dmap=1, pairs=0) == 2                  # the unbounded map needs the pair path
    assert _variant(lib, dt=0) == 2                             # fp32: not on the tensor-core path
    assert _variant(lib, dk=64) == 2
    assert _variant(lib, dmap=0, pairs=1, dv=96) == 2
    assert _variant(lib, q=None) == 1                           # the kda_chunk_fwd checks still apply
    assert _variant(lib, dmap=2, B=0, num_seqs=0) == 1          # checked before the empty-batch return
    assert _variant(lib, B=0, num_seqs=0) == 0                  # nothing to do, no CUDA call


def test_decode_rejects_bad_arguments_on_host():
    lib = kda.load_library()
    f = lib.kda_decode_step
    p = [FAKE + (i << 30) for i in range(8)]
    assert f(p[0], p[1], p[2], p[3], p[4], p[5], 0, 96, 128, 128, 1, p[6], None) == 0     # N = 0: no-op
    assert f(None, p[1], p[2], p[3], p[4], p[5], 4, 96, 128, 128, 1, p[6], None) == 1
    assert f(p[0], p[1], p[2], p[3], p[4], p[5], 4, 96, 80, 128, 1, p[6], None) == 2
    assert f(p[0], p[1], p[2], p[3], p[4], p[5], 4, 0, 128, 128, 1, p[6], None) == 1
    assert f(p[0], p[1], p[2], p[3], p[4], p[5] + 4, 4, 96, 128, 128, 1, p[6], None) == 1  # misaligned state
    assert f(p[0], p[1], p[2], p[3], p[4], p[5], 4, 96, 128, 128, 1, p[5], None) == 1      # o overlaps state
    assert f(p[0], p[1], p[2], p[3], p[4], p[5], 4, 96, 128, 128, 3, p[6], None) == 1      # bad dtype


def _layer(lib, **kw):
    p = [FAKE + (i << 30) for i in range(14)]
    a = dict(q=p[0], k=p[1], v=p[2], z=p[3], A=p[4], bl=p[5], cache=p[6], w=p[7], W=4, state=p[8], gate=p[9],
             nw=p[10], e1=1e-6, e2=1e-6, N=4, H=8, dk=128, dv=128, dt=1, o=p[11])
    a.update(kw)
    return lib.kda_decode_layer_step(a["q"], a["k"], a["v"], a["z"], a["A"], a["bl"], a["cache"], a["w"], a["W"],
                                     a["state"], a["gate"], a["nw"], a["e1"], a["e2"], a["N"], a["H"], a["dk"],
                                     a["dv"], a["dt"], a["o"], None)


def test_decode_layer_step_rejects_bad_arguments_on_host():
    lib = kda.load_library()
    assert _layer(lib, N=0) == 0                                   # no-op, no CUDA call
    assert _layer(lib, q=None) == 1
    assert _layer(lib, W=0) == 1 and _layer(lib, W=9) == 1          # conv width 1..8
    assert _layer(lib, cache=None) == 1                             # width 4 needs the cache
    assert _layer(lib, dk=96) == 2
    assert _layer(lib, dt=7) == 1
    assert _layer(lib, e1=-1.0) == 1 and _layer(lib, e2=float("nan")) == 1
    assert _layer(lib, state=FAKE + (8 << 30) + 4) == 1             # state: 16-byte alignment
    assert _layer(lib, q=FAKE + 1) == 1                             # bf16 element alignment
    assert _layer(lib, A=FAKE + (4 << 30) + 2) == 1                 # fp32 alignment
    assert _layer(lib, o=FAKE + (2 << 30) + 64) == 1                # o overlaps v_in
    assert _layer(lib, cache=FAKE + (8 << 30) + 256) == 1           # the cache overlaps the state
    assert _layer(lib, H=0) == 1


def test_wait_timeout_check_rejects_bad_limits_on_host():
    lib = kda.load_library()
    assert lib.kda_check_wait_timeout(0, None) == 1
    assert lib.kda_check_wait_timeout(-5, None) == 1
    assert lib.kda_check_wait_timeout(10**9 + 1, None) == 1


def test_python_binding_has_no_cpu_path():
    """The binding's functions only marshal: on CPU tensors the library must
    refuse (the pointers are host pointers), never compute on the host."""
    import torch

    if torch.cuda.is_available():
        pytest.skip("checks the no-GPU behaviour")
    q = torch.zeros(1, 4, 1, 64)
    with pytest.raises(Exception):
        kda.kda_chunk_fwd(q, q, q, q, torch.zeros(1, 4, 1))
