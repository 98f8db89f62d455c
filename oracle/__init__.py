"""fp64 CPU oracle of the KDA recurrence -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  It shares no code with the CUDA library (the
library never imports it) and follows the recurrence token by token as
written on the page "Kimi K3：架构、训练与百万 Token Agentic RL 技术解读":
§3.1 (the KDA update ``S_t = (I - beta k k^T) Diag(alpha) S_{t-1} + beta k v^T``,
``o_t = S_t^T q_t``), §3.2 (the order decay -> read -> write error -> read out)
and §3.3 (``log alpha = -5 * Sigmoid(logit)``); optionally the unbounded
``log alpha = -Softplus(logit)`` of the predecessor model (page "Kimi K3 架构篇：
一文详解 2.8 万亿参数的巨型怪兽", "最被低估的一个细节：下界衰减").  The arithmetic is in
``kda_oracle.c``; this module compiles it with gcc and marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_SO = os.path.join(_HERE, "libkda_oracle.so")

F32, BF16, F64 = 0, 1, 2
DECAY_BOUNDED, DECAY_SOFTPLUS = 0, 1
_NP = {F32: np.float32, BF16: np.uint16, F64: np.float64}


def build(force: bool = False) -> str:
    """Compile the oracle into ``libkda_oracle.so`` (gcc -O3, OpenMP, no FMA
    contraction so x86-64 and aarch64 agree)."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    subprocess.run(["gcc", "-O3", "-std=c99", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", _SRC,
                    "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _SO)
    return _SO


_handle = None


def _lib():
    global _handle
    if _handle is None:
        lib = ctypes.CDLL(build())
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        lib.kda_oracle_chains.argtypes = [vp, vp, vp, vp, i32, vp, i64, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        lib.kda_oracle_chains.restype = ctypes.c_int
        lib.kda_oracle_chains_snap.argtypes = [vp, vp, vp, vp, i32, vp, i64, i32, i32, i32, vp, vp, vp, vp, vp, vp,
                                               i64, vp, vp]
        lib.kda_oracle_chains_snap.restype = ctypes.c_int
        lib.kda_oracle_chains_map.argtypes = [vp, vp, vp, vp, i32, vp, i64, i32, i32, i32, vp, vp, vp, vp, vp, vp,
                                              i64, vp, vp, i32]
        lib.kda_oracle_chains_map.restype = ctypes.c_int
        lib.kda_oracle_max_threads.argtypes = []
        lib.kda_oracle_max_threads.restype = ctypes.c_int
        _handle = lib
    return _handle


def max_threads() -> int:
    return int(_lib().kda_oracle_max_threads())


def _arr(x, dtype_code):
    a = np.ascontiguousarray(x)
    if a.dtype != _NP[dtype_code]:
        raise TypeError(f"expected {_NP[dtype_code]}, got {a.dtype}")
    return a


def chains(q, k, v, g, beta, dtype: int, d_k: int, d_v: int, row_stride: int,
           row0: Sequence[int], n: Sequence[int], s0: Optional[np.ndarray] = None, snap_every: int = 0,
           decay_map: int = DECAY_BOUNDED):
    """Run independent chains over shared token arrays.

    ``q, k, g``: rows of ``d_k`` values, ``v``: rows of ``d_v`` (storage dtype:
    float32, bfloat16 bits as uint16, or float64); ``beta`` float32 per row.
    Chain c reads rows ``row0[c] + j*row_stride`` for ``j < n[c]``; ``s0`` is
    ``[nchains, d_k, d_v]`` fp64 (or None = zeros).
    Returns (list of ``[n[c], d_v]`` fp64 outputs, ``[nchains, d_k, d_v]`` fp64
    final states, threads used); with ``snap_every > 0`` a fourth item, the list
    of ``[n[c] // snap_every, d_k, d_v]`` fp64 states after every ``snap_every``
    tokens of each chain.  ``decay_map``: ``DECAY_BOUNDED`` (-5 Sigmoid) or
    ``DECAY_SOFTPLUS`` (-Softplus)."""
    q, k, g = _arr(q, dtype), _arr(k, dtype), _arr(g, dtype)
    v = _arr(v, dtype)
    beta = np.ascontiguousarray(beta, dtype=np.float32)
    nc = len(row0)
    r0 = np.ascontiguousarray(row0, dtype=np.int64)
    nn = np.ascontiguousarray(n, dtype=np.int64)
    assert len(nn) == nc
    off = np.zeros(nc, dtype=np.int64)
    if nc > 1:
        off[1:] = np.cumsum(nn[:-1] * d_v)
    o = np.zeros(int(nn.sum()) * d_v, dtype=np.float64)
    s_out = np.zeros((nc, d_k, d_v), dtype=np.float64)
    s0p = None
    if s0 is not None:
        s0 = np.ascontiguousarray(s0, dtype=np.float64).reshape(nc, d_k, d_v)
        s0p = s0.ctypes.data
    snap_every = int(snap_every)
    if snap_every < 0:
        raise ValueError("snap_every must be >= 0")
    counts = nn // snap_every if snap_every > 0 else np.zeros(nc, dtype=np.int64)
    soff = np.zeros(nc, dtype=np.int64)
    if nc > 1:
        soff[1:] = np.cumsum(counts[:-1])
    snaps = np.zeros((max(int(counts.sum()), 1), d_k, d_v), dtype=np.float64)
    used = _lib().kda_oracle_chains_map(q.ctypes.data, k.ctypes.data, v.ctypes.data, g.ctypes.data, dtype,
                                        beta.ctypes.data, row_stride, d_k, d_v, nc, r0.ctypes.data,
                                        nn.ctypes.data, s0p, o.ctypes.data, off.ctypes.data, s_out.ctypes.data,
                                        snap_every, snaps.ctypes.data, soff.ctypes.data, int(decay_map))
    if used < 0:
        raise ValueError("kda_oracle_chains: bad arguments")
    outs = [o[off[c]: off[c] + nn[c] * d_v].reshape(int(nn[c]), d_v) for c in range(nc)]
    if snap_every > 0:
        return outs, s_out, used, [snaps[soff[c]: soff[c] + counts[c]] for c in range(nc)]
    return outs, s_out, used


def recurrence(q, k, v, g, beta, s0=None, dtype: int = F64, decay_map: int = DECAY_BOUNDED):
    """One chain: ``q, k, g`` ``[n, d_k]``, ``v`` ``[n, d_v]``, ``beta`` ``[n]``,
    ``s0`` ``[d_k, d_v]`` or None.  Returns (o ``[n, d_v]``, S ``[d_k, d_v]``), fp64."""
    q = np.asarray(q)
    n, d_k = q.shape
    d_v = np.asarray(v).shape[1]
    outs, s_out, _ = chains(q, k, v, g, beta, dtype, d_k, d_v, 1, [0], [n],
                            None if s0 is None else np.asarray(s0, dtype=np.float64)[None], decay_map=decay_map)
    return outs[0], s_out[0]
