"""Seeded synthetic inputs for the KDA recurrence.

This module only draws numbers (SplitMix64 + Box-Muller, see ``synth.c``) and
lays them out in the shapes of the workloads; it holds none of the recurrence's
arithmetic.  Both the fp64 oracle's tests and the GPU tests / benchmark use it,
so the two sides always see the same stored values.

Recipe (per workload, every tensor is its own counter stream, so any slice can
be regenerated alone):

* q, k ~ N(0, 1) per element, each (token, head) row divided by its fp64 norm,
  then stored in the workload dtype (fp64 -> fp32 -> bf16, round to nearest even);
* v ~ N(0, 1); g ~ N(0, std 2) (the raw decay logit); stored in the workload dtype;
* beta = sigmoid(N(0, 1)) in fp32, one per (token, head);
* initial state S0 ~ N(0, std s0_std) in fp32 ([state, H, d_k, d_v], d_v
  contiguous), or no initial state at all;
* varlen: 12 lengths exp(U(ln 4096, ln 524288)), scaled to the total token
  count and floored, the remainder added to the longest.

Layouts are token-major and head-interleaved: q, k, g ``[tokens, H, d_k]``,
v ``[tokens, H, d_v]``, beta ``[tokens, H]`` where ``tokens = B*T`` (batched)
or the packed total (varlen).  Logical row ``tok*H + h`` of a stream holds the
``d`` values of token ``tok``, head ``h``.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import tempfile
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_SO = os.path.join(_HERE, "libkda_synth.so")

F32, BF16, F64 = 0, 1, 2
DTYPE_CODES = {"f32": F32, "bf16": BF16, "f64": F64}

# stream ids of the tensors of one workload
STREAM_Q, STREAM_K, STREAM_V, STREAM_G, STREAM_BETA, STREAM_S0, STREAM_LENS = 1, 2, 3, 4, 5, 6, 7


def build(force: bool = False) -> str:
    """Compile ``synth.c`` into ``libkda_synth.so`` beside it (plain gcc, OpenMP)."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    cmd = ["gcc", "-O3", "-std=c99", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


_lib_handle = None


def _lib():
    global _lib_handle
    if _lib_handle is None:
        lib = ctypes.CDLL(build())
        i64, i32, u64, dbl, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64, ctypes.c_double, ctypes.c_void_p
        lib.synth_stream_key.argtypes = [u64, u64]
        lib.synth_stream_key.restype = u64
        lib.synth_normal_f64.argtypes = [u64, u64, i64, i64, vp]
        lib.synth_normal_f64.restype = None
        lib.synth_rows.argtypes = [u64, u64, i64, i64, i64, i32, dbl, i32, i32, vp]
        lib.synth_rows.restype = ctypes.c_int
        lib.synth_sigmoid_normal_f32.argtypes = [u64, u64, i64, i64, i64, vp]
        lib.synth_sigmoid_normal_f32.restype = ctypes.c_int
        lib.synth_f32_to_bf16.argtypes = [vp, i64, vp]
        lib.synth_f32_to_bf16.restype = None
        lib.synth_uniform_f64.argtypes = [u64, u64, i64, i64, vp]
        lib.synth_uniform_f64.restype = None
        _lib_handle = lib
    return _lib_handle


def _ptr(out) -> int:
    if isinstance(out, np.ndarray):
        assert out.flags["C_CONTIGUOUS"]
        return out.ctypes.data
    return int(out)


def _np_dtype(code: int):
    return {F32: np.float32, BF16: np.uint16, F64: np.float64}[code]


def rows(seed: int, stream: int, first_row: int, row_stride: int, nrows: int, d: int,
         scale: float = 1.0, unit_norm: bool = False, dtype: int = F64, out=None):
    """``nrows`` rows of ``d`` values (logical rows ``first_row + r*row_stride``).

    ``out`` is a C-contiguous numpy array or a raw host address; when omitted a
    numpy array (bf16 stored as uint16 bits) is returned."""
    if out is None:
        out = np.empty((nrows, d), dtype=_np_dtype(dtype))
    rc = _lib().synth_rows(seed, stream, first_row, row_stride, nrows, d, float(scale), int(unit_norm), dtype,
                           _ptr(out))
    if rc != 0:
        raise ValueError("synth_rows: bad arguments")
    return out


def sigmoid_normal(seed: int, stream: int, first: int, stride: int, n: int, out=None):
    if out is None:
        out = np.empty((n,), dtype=np.float32)
    if _lib().synth_sigmoid_normal_f32(seed, stream, first, stride, n, _ptr(out)) != 0:
        raise ValueError("synth_sigmoid_normal_f32: bad arguments")
    return out


def normals(seed: int, stream: int, offset: int, n: int) -> np.ndarray:
    out = np.empty((n,), dtype=np.float64)
    _lib().synth_normal_f64(seed, stream, offset, n, out.ctypes.data)
    return out


def uniforms(seed: int, stream: int, first: int, n: int) -> np.ndarray:
    out = np.empty((n,), dtype=np.float64)
    _lib().synth_uniform_f64(seed, stream, first, n, out.ctypes.data)
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _lib().synth_f32_to_bf16(x.ctypes.data, x.size, out.ctypes.data)
    return out


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def varlen_lengths(seed: int, total: int, n: int = 12, lo: int = 4096, hi: int = 524288) -> np.ndarray:
    """n lengths exp(U(ln lo, ln hi)), scaled to sum to ``total`` and floored;
    the remainder goes to the (first) longest."""
    u = uniforms(seed, STREAM_LENS, 0, n)
    raw = np.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
    lens = np.floor(raw * (total / raw.sum())).astype(np.int64)
    lens[int(np.argmax(lens))] += total - int(lens.sum())
    assert int(lens.sum()) == total and (lens >= 0).all()
    return lens


@dataclass
class PrefillWorkload:
    """One chunked-prefill workload.  ``seq_lens`` set => packed varlen (B = 1)."""
    name: str
    dtype: str
    B: int
    T: int
    H: int
    d_k: int
    d_v: int
    seed: int
    s0_std: Optional[float]          # None: no initial state (zeros)
    seq_lens: Optional[np.ndarray] = None
    extra: dict = field(default_factory=dict)
    # A shard of a larger workload (see ``shard``): this workload's token 0 and
    # sequence 0 are token ``tok_base`` and sequence ``seq_base`` of the
    # generator streams, so its values are exactly that slice of the whole.
    tok_base: int = 0
    seq_base: int = 0

    @property
    def dcode(self) -> int:
        return DTYPE_CODES[self.dtype]

    @property
    def tokens(self) -> int:
        return self.B * self.T

    @property
    def num_seqs(self) -> int:
        return len(self.seq_lens) if self.seq_lens is not None else self.B

    def cu_seqlens(self) -> Optional[np.ndarray]:
        if self.seq_lens is None:
            return None
        return np.concatenate([[0], np.cumsum(self.seq_lens)]).astype(np.int32)

    def seq_bounds(self, s: int):
        """(first packed token, length) of sequence s."""
        if self.seq_lens is None:
            return s * self.T, self.T
        cu = self.cu_seqlens()
        return int(cu[s]), int(cu[s + 1] - cu[s])

    # ---- whole tensors -------------------------------------------------
    def fill(self, name: str, out, tok0: int = 0, ntok: Optional[int] = None):
        """Generate tensor ``name`` (q, k, v, g, beta, s0) for packed tokens
        [tok0, tok0 + ntok) of all heads (s0: all states) into ``out``."""
        ntok = self.tokens - tok0 if ntok is None else ntok
        H = self.H
        tok0 = tok0 + self.tok_base
        if name == "q":
            return rows(self.seed, STREAM_Q, tok0 * H, 1, ntok * H, self.d_k, 1.0, True, self.dcode, out)
        if name == "k":
            return rows(self.seed, STREAM_K, tok0 * H, 1, ntok * H, self.d_k, 1.0, True, self.dcode, out)
        if name == "v":
            return rows(self.seed, STREAM_V, tok0 * H, 1, ntok * H, self.d_v, 1.0, False, self.dcode, out)
        if name == "g":
            return rows(self.seed, STREAM_G, tok0 * H, 1, ntok * H, self.d_k, 2.0, False, self.dcode, out)
        if name == "beta":
            return sigmoid_normal(self.seed, STREAM_BETA, tok0 * H, 1, ntok * H, out)
        if name == "s0":
            assert self.s0_std is not None
            n = self.num_seqs * H * self.d_k
            return rows(self.seed, STREAM_S0, self.seq_base * H * self.d_k, 1, n, self.d_v, self.s0_std, False, F32,
                        out)
        raise KeyError(name)

    # ---- one (sequence, head) chain, for the oracle -----------------------
    def chain_inputs(self, s: int, h: int, ntok: Optional[int] = None):
        """Stored values of sequence s, head h (first ``ntok`` tokens):
        dict of numpy arrays q, k [n, d_k], v [n, d_v], g [n, d_k] (storage
        dtype; bf16 as uint16 bits), beta [n] fp32, s0 [d_k, d_v] fp32 or None."""
        tok0, L = self.seq_bounds(s)
        n = L if ntok is None else min(ntok, L)
        H = self.H
        tok0 += self.tok_base
        out = {
            "q": rows(self.seed, STREAM_Q, tok0 * H + h, H, n, self.d_k, 1.0, True, self.dcode),
            "k": rows(self.seed, STREAM_K, tok0 * H + h, H, n, self.d_k, 1.0, True, self.dcode),
            "v": rows(self.seed, STREAM_V, tok0 * H + h, H, n, self.d_v, 1.0, False, self.dcode),
            "g": rows(self.seed, STREAM_G, tok0 * H + h, H, n, self.d_k, 2.0, False, self.dcode),
            "beta": sigmoid_normal(self.seed, STREAM_BETA, tok0 * H + h, H, n),
            "s0": None,
        }
        if self.s0_std is not None:
            out["s0"] = rows(self.seed, STREAM_S0, ((self.seq_base + s) * H + h) * self.d_k, 1, self.d_k, self.d_v,
                             self.s0_std, False, F32)
        return out

    def shard(self, first_seq: int, count: int, name: Optional[str] = None) -> "PrefillWorkload":
        """Sequences [first_seq, first_seq + count) of this workload (all their
        heads) as a workload of their own, with exactly the same values."""
        assert 0 <= first_seq and count >= 0 and first_seq + count <= self.num_seqs
        import dataclasses

        tok0, _ = self.seq_bounds(first_seq) if count else (0, 0)
        if self.seq_lens is None:
            B, T, lens = count, self.T, None
        else:
            lens = np.asarray(self.seq_lens[first_seq: first_seq + count])
            B, T = 1, int(lens.sum())
        return dataclasses.replace(self, name=name or f"{self.name}[{first_seq}:{first_seq + count}]", B=B, T=T,
                                   seq_lens=lens, tok_base=self.tok_base + tok0,
                                   seq_base=self.seq_base + first_seq, extra=dict(self.extra))


@dataclass
class DecodeWorkload:
    """``steps`` decode steps of N sequences x H heads, one token each."""
    name: str
    dtype: str
    N: int
    H: int
    d_k: int
    d_v: int
    seed: int
    state_std: float
    steps: int

    @property
    def dcode(self) -> int:
        return DTYPE_CODES[self.dtype]

    def _stream(self, step: int, base: int) -> int:
        return 1000 * (step + 1) + base

    def fill_step(self, step: int, name: str, out=None, first: int = 0, count: Optional[int] = None,
                  stride: int = 1):
        """Tensor ``name`` of decode step ``step`` for (seq, head) rows
        first + r*stride, r < count (row index n*H + h)."""
        count = self.N * self.H if count is None else count
        if name == "q":
            return rows(self.seed, self._stream(step, STREAM_Q), first, stride, count, self.d_k, 1.0, True,
                        self.dcode, out)
        if name == "k":
            return rows(self.seed, self._stream(step, STREAM_K), first, stride, count, self.d_k, 1.0, True,
                        self.dcode, out)
        if name == "v":
            return rows(self.seed, self._stream(step, STREAM_V), first, stride, count, self.d_v, 1.0, False,
                        self.dcode, out)
        if name == "g":
            return rows(self.seed, self._stream(step, STREAM_G), first, stride, count, self.d_k, 2.0, False,
                        self.dcode, out)
        if name == "beta":
            return sigmoid_normal(self.seed, self._stream(step, STREAM_BETA), first, stride, count, out)
        raise KeyError(name)

    def fill_state(self, out=None, first_head: int = 0, count: Optional[int] = None):
        """Initial states of (seq, head) rows [first_head, first_head + count), fp32 [count*d_k, d_v]."""
        count = self.N * self.H if count is None else count
        return rows(self.seed, STREAM_S0, first_head * self.d_k, 1, count * self.d_k, self.d_v, self.state_std,
                    False, F32, out)


def workloads() -> dict:
    """The five workloads, by name (sizes as the method's pages describe them:
    head dim 128, 32 or 96 heads, up to a million packed tokens)."""
    return {
        "fp32_b1_h2_t256_d64": PrefillWorkload("fp32_b1_h2_t256_d64", "f32", 1, 256, 2, 64, 64, seed=0, s0_std=None),
        "prefill_b1_h32_t65536_d128": PrefillWorkload("prefill_b1_h32_t65536_d128", "bf16", 1, 65536, 32, 128, 128,
                                                      seed=1, s0_std=0.01),
        "prefill_b8_h96_t8192_d128": PrefillWorkload("prefill_b8_h96_t8192_d128", "bf16", 8, 8192, 96, 128, 128,
                                                     seed=2, s0_std=None),
        "decode_n256_h96_d128_x100": DecodeWorkload("decode_n256_h96_d128_x100", "bf16", 256, 96, 128, 128, seed=3,
                                                    state_std=0.05, steps=100),
        "varlen_12seq_1m_h32_d128": PrefillWorkload("varlen_12seq_1m_h32_d128", "bf16", 1, 1 << 20, 32, 128, 128,
                                                    seed=4, s0_std=0.01, seq_lens=varlen_lengths(4, 1 << 20)),
    }
