"""KDA (Kimi Delta Attention) recurrence on one GB300 GPU.

Thin ctypes binding of the C ABI in ``include/kda.h`` (``libkda_gb300.so``,
built in-tree by ``_build.build()``).  This module only marshals arguments:
torch supplies device memory and the current CUDA stream; every step of the
recurrence runs in the library's CUDA kernels.  There is no CPU fallback: if
the library is missing or fails to load, the functions raise.

Functions keep the C names:

* ``kda_chunk_fwd(q, k, v, g, beta, initial_state=None, cu_seqlens=None, ...)``
  -> ``(o, final_state)``: chunked prefill (page "Kimi K3：架构、训练与百万 Token
  Agentic RL 技术解读" §3.3), q/k/g ``[B, T, H, d_k]``, v ``[B, T, H, d_v]``,
  beta ``[B, T, H]`` fp32, states ``[S, H, d_k, d_v]`` fp32.
* ``kda_chunk_fwd_snapshots(q, k, v, g, beta, snapshot_interval, ...)`` ->
  ``(o, final_state, snapshots)``: the same, also keeping the state every
  ``snapshot_interval`` tokens of each sequence (same page §9, prefix cache).
* ``kda_chunk_fwd_gated(q, k, v, g, beta, out_gate, norm_weight=None, ...)`` ->
  ``(o, final_state)``: the same with the output epilogue (Sigmoid gate times
  the per-head RMSNorm of o) applied before o is written (same page §3.2).
* ``kda_chunk_fwd_decay_variant(q, k, v, g, beta, decay_map, diag_by_pairs, ...)``
  -> ``(o, final_state)``: the same under the unbounded -Softplus decay map or
  with the diagonal tiles formed by position pairs, the ablation of the lower
  bound (page "Kimi K3 架构篇：一文详解 2.8 万亿参数的巨型怪兽", "最被低估的一个细节：下界衰减").
* ``kda_decode_step(q, k, v, g, beta, state, o=None)`` -> ``o``: one token per
  sequence (same page §3.2), state updated in place.
* ``kda_decode_layer_step(q_in, k_in, v_in, z, A_log, beta_logit, conv_cache,
  conv_weight, state, out_gate=None, norm_weight=None)`` -> ``o``: the decode
  step of a whole layer from the token's projections (ShortConv with its cache,
  Swish, L2Norm, gate scale, recurrence, Sigmoid-gated RMSNorm output).
* ``kda_chunk_fwd_workspace_size(...)``, ``kda_device_error()``,
  ``kda_check_wait_timeout(limit_cycles)`` (failure-detection check).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

from . import _build

__all__ = ["kda_chunk_fwd", "kda_chunk_fwd_snapshots", "kda_chunk_fwd_gated", "kda_chunk_fwd_decay_variant",
           "DECAY_BOUNDED", "DECAY_SOFTPLUS", "kda_decode_step", "kda_decode_layer_step", "kda_chunk_fwd_workspace_size", "kda_device_error",
           "kda_check_wait_timeout", "KdaError", "library_path", "load_library", "STATUS"]

DECAY_BOUNDED, DECAY_SOFTPLUS = 0, 1   # kda_decay_map
STATUS = {0: "KDA_OK", 1: "KDA_ERR_INVALID_ARG", 2: "KDA_ERR_UNSUPPORTED", 3: "KDA_ERR_CUDA",
          4: "KDA_ERR_DEVICE_TIMEOUT", 5: "KDA_ERR_NONFINITE"}
_DT = {torch.float32: 0, torch.bfloat16: 1}
SIZE_MAX = (1 << 64) - 1


class KdaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


def library_path() -> str:
    return _build.LIB


_lib = None


def load_library():
    """Load ``libkda_gb300.so`` (building it first if it is missing or stale and
    nvcc is available).  Raises if it cannot be loaded."""
    global _lib
    if _lib is not None:
        return _lib
    if not _build.up_to_date():
        _build.build()
    lib = ctypes.CDLL(_build.LIB)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    lib.kda_status_string.argtypes = [ctypes.c_int]
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_chunk_fwd_workspace_size.argtypes = [i64, i64, i32, i32, i32, i32, ctypes.c_int]
    lib.kda_chunk_fwd_workspace_size.restype = sz
    lib.kda_chunk_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i64, i64, i32, i32, i32, ctypes.c_int, vp, vp,
                                  vp, sz, vp]
    lib.kda_chunk_fwd.restype = ctypes.c_int
    lib.kda_chunk_fwd_snapshots.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i64, i64, i32, i32, i32, ctypes.c_int,
                                            vp, vp, vp, i32, i64, vp, sz, vp]
    lib.kda_chunk_fwd_snapshots.restype = ctypes.c_int
    lib.kda_chunk_fwd_gated.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i64, i64, i32, i32, i32, ctypes.c_int,
                                        vp, vp, vp, vp, ctypes.c_float, vp, sz, vp]
    lib.kda_chunk_fwd_gated.restype = ctypes.c_int
    lib.kda_chunk_fwd_decay_variant.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i64, i64, i32, i32, i32,
                                                ctypes.c_int, vp, vp, i32, i32, vp, sz, vp]
    lib.kda_chunk_fwd_decay_variant.restype = ctypes.c_int
    lib.kda_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, ctypes.c_int, vp, vp]
    lib.kda_decode_step.restype = ctypes.c_int
    f32 = ctypes.c_float
    lib.kda_decode_layer_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, f32, f32, i32, i32, i32,
                                          i32, ctypes.c_int, vp, vp]
    lib.kda_decode_layer_step.restype = ctypes.c_int
    lib.kda_device_error.argtypes = [vp, ctypes.POINTER(i32)]
    lib.kda_device_error.restype = ctypes.c_int
    lib.kda_check_wait_timeout.argtypes = [i64, vp]
    lib.kda_check_wait_timeout.restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(status: int, where: str):
    if status != 0:
        raise KdaError(status, where)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _DT:
        raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")
    return _DT[t.dtype]


def kda_chunk_fwd_workspace_size(B: int, T: int, H: int, d_k: int, d_v: int, num_seqs: int,
                                 dtype: torch.dtype) -> int:
    n = load_library().kda_chunk_fwd_workspace_size(B, T, H, d_k, d_v, num_seqs, _DT[dtype])
    if n == SIZE_MAX:
        raise KdaError(1, "kda_chunk_fwd_workspace_size")
    return int(n)


def kda_chunk_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
                  initial_state: Optional[torch.Tensor] = None, cu_seqlens: Optional[torch.Tensor] = None,
                  output_final_state: bool = True, o: Optional[torch.Tensor] = None,
                  final_state: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                  stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Chunked prefill.  Returns ``(o, final_state)`` (``final_state`` is None
    when ``output_final_state`` is False).  ``final_state`` may be passed as the
    same tensor as ``initial_state`` to update it in place."""
    lib = load_library()
    B, T, H, d_k = q.shape
    d_v = v.shape[-1]
    num_seqs = B if cu_seqlens is None else cu_seqlens.numel() - 1
    if o is None:
        o = torch.empty(v.shape, dtype=v.dtype, device=v.device)
    if output_final_state and final_state is None:
        final_state = torch.empty((num_seqs, H, d_k, d_v), dtype=torch.float32, device=q.device)
    if not output_final_state:
        final_state = None
    ws_bytes = kda_chunk_fwd_workspace_size(B, T, H, d_k, d_v, num_seqs, q.dtype)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
    st = lib.kda_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state), _ptr(cu_seqlens),
                           num_seqs, B, T, H, d_k, d_v, _dtype_code(q), _ptr(o), _ptr(final_state),
                           _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "kda_chunk_fwd")
    return o, final_state


def kda_chunk_fwd_snapshots(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                            beta: torch.Tensor, snapshot_interval: int, initial_state: Optional[torch.Tensor] = None,
                            cu_seqlens: Optional[torch.Tensor] = None, output_final_state: bool = True,
                            o: Optional[torch.Tensor] = None, final_state: Optional[torch.Tensor] = None,
                            snapshots: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                            stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor], torch.Tensor]:
    """Chunked prefill that also keeps the state every ``snapshot_interval``
    tokens (a multiple of 64) of each sequence.  Returns ``(o, final_state,
    snapshots)``; ``snapshots`` is ``[slots, H, d_k, d_v]`` fp32 with
    ``slots = B * (T // snapshot_interval)`` (batched) or ``T // snapshot_interval``
    (``cu_seqlens``: an upper bound, the sequences' snapshots come first, in
    sequence order)."""
    lib = load_library()
    B, T, H, d_k = q.shape
    d_v = v.shape[-1]
    num_seqs = B if cu_seqlens is None else cu_seqlens.numel() - 1
    if o is None:
        o = torch.empty(v.shape, dtype=v.dtype, device=v.device)
    if output_final_state and final_state is None:
        final_state = torch.empty((num_seqs, H, d_k, d_v), dtype=torch.float32, device=q.device)
    if not output_final_state:
        final_state = None
    interval = int(snapshot_interval)
    cap = (B * (T // interval) if cu_seqlens is None else (B * T) // interval) if interval > 0 else 0
    if snapshots is None:
        snapshots = torch.empty((max(cap, 1), H, d_k, d_v), dtype=torch.float32, device=q.device)
    ws_bytes = kda_chunk_fwd_workspace_size(B, T, H, d_k, d_v, num_seqs, q.dtype)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
    st = lib.kda_chunk_fwd_snapshots(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state),
                                     _ptr(cu_seqlens), num_seqs, B, T, H, d_k, d_v, _dtype_code(q), _ptr(o),
                                     _ptr(final_state), _ptr(snapshots), interval,
                                     snapshots.shape[0] if cap > 0 else 0, _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "kda_chunk_fwd_snapshots")
    return o, final_state, snapshots[:cap]


def kda_chunk_fwd_gated(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
                        out_gate: torch.Tensor, norm_weight: Optional[torch.Tensor] = None, eps_rms: float = 1e-6,
                        initial_state: Optional[torch.Tensor] = None, cu_seqlens: Optional[torch.Tensor] = None,
                        output_final_state: bool = True, o: Optional[torch.Tensor] = None,
                        final_state: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                        stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Chunked prefill with ``o = Sigmoid(out_gate) * RMSNorm(o~) * norm_weight``
    (per token and head over d_v) applied before o is written.  ``out_gate`` is
    ``[B, T, H, d_v]`` in the input dtype, ``norm_weight`` ``[H, d_v]`` fp32."""
    lib = load_library()
    B, T, H, d_k = q.shape
    d_v = v.shape[-1]
    num_seqs = B if cu_seqlens is None else cu_seqlens.numel() - 1
    if o is None:
        o = torch.empty(v.shape, dtype=v.dtype, device=v.device)
    if output_final_state and final_state is None:
        final_state = torch.empty((num_seqs, H, d_k, d_v), dtype=torch.float32, device=q.device)
    if not output_final_state:
        final_state = None
    ws_bytes = kda_chunk_fwd_workspace_size(B, T, H, d_k, d_v, num_seqs, q.dtype)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
    st = lib.kda_chunk_fwd_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state),
                                 _ptr(cu_seqlens), num_seqs, B, T, H, d_k, d_v, _dtype_code(q), _ptr(o),
                                 _ptr(final_state), _ptr(out_gate), _ptr(norm_weight), float(eps_rms),
                                 _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "kda_chunk_fwd_gated")
    return o, final_state


def kda_chunk_fwd_decay_variant(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                                beta: torch.Tensor, decay_map: int = DECAY_BOUNDED, diag_by_pairs: bool = True,
                                initial_state: Optional[torch.Tensor] = None,
                                cu_seqlens: Optional[torch.Tensor] = None, output_final_state: bool = True,
                                o: Optional[torch.Tensor] = None, final_state: Optional[torch.Tensor] = None,
                                workspace: Optional[torch.Tensor] = None,
                                stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Chunked prefill under ``decay_map`` (``DECAY_BOUNDED``: -5 Sigmoid,
    ``DECAY_SOFTPLUS``: -Softplus) with the diagonal 16x16 tiles either on the
    tensor cores (``diag_by_pairs=False``, bounded map only) or formed pair by
    pair on the CUDA cores.  Arguments otherwise as ``kda_chunk_fwd``."""
    lib = load_library()
    B, T, H, d_k = q.shape
    d_v = v.shape[-1]
    num_seqs = B if cu_seqlens is None else cu_seqlens.numel() - 1
    if o is None:
        o = torch.empty(v.shape, dtype=v.dtype, device=v.device)
    if output_final_state and final_state is None:
        final_state = torch.empty((num_seqs, H, d_k, d_v), dtype=torch.float32, device=q.device)
    if not output_final_state:
        final_state = None
    ws_bytes = kda_chunk_fwd_workspace_size(B, T, H, d_k, d_v, num_seqs, q.dtype)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
    st = lib.kda_chunk_fwd_decay_variant(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state),
                                         _ptr(cu_seqlens), num_seqs, B, T, H, d_k, d_v, _dtype_code(q), _ptr(o),
                                         _ptr(final_state), int(decay_map), int(bool(diag_by_pairs)),
                                         _ptr(workspace), workspace.numel() * workspace.element_size(),
                                         _stream(stream))
    _check(st, "kda_chunk_fwd_decay_variant")
    return o, final_state


def kda_decode_step(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
                    state: torch.Tensor, o: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """One decode step: q/k/g ``[N, H, d_k]``, v ``[N, H, d_v]``, beta ``[N, H]``
    fp32, state ``[N, H, d_k, d_v]`` fp32 (updated in place).  Returns o."""
    lib = load_library()
    N, H, d_k = q.shape
    d_v = v.shape[-1]
    if o is None:
        o = torch.empty(v.shape, dtype=v.dtype, device=v.device)
    st = lib.kda_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state), N, H, d_k, d_v,
                             _dtype_code(q), _ptr(o), _stream(stream))
    _check(st, "kda_decode_step")
    return o


def kda_decode_layer_step(q_in: torch.Tensor, k_in: torch.Tensor, v_in: torch.Tensor, z: torch.Tensor,
                          A_log: torch.Tensor, beta_logit: torch.Tensor, conv_cache: Optional[torch.Tensor],
                          conv_weight: torch.Tensor, state: torch.Tensor, out_gate: Optional[torch.Tensor] = None,
                          norm_weight: Optional[torch.Tensor] = None, eps_l2: float = 1e-6, eps_rms: float = 1e-6,
                          o: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """One decode step of a KDA layer from the token's projections.
    q_in/k_in/z ``[N, H, d_k]``, v_in/out_gate ``[N, H, d_v]`` (input dtype),
    A_log ``[H]``, beta_logit ``[N, H]`` fp32, conv_cache ``[N, H, W-1, 2 d_k + d_v]``
    (input dtype, updated in place), conv_weight ``[H, 2 d_k + d_v, W]`` fp32,
    state ``[N, H, d_k, d_v]`` fp32 (updated in place), norm_weight ``[H, d_v]``
    fp32.  Returns o ``[N, H, d_v]``."""
    lib = load_library()
    N, H, d_k = q_in.shape
    d_v = v_in.shape[-1]
    W = conv_weight.shape[-1]
    if o is None:
        o = torch.empty(v_in.shape, dtype=v_in.dtype, device=v_in.device)
    st = lib.kda_decode_layer_step(_ptr(q_in), _ptr(k_in), _ptr(v_in), _ptr(z), _ptr(A_log), _ptr(beta_logit),
                                   _ptr(conv_cache), _ptr(conv_weight), W, _ptr(state), _ptr(out_gate),
                                   _ptr(norm_weight), float(eps_l2), float(eps_rms), N, H, d_k, d_v,
                                   _dtype_code(q_in), _ptr(o), _stream(stream))
    _check(st, "kda_decode_layer_step")
    return o


def kda_device_error(stream=None) -> Tuple[int, int]:
    """(status, raw device error word) after waiting for ``stream``; clears the word."""
    code = ctypes.c_int32(0)
    st = load_library().kda_device_error(_stream(stream), ctypes.byref(code))
    return int(st), int(code.value)


def kda_check_wait_timeout(limit_cycles: int, stream=None) -> None:
    """Launch the failure-detection check: a bounded wait that runs out after
    ``limit_cycles`` SM cycles and reports through the device error word."""
    _check(load_library().kda_check_wait_timeout(int(limit_cycles), _stream(stream)), "kda_check_wait_timeout")
