"""Move seeded workload tensors into torch tensors (device or pinned host).

Pure data movement: values come from the generator in this package, slice by
slice through one pinned host buffer, so host memory stays bounded even for
the million-token workload."""
from __future__ import annotations

import numpy as np
import torch

from . import PrefillWorkload

_TORCH = {"f32": torch.float32, "bf16": torch.bfloat16}
_HOST = {"f32": torch.float32, "bf16": torch.int16}


def _fill(w: PrefillWorkload, name: str, out: torch.Tensor, d: int, slice_tokens: int = 1 << 15):
    tokens, H = w.tokens, w.H
    rows = min(slice_tokens, max(tokens, 1)) * H
    if name == "beta":
        host = torch.empty((rows,), dtype=torch.float32).pin_memory()
        flat = out.view(tokens * H)
    else:
        host = torch.empty((rows, d), dtype=_HOST[w.dtype]).pin_memory()
        flat = out.view(tokens * H, d)
    for t0 in range(0, tokens, slice_tokens):
        n = min(slice_tokens, tokens - t0)
        w.fill(name, host.data_ptr(), t0, n)
        src = host[: n * H]
        if name != "beta" and w.dtype == "bf16":
            src = src.view(torch.bfloat16)
        flat[t0 * H: (t0 + n) * H].copy_(src)


def prefill_inputs(w: PrefillWorkload, device="cuda", pin: bool = False):
    """q, k, v, g ``[B, T, H, d]``, beta ``[B, T, H]``, s0 ``[S, H, d_k, d_v]``
    (or None) and cu_seqlens (or None) as torch tensors on ``device``
    (``device="cpu", pin=True`` gives pinned host tensors)."""
    dt = _TORCH[w.dtype]
    B, T, H = w.B, w.T, w.H

    def empty(shape, dtype):
        t = torch.empty(shape, dtype=dtype, device=device)
        return t.pin_memory() if pin else t

    t = {}
    for name, d in (("q", w.d_k), ("k", w.d_k), ("v", w.d_v), ("g", w.d_k)):
        t[name] = empty((B, T, H, d), dt)
        _fill(w, name, t[name], d)
    t["beta"] = empty((B, T, H), torch.float32)
    _fill(w, "beta", t["beta"], 1)
    t["s0"] = None
    if w.s0_std is not None:
        s0 = w.fill("s0", np.empty((w.num_seqs * H * w.d_k, w.d_v), np.float32))
        t["s0"] = empty((w.num_seqs, H, w.d_k, w.d_v), torch.float32)
        t["s0"].copy_(torch.from_numpy(s0).reshape(w.num_seqs, H, w.d_k, w.d_v))
    cu = w.cu_seqlens()
    t["cu"] = None if cu is None else torch.from_numpy(cu).to(device)
    return t
