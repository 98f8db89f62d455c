"""fp64 oracle of the fused decode layer step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU legs may
import it; it shares no code with the CUDA library.  One decode step of a KDA
layer from the per-head projections of the token, as page "Kimi K3：架构、训练与百万
Token Agentic RL 技术解读" writes it:

* §3.2, the input branches: ``q, k = L2Norm(Swish(ShortConv(W_{q/k} x)))``,
  ``v = Swish(ShortConv(W_v x))``, ``beta = Sigmoid(W_beta x)``; ShortConv also
  reads the conv cache ``C^conv_{t-1}`` of recent tokens and leaves
  ``C^conv_t`` for the next one (the interface ``(x_t, S_{t-1}, C_{t-1}) ->
  (y_t, S_t, C_t)``).
* §3.3, the gate: ``g = g_min * Sigmoid(e^{A^h} z)``, ``g_min = -5``.
* §3.1 / §3.2, the recurrence step (the C oracle in ``kda_oracle.c``).
* §3.2, the output: ``Sigmoid(W_g x) * RMSNorm(o~)`` before ``W_o``.

Readings where the page leaves a step open (each listed in the design notes):
ShortConv is a causal depthwise convolution per channel of width ``W``
(``y[c] = sum_j w[c][j] * x_{t-W+1+j}[c]``, the last tap on the current token),
its cache holds the ``W - 1`` previous inputs (oldest first); the width is a
parameter (the page says only "the most recent few positions"); Swish is
``x * Sigmoid(x)``; ``L2Norm(x) = x / sqrt(sum x^2 + eps)``; ``RMSNorm(x) = x /
sqrt(mean x^2 + eps) * w`` over each head's ``d_v`` outputs with a per-head
weight ``w``; the projections ``W x`` are inputs (no weights are trained here).
"""
from __future__ import annotations

from typing import Optional

import numpy as np

from . import F64, chains


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-np.asarray(x, dtype=np.float64)))


def swish(x):
    x = np.asarray(x, dtype=np.float64)
    return x * sigmoid(x)


def l2norm(x, eps: float):
    """Over the last axis."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def rmsnorm(x, w, eps: float):
    """Over the last axis, times the weight ``w`` (broadcast)."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * np.asarray(w, dtype=np.float64)


def short_conv_step(x_new, cache, weight):
    """Causal depthwise convolution for one new token.

    ``x_new`` [..., C]; ``cache`` [..., W-1, C] (the previous inputs, oldest
    first); ``weight`` [..., C, W] (tap W-1 multiplies the current token).
    Returns (y [..., C], the new cache [..., W-1, C]: shifted by one, x_new last)."""
    x_new = np.asarray(x_new, dtype=np.float64)
    cache = np.asarray(cache, dtype=np.float64)
    weight = np.asarray(weight, dtype=np.float64)
    W = weight.shape[-1]
    window = np.concatenate([cache, x_new[..., None, :]], axis=-2)   # [..., W, C], oldest first
    y = np.sum(window * np.swapaxes(weight, -1, -2), axis=-2)
    return y, window[..., 1:, :] if W > 1 else cache


def decode_layer_step(q_in, k_in, v_in, z, A_log, beta_logit, conv_cache, conv_weight, state,
                      out_gate=None, norm_weight=None, eps_l2: float = 1e-6, eps_rms: float = 1e-6):
    """One fused decode step for N sequences x H heads, all fp64 values.

    q_in, k_in, z: [N, H, d_k]; v_in: [N, H, d_v]; A_log: [H]; beta_logit: [N, H];
    conv_cache: [N, H, W-1, 2*d_k + d_v] (channels q, then k, then v);
    conv_weight: [H, 2*d_k + d_v, W]; state: [N, H, d_k, d_v];
    out_gate: [N, H, d_v] or None (then o = o~); norm_weight: [H, d_v] or None (ones).
    Returns (o [N, H, d_v], new state, new conv cache)."""
    q_in, k_in, v_in = (np.asarray(a, dtype=np.float64) for a in (q_in, k_in, v_in))
    N, H, d_k = q_in.shape
    d_v = v_in.shape[-1]
    x = np.concatenate([q_in, k_in, v_in], axis=-1)                    # [N, H, 2 d_k + d_v]
    y, new_cache = short_conv_step(x, conv_cache, np.broadcast_to(conv_weight, (N,) + np.shape(conv_weight)))
    act = swish(y)
    q = l2norm(act[..., :d_k], eps_l2)
    k = l2norm(act[..., d_k:2 * d_k], eps_l2)
    v = act[..., 2 * d_k:]
    g = np.exp(np.asarray(A_log, dtype=np.float64))[None, :, None] * np.asarray(z, dtype=np.float64)
    beta = sigmoid(beta_logit).astype(np.float32)   # the recurrence oracle takes beta as fp32
    rows = N * H
    outs, s_new, _ = chains(q.reshape(rows, d_k), k.reshape(rows, d_k), v.reshape(rows, d_v),
                            g.reshape(rows, d_k), beta.reshape(rows), F64, d_k, d_v, 1,
                            list(range(rows)), [1] * rows, np.asarray(state, dtype=np.float64).reshape(rows, d_k, d_v))
    o = np.stack([x_[0] for x_ in outs]).reshape(N, H, d_v)
    if out_gate is not None:
        w = np.ones((H, d_v)) if norm_weight is None else np.asarray(norm_weight, dtype=np.float64)
        o = sigmoid(out_gate) * rmsnorm(o, w[None], eps_rms)
    return o, s_new.reshape(N, H, d_k, d_v), new_cache
