"""The chunked algebra of the prefill path, stated in plain fp64 numpy and
checked against the token-by-token oracle on the CPU.

Page "Kimi K3：架构、训练与百万 Token Agentic RL 技术解读" §3.3 describes prefill as
chunks processed in parallel inside and chained by their boundary states,
(X_[c], S_in) -> (Y_[c], S_out), in a WY/UT organisation.  Written out for one
chunk with G the inclusive cumulative log-decay (per key channel):

    A_ri = beta_r sum_c k_rc k_ic e^{G_rc - G_ic}          (i < r)
    P_ri =        sum_c q_rc k_ic e^{G_rc - G_ic}          (i <= r)
    X    = (I + A)^{-1}
    w    = X Diag(beta) (k e^G),   u = X Diag(beta) V
    V_new = u - w S,   O = (q e^G) S + P V_new
    S'   = Diag(e^{G_last}) S + (k e^{G_last - G})^T V_new

The diagonal 16-token sub-tiles can be formed two ways: as a product of two
factored operands referenced to the sub-tile start (k_r e^{G_r - G_s}) .
(k_i e^{G_s - G_i}), the dense form that tensor cores take, whose second factor
grows like e^{-(G_i - G_s)}; or pair by pair with e^{G_r - G_i} <= 1.  Page
"Kimi K3 架构篇：一文详解 2.8 万亿参数的巨型怪兽" ("最被低估的一个细节：下界衰减") states
that the lower bound g_min = -5 keeps the first form in range (e^80 over 16
tokens); without a bound only the second one stays finite.  These tests pin
both forms to the oracle and show the overflow.
"""
import math

import numpy as np
import pytest

import oracle

SUB = 16


def _log_decay(g, decay_map):
    if decay_map == oracle.DECAY_SOFTPLUS:
        return -np.logaddexp(0.0, g)
    return -5.0 / (1.0 + np.exp(-g))


def _intra(k, q, G, beta, diag):
    """A (beta-weighted, strictly lower) and P (inclusive lower) of one chunk."""
    L = len(k)
    A = np.zeros((L, L))
    P = np.zeros((L, L))
    with np.errstate(over="ignore", invalid="ignore"):
        for r in range(L):
            a = r // SUB
            Gs = G[SUB * a - 1] if a > 0 else np.zeros_like(G[0])   # decay before sub-tile a
            for i in range(r + 1):
                if i // SUB < a:        # below the diagonal sub-tile: both factors <= 1
                    f = np.exp(G[r] - Gs) * np.exp(Gs - G[i])
                elif diag == "pairs":   # the diagonal sub-tile pair by pair: e^{G_r - G_i} <= 1
                    f = np.exp(G[r] - G[i])
                else:                   # the diagonal sub-tile factored: e^{G_s - G_i} >= 1
                    f = np.exp(G[r] - Gs) * np.exp(Gs - G[i])
                if i < r:
                    A[r, i] = beta[r] * np.dot(k[r] * f, k[i])
                P[r, i] = np.dot(q[r] * f, k[i])
    return A, P


def chunked(q, k, v, g, beta, s0, C, decay_map=oracle.DECAY_BOUNDED, diag="factored"):
    """Outputs and final state of one sequence by the chunked form above."""
    T, d_k = q.shape
    S = np.array(s0, dtype=np.float64)
    ld = _log_decay(g, decay_map)
    outs = []
    for c0 in range(0, T, C):
        sl = slice(c0, min(c0 + C, T))
        kc, qc, vc, bc = k[sl], q[sl], v[sl], beta[sl].astype(np.float64)
        G = np.cumsum(ld[sl], axis=0)
        A, P = _intra(kc, qc, G, bc, diag)
        X = np.linalg.inv(np.eye(len(kc)) + A)
        w = X @ (bc[:, None] * kc * np.exp(G))
        u = X @ (bc[:, None] * vc)
        Vn = u - w @ S
        outs.append((qc * np.exp(G)) @ S + P @ Vn)
        S = np.exp(G[-1])[:, None] * S + (kc * np.exp(G[-1] - G)).T @ Vn
    return np.concatenate(outs), S


def _inputs(rng, T, d_k, d_v, g_scale=2.0):
    q = rng.normal(size=(T, d_k))
    k = rng.normal(size=(T, d_k))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.normal(size=(T, d_v))
    g = g_scale * rng.normal(size=(T, d_k))
    beta = (1.0 / (1.0 + np.exp(-rng.normal(size=T)))).astype(np.float32)
    s0 = 0.1 * rng.normal(size=(d_k, d_v))
    return q, k, v, g, beta, s0


@pytest.mark.parametrize("C", [16, 32, 64])
@pytest.mark.parametrize("decay_map", [oracle.DECAY_BOUNDED, oracle.DECAY_SOFTPLUS])
@pytest.mark.parametrize("diag", ["factored", "pairs"])
def test_chunked_form_equals_the_recurrence(C, decay_map, diag):
    """Both ways of forming the diagonal sub-tiles, every chunk size, a ragged
    last chunk, d_k != d_v: the chunked outputs and final state equal the
    token-by-token oracle to fp64 rounding."""
    rng = np.random.default_rng(50 + C + 7 * decay_map + (diag == "pairs"))
    T, d_k, d_v = 150, 6, 5
    q, k, v, g, beta, s0 = _inputs(rng, T, d_k, d_v)
    o, S = chunked(q, k, v, g, beta, s0, C, decay_map, diag)
    o_ref, S_ref = oracle.recurrence(q, k, v, g, beta, s0, decay_map=decay_map)
    np.testing.assert_allclose(o, o_ref, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(S, S_ref, rtol=1e-9, atol=1e-11)


def test_bounded_map_keeps_the_factored_diagonal_in_range():
    """Every logit +30 (alpha on its e^-5 bound): the largest factored column
    factor inside a sub-tile, e^{-G} after its 16 tokens, is e^{80 Sigmoid(30)},
    just under the e^80 of the page, and the factored form still matches the
    oracle."""
    rng = np.random.default_rng(60)
    T, d_k, d_v = 64, 4, 3
    q, k, v, _, beta, s0 = _inputs(rng, T, d_k, d_v)
    g = np.full((T, d_k), 30.0)
    G = np.cumsum(_log_decay(g, oracle.DECAY_BOUNDED), axis=0)
    assert np.max(-(G[SUB - 1] - 0.0)) < 80.0
    o, S = chunked(q, k, v, g, beta, s0, 64, oracle.DECAY_BOUNDED, "factored")
    o_ref, S_ref = oracle.recurrence(q, k, v, g, beta, s0)
    np.testing.assert_allclose(o, o_ref, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(S, S_ref, rtol=1e-9, atol=1e-12)


def test_unbounded_map_overflows_the_factored_diagonal_but_not_the_pairs():
    """Logits +60 on half of the key channels under -Softplus: those channels
    decay by e^-60 per token, so inside a 16-token sub-tile the factored column
    factor reaches e^{900}, beyond fp64 itself (e^709).  The factored form
    yields non-finite values; the pair form, whose every factor is <= 1,
    matches the oracle."""
    rng = np.random.default_rng(61)
    T, d_k, d_v = 48, 4, 3
    q, k, v, g, beta, s0 = _inputs(rng, T, d_k, d_v)
    g[:, :2] = 60.0
    assert 15 * 60.0 > math.log(np.finfo(np.float64).max)
    o_f, S_f = chunked(q, k, v, g, beta, s0, 16, oracle.DECAY_SOFTPLUS, "factored")
    assert not (np.isfinite(o_f).all() and np.isfinite(S_f).all())
    o_p, S_p = chunked(q, k, v, g, beta, s0, 16, oracle.DECAY_SOFTPLUS, "pairs")
    o_ref, S_ref = oracle.recurrence(q, k, v, g, beta, s0, decay_map=oracle.DECAY_SOFTPLUS)
    np.testing.assert_allclose(o_p, o_ref, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(S_p, S_ref, rtol=1e-9, atol=1e-12)
