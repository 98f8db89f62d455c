"""Pins of the fused decode layer oracle (``oracle.decode_layer``) against what
the mathematics fixes: the conv cache reproduces a whole-sequence causal
convolution computed by numpy, the activations and norms meet their closed
forms and defining properties, the gate scale and a delta conv kernel reduce
the layer step to the plain recurrence step, and the output epilogue has the
RMS and gate behaviour its definition gives."""
import numpy as np
import pytest

import oracle
from oracle import decode_layer as dl


@pytest.mark.parametrize("W", [1, 2, 4])
def test_conv_cache_matches_whole_sequence_convolution(W):
    rng = np.random.default_rng(40 + W)
    T, C = 11, 5
    x = rng.normal(size=(T, C))
    w = rng.normal(size=(C, W))
    cache = np.zeros((W - 1, C))
    ys = []
    for t in range(T):
        y, cache = dl.short_conv_step(x[t], cache, w)
        ys.append(y)
    ys = np.array(ys)
    for c in range(C):   # y_t = sum_j w[j] x_{t-W+1+j}: np.convolve with the taps reversed, zeros before t = 0
        np.testing.assert_allclose(ys[:, c], np.convolve(x[:, c], w[c, ::-1])[:T], rtol=1e-13, atol=1e-13)
    if W > 1:   # the cache holds the last W-1 inputs, oldest first
        np.testing.assert_array_equal(cache, x[T - (W - 1):])


def test_activation_and_norm_closed_forms():
    assert dl.swish(0.0) == 0.0
    assert abs(dl.swish(40.0) - 40.0) < 1e-12 and abs(dl.swish(-40.0)) < 1e-15
    assert abs(dl.swish(1.0) - 1.0 / (1.0 + np.exp(-1.0))) < 1e-15
    rng = np.random.default_rng(3)
    x = rng.normal(size=(4, 7))
    np.testing.assert_allclose(np.linalg.norm(dl.l2norm(x, 1e-30), axis=-1), 1.0, rtol=1e-14)
    np.testing.assert_array_equal(dl.l2norm(np.zeros(5), 1e-6), np.zeros(5))
    r = dl.rmsnorm(x, np.ones(7), 1e-30)
    np.testing.assert_allclose(np.mean(r * r, axis=-1), 1.0, rtol=1e-14)
    w = rng.normal(size=7)
    np.testing.assert_allclose(dl.rmsnorm(x, w, 1e-30), r * w, rtol=1e-14)
    np.testing.assert_allclose(dl.rmsnorm(3.0 * x, np.ones(7), 1e-30), r, rtol=1e-13)   # scale invariant


def _layer_inputs(rng, N, H, d_k, d_v, W):
    C = 2 * d_k + d_v
    return dict(q_in=rng.normal(size=(N, H, d_k)), k_in=rng.normal(size=(N, H, d_k)), v_in=rng.normal(size=(N, H, d_v)),
                z=2.0 * rng.normal(size=(N, H, d_k)), A_log=0.3 * rng.normal(size=H), beta_logit=rng.normal(size=(N, H)),
                conv_cache=rng.normal(size=(N, H, W - 1, C)), conv_weight=rng.normal(size=(H, C, W)) / W,
                state=0.1 * rng.normal(size=(N, H, d_k, d_v)))


@pytest.mark.parametrize("scale", [1.0, 2.0])
def test_delta_kernel_and_gate_scale_reduce_to_the_plain_step(scale):
    """Conv taps (0, ..., 0, 1) pass the current token through, and e^{A^h}
    with A^h = ln(scale) multiplies the gate logit: the layer step is then the
    plain recurrence step on L2Norm(Swish(q)), L2Norm(Swish(k)), Swish(v),
    logit scale * z and beta = Sigmoid(logit), head by head."""
    rng = np.random.default_rng(11)
    N, H, d_k, d_v, W = 2, 3, 4, 5, 3
    a = _layer_inputs(rng, N, H, d_k, d_v, W)
    a["conv_weight"] = np.zeros_like(a["conv_weight"])
    a["conv_weight"][..., W - 1] = 1.0
    a["A_log"] = np.full(H, np.log(scale))
    o, S, cache = dl.decode_layer_step(**a)
    for n in range(N):
        for h in range(H):
            q = a["q_in"][n, h] / (1 + np.exp(-a["q_in"][n, h]))
            k = a["k_in"][n, h] / (1 + np.exp(-a["k_in"][n, h]))
            q, k = q / np.sqrt(q @ q + 1e-6), k / np.sqrt(k @ k + 1e-6)
            v = a["v_in"][n, h] / (1 + np.exp(-a["v_in"][n, h]))
            beta = np.float32(1 / (1 + np.exp(-a["beta_logit"][n, h])))
            o_ref, S_ref = oracle.recurrence(q[None], k[None], v[None], scale * a["z"][n, h][None], np.array([beta]),
                                             a["state"][n, h])
            np.testing.assert_allclose(o[n, h], o_ref[0], rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(S[n, h], S_ref, rtol=1e-12, atol=1e-14)
    x = np.concatenate([a["q_in"], a["k_in"], a["v_in"]], axis=-1)
    np.testing.assert_array_equal(cache[:, :, -1], x)                      # the new token enters last
    np.testing.assert_array_equal(cache[:, :, :-1], a["conv_cache"][:, :, 1:])


def test_output_epilogue_gate_and_rms():
    """Sigmoid(gate) * RMSNorm(o~): an open gate (large logit) with unit weight
    leaves outputs of unit RMS per head; a zero logit halves them; the weight
    scales each channel."""
    rng = np.random.default_rng(12)
    N, H, d_k, d_v, W = 2, 2, 4, 6, 2
    a = _layer_inputs(rng, N, H, d_k, d_v, W)
    o_raw, _, _ = dl.decode_layer_step(**a)
    o_open, _, _ = dl.decode_layer_step(**a, out_gate=np.full((N, H, d_v), 60.0), eps_rms=1e-30)
    np.testing.assert_allclose(np.mean(o_open ** 2, axis=-1), 1.0, rtol=1e-12)
    np.testing.assert_allclose(o_open, o_raw / np.sqrt(np.mean(o_raw ** 2, axis=-1, keepdims=True)), rtol=1e-12)
    o_half, _, _ = dl.decode_layer_step(**a, out_gate=np.zeros((N, H, d_v)), eps_rms=1e-30)
    np.testing.assert_allclose(o_half, 0.5 * o_open, rtol=1e-12)
    w = rng.normal(size=(H, d_v))
    o_w, _, _ = dl.decode_layer_step(**a, out_gate=np.full((N, H, d_v), 60.0), norm_weight=w, eps_rms=1e-30)
    np.testing.assert_allclose(o_w, o_open * w[None], rtol=1e-12)
