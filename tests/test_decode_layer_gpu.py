"""GPU parity of the fused decode layer step (``kda_decode_layer_step``) with
the fp64 oracle ``oracle.decode_layer``: several consecutive steps, so that the
conv cache and the state evolve, for both dtypes, every head size, conv widths
1, 2 and 4, with and without the gated RMSNorm output.  The conv cache holds
copies of past inputs and is compared bit for bit; o and the state use the
tolerances of kda_testutil."""
import numpy as np
import pytest
import torch

from oracle import decode_layer as dl
import linear_attention_recurrence_chunk_gb300 as kda
from kda_testutil import assert_o_close, assert_state_close

pytestmark = pytest.mark.gpu

DEV = "cuda"
TDT = {"f32": torch.float32, "bf16": torch.bfloat16}


def _stored(x, dtype):
    """Device tensor in the storage dtype and its exact values as fp64."""
    t = torch.from_numpy(np.asarray(x, dtype=np.float32)).to(TDT[dtype])
    return t.to(DEV), t.to(torch.float64).numpy()


def _case(rng, dtype, N, H, d_k, d_v, W, gated, weighted):
    C = 2 * d_k + d_v
    A_log = torch.from_numpy((0.3 * rng.normal(size=H)).astype(np.float32)).to(DEV)
    conv_w = torch.from_numpy((rng.normal(size=(H, C, W)) / W).astype(np.float32)).to(DEV)
    cache_d, cache_h = _stored(rng.normal(size=(N, H, W - 1, C)), dtype)
    state = torch.from_numpy((0.05 * rng.normal(size=(N, H, d_k, d_v))).astype(np.float32)).to(DEV)
    nw = torch.from_numpy((1 + 0.1 * rng.normal(size=(H, d_v))).astype(np.float32)).to(DEV) if weighted else None
    return dict(A_log=A_log, conv_w=conv_w, cache_d=cache_d, cache_h=cache_h, state=state, nw=nw, gated=gated)


def _token(rng, dtype, N, H, d_k, d_v):
    q = _stored(rng.normal(size=(N, H, d_k)), dtype)
    k = _stored(rng.normal(size=(N, H, d_k)), dtype)
    v = _stored(rng.normal(size=(N, H, d_v)), dtype)
    z = _stored(2.0 * rng.normal(size=(N, H, d_k)), dtype)
    gate = _stored(rng.normal(size=(N, H, d_v)), dtype)
    bl = torch.from_numpy(rng.normal(size=(N, H)).astype(np.float32)).to(DEV)
    return q, k, v, z, gate, bl


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("d_k,d_v", [(128, 128), (64, 128), (128, 64), (64, 64)])
@pytest.mark.parametrize("W,gated,weighted", [(4, True, True), (1, False, False), (2, True, False)])
def test_decode_layer_steps_match_oracle(dtype, d_k, d_v, W, gated, weighted):
    rng = np.random.default_rng(1000 + 7 * d_k + 3 * d_v + 11 * W + int(gated) + (500 if dtype == "bf16" else 0))
    N, H, steps = 5, 3, 4
    c = _case(rng, dtype, N, H, d_k, d_v, W, gated, weighted)
    S_ref = c["state"].double().cpu().numpy()
    cache_ref = c["cache_h"]
    for _ in range(steps):
        (qd, qh), (kd, kh), (vd, vh), (zd, zh), (gd, gh), bl = _token(rng, dtype, N, H, d_k, d_v)
        o = kda.kda_decode_layer_step(qd, kd, vd, zd, c["A_log"], bl, c["cache_d"] if W > 1 else None, c["conv_w"],
                                      c["state"], out_gate=gd if gated else None, norm_weight=c["nw"])
        torch.cuda.synchronize()
        o_ref, S_ref, cache_ref = dl.decode_layer_step(
            qh, kh, vh, zh, c["A_log"].double().cpu().numpy(), bl.double().cpu().numpy(), cache_ref,
            c["conv_w"].double().cpu().numpy(), S_ref, out_gate=gh if gated else None,
            norm_weight=None if c["nw"] is None else c["nw"].double().cpu().numpy())
        assert_o_close([o.double().cpu().numpy()], [o_ref], dtype)
        assert_state_close(c["state"].double().cpu().numpy(), S_ref)
        if W > 1:
            np.testing.assert_array_equal(c["cache_d"].double().cpu().numpy(), cache_ref)
    assert kda.kda_device_error() == (0, 0)


def test_decode_layer_full_decode_size():
    """The decode workload's size (256 sequences x 96 heads, d = 128, bf16),
    one gated step with the conv width 4, every head against the oracle."""
    rng = np.random.default_rng(2024)
    N, H, d_k, d_v, W = 256, 96, 128, 128, 4
    c = _case(rng, "bf16", N, H, d_k, d_v, W, True, True)
    S0 = c["state"].double().cpu().numpy()
    (qd, qh), (kd, kh), (vd, vh), (zd, zh), (gd, gh), bl = _token(rng, "bf16", N, H, d_k, d_v)
    o = kda.kda_decode_layer_step(qd, kd, vd, zd, c["A_log"], bl, c["cache_d"], c["conv_w"], c["state"],
                                  out_gate=gd, norm_weight=c["nw"])
    torch.cuda.synchronize()
    o_ref, S_ref, cache_ref = dl.decode_layer_step(
        qh, kh, vh, zh, c["A_log"].double().cpu().numpy(), bl.double().cpu().numpy(), c["cache_h"],
        c["conv_w"].double().cpu().numpy(), S0, out_gate=gh, norm_weight=c["nw"].double().cpu().numpy())
    assert_o_close([o.double().cpu().numpy()], [o_ref], "bf16")
    assert_state_close(c["state"].double().cpu().numpy(), S_ref)
    np.testing.assert_array_equal(c["cache_d"].double().cpu().numpy(), cache_ref)
    assert kda.kda_device_error() == (0, 0)


def test_delta_conv_no_gate_equals_the_plain_decode_step():
    """Conv taps (0, 0, 0, 1), e^{A} = 1 and no output gate: the layer step
    gives what kda_decode_step gives on the activated, normalised inputs."""
    rng = np.random.default_rng(7)
    N, H, d, W = 6, 4, 128, 4
    c = _case(rng, "f32", N, H, d, d, W, False, False)
    c["conv_w"].zero_()
    c["conv_w"][..., W - 1] = 1.0
    c["A_log"].zero_()
    (qd, _), (kd, _), (vd, _), (zd, _), _, bl = _token(rng, "f32", N, H, d, d)
    state2 = c["state"].clone()
    o = kda.kda_decode_layer_step(qd, kd, vd, zd, c["A_log"], bl, c["cache_d"], c["conv_w"], c["state"])
    sw = lambda x: x * torch.sigmoid(x)
    l2 = lambda x: x / torch.sqrt((x * x).sum(-1, keepdim=True) + 1e-6)
    o2 = kda.kda_decode_step(l2(sw(qd)), l2(sw(kd)), sw(vd), zd, torch.sigmoid(bl), state2)
    torch.cuda.synchronize()
    torch.testing.assert_close(o, o2, rtol=1e-5, atol=1e-6)
    torch.testing.assert_close(c["state"], state2, rtol=1e-5, atol=1e-6)
