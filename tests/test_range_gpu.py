"""GPU checks of the fp16 range of the tensor-core prefill (bf16, d_k = 128).

The chain multiplies fp16 copies of u = (I + A)^{-1} Diag(beta) V, of
V_new = u - w S and of the state.  The state of the recurrence is not
normalised (page "Kimi K3：架构、训练与百万 Token Agentic RL 技术解读" §3.1: it
accumulates beta k v^T with decays at most 1), so large values and large
initial states are legitimate inputs.  These tests take v scaled by powers of
two (exact in bf16) and large initial states:
  - well inside the range (v x 128, S0 of std 10): parity with the oracle at
    the usual tolerances, on every chain width;
  - near the documented limit (v x 4096, |beta v| up to ~2e4): parity;
  - beyond it (v x 32768: beta v itself exceeds fp16's 65504): the call must
    report KDA_ERR_NONFINITE through the device error word instead of
    returning inf silently, and the next call must be clean.
"""
import numpy as np
import pytest
import torch

import kda_synth as ks
import oracle
import linear_attention_recurrence_chunk_gb300 as kda
from kda_testutil import assert_o_close, assert_state_close, prefill_device_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _scaled_bits(bits: np.ndarray, scale: float) -> np.ndarray:
    """bf16 bit patterns of the stored values times a power of two (exact)."""
    x = (ks.bf16_bits_to_f64(bits) * scale).astype(np.float32)
    out = ks.f32_to_bf16_bits(x)
    assert np.array_equal(ks.bf16_bits_to_f64(out), ks.bf16_bits_to_f64(bits) * scale)
    return out


def _run(t, v):
    o, sf = kda.kda_chunk_fwd(t["q"], t["k"], v, t["g"], t["beta"], initial_state=t["s0"], cu_seqlens=t["cu"])
    torch.cuda.synchronize()
    return o, sf, kda.kda_device_error()


@pytest.mark.parametrize("chain_cols", ["32", "64", "128"])
@pytest.mark.parametrize("v_scale,s0_std", [(128.0, 10.0), (4096.0, 10.0)])
def test_large_values_match_oracle(monkeypatch, chain_cols, v_scale, s0_std):
    monkeypatch.setenv("KDA_CHAIN_COLUMNS", chain_cols)
    w = ks.PrefillWorkload("range", "bf16", 2, 400, 2, 128, 128, seed=600 + int(v_scale), s0_std=s0_std)
    t = prefill_device_inputs(w, DEV)
    v = (t["v"].float() * v_scale).to(torch.bfloat16)
    o, sf, (st, code) = _run(t, v)
    assert st == 0 and code == 0, (kda.STATUS.get(st, st), code)
    for s in range(w.num_seqs):
        for h in range(w.H):
            ci = w.chain_inputs(s, h)
            o_ref, s_ref = oracle.recurrence(ci["q"], ci["k"], _scaled_bits(ci["v"], v_scale), ci["g"], ci["beta"],
                                             ci["s0"].astype(np.float64), dtype=oracle.BF16)
            tok0, L = w.seq_bounds(s)
            got = o.reshape(w.tokens, w.H, w.d_v)[tok0: tok0 + L, h].float().cpu().numpy()
            assert_o_close([got], [o_ref], "bf16", record=f"range: v x {int(v_scale)}, S0 std {s0_std}")
            assert_state_close(sf[s, h].cpu().numpy(), s_ref, record=f"range: v x {int(v_scale)}, S0 std {s0_std}")
            assert np.abs(s_ref).max() > 0.1 * v_scale   # the state really is large (about 0.5 max|S| at v x 1)


@pytest.mark.parametrize("chain_cols", ["32", "128"])
def test_out_of_range_reports_nonfinite(monkeypatch, chain_cols):
    monkeypatch.setenv("KDA_CHAIN_COLUMNS", chain_cols)
    w = ks.PrefillWorkload("range_over", "bf16", 1, 200, 2, 128, 128, seed=77, s0_std=0.05)
    t = prefill_device_inputs(w, DEV)
    assert float(t["v"].float().abs().max()) * 32768.0 > 65504.0
    v = (t["v"].float() * 32768.0).to(torch.bfloat16)
    o, sf, (st, code) = _run(t, v)
    assert kda.STATUS[st] == "KDA_ERR_NONFINITE" and code == 3, (st, code)
    assert not (torch.isfinite(o.float()).all() and torch.isfinite(sf).all())
    # the word was read and cleared: an in-range call afterwards is clean
    o2, sf2, (st2, code2) = _run(t, t["v"])
    assert st2 == 0 and code2 == 0
    assert torch.isfinite(o2.float()).all() and torch.isfinite(sf2).all()
