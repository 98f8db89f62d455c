"""GPU parity of the chunked prefill with the output epilogue
(``kda_chunk_fwd_gated``: ``o = Sigmoid(gate) * RMSNorm(o~) * w`` per token and
head before o is written, page "Kimi K3：架构、训练与百万 Token Agentic RL 技术解读"
§3.2) against the fp64 oracle's o~ put through the same definitions
(``oracle.decode_layer``'s pinned ``sigmoid`` and ``rmsnorm``): batched and
varlen (empty sequences, ragged tails), d_v = 128 and 64, with and without the
norm weight; final states as the oracle's."""
import numpy as np
import pytest
import torch

import kda_synth as ks
from oracle import decode_layer as dl
import linear_attention_recurrence_chunk_gb300 as kda
from kda_testutil import (assert_state_close, gpu_chain_outputs, half_ulp_bf16, oracle_chains,
                          prefill_device_inputs)

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _assert_gated_close(got_rows, ref_rows, o_ref_rows, gate_rows, w_rows):
    """The per-row RMSNorm divides o~'s error by the row's own RMS: o~ meets
    |d o~| <= 2e-2 rms(o~) (over all rows), allowed here with the half-ulp of a
    bf16 value on top, so the gated output may differ by
    (2e-2 rms(o~) + ulp(o~)/2) / rms(o~ row) * Sigmoid(gate) * |w| per element,
    plus the half-ulp of its own rounding."""
    rms = np.sqrt(np.mean(np.concatenate([x.reshape(-1) for x in o_ref_rows]) ** 2))
    worst = 0.0
    for got, ref, oref, g, wr in zip(got_rows, ref_rows, o_ref_rows, gate_rows, w_rows):
        row_rms = np.sqrt(np.mean(oref ** 2, axis=-1, keepdims=True) + 1e-6)
        bound = (2e-2 * rms + half_ulp_bf16(oref)) / row_rms * dl.sigmoid(g) * np.abs(wr)
        excess = np.abs(got - ref) - half_ulp_bf16(got)
        worst = max(worst, float((excess / bound).max()) if excess.size else 0.0)
    assert worst <= 1.0, f"gated o: error {worst:.3f} x its bound"


def _gate_inputs(w, seed, weighted):
    rng = np.random.default_rng(seed)
    gate = torch.from_numpy(rng.normal(size=(w.tokens, w.H, w.d_v)).astype(np.float32)).to(torch.bfloat16)
    nw = None
    if weighted:
        nw = torch.from_numpy((1 + 0.2 * rng.normal(size=(w.H, w.d_v))).astype(np.float32))
    return gate, nw


# the epilogue fused into the 32-column chain (row sums exchanged within each
# head's cluster of CTAs), into the all-columns chain, and a forced 64-column
# width (which the gated call replaces by the all-columns chain)
@pytest.mark.parametrize("chain_cols", ["32", "64", "full"])
@pytest.mark.parametrize("d_v,B,T,lens,weighted", [
    (128, 2, 300, None, True),
    (128, 1, None, [0, 1, 63, 64, 65, 200, 0, 17], False),
    (64, 1, 200, None, True),
    (64, 1, None, [130, 0, 64], False),
])
def test_gated_prefill_matches_oracle(monkeypatch, chain_cols, d_v, B, T, lens, weighted):
    monkeypatch.setenv("KDA_CHAIN_COLUMNS", str(d_v) if chain_cols == "full" else chain_cols)
    if lens is not None:
        lens = np.array(lens)
        w = ks.PrefillWorkload("gated", "bf16", 1, int(lens.sum()), 3, 128, d_v, seed=611, s0_std=0.05, seq_lens=lens)
    else:
        w = ks.PrefillWorkload("gated", "bf16", B, T, 3, 128, d_v, seed=610 + T, s0_std=0.05)
    t = prefill_device_inputs(w, DEV)
    gate, nw = _gate_inputs(w, 620 + w.tokens, weighted)
    gate_d = gate.reshape(t["v"].shape).to(DEV)
    o, sf = kda.kda_chunk_fwd_gated(t["q"], t["k"], t["v"], t["g"], t["beta"], gate_d,
                                    norm_weight=None if nw is None else nw.to(DEV), eps_rms=1e-6,
                                    initial_state=t["s0"], cu_seqlens=t["cu"])
    torch.cuda.synchronize()
    assert kda.kda_device_error() == (0, 0)
    pairs = [(s, h) for s in range(w.num_seqs) for h in range(w.H)]
    o_ref, s_ref = oracle_chains(w, pairs)
    gate64 = gate.double().numpy()
    w64 = np.ones((w.H, d_v)) if nw is None else nw.double().numpy()
    gated_ref, g_rows, w_rows = [], [], []
    for (s, h), orow in zip(pairs, o_ref):
        tok0, L = w.seq_bounds(s)
        g_rows.append(gate64[tok0: tok0 + L, h])
        w_rows.append(np.broadcast_to(w64[h], orow.shape))
        gated_ref.append(dl.sigmoid(g_rows[-1]) * dl.rmsnorm(orow, w64[h][None], 1e-6))
    got = gpu_chain_outputs(w, o, pairs)
    _assert_gated_close(got, gated_ref, o_ref, g_rows, w_rows)
    assert_state_close(np.stack([sf[s, h].cpu().numpy() for s, h in pairs]), s_ref)

    # The epilogue itself, against the GPU's own o~ from a plain call whose chain
    # does the same arithmetic: equal up to the bf16 roundings of o~ and of o.
    # (For any width but 32 the gated call runs the wide chain over all columns;
    # its 64-column form matches it column for column, while a plain call over
    # all 128 columns runs the value-major chain, which forms V_new in fp32.)
    if chain_cols != "32":
        monkeypatch.setenv("KDA_CHAIN_COLUMNS", "64")
    o_plain, _ = kda.kda_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], initial_state=t["s0"],
                                   cu_seqlens=t["cu"])
    torch.cuda.synchronize()
    op = o_plain.double().cpu().numpy().reshape(w.tokens, w.H, d_v)
    og = o.double().cpu().numpy().reshape(w.tokens, w.H, d_v)
    ref = dl.sigmoid(gate64) * dl.rmsnorm(op, w64[None], 1e-6)
    # o~ rounded to bf16 moves each value and the row RMS by at most 2^-9 relative, and o's own
    # rounding adds half an ulp: allowed twice over (binade edges, fast exp / rsqrt)
    allow = 2 * half_ulp_bf16(og) + (2.0 ** -7) * np.abs(ref) + 1e-6
    assert (np.abs(og - ref) <= allow).all(), float((np.abs(og - ref) / allow).max())


def test_gated_prefill_many_heads_sampled():
    """A grid that already selects the all-columns chain (B=4, H=48, T=1000),
    sampled heads against the oracle."""
    w = ks.PrefillWorkload("gated_big", "bf16", 4, 1000, 48, 128, 128, seed=640, s0_std=0.01)
    t = prefill_device_inputs(w, DEV)
    gate, nw = _gate_inputs(w, 641, True)
    o, sf = kda.kda_chunk_fwd_gated(t["q"], t["k"], t["v"], t["g"], t["beta"], gate.reshape(t["v"].shape).to(DEV),
                                    norm_weight=nw.to(DEV), initial_state=t["s0"])
    torch.cuda.synchronize()
    assert kda.kda_device_error() == (0, 0)
    pairs = [(0, 0), (1, 17), (3, 47), (2, 30)]
    o_ref, s_ref = oracle_chains(w, pairs)
    gate64, w64 = gate.double().numpy(), nw.double().numpy()
    gated_ref, g_rows, w_rows = [], [], []
    for (s, h), orow in zip(pairs, o_ref):
        tok0, L = w.seq_bounds(s)
        g_rows.append(gate64[tok0: tok0 + L, h])
        w_rows.append(np.broadcast_to(w64[h], orow.shape))
        gated_ref.append(dl.sigmoid(g_rows[-1]) * dl.rmsnorm(orow, w64[h][None], 1e-6))
    _assert_gated_close(gpu_chain_outputs(w, o, pairs), gated_ref, o_ref, g_rows, w_rows)
    assert_state_close(np.stack([sf[s, h].cpu().numpy() for s, h in pairs]), s_ref)
