"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs, element by element, plus cross-call invariants and edge
cases.  Tolerances are those of kda_testutil (fp32: 1e-4 rms, bf16: 2e-2 rms,
state: 1e-2 relative Frobenius)."""
import numpy as np
import pytest
import torch

import kda_synth as ks
import oracle
import linear_attention_recurrence_chunk_gb300 as kda
from kda_testutil import (assert_o_close, assert_state_close, gpu_chain_outputs, o_excess, oracle_chains,
                          prefill_device_inputs)

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _run_prefill(w, t, **kw):
    o, sf = kda.kda_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], initial_state=t["s0"],
                              cu_seqlens=t["cu"], **kw)
    torch.cuda.synchronize()
    st, code = kda.kda_device_error()
    assert st == 0 and code == 0, (st, code)
    return o, sf


def _check_all_chains(w, o, sf, pairs=None, ntok=None, record=None):
    pairs = pairs or [(s, h) for s in range(w.num_seqs) for h in range(w.H)]
    o_ref, s_ref = oracle_chains(w, pairs, ntok)
    assert_o_close(gpu_chain_outputs(w, o, pairs, ntok), o_ref, w.dtype, record=record)
    if ntok is None and sf is not None:
        s_gpu = np.stack([sf[s, h].cpu().numpy() for s, h in pairs])
        assert_state_close(s_gpu, s_ref, record=record)


# --------------------------------------------------------------------- prefill
SMALL = [  # (dtype, d_k, d_v, B, T, s0_std)
    ("f32", 64, 64, 1, 256, None),
    ("f32", 128, 128, 2, 130, 0.1),
    ("f32", 64, 128, 1, 17, 0.1),
    ("f32", 128, 64, 1, 64, 0.1),
    ("bf16", 128, 128, 2, 1, 0.05),
    ("bf16", 128, 128, 1, 15, None),
    ("bf16", 128, 128, 1, 16, 0.05),
    ("bf16", 128, 128, 2, 63, 0.05),
    ("bf16", 128, 128, 1, 65, 0.05),
    ("bf16", 128, 128, 3, 200, 0.05),
    ("bf16", 64, 64, 2, 300, 0.05),
    ("bf16", 64, 128, 1, 129, 0.05),
    ("bf16", 128, 64, 1, 191, None),
]


@pytest.mark.parametrize("dtype,d_k,d_v,B,T,s0_std", SMALL)
def test_prefill_small_all_outputs(dtype, d_k, d_v, B, T, s0_std):
    w = ks.PrefillWorkload("small", dtype, B, T, 3, d_k, d_v, seed=1000 + T + d_k, s0_std=s0_std)
    t = prefill_device_inputs(w, DEV)
    o, sf = _run_prefill(w, t)
    _check_all_chains(w, o, sf)


@pytest.mark.parametrize("chain_cols", ["32", "64", "full"])
@pytest.mark.parametrize("d_v,B,T,lens", [(128, 2, 1, None), (128, 3, 200, None), (64, 1, 191, None),
                                          (128, 1, None, [0, 1, 63, 64, 65, 200, 0, 17])])
def test_prefill_both_chain_widths(monkeypatch, chain_cols, d_v, B, T, lens):
    """Every inter-chunk variant (32, 64 or all value columns per CTA) on the
    same small cases: full tiles, ragged tails, empty sequences."""
    monkeypatch.setenv("KDA_CHAIN_COLUMNS", str(d_v) if chain_cols == "full" else chain_cols)
    if lens is not None:
        lens = np.array(lens)
        w = ks.PrefillWorkload("widths", "bf16", 1, int(lens.sum()), 3, 128, d_v, seed=321, s0_std=0.05,
                               seq_lens=lens)
    else:
        w = ks.PrefillWorkload("widths", "bf16", B, T, 3, 128, d_v, seed=123 + T, s0_std=0.05)
    t = prefill_device_inputs(w, DEV)
    o, sf = _run_prefill(w, t)
    _check_all_chains(w, o, sf)


@pytest.mark.parametrize("streams", ["1", "2"])
@pytest.mark.parametrize("d_v,B,T,lens", [(128, 1, 1, None), (128, 3, 200, None), (64, 1, 191, None),
                                          (64, 2, 130, None), (128, 1, None, [0, 1, 63, 64, 65, 200, 0, 17])])
def test_prefill_both_prep_kernels(monkeypatch, streams, d_v, B, T, lens):
    """The bounded map's prep with two task streams per CTA (the default) and
    with one (KDA_PREP_STREAMS=1) on the same small cases: fewer tasks than
    streams, odd task counts, ragged tails, empty sequences."""
    monkeypatch.setenv("KDA_PREP_STREAMS", streams)
    if lens is not None:
        lens = np.array(lens)
        w = ks.PrefillWorkload("streams", "bf16", 1, int(lens.sum()), 3, 128, d_v, seed=654, s0_std=0.05,
                               seq_lens=lens)
    else:
        w = ks.PrefillWorkload("streams", "bf16", B, T, 3, 128, d_v, seed=456 + T, s0_std=0.05)
    t = prefill_device_inputs(w, DEV)
    o, sf = _run_prefill(w, t)
    _check_all_chains(w, o, sf)


def test_fp32_b1_h2_t256_d64_workload():
    """The fp32 workload in full (B=1, H=2, T=256, d=64, S0 = 0)."""
    w = ks.workloads()["fp32_b1_h2_t256_d64"]
    t = prefill_device_inputs(w, DEV)
    o, sf = _run_prefill(w, t)
    _check_all_chains(w, o, sf, record="fp32_b1_h2_t256_d64 (all chains)")


@pytest.mark.parametrize("lens", [[0, 1, 63, 64, 65, 200, 0, 17], [128], [5, 0, 0, 300]])
def test_prefill_varlen_small(lens):
    lens = np.array(lens)
    w = ks.PrefillWorkload("varlen_small", "bf16", 1, int(lens.sum()), 4, 128, 128, seed=77 + len(lens),
                           s0_std=0.05, seq_lens=lens)
    t = prefill_device_inputs(w, DEV)
    o, sf = _run_prefill(w, t)
    _check_all_chains(w, o, sf)
    # empty sequences hand their initial state straight through
    for s in np.flatnonzero(lens == 0):
        torch.testing.assert_close(sf[s], t["s0"][s], rtol=0, atol=0)


def test_prefill_h32_t65536_full_size_sampled():
    """Full-size B=1, H=32, T=65536 bf16: every output and the final state of
    four sampled heads against the oracle."""
    w = ks.workloads()["prefill_b1_h32_t65536_d128"]
    t = prefill_device_inputs(w, DEV)
    o, sf = _run_prefill(w, t)
    _check_all_chains(w, o, sf, pairs=[(0, 0), (0, 7), (0, 19), (0, 31)],
                      record="prefill_b1_h32_t65536_d128 (4 heads)")


def test_prefill_b8_h96_t8192_full_size_sampled():
    """Full-size B=8, H=96, T=8192 bf16, no initial state: 32 chains, four on
    each of the eight sequences, every output and final state."""
    w = ks.workloads()["prefill_b8_h96_t8192_d128"]
    t = prefill_device_inputs(w, DEV)
    o, sf = _run_prefill(w, t)
    rng = np.random.default_rng(2)
    pairs = [(s, int(h)) for s in range(w.num_seqs) for h in rng.choice(w.H, 4, replace=False)]
    _check_all_chains(w, o, sf, pairs=pairs, record="prefill_b8_h96_t8192_d128 (32 chains)")


def test_varlen_1m_full_size_sampled():
    """Full-size packed varlen (12 sequences, 1,048,576 tokens, H=32): the
    three shortest sequences in full on every fourth head, and the longest
    sequence (the deepest chain, thousands of chunks) in full on two heads,
    every output row and its final state."""
    w = ks.workloads()["varlen_12seq_1m_h32_d128"]
    t = prefill_device_inputs(w, DEV)
    o, sf = _run_prefill(w, t)
    order = np.argsort(w.seq_lens)
    short = [int(s) for s in order[:3]]
    _check_all_chains(w, o, sf, pairs=[(s, h) for s in short for h in range(0, w.H, 4)],
                      record="varlen_12seq_1m_h32_d128 (3 shortest seqs)")
    longest = int(order[-1])
    assert w.seq_lens[longest] > 200_000
    _check_all_chains(w, o, sf, pairs=[(longest, 3), (longest, 30)],
                      record="varlen_12seq_1m_h32_d128 (longest seq, 2 heads)")


# ---------------------------------------------------------- prefill invariants
def _bf16_case(B=1, T=300, H=2, seed=5, s0=0.05, lens=None):
    return ks.PrefillWorkload("inv", "bf16", B, T, H, 128, 128, seed=seed, s0_std=s0,
                              seq_lens=None if lens is None else np.array(lens))


def test_split_prefill_hands_state_over():
    """prefill(T1) then prefill(T2, initial_state = its final state) equals
    prefill(T1 + T2), and in-place state update (final_state aliasing
    initial_state) gives the same result."""
    w = _bf16_case(T=320)
    t = prefill_device_inputs(w, DEV)
    o_full, s_full = _run_prefill(w, t)
    T1 = 136
    part = {k_: (v_[:, :T1].contiguous() if k_ in ("q", "k", "v", "g", "beta") else v_) for k_, v_ in t.items()}
    o1, s1 = _run_prefill(w, part)
    rest = {k_: (v_[:, T1:].contiguous() if k_ in ("q", "k", "v", "g", "beta") else v_) for k_, v_ in t.items()}
    rest["s0"] = s1.clone()
    o2, _ = kda.kda_chunk_fwd(rest["q"], rest["k"], rest["v"], rest["g"], rest["beta"],
                              initial_state=rest["s0"], final_state=rest["s0"])
    torch.cuda.synchronize()
    ref = o_full.float().cpu().numpy()
    rms = float(np.sqrt(np.mean(ref.astype(np.float64) ** 2)))
    got = torch.cat([o1, o2], dim=1).float().cpu().numpy()
    assert o_excess(got, ref, "bf16").max() <= 2e-2 * rms
    rel = ((rest["s0"] - s_full).norm() / s_full.norm()).item()
    assert rel <= 1e-2


def test_varlen_equals_separate_calls():
    lens = [70, 0, 129, 64]
    w = _bf16_case(T=sum(lens), H=3, lens=lens, seed=9)
    t = prefill_device_inputs(w, DEV)
    o, sf = _run_prefill(w, t)
    cu = w.cu_seqlens()
    for s, L in enumerate(lens):
        a, b = int(cu[s]), int(cu[s + 1])
        sub = {k_: v_[:, a:b].contiguous() for k_, v_ in t.items() if k_ in ("q", "k", "v", "g", "beta")}
        o_s, s_s = kda.kda_chunk_fwd(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"],
                                     initial_state=t["s0"][s:s + 1].contiguous())
        torch.cuda.synchronize()
        if L:
            ref = o[:, a:b].float().cpu().numpy()
            rms = float(np.sqrt(np.mean(ref.astype(np.float64) ** 2)))
            assert o_excess(o_s.float().cpu().numpy(), ref, "bf16").max() <= 2e-2 * rms
        assert ((s_s[0] - sf[s]).norm() / sf[s].norm()).item() <= 1e-2


def test_gate_on_lower_bound_stays_finite():
    """All logits +30 (every alpha on the e^-5 bound): the diagonal sub-tile
    factors reach e^80, the edge of the bf16/fp32 range argument."""
    w = _bf16_case(T=200, H=2, seed=21)
    t = prefill_device_inputs(w, DEV)
    t["g"].fill_(30.0)
    o, sf = _run_prefill(w, t)
    assert torch.isfinite(o.float()).all() and torch.isfinite(sf).all()
    g_host = np.full((w.T, w.d_k), ks.f32_to_bf16_bits(np.array([30.0], np.float32))[0], np.uint16)
    for h in range(w.H):
        ci = w.chain_inputs(0, h)
        o_ref, s_ref = oracle.recurrence(ci["q"], ci["k"], ci["v"], g_host, ci["beta"],
                                         ci["s0"].astype(np.float64), dtype=oracle.BF16)
        assert_o_close([o[0, :, h].float().cpu().numpy()], [o_ref], "bf16")
        assert_state_close(sf[0, h].cpu().numpy(), s_ref)


def test_no_decay_no_initial_state_and_t0():
    """T = 0 writes the initial state to final_state; no initial state means zeros."""
    w = _bf16_case(T=0, H=2, seed=3)
    t = prefill_device_inputs(w, DEV)
    o, sf = _run_prefill(w, t)
    torch.testing.assert_close(sf, t["s0"], rtol=0, atol=0)
    w2 = _bf16_case(T=0, H=2, seed=3, s0=None)
    t2 = prefill_device_inputs(w2, DEV)
    _, sf2 = _run_prefill(w2, t2)
    assert (sf2 == 0).all()


def test_malformed_cu_seqlens_reported_on_device():
    lens = [10, 20]
    w = _bf16_case(T=30, H=2, lens=lens)
    t = prefill_device_inputs(w, DEV)
    t["cu"] = torch.tensor([0, 25, 20], dtype=torch.int32, device=DEV)   # decreasing
    o = torch.full_like(t["v"], 7.0)
    sf = torch.full((2, 2, 128, 128), 3.0, device=DEV)
    kda.kda_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], initial_state=t["s0"], cu_seqlens=t["cu"], o=o,
                      final_state=sf)
    torch.cuda.synchronize()
    st, code = kda.kda_device_error()
    assert st == 1 and code != 0
    assert (o.float() == 7.0).all() and (sf == 3.0).all()
    st, code = kda.kda_device_error()
    assert st == 0 and code == 0


# ---------------------------------------------------------------------- decode
def _decode_inputs(d, step, first=0, count=None):
    count = d.N * d.H if count is None else count
    tdt = torch.bfloat16 if d.dtype == "bf16" else torch.float32

    def dv(name, width):
        a = d.fill_step(step, name, first=first, count=count)
        if d.dtype == "bf16":
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).reshape(count, width)
        return torch.from_numpy(a).reshape(count, width)

    return {"q": dv("q", d.d_k), "k": dv("k", d.d_k), "v": dv("v", d.d_v), "g": dv("g", d.d_k),
            "beta": torch.from_numpy(d.fill_step(step, "beta", first=first, count=count))}, tdt


@pytest.mark.parametrize("dtype,d_k,d_v", [("f32", 64, 64), ("f32", 128, 128), ("bf16", 128, 64),
                                           ("bf16", 64, 128), ("bf16", 128, 128)])
def test_decode_small_all_heads(dtype, d_k, d_v):
    d = ks.DecodeWorkload("dsmall", dtype, 5, 3, d_k, d_v, seed=40 + d_k, state_std=0.05, steps=4)
    heads = d.N * d.H
    st0 = d.fill_state()
    state = torch.from_numpy(st0).reshape(d.N, d.H, d_k, d_v).to(DEV)
    ref = st0.reshape(heads, d_k, d_v).astype(np.float64)
    odt = oracle.F32 if dtype == "f32" else oracle.BF16
    for step in range(d.steps):
        x, _ = _decode_inputs(d, step)
        o = kda.kda_decode_step(*(x[n].reshape(d.N, d.H, -1).to(DEV) for n in ("q", "k", "v", "g")),
                                x["beta"].reshape(d.N, d.H).to(DEV), state)
        host = {n: d.fill_step(step, n) for n in ("q", "k", "v", "g", "beta")}
        outs, ref, _ = oracle.chains(host["q"], host["k"], host["v"], host["g"], host["beta"], odt, d_k, d_v, 1,
                                     list(range(heads)), [1] * heads, ref)
        assert_o_close([o.float().cpu().numpy().reshape(heads, d_v)], [np.concatenate(outs)], dtype)
    assert_state_close(state.cpu().numpy().reshape(heads, d_k, d_v), ref)


def test_decode_n256_h96_100_steps_sampled():
    """Full-size decode (256 sequences x 96 heads, fp32 state N(0, 0.05)), 100
    steps with fresh tokens, every head on the GPU; o of every step and the
    state after step 100 of 384 sampled heads against the oracle."""
    d = ks.workloads()["decode_n256_h96_d128_x100"]
    heads = d.N * d.H
    state = torch.from_numpy(d.fill_state()).reshape(d.N, d.H, 128, 128).to(DEV)
    sample = np.arange(0, heads, 64)       # 384 heads spread over sequences and heads
    ref = np.stack([d.fill_state(first_head=int(hd), count=1).reshape(128, 128) for hd in sample]).astype(np.float64)
    for step in range(d.steps):
        x, _ = _decode_inputs(d, step)
        o = kda.kda_decode_step(*(x[n].reshape(d.N, d.H, -1).to(DEV) for n in ("q", "k", "v", "g")),
                                x["beta"].reshape(d.N, d.H).to(DEV), state)
        sub = {n: np.ascontiguousarray(d.fill_step(step, n)[sample]) for n in ("q", "k", "v", "g", "beta")}
        outs, ref, _ = oracle.chains(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], oracle.BF16, 128, 128, 1,
                                     list(range(len(sample))), [1] * len(sample), ref)
        got = o.reshape(heads, 128)[torch.from_numpy(sample).to(DEV)].float().cpu().numpy()
        assert_o_close([got], [np.concatenate(outs)], "bf16", what=f"o at step {step}",
                       record="decode_n256_h96_d128_x100 (384 heads)")
    s_gpu = state.reshape(heads, 128, 128)[torch.from_numpy(sample).to(DEV)].cpu().numpy()
    assert_state_close(s_gpu, ref, record="decode_n256_h96_d128_x100 (384 heads)")


def test_decode_steps_equal_prefill():
    """N decode steps on one sequence equal a prefill over the same N tokens."""
    w = _bf16_case(T=40, H=4, seed=31)
    t = prefill_device_inputs(w, DEV)
    o_p, s_p = _run_prefill(w, t)
    state = t["s0"].clone()
    outs = []
    for i in range(w.T):
        outs.append(kda.kda_decode_step(t["q"][:, i].contiguous(), t["k"][:, i].contiguous(),
                                        t["v"][:, i].contiguous(), t["g"][:, i].contiguous(),
                                        t["beta"][:, i].contiguous(), state))
    torch.cuda.synchronize()
    o_d = torch.stack(outs, dim=1).float().cpu().numpy()
    o_pn = o_p.float().cpu().numpy()
    rms = float(np.sqrt(np.mean(o_pn.astype(np.float64) ** 2)))
    assert o_excess(o_d, o_pn, "bf16").max() <= 2e-2 * rms
    assert ((state - s_p).norm() / s_p.norm()).item() <= 1e-2
