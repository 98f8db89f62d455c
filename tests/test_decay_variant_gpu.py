"""GPU parity of the decay-map ablation (``kda_chunk_fwd_decay_variant``): the
diagonal 16x16 tiles formed by position pairs on the CUDA cores, under the
bounded -5 Sigmoid map and under the unbounded -Softplus map of the
predecessor model (page "Kimi K3 架构篇：一文详解 2.8 万亿参数的巨型怪兽", section
"最被低估的一个细节：下界衰减"), against the fp64 oracle under the same map:
batched and varlen (empty sequences, ragged tails), d_v = 128 and 64, in-tile
decays far past the e^80 that the bound guarantees, and the benchmark's full
size on sampled heads.  Tolerances are those of kda_testutil."""
import numpy as np
import pytest
import torch

import kda_synth as ks
import oracle
import linear_attention_recurrence_chunk_gb300 as kda
from kda_testutil import assert_o_close, assert_state_close, gpu_chain_outputs, oracle_chains, prefill_device_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"
MAPS = {"bounded": (kda.DECAY_BOUNDED, oracle.DECAY_BOUNDED), "softplus": (kda.DECAY_SOFTPLUS, oracle.DECAY_SOFTPLUS)}


def _run(t, dmap, pairs=True):
    o, sf = kda.kda_chunk_fwd_decay_variant(t["q"], t["k"], t["v"], t["g"], t["beta"], decay_map=dmap,
                                            diag_by_pairs=pairs, initial_state=t["s0"], cu_seqlens=t["cu"])
    torch.cuda.synchronize()
    assert kda.kda_device_error() == (0, 0)
    return o, sf


def _check(w, o, sf, omap, pairs=None, ntok=None):
    pairs = pairs or [(s, h) for s in range(w.num_seqs) for h in range(w.H)]
    o_ref, s_ref = oracle_chains(w, pairs, ntok, decay_map=omap)
    assert_o_close(gpu_chain_outputs(w, o, pairs, ntok), o_ref, w.dtype)
    if ntok is None:
        assert_state_close(np.stack([sf[s, h].cpu().numpy() for s, h in pairs]), s_ref)


@pytest.mark.parametrize("gate", sorted(MAPS))
@pytest.mark.parametrize("d_v,B,T,lens", [
    (128, 2, 300, None),
    (128, 1, None, [0, 1, 63, 64, 65, 200, 0, 17]),
    (64, 1, 200, None),
    (64, 1, None, [130, 0, 64]),
])
def test_pair_diagonal_matches_oracle(gate, d_v, B, T, lens):
    dmap, omap = MAPS[gate]
    if lens is not None:
        lens = np.array(lens)
        w = ks.PrefillWorkload("pairs", "bf16", 1, int(lens.sum()), 3, 128, d_v, seed=711, s0_std=0.05, seq_lens=lens)
    else:
        w = ks.PrefillWorkload("pairs", "bf16", B, T, 3, 128, d_v, seed=710 + T, s0_std=0.05)
    t = prefill_device_inputs(w, DEV)
    o, sf = _run(t, dmap)
    _check(w, o, sf, omap)


def test_bounded_tensor_core_diagonal_is_the_plain_call():
    """decay_map = bounded with the tensor-core diagonal is kda_chunk_fwd: the
    same kernels, bit for bit."""
    w = ks.PrefillWorkload("pairs", "bf16", 2, 200, 2, 128, 128, seed=720, s0_std=0.05)
    t = prefill_device_inputs(w, DEV)
    o1, s1 = _run(t, kda.DECAY_BOUNDED, pairs=False)
    o2, s2 = kda.kda_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], initial_state=t["s0"])
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_softplus_in_tile_decay_far_past_the_bound():
    """Logits +40 on the first 32 key channels (N(0, 2^2) elsewhere): those
    channels decay by e^-40 per token, so inside a 16-token tile the cumulative
    decay reaches e^-640, where the tensor-core diagonal's factors
    e^{G_s - G_i} would be e^{+600} and overflow.  The pair path stays finite
    and matches the oracle on every head."""
    w = ks.PrefillWorkload("stress", "bf16", 1, 200, 2, 128, 128, seed=730, s0_std=0.05)
    t = prefill_device_inputs(w, DEV)
    t["g"][..., :32] = 40.0
    o, sf = _run(t, kda.DECAY_SOFTPLUS)
    assert torch.isfinite(o.float()).all() and torch.isfinite(sf).all()
    forty = ks.f32_to_bf16_bits(np.array([40.0], np.float32))[0]
    for h in range(w.H):
        ci = w.chain_inputs(0, h)
        g_host = ci["g"].copy()
        g_host[:, :32] = forty
        o_ref, s_ref = oracle.recurrence(ci["q"], ci["k"], ci["v"], g_host, ci["beta"], ci["s0"].astype(np.float64),
                                         dtype=oracle.BF16, decay_map=oracle.DECAY_SOFTPLUS)
        assert_o_close([o[0, :, h].float().cpu().numpy()], [o_ref], "bf16")
        assert_state_close(sf[0, h].cpu().numpy(), s_ref)


@pytest.mark.parametrize("gate", sorted(MAPS))
def test_pairs_full_size_sampled(gate):
    """The benchmark's workload (B=1, H=32, T=65536, bf16) with the pair
    diagonal: every output and the final state of two sampled heads."""
    dmap, omap = MAPS[gate]
    w = ks.workloads()["prefill_b1_h32_t65536_d128"]
    t = prefill_device_inputs(w, DEV)
    o, sf = _run(t, dmap)
    _check(w, o, sf, omap, pairs=[(0, 3), (0, 28)])
