"""GPU parity of the state snapshots (``kda_chunk_fwd_snapshots``, the
prefix-cache states of page "Kimi K3：架构、训练与百万 Token Agentic RL 技术解读" §9):
every stored snapshot against the oracle's state after the same number of
tokens, on the tensor-core path at every chain width and on the SIMT path,
batched and varlen (empty sequences, ragged tails, lengths that are exact
multiples of the interval); outputs and final states are those of
``kda_chunk_fwd``."""
import numpy as np
import pytest
import torch

import kda_synth as ks
import oracle
import linear_attention_recurrence_chunk_gb300 as kda
from kda_testutil import ORACLE_DT, assert_state_close, prefill_device_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _oracle_snapshots(w, pairs, every):
    """Oracle states after every ``every`` tokens of each (seq, head) chain."""
    ins = [w.chain_inputs(s, h) for s, h in pairs]
    n = [len(x["beta"]) for x in ins]
    cat = {k: np.concatenate([x[k] for x in ins]) for k in ("q", "k", "v", "g", "beta")}
    s0 = None if w.s0_std is None else np.stack([x["s0"] for x in ins]).astype(np.float64)
    row0 = np.concatenate([[0], np.cumsum(n)[:-1]])
    _, states, _, snaps = oracle.chains(cat["q"], cat["k"], cat["v"], cat["g"], cat["beta"], ORACLE_DT[w.dtype],
                                        w.d_k, w.d_v, 1, row0, n, s0, snap_every=every)
    return snaps, states


def _first_slots(w, every):
    """First snapshot slot of each sequence: the snapshots of the earlier ones."""
    counts = [w.seq_bounds(s)[1] // every for s in range(w.num_seqs)]
    return np.concatenate([[0], np.cumsum(counts)[:-1]]).astype(int), counts


def _run(w, every, **kw):
    t = prefill_device_inputs(w, DEV)
    o, sf, snaps = kda.kda_chunk_fwd_snapshots(t["q"], t["k"], t["v"], t["g"], t["beta"], every,
                                               initial_state=t["s0"], cu_seqlens=t["cu"], **kw)
    torch.cuda.synchronize()
    st, code = kda.kda_device_error()
    assert st == 0 and code == 0, (st, code)
    return t, o, sf, snaps


def _check(w, every, snaps, sf, pairs=None):
    pairs = pairs or [(s, h) for s in range(w.num_seqs) for h in range(w.H)]
    ref, s_ref = _oracle_snapshots(w, pairs, every)
    first, counts = _first_slots(w, every)
    total = int(sum(counts))
    assert snaps.shape[0] >= total
    got_all = snaps.cpu().numpy()
    n_checked = 0
    for (s, h), r, sr in zip(pairs, ref, s_ref):
        assert r.shape[0] == counts[s]
        for m in range(counts[s]):
            assert_state_close(got_all[first[s] + m, h], r[m], what=f"snapshot {m + 1} of seq {s} head {h}")
            n_checked += 1
        L = w.seq_bounds(s)[1]
        if counts[s] and L % every == 0:   # the last snapshot is the final state
            np.testing.assert_array_equal(got_all[first[s] + counts[s] - 1, h], sf[s, h].cpu().numpy())
    return n_checked


@pytest.mark.parametrize("chain_cols", ["32", "64", "full"])
@pytest.mark.parametrize("d_v,B,T,lens,every", [
    (128, 2, 1100, None, 256),
    (64, 1, 640, None, 128),
    (128, 1, None, [0, 64, 512, 513, 700, 1024, 100], 128),
])
def test_snapshots_tensor_core_path(monkeypatch, chain_cols, d_v, B, T, lens, every):
    monkeypatch.setenv("KDA_CHAIN_COLUMNS", str(d_v) if chain_cols == "full" else chain_cols)
    if lens is not None:
        lens = np.array(lens)
        w = ks.PrefillWorkload("snap", "bf16", 1, int(lens.sum()), 3, 128, d_v, seed=901, s0_std=0.05,
                               seq_lens=lens)
    else:
        w = ks.PrefillWorkload("snap", "bf16", B, T, 3, 128, d_v, seed=900 + T, s0_std=0.05)
    _, o, sf, snaps = _run(w, every)
    assert _check(w, every, snaps, sf) > 0


@pytest.mark.parametrize("d_k,d_v,B,T,every", [(64, 64, 1, 300, 64), (128, 128, 2, 130, 128), (64, 128, 1, 256, 128)])
def test_snapshots_simt_path(d_k, d_v, B, T, every):
    w = ks.PrefillWorkload("snap_f32", "f32", B, T, 2, d_k, d_v, seed=950 + T, s0_std=0.1)
    _, o, sf, snaps = _run(w, every)
    assert _check(w, every, snaps, sf) > 0


def test_snapshots_leave_outputs_unchanged():
    """Outputs and final states are bit-identical to kda_chunk_fwd's."""
    lens = np.array([300, 0, 1024, 77])
    w = ks.PrefillWorkload("snap_same", "bf16", 1, int(lens.sum()), 4, 128, 128, seed=960, s0_std=0.05,
                           seq_lens=lens)
    t, o, sf, snaps = _run(w, 256)
    o2, sf2 = kda.kda_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], initial_state=t["s0"],
                                cu_seqlens=t["cu"])
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(sf, sf2)


def test_snapshots_every_512_tokens_sampled():
    """The pages' interval (512 tokens) on a longer sequence, sampled heads."""
    w = ks.PrefillWorkload("snap_512", "bf16", 1, 4096 + 200, 32, 128, 128, seed=970, s0_std=0.01)
    _, o, sf, snaps = _run(w, 512)
    assert snaps.shape[0] == (4096 + 200) // 512
    assert _check(w, 512, snaps, sf, pairs=[(0, 0), (0, 13), (0, 31)]) == 3 * 8


def test_no_snapshot_when_sequences_are_shorter_than_the_interval():
    lens = np.array([63, 0, 500])
    w = ks.PrefillWorkload("snap_none", "bf16", 1, int(lens.sum()), 2, 128, 128, seed=980, s0_std=0.05,
                           seq_lens=lens)
    t = prefill_device_inputs(w, DEV)
    sentinel = torch.full((1, w.H, 128, 128), 7.0, device=DEV)
    _, _, snaps = kda.kda_chunk_fwd_snapshots(t["q"], t["k"], t["v"], t["g"], t["beta"], 512,
                                              initial_state=t["s0"], cu_seqlens=t["cu"], snapshots=sentinel)
    torch.cuda.synchronize()
    assert kda.kda_device_error() == (0, 0)
    assert snaps.shape[0] == 1 and bool((sentinel == 7.0).all())   # the slot is not written
