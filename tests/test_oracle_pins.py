"""Pins of the fp64 oracle against what the pages and plain mathematics fix.

None of these re-types the oracle's step loop: each compares it with a
different statement of the same quantity (a closed form, a hand-worked
example, a special case that reduces to the textbook delta rule, an explicit
product of transition matrices, or an invariant).  Sources: page
"Kimi K3：架构、训练与百万 Token Agentic RL 技术解读" §3.1 (KDA update, delta rule),
§3.2 (step order), §3.3 (lower-bounded gate, 16-token tile bound), and page
"Kimi K3 架构篇：一文详解 2.8 万亿参数的巨型怪兽" ("KDA 到底在算什么",
"最被低估的一个细节：下界衰减").
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_inputs(rng, n, d_k, d_v, unit=True):
    q = rng.normal(size=(n, d_k))
    k = rng.normal(size=(n, d_k))
    if unit:
        q /= np.linalg.norm(q, axis=1, keepdims=True)
        k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.normal(size=(n, d_v))
    g = 2.0 * rng.normal(size=(n, d_k))
    beta = (1.0 / (1.0 + np.exp(-rng.normal(size=n)))).astype(np.float32)
    return q, k, v, g, beta


@pytest.mark.parametrize("name", ["delta_rule_worked_example.json", "erase_full_decay_example.json"])
def test_hand_worked_examples(name):
    """Hand-derived values (derivation stored with each fixture)."""
    fx = json.load(open(os.path.join(GOLDEN, name)))
    q = np.array(fx["q"], dtype=np.float64)
    k = np.array(fx["k"], dtype=np.float64)
    v = np.array(fx["v"], dtype=np.float64)
    if fx["g"] == "-inf":
        g = np.full(q.shape, -np.inf)
    else:
        g = np.array(fx["g"], dtype=np.float64)
    beta = np.array(fx["beta"], dtype=np.float32)
    s0 = np.array(fx["S0"], dtype=np.float64) if "S0" in fx else None
    o, S = oracle.recurrence(q, k, v, g, beta, s0)
    np.testing.assert_allclose(o, np.array(fx["o"]), rtol=0, atol=1e-13)
    np.testing.assert_allclose(S, np.array(fx["S_final"]), rtol=0, atol=1e-13)


def test_gate_special_values():
    """Gate map of §3.3: logit 0 -> alpha = e^{-5/2}; +inf -> e^{-5} (the
    lower bound); -inf -> 1.  Probed through beta = 0 (pure decay), where
    S_1 = Diag(alpha) S_0 and o_1 = S_1^T q."""
    d = 3
    s0 = np.arange(1.0, 1.0 + d * d).reshape(d, d)
    g = np.array([[0.0, np.inf, -np.inf]])
    q = np.eye(d)[[0]]  # o_1 = S_1^T e_0 = row 0 of S_1
    o, S = oracle.recurrence(q, np.zeros((1, d)), np.zeros((1, d)), g, np.zeros(1, np.float32), s0)
    expect = s0 * np.array([math.exp(-2.5), math.exp(-5.0), 1.0])[:, None]
    np.testing.assert_allclose(S, expect, rtol=1e-15, atol=0)
    np.testing.assert_allclose(o[0], expect[0], rtol=1e-15, atol=0)


def test_pure_decay_closed_form():
    """beta = 0: S_t = Diag(exp(sum_{tau<=t} log alpha_tau)) S_0 and
    o_t = S_t^T q_t, with log alpha = -5 * Sigmoid(logit)."""
    rng = np.random.default_rng(11)
    n, d_k, d_v = 40, 5, 7
    q, k, v, g, _ = _rand_inputs(rng, n, d_k, d_v)
    s0 = rng.normal(size=(d_k, d_v))
    o, S = oracle.recurrence(q, k, v, g, np.zeros(n, np.float32), s0)
    logdecay = -5.0 / (1.0 + np.exp(-g))              # [n, d_k]
    cum = np.cumsum(logdecay, axis=0)
    for t in range(n):
        St = np.exp(cum[t])[:, None] * s0
        np.testing.assert_allclose(o[t], St.T @ q[t], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(S, np.exp(cum[-1])[:, None] * s0, rtol=1e-12, atol=1e-300)


def test_no_decay_is_textbook_delta_rule():
    """alpha == 1 (logit -1e4 => Sigmoid underflows to 0 in fp64) reduces KDA to
    the ungated delta rule of §3.1, written here in its projector form
    S_t = (I - beta k k^T) S_{t-1} + beta k v^T."""
    rng = np.random.default_rng(12)
    n, d_k, d_v = 30, 6, 4
    q, k, v, _, beta = _rand_inputs(rng, n, d_k, d_v)
    g = np.full((n, d_k), -1.0e4)
    s0 = rng.normal(size=(d_k, d_v))
    o, S = oracle.recurrence(q, k, v, g, beta, s0)
    St = s0.copy()
    for t in range(n):
        b = float(beta[t])
        St = (np.eye(d_k) - b * np.outer(k[t], k[t])) @ St + b * np.outer(k[t], v[t])
        np.testing.assert_allclose(o[t], St.T @ q[t], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(S, St, rtol=1e-11, atol=1e-12)


def test_full_write_recalls_value():
    """beta = 1 and unit-norm k: the erase removes the whole old prediction along
    k, so S_t^T k_t = v_t.  Read through o_t with q_t = k_t."""
    rng = np.random.default_rng(13)
    n, d_k, d_v = 50, 8, 5
    _, k, v, g, _ = _rand_inputs(rng, n, d_k, d_v)
    s0 = rng.normal(size=(d_k, d_v))
    o, _ = oracle.recurrence(k, k, v, g, np.ones(n, np.float32), s0)
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-12 * np.abs(v).max())


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_brute_force_transition_product(seed):
    """Tiny inputs, d_k != d_v so a transposed operand cannot pass: build
    M_t = (I - beta_t k_t k_t^T) Diag(alpha_t) explicitly and compare
    S_t = M_t...M_1 S_0 + sum_{tau<=t} M_t...M_{tau+1} beta_tau k_tau v_tau^T
    and o_t = S_t^T q_t with the oracle at every t."""
    rng = np.random.default_rng(100 + seed)
    n, d_k, d_v = 8, 3, 4
    q, k, v, g, beta = _rand_inputs(rng, n, d_k, d_v, unit=False)
    s0 = rng.normal(size=(d_k, d_v))
    alpha = np.exp(-5.0 / (1.0 + np.exp(-g)))
    Ms = [(np.eye(d_k) - float(beta[t]) * np.outer(k[t], k[t])) @ np.diag(alpha[t]) for t in range(n)]

    def prod(a, b):  # M_b ... M_a (a <= b), identity if empty
        P = np.eye(d_k)
        for t in range(a, b + 1):
            P = Ms[t] @ P
        return P

    for m in range(1, n + 1):
        o, S = oracle.recurrence(q[:m], k[:m], v[:m], g[:m], beta[:m], s0)
        St = prod(0, m - 1) @ s0
        for tau in range(m):
            St = St + prod(tau + 1, m - 1) @ (float(beta[tau]) * np.outer(k[tau], v[tau]))
        np.testing.assert_allclose(S, St, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(o[m - 1], St.T @ q[m - 1], rtol=1e-12, atol=1e-13)


def _brute_states(q, k, v, g, beta, s0):
    """S_t for t = 1..n from explicit transition matrices M_t = (I - beta_t k_t k_t^T) Diag(alpha_t)."""
    alpha = np.exp(-5.0 / (1.0 + np.exp(-g)))
    d_k = k.shape[1]
    St, out = np.array(s0, dtype=np.float64), []
    for t in range(len(q)):
        M = (np.eye(d_k) - float(beta[t]) * np.outer(k[t], k[t])) @ np.diag(alpha[t])
        St = M @ St + float(beta[t]) * np.outer(k[t], v[t])
        out.append(St.copy())
    return out


@pytest.mark.parametrize("every", [1, 2, 3, 7])
def test_snapshots_match_brute_force_states(every):
    """State snapshots (the prefix-cache states of the first page's §9): the
    m-th snapshot of a chain is S after its first m*every tokens, checked
    against explicit transition-matrix products for several chains of
    different lengths (one of them empty) sharing the token arrays."""
    rng = np.random.default_rng(300 + every)
    H, d_k, d_v = 3, 3, 4
    lens = [9, 0, 14]
    n = max(lens)
    q, k, v, g, beta = _rand_inputs(rng, n * H, d_k, d_v, unit=False)
    s0 = rng.normal(size=(H, d_k, d_v))
    outs, S, _, snaps = oracle.chains(q, k, v, g, beta, oracle.F64, d_k, d_v, H, list(range(H)), lens, s0,
                                      snap_every=every)
    for h, L in enumerate(lens):
        rows = slice(h, h + H * L, H) if L else slice(0, 0)
        ref = _brute_states(q[rows], k[rows], v[rows], g[rows], beta[rows], s0[h])
        assert snaps[h].shape == (L // every, d_k, d_v)
        for m in range(1, L // every + 1):
            np.testing.assert_allclose(snaps[h][m - 1], ref[m * every - 1], rtol=1e-12, atol=1e-13)
        if L and L % every == 0:
            np.testing.assert_array_equal(snaps[h][-1], S[h])


def test_snapshot_planted_off_by_one_fails_the_pin(tmp_path):
    """A snapshot taken one token early, planted in a compiled copy of the
    oracle, is rejected by the brute-force state comparison."""
    import ctypes
    import subprocess

    src = open(oracle._SRC).read()
    old = "(j + 1) % snap_every == 0)"
    assert src.count(old) == 1
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, "(j + 2) % snap_every == 0 && j + 2 <= n)").replace(
        "memcpy(snaps + ((j + 1) / snap_every - 1)", "memcpy(snaps + ((j + 2) / snap_every - 1)"))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c99", "-fopenmp", "-fPIC", "-shared", str(mpath), "-o", str(so), "-lm"],
                   check=True)
    lib = ctypes.CDLL(str(so))
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.kda_oracle_chains_snap.argtypes = [vp, vp, vp, vp, i32, vp, i64, i32, i32, i32, vp, vp, vp, vp, vp, vp,
                                           i64, vp, vp]
    lib.kda_oracle_chains_snap.restype = ctypes.c_int
    rng = np.random.default_rng(17)
    n, d_k, d_v, every = 8, 3, 4, 4
    q, k, v, g, beta = _rand_inputs(rng, n, d_k, d_v, unit=False)
    s0 = rng.normal(size=(d_k, d_v))
    o, S = np.zeros((n, d_v)), np.zeros((d_k, d_v))
    snaps = np.zeros((n // every, d_k, d_v))
    z, nn = np.zeros(1, np.int64), np.array([n], np.int64)
    arrs = [np.ascontiguousarray(x, dtype=np.float64) for x in (q, k, v, g)]
    assert lib.kda_oracle_chains_snap(*(a.ctypes.data for a in arrs), oracle.F64, beta.ctypes.data, 1, d_k, d_v, 1,
                                      z.ctypes.data, nn.ctypes.data, s0.ctypes.data, o.ctypes.data, z.ctypes.data,
                                      S.ctypes.data, every, snaps.ctypes.data, z.ctypes.data) > 0
    ref = _brute_states(q, k, v, g, beta, s0)
    err = max(np.abs(snaps[m - 1] - ref[m * every - 1]).max() for m in range(1, n // every + 1))
    assert err > 1e-6, f"off-by-one snapshot was not caught (err {err:g})"


def test_gate_lower_bound_tile_edge():
    """All logits +30: alpha sits on the e^{-5} bound, and 16 steps reach a
    cumulative log-decay of -80, the edge of the 16-token tile bound (§3.3).
    The oracle stays finite and matches the closed form there."""
    n, d = 16, 4
    s0 = np.full((d, d), 1.0e30)
    g = np.full((n, d), 30.0)
    o, S = oracle.recurrence(np.ones((n, d)), np.zeros((n, d)), np.zeros((n, d)), g, np.zeros(n, np.float32), s0)
    sig30 = 1.0 / (1.0 + math.exp(-30.0))
    expect = math.exp(-5.0 * sig30 * n) * 1.0e30
    assert np.isfinite(S).all() and np.isfinite(o).all()
    np.testing.assert_allclose(S, expect, rtol=1e-12)
    assert abs(-5.0 * sig30 * n + 80.0) < 1e-11


def test_storage_dtypes_read_exactly():
    """bf16 inputs (bit patterns) and fp32 inputs give the same result as the
    same values passed in fp64 (the oracle widens exactly)."""
    rng = np.random.default_rng(14)
    n, d_k, d_v = 20, 4, 3
    q, k, v, g, beta = _rand_inputs(rng, n, d_k, d_v)
    s0 = rng.normal(size=(d_k, d_v))
    q32, k32, v32, g32 = (x.astype(np.float32) for x in (q, k, v, g))
    o32, S32 = oracle.recurrence(q32, k32, v32, g32, beta, s0, dtype=oracle.F32)
    o64, S64 = oracle.recurrence(*(x.astype(np.float64) for x in (q32, k32, v32, g32)), beta, s0)
    np.testing.assert_array_equal(o32, o64)
    np.testing.assert_array_equal(S32, S64)
    # bf16: truncate fp32 bit patterns (exactly representable values)
    def tobits(x):
        return (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)

    def widen(b):
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)

    qb, kb, vb, gb = (tobits(x) for x in (q, k, v, g))
    ob, Sb = oracle.recurrence(qb, kb, vb, gb, beta, s0, dtype=oracle.BF16)
    ow, Sw = oracle.recurrence(*(widen(x) for x in (qb, kb, vb, gb)), beta, s0)
    np.testing.assert_array_equal(ob, ow)
    np.testing.assert_array_equal(Sb, Sw)


def test_chains_match_single_runs_and_split():
    """Batch entry point: strided chains equal separate calls, and running a
    sequence in two pieces with the state handed over equals one run."""
    rng = np.random.default_rng(15)
    T, H, d_k, d_v = 24, 3, 4, 5
    q, k, v, g, beta = _rand_inputs(rng, T * H, d_k, d_v)
    s0 = rng.normal(size=(H, d_k, d_v))
    outs, S, _ = oracle.chains(q, k, v, g, beta, oracle.F64, d_k, d_v, H, list(range(H)), [T] * H, s0)
    for h in range(H):
        sl = slice(h, None, H)
        o1, S1 = oracle.recurrence(q[sl], k[sl], v[sl], g[sl], beta[sl], s0[h])
        np.testing.assert_array_equal(outs[h], o1)
        np.testing.assert_array_equal(S[h], S1)
        oa, Sa = oracle.recurrence(q[sl][:10], k[sl][:10], v[sl][:10], g[sl][:10], beta[sl][:10], s0[h])
        ob, Sb = oracle.recurrence(q[sl][10:], k[sl][10:], v[sl][10:], g[sl][10:], beta[sl][10:], Sa)
        np.testing.assert_allclose(np.concatenate([oa, ob]), o1, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(Sb, S1, rtol=1e-13, atol=1e-14)


MUTANTS = {
    "decay scales columns": ("S[(int64_t)i * d_v + c] *= alpha[i];", "S[(int64_t)i * d_v + c] *= alpha[c % d_k];"),
    "beta dropped": ("err[c] = b * (", "err[c] = ("),
    "write sign": ("S[(int64_t)i * d_v + c] += kk[i] * err[c];", "S[(int64_t)i * d_v + c] -= kk[i] * err[c];"),
    "transposed read": ("vhat += S[(int64_t)i * d_v + c] * kk[i];",
                        "vhat += S[(int64_t)(c % d_k) * d_v + (i % d_v)] * kk[i];"),
    "gate complement": ("return exp(-5.0 * sig);", "return exp(-5.0 * (1.0 - sig));"),
    "read-out with k": ("acc += S[(int64_t)i * d_v + c] * qq[i];", "acc += S[(int64_t)i * d_v + c] * kk[i];"),
    "no erase": ("vhat += S[(int64_t)i * d_v + c] * kk[i];", "vhat += 0.0 * S[(int64_t)i * d_v + c] * kk[i];"),
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistakes_fail_a_pin(mutant, tmp_path):
    """Plant one plausible mistake in a compiled copy of the oracle's C source
    and check that the brute-force transition-product pin rejects it."""
    import ctypes
    import subprocess

    src = open(oracle._SRC).read()
    old, new = MUTANTS[mutant]
    assert src.count(old) == 1, mutant
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c99", "-fopenmp", "-fPIC", "-shared", str(mpath), "-o", str(so), "-lm"],
                   check=True)
    lib = ctypes.CDLL(str(so))
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.kda_oracle_chains.argtypes = [vp, vp, vp, vp, i32, vp, i64, i32, i32, i32, vp, vp, vp, vp, vp, vp]
    lib.kda_oracle_chains.restype = ctypes.c_int

    rng = np.random.default_rng(16)
    n, d_k, d_v = 8, 3, 4
    q, k, v, g, beta = _rand_inputs(rng, n, d_k, d_v, unit=False)
    s0 = rng.normal(size=(d_k, d_v))
    o = np.zeros((n, d_v))
    S = np.zeros((d_k, d_v))
    r0 = np.zeros(1, np.int64)
    nn = np.array([n], np.int64)
    off = np.zeros(1, np.int64)
    arrs = [np.ascontiguousarray(x, dtype=np.float64) for x in (q, k, v, g)]
    lib.kda_oracle_chains(*(a.ctypes.data for a in arrs), oracle.F64, beta.ctypes.data, 1, d_k, d_v, 1,
                          r0.ctypes.data, nn.ctypes.data, s0.ctypes.data, o.ctypes.data, off.ctypes.data,
                          S.ctypes.data)
    alpha = np.exp(-5.0 / (1.0 + np.exp(-g)))
    St = s0.copy()
    o_ref = np.zeros((n, d_v))
    for t in range(n):
        M = (np.eye(d_k) - float(beta[t]) * np.outer(k[t], k[t])) @ np.diag(alpha[t])
        St = M @ St + float(beta[t]) * np.outer(k[t], v[t])
        o_ref[t] = St.T @ q[t]
    err = max(np.abs(o - o_ref).max(), np.abs(S - St).max())
    assert err > 1e-6, f"mutant '{mutant}' was not caught (err {err:g})"


def test_bf16_rounding_reading():
    """Reading of the bf16 output tolerance: rounding the exact (fp64 oracle)
    outputs of a bf16 workload to bf16 already moves them by more than
    2e-2 * rms(o) (max|o| is 10-20x rms here), so the bound can only apply to
    the computation with each stored value's half-ulp rounding allowed on top;
    with that allowance the exactly rounded result passes (excess at the fp32
    rounding level only)."""
    import kda_synth as ks
    from kda_testutil import half_ulp_bf16, o_excess

    w = ks.PrefillWorkload("x", "bf16", 1, 300, 3, 128, 128, seed=5, s0_std=0.05)
    worst_bare = 0.0
    for h in range(w.H):
        ci = w.chain_inputs(0, h)
        o, _ = oracle.recurrence(ci["q"], ci["k"], ci["v"], ci["g"], ci["beta"], ci["s0"].astype(np.float64),
                                 dtype=oracle.BF16)
        ob = ks.bf16_bits_to_f64(ks.f32_to_bf16_bits(o.astype(np.float32)))
        rms = np.sqrt(np.mean(o ** 2))
        worst_bare = max(worst_bare, np.abs(ob - o).max() / rms)
        # (fp64 -> fp32 -> bf16 double rounding adds at most an fp32 ulp)
        assert o_excess(ob, o, "bf16").max() <= 1e-6 * rms
        assert (np.abs(ob - o) <= half_ulp_bf16(ob) * (1 + 2.0 ** -13)).all()
    assert worst_bare > 2e-2


# ---- the unbounded -Softplus decay map (the predecessor model's gate that the
# ---- second page contrasts with the lower bound, "最被低估的一个细节：下界衰减")

def test_softplus_gate_special_values():
    """log alpha = -ln(1 + e^x): logit 0 -> alpha = 1/2; ln(e - 1) -> 1/e;
    +inf -> 0 (no lower limit); -inf -> 1.  Probed through beta = 0, where
    S_1 = Diag(alpha) S_0."""
    d = 4
    s0 = np.arange(1.0, 1.0 + d * d).reshape(d, d)
    g = np.array([[0.0, math.log(math.e - 1.0), np.inf, -np.inf]])
    o, S = oracle.recurrence(np.eye(d)[[1]], np.zeros((1, d)), np.zeros((1, d)), g, np.zeros(1, np.float32), s0,
                             decay_map=oracle.DECAY_SOFTPLUS)
    expect = s0 * np.array([0.5, 1.0 / math.e, 0.0, 1.0])[:, None]
    np.testing.assert_allclose(S, expect, rtol=1e-15, atol=0)
    np.testing.assert_allclose(o[0], expect[1], rtol=1e-15, atol=0)


def test_softplus_pure_decay_closed_form():
    """beta = 0: S_t = Diag(exp(-sum_{tau<=t} Softplus(logit_tau))) S_0, with
    Softplus from numpy's logaddexp(0, x)."""
    rng = np.random.default_rng(21)
    n, d_k, d_v = 40, 5, 7
    q, k, v, g, _ = _rand_inputs(rng, n, d_k, d_v)
    s0 = rng.normal(size=(d_k, d_v))
    o, S = oracle.recurrence(q, k, v, g, np.zeros(n, np.float32), s0, decay_map=oracle.DECAY_SOFTPLUS)
    cum = np.cumsum(-np.logaddexp(0.0, g), axis=0)
    for t in range(n):
        St = np.exp(cum[t])[:, None] * s0
        np.testing.assert_allclose(o[t], St.T @ q[t], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(S, np.exp(cum[-1])[:, None] * s0, rtol=1e-12, atol=1e-14)


def _brute_states_alpha(q, k, v, alpha, beta, s0):
    """S_t (t = 1..n) from explicit M_t = (I - beta_t k_t k_t^T) Diag(alpha_t)."""
    d_k = k.shape[1]
    St, out = np.array(s0, dtype=np.float64), []
    for t in range(len(q)):
        M = (np.eye(d_k) - float(beta[t]) * np.outer(k[t], k[t])) @ np.diag(alpha[t])
        St = M @ St + float(beta[t]) * np.outer(k[t], v[t])
        out.append(St.copy())
    return out


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_softplus_brute_force_transition_product(seed):
    """Tiny inputs, d_k != d_v: the oracle under the -Softplus map against
    explicit transition products with alpha = 1 / (1 + e^x) (= e^{-Softplus(x)},
    written without a logarithm), every o_t and the final state."""
    rng = np.random.default_rng(400 + seed)
    n, d_k, d_v = 8, 3, 4
    q, k, v, g, beta = _rand_inputs(rng, n, d_k, d_v, unit=False)
    s0 = rng.normal(size=(d_k, d_v))
    o, S = oracle.recurrence(q, k, v, g, beta, s0, decay_map=oracle.DECAY_SOFTPLUS)
    ref = _brute_states_alpha(q, k, v, 1.0 / (1.0 + np.exp(g)), beta, s0)
    for t in range(n):
        np.testing.assert_allclose(o[t], ref[t].T @ q[t], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(S, ref[-1], rtol=1e-12, atol=1e-13)


def test_softplus_passes_the_tile_bound():
    """All logits +40: each step decays by about e^{-40}, so 16 steps reach a
    cumulative log-decay of -640, far past the -80 that the lower bound
    guarantees for a 16-token tile (and past fp32's e^{-103}).  The fp64 oracle
    stays finite and matches the closed form."""
    n, d = 16, 4
    s0 = np.full((d, d), 1.0e300)
    g = np.full((n, d), 40.0)
    o, S = oracle.recurrence(np.ones((n, d)), np.zeros((n, d)), np.zeros((n, d)), g, np.zeros(n, np.float32), s0,
                             decay_map=oracle.DECAY_SOFTPLUS)
    logdecay = -n * (40.0 + math.log1p(math.exp(-40.0)))
    assert logdecay <= -640.0
    assert np.isfinite(S).all() and np.isfinite(o).all()
    np.testing.assert_allclose(S, math.exp(logdecay) * 1.0e300, rtol=1e-12)


def test_decay_map_is_checked():
    with pytest.raises(ValueError):
        oracle.recurrence(np.ones((1, 2)), np.ones((1, 2)), np.ones((1, 2)), np.zeros((1, 2)),
                          np.zeros(1, np.float32), decay_map=2)


SOFTPLUS_MUTANTS = {
    "positive part dropped": ("(logit > 0.0 ? logit : 0.0) + log1p", "0.0 + log1p"),
    "tail sign": ("log1p(exp(-fabs(logit)))", "log1p(exp(fabs(logit)))"),
    "tail without abs": ("log1p(exp(-fabs(logit)))", "log1p(exp(-logit))"),
    "decay inverted": ("return exp(-softplus);", "return exp(softplus);"),
}


@pytest.mark.parametrize("mutant", sorted(SOFTPLUS_MUTANTS))
def test_softplus_planted_mistakes_fail_a_pin(mutant, tmp_path):
    """A plausible mistake planted in the -Softplus branch of a compiled copy of
    the oracle is rejected by the transition-product pin above."""
    import ctypes
    import subprocess

    src = open(oracle._SRC).read()
    old, new = SOFTPLUS_MUTANTS[mutant]
    assert src.count(old) == 1, mutant
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c99", "-fopenmp", "-fPIC", "-shared", str(mpath), "-o", str(so), "-lm"],
                   check=True)
    lib = ctypes.CDLL(str(so))
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.kda_oracle_chains_map.argtypes = [vp, vp, vp, vp, i32, vp, i64, i32, i32, i32, vp, vp, vp, vp, vp, vp,
                                          i64, vp, vp, i32]
    lib.kda_oracle_chains_map.restype = ctypes.c_int
    rng = np.random.default_rng(410)
    n, d_k, d_v = 8, 3, 4
    q, k, v, g, beta = _rand_inputs(rng, n, d_k, d_v, unit=False)
    s0 = rng.normal(size=(d_k, d_v))
    o, S = np.zeros((n, d_v)), np.zeros((d_k, d_v))
    z, nn = np.zeros(1, np.int64), np.array([n], np.int64)
    arrs = [np.ascontiguousarray(x, dtype=np.float64) for x in (q, k, v, g)]
    assert lib.kda_oracle_chains_map(*(a.ctypes.data for a in arrs), oracle.F64, beta.ctypes.data, 1, d_k, d_v, 1,
                                     z.ctypes.data, nn.ctypes.data, s0.ctypes.data, o.ctypes.data, z.ctypes.data,
                                     S.ctypes.data, 0, None, None, oracle.DECAY_SOFTPLUS) > 0
    ref = _brute_states_alpha(q, k, v, 1.0 / (1.0 + np.exp(g)), beta, s0)
    o_ref = np.stack([ref[t].T @ q[t] for t in range(n)])
    err = max(np.abs(o - o_ref).max(), np.abs(S - ref[-1]).max())
    assert err > 1e-6, f"mutant '{mutant}' was not caught (err {err:g})"
