"""The seeded input generator: deterministic, counter based (slices equal the
whole), unit-norm q/k rows, bf16 rounding, varlen lengths."""
import numpy as np

import kda_synth as ks


def test_deterministic_and_sliceable():
    a = ks.rows(7, 1, 0, 1, 64, 16)
    b = ks.rows(7, 1, 0, 1, 64, 16)
    np.testing.assert_array_equal(a, b)
    c = ks.rows(7, 1, 10, 3, 5, 16)          # rows 10, 13, ..., 22
    np.testing.assert_array_equal(c, a[10:25:3])
    assert not np.array_equal(ks.rows(8, 1, 0, 1, 4, 16), a[:4])
    assert not np.array_equal(ks.rows(7, 2, 0, 1, 4, 16), a[:4])


def test_normal_moments():
    x = ks.normals(3, 1, 0, 400_000)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    assert abs(np.mean(x ** 3)) < 0.02 and abs(np.mean(x ** 4) - 3.0) < 0.05


def test_unit_rows_and_storage():
    r64 = ks.rows(1, 2, 0, 1, 100, 128, unit_norm=True)
    np.testing.assert_allclose(np.linalg.norm(r64, axis=1), 1.0, rtol=1e-14)
    r32 = ks.rows(1, 2, 0, 1, 100, 128, unit_norm=True, dtype=ks.F32)
    np.testing.assert_array_equal(r32, r64.astype(np.float32))
    rb = ks.rows(1, 2, 0, 1, 100, 128, unit_norm=True, dtype=ks.BF16)
    np.testing.assert_array_equal(rb, ks.f32_to_bf16_bits(r32))
    assert np.abs(ks.bf16_bits_to_f64(rb) - r64).max() <= 2.0 ** -9


def test_bf16_round_to_nearest_even():
    x = np.array([1.0, -2.5, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -8 + 2 ** -20, np.inf, 0.0],
                 dtype=np.float32)
    bits = ks.f32_to_bf16_bits(x)
    # 1 + 2^-8 is a tie -> even (1.0); 1 + 3*2^-8 is a tie -> even (1 + 2^-6... i.e. 1 + 4*2^-8)
    np.testing.assert_array_equal(ks.bf16_bits_to_f64(bits),
                                  [1.0, -2.5, 1.0, 1.0 + 4 * 2 ** -8, 1.0 + 2 ** -7, np.inf, 0.0])


def test_sigmoid_normal_range():
    b = ks.sigmoid_normal(0, 5, 0, 1, 10000)
    assert b.dtype == np.float32 and (b > 0).all() and (b < 1).all()
    assert abs(float(b.mean()) - 0.5) < 0.02


def test_varlen_lengths():
    lens = ks.varlen_lengths(4, 1 << 20)
    assert len(lens) == 12 and int(lens.sum()) == 1 << 20 and (lens > 0).all()
    w = ks.workloads()["varlen_12seq_1m_h32_d128"]
    cu = w.cu_seqlens()
    assert cu[0] == 0 and cu[-1] == 1 << 20 and (np.diff(cu) >= 0).all()


def test_chain_slices_match_whole_tensor():
    w = ks.PrefillWorkload("t", "bf16", 2, 40, 3, 16, 8, seed=5, s0_std=0.5)
    q = w.fill("q", None if False else np.empty((w.tokens * w.H, 16), np.uint16))
    v = w.fill("v", np.empty((w.tokens * w.H, 8), np.uint16))
    beta = w.fill("beta", np.empty((w.tokens * w.H,), np.float32))
    s0 = w.fill("s0", np.empty((w.num_seqs * w.H * 16, 8), np.float32))
    ci = w.chain_inputs(1, 2)
    rows = [(1 * 40 + t) * 3 + 2 for t in range(40)]
    np.testing.assert_array_equal(ci["q"], q[rows])
    np.testing.assert_array_equal(ci["v"], v[rows])
    np.testing.assert_array_equal(ci["beta"], beta[rows])
    np.testing.assert_array_equal(ci["s0"], s0.reshape(2, 3, 16, 8)[1, 2])
