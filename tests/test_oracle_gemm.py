"""Pins for the oracle's GEMM and acceptance check.

* tiny cases against exact rational arithmetic (fractions.Fraction), written here with
  plain Python loops from the definition Y = c * sum_k A W;
* one-hot rows of A return the dequantised weight column exactly;
* q == z everywhere gives Y == 0;
* a group scale constant along K equals the same factor applied per channel in the
  epilogue, within the acceptance bound (the two round differently, so not bitwise);
* the sampled path agrees bit for bit with the full path;
* the acceptance check rejects a planted error.
"""
from fractions import Fraction

import numpy as np
import pytest

import synth_inputs as si

FP16, BF16 = 0, 1


def _exact_dot(a_vals, w_vals):
    return sum((Fraction(float(a)) * Fraction(float(w)) for a, w in zip(a_vals, w_vals)),
               Fraction(0))


@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("shape", [(1, 8, 32, 32), (3, 8, 64, 32), (4, 16, 128, 64)])
def test_tiny_against_rationals(orc, dtype, shape):
    M, N, K, g = shape
    c = si.make_case(M, N, K, g, dtype, seed=17 + M, channel_scale=(0.5, 2.0))
    wd = orc.dequant(c.qweight, c.scales, c.qzeros, N, K, g, dtype)
    yd, bb, yr = orc.gemm(c.A, wd, M, N, K, dtype, cscale=c.cscale)
    A = orc.decode(c.A, dtype)
    W = orc.decode(wd, dtype)
    C = orc.decode(c.cscale, dtype)
    for m in range(M):
        for n in range(N):
            ex = Fraction(float(C[n])) * _exact_dot(A[m], W[n])
            mag = abs(Fraction(float(C[n]))) * sum(
                (abs(Fraction(float(a)) * Fraction(float(w))) for a, w in zip(A[m], W[n])),
                Fraction(0))
            assert abs(Fraction(yd[m, n]) - ex) <= Fraction(2.0 ** -40) * (mag + 1)
            assert abs(Fraction(bb[m, n]) - mag) <= Fraction(2.0 ** -40) * (mag + 1)
            assert yr[m, n] == orc.encode(np.array([float(ex)]), dtype)[0]


@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_one_hot_rows_return_weight_columns(orc, dtype):
    N, K, g = 64, 256, 64
    c = si.make_case(1, N, K, g, dtype, seed=3)
    wd = orc.dequant(c.qweight, c.scales, c.qzeros, N, K, g, dtype)
    ks = [0, 1, 63, 64, 200, 255]
    A = np.zeros((len(ks), K), dtype=np.uint16)
    one = 0x3C00 if dtype == FP16 else 0x3F80
    for i, k in enumerate(ks):
        A[i, k] = one
    yd, _, yr = orc.gemm(A, wd, len(ks), N, K, dtype)
    for i, k in enumerate(ks):
        assert np.array_equal(yr[i], wd[:, k])
        assert np.array_equal(yd[i], orc.decode(wd[:, k], dtype))


def test_q_equals_z_gives_zero_output(orc):
    M, N, K, g = 4, 32, 256, 128
    c = si.make_case(M, N, K, g, FP16, seed=9)
    # every nibble 5, every zero 5
    qw = np.full((N, K // 8), 0x55555555, dtype=np.uint32)
    qz = np.full((K // g, N // 8), 0x55555555, dtype=np.uint32)
    wd = orc.dequant(qw, c.scales, qz, N, K, g, FP16)
    yd, bb, yr = orc.gemm(c.A, wd, M, N, K, FP16)
    assert (yd == 0).all() and (bb == 0).all()
    assert (orc.decode(yr, FP16) == 0).all()


@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_constant_group_scale_equals_channel_scale(orc, dtype):
    M, N, K, g = 4, 64, 512, 128
    c = si.make_case(M, N, K, g, dtype, seed=21)
    G = K // g
    cvals = np.random.default_rng(2).uniform(0.005, 0.02, size=N)
    cbits = si.to_dtype_bits(cvals, dtype)
    # (1) the factor as a group scale, identical for every group
    s_const = np.tile(cbits[None, :], (G, 1))
    wd1 = orc.dequant(c.qweight, s_const, c.qzeros, N, K, g, dtype)
    y1, b1, _ = orc.gemm(c.A, wd1, M, N, K, dtype)
    # (2) unit group scale, the factor applied per channel after the k-sum
    one = 0x3C00 if dtype == FP16 else 0x3F80
    s_one = np.full((G, N), one, dtype=np.uint16)
    wd2 = orc.dequant(c.qweight, s_one, c.qzeros, N, K, g, dtype)
    y2, b2, yr2 = orc.gemm(c.A, wd2, M, N, K, dtype, cscale=cbits)
    bad, first, worst = orc.check(orc.encode(y1, dtype), y2, b2, dtype)
    assert bad == 0, (first, worst)
    assert not np.array_equal(y1, y2)  # they round differently: equal only within bound


def test_sampled_matches_full(orc):
    M, N, K, g = 5, 64, 256, 32
    for asym in (True, False):
        c = si.make_case(M, N, K, g, BF16, seed=4, asym=asym, channel_scale=(0.9, 1.1))
        wd = orc.dequant(c.qweight, c.scales, c.qzeros, N, K, g, BF16)
        yd, bb, yr = orc.gemm(c.A, wd, M, N, K, BF16, cscale=c.cscale)
        rng = np.random.default_rng(0)
        im = rng.integers(0, M, 200)
        inn = rng.integers(0, N, 200)
        sd, sb, sr = orc.gemm_sampled(c.A, c.qweight, c.scales, c.qzeros, M, N, K, g, BF16,
                                      im, inn, cscale=c.cscale)
        assert np.array_equal(sd, yd[im, inn])
        assert np.array_equal(sb, bb[im, inn])
        assert np.array_equal(sr, yr[im, inn])


def test_check_accepts_reference_and_rejects_planted_error(orc):
    M, N, K, g = 2, 32, 256, 128
    c = si.make_case(M, N, K, g, FP16, seed=8)
    wd = orc.dequant(c.qweight, c.scales, c.qzeros, N, K, g, FP16)
    yd, bb, yr = orc.gemm(c.A, wd, M, N, K, FP16)
    assert orc.check(yr, yd, bb, FP16)[0] == 0
    y = orc.decode(yr, FP16).copy()
    y[1, 7] += 2e-3 * bb[1, 7] + 1.0
    bad, first, worst = orc.check(orc.encode(y, FP16), yd, bb, FP16)
    assert bad == 1 and first == 1 * N + 7 and worst > 1.0


def test_transposed_operand_is_caught(orc):
    """A plausible oracle mistake -- indexing the scale as s[n, k/g] instead of
    s[k/g, n] -- changes the result, so the one-hot pin would catch it."""
    N, K, g = 16, 64, 32
    c = si.make_case(1, N, K, g, FP16, seed=12)
    G = K // g
    wd = orc.dequant(c.qweight, c.scales, c.qzeros, N, K, g, FP16)
    q = orc.unpack_q(c.qweight, N, K).astype(np.float64)
    z = orc.unpack_z(c.qzeros, G, N).astype(np.float64)
    s = orc.decode(c.scales, FP16)  # [G, N]
    n_idx = np.arange(N)[:, None]
    k_idx = np.arange(K)[None, :]
    right = (q - z[k_idx // g, n_idx]) * s[k_idx // g, n_idx]
    assert np.array_equal(orc.decode(wd, FP16),
                          right.astype(np.float16).astype(np.float64))
    flat = s.reshape(-1)
    wrong = (q - z[k_idx // g, n_idx]) * flat[(n_idx * G + k_idx // g) % flat.size]
    assert not np.array_equal(orc.decode(wd, FP16),
                              wrong.astype(np.float16).astype(np.float64))


# ---- the product with unrounded weights (integer-operand variant) -------------------

def _nibble(words, idx):
    """Nibble idx of a flat little-endian array of uint32 words (8 per word)."""
    return (int(words[idx // 8]) >> (4 * (idx % 8))) & 0xF


@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("asym", [True, False])
def test_exact_w_tiny_brute_force(orc, dtype, asym):
    """Plain loops over the canonical inputs (nibbles read here, not through the
    oracle's unpack), exact rational arithmetic: sum_k A (q - z) s."""
    M, N, K, g = 2, 8, 64, 32
    c = si.make_case(M, N, K, g, dtype, seed=5 + dtype, asym=asym, channel_scale=(0.5, 2.0))
    yd, bb, yr = orc.gemm_exact_w(c.A, c.qweight, c.scales, c.qzeros, M, N, K, g, dtype,
                                  cscale=c.cscale)
    A = orc.decode(c.A, dtype)
    S = orc.decode(c.scales, dtype)
    C = orc.decode(c.cscale, dtype)
    qw = c.qweight.ravel()
    qz = None if c.qzeros is None else c.qzeros.ravel()
    for m in range(M):
        for n in range(N):
            ex, mag = Fraction(0), Fraction(0)
            for k in range(K):
                q = _nibble(qw, n * K + k)
                gi = k // g
                z = 8 if qz is None else _nibble(qz, gi * N + n)
                t = Fraction(float(A[m, k])) * (q - z) * Fraction(float(S[gi, n]))
                ex += t
                mag += abs(t)
            ex *= Fraction(float(C[n]))
            mag *= abs(Fraction(float(C[n])))
            assert abs(Fraction(yd[m, n]) - ex) <= Fraction(2.0 ** -40) * (mag + 1)
            assert abs(Fraction(bb[m, n]) - mag) <= Fraction(2.0 ** -40) * (mag + 1)
            assert yr[m, n] == orc.encode(np.array([float(ex)]), dtype)[0]


@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_exact_w_equals_rounded_for_power_of_two_scales(orc, dtype):
    """With scales 2^e every (q - z) s is exact in the dtype, so rounding the weight is the
    identity and both products agree bit for bit."""
    M, N, K, g = 3, 32, 256, 64
    c = si.make_case(M, N, K, g, dtype, seed=9)
    rng = np.random.default_rng(1)
    e = rng.integers(-8, -2, size=c.scales.shape)
    c.scales = orc.encode(np.ldexp(1.0, e) * rng.choice([-1.0, 1.0], size=e.shape), dtype)
    wd = orc.dequant(c.qweight, c.scales, c.qzeros, N, K, g, dtype)
    y1, b1, r1 = orc.gemm(c.A, wd, M, N, K, dtype)
    y2, b2, r2 = orc.gemm_exact_w(c.A, c.qweight, c.scales, c.qzeros, M, N, K, g, dtype)
    assert np.array_equal(y1, y2) and np.array_equal(b1, b2) and np.array_equal(r1, r2)


def test_exact_w_is_linear_in_the_scales(orc):
    """Doubling every scale doubles the exact product (a power-of-two factor is exact)."""
    M, N, K, g = 2, 16, 128, 32
    c = si.make_case(M, N, K, g, FP16, seed=4)
    y1, b1, _ = orc.gemm_exact_w(c.A, c.qweight, c.scales, c.qzeros, M, N, K, g, FP16)
    s2 = orc.encode(2.0 * orc.decode(c.scales, FP16), FP16)
    y2, b2, _ = orc.gemm_exact_w(c.A, c.qweight, s2, c.qzeros, M, N, K, g, FP16)
    assert np.array_equal(2.0 * y1, y2) and np.array_equal(2.0 * b1, b2)
