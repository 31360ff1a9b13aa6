"""Pins of the W4A8 (LiquidQuant) oracle against facts that do not come from it: the plain
integer value the page's congruence stands for, brute-force searches over every code,
exact integer dot products in pure Python, and closed forms.

Source: "W4A8量化计算优化：提升LLM推理效率的关键技术", §2.1 (Q_i8 = (Q_u4 * s_u8 + a) XOR 0x80
mod 256, a = 128 + min(Q_i8), s_u8 <= 16)."""
import itertools

import numpy as np
import pytest

from oracle import w4a8


def test_congruence_equals_the_plain_affine_value_everywhere():
    """For every code q, step s <= 16 and minimum mn whose values stay in int8, the XOR
    form gives q * s + mn: the byte (q * s + 128 + mn) never wraps, and flipping its top
    bit is subtracting 128."""
    n = 0
    for s in range(1, 17):
        for mn in range(-128, 128):
            q = np.arange(16)
            ok = q * s + mn <= 127
            if not ok.any():
                continue
            got = w4a8.congruence_dequant(q[ok], s, 128 + mn)
            assert np.array_equal(got, q[ok] * s + mn), (s, mn)
            n += int(ok.sum())
    assert n > 30000


def test_congruence_products_fit_a_byte_when_the_step_is_at_most_16():
    """The page's reason for s_u8 <= 16: 15 * 16 + a stays below 256 for every a the
    quantiser can produce with that step (a <= 255 - 15 s), so the 8-bit lanes of one
    32-bit multiply-add never carry into each other."""
    for s in range(1, 17):
        for mn in range(-128, 128 - 15 * s):
            a = 128 + mn
            assert 15 * s + a <= 255
    # and the packed form: four codes in the bytes of one word, one multiply-add
    rng = np.random.default_rng(1)
    for _ in range(2000):
        s = int(rng.integers(1, 17))
        mn = int(rng.integers(-128, 128 - 15 * s))
        q = rng.integers(0, 16, size=4)
        word = int(q[0] | (q[1] << 8) | (q[2] << 16) | (q[3] << 24))
        packed = (word * s + (128 + mn) * 0x01010101) & 0xFFFFFFFF
        packed ^= 0x80808080
        lanes = [(packed >> (8 * i)) & 0xFF for i in range(4)]
        lanes = [v - 256 if v >= 128 else v for v in lanes]
        assert lanes == [int(x) * s + mn for x in q]


def test_group_quantiser_picks_the_nearest_representable_code():
    """Brute force: for random int8 groups the chosen code is, element by element, the
    code in 0..qmax whose value min + code * s is nearest (ties: the larger), where qmax
    keeps values in int8; and the step is the smallest that covers the range, capped at
    16."""
    rng = np.random.default_rng(2)
    for trial in range(60):
        lo = int(rng.integers(-127, 100))
        hi = int(rng.integers(lo, 128))
        Q = rng.integers(lo, hi + 1, size=(2, 256))
        q, s, a = w4a8.quantize_groups_u4(Q, group=128)
        for n, g in itertools.product(range(2), range(2)):
            grp = Q[n, g * 128:(g + 1) * 128]
            mn, mx = int(grp.min()), int(grp.max())
            step = next((t for t in range(1, 17) if 15 * t >= mx - mn), 16)
            assert s[n, g] == step and a[n, g] == 128 + mn
            for j, v in enumerate(grp):
                cands = [c for c in range(16) if mn + c * step <= 127]
                best = min(cands, key=lambda c: (abs(mn + c * step - int(v)), -c))
                assert q[n, g * 128 + j] == best, (v, mn, step)


def test_group_quantiser_is_exact_where_the_step_is_one():
    """A group spanning at most 15 values has step 1 and reconstructs exactly."""
    rng = np.random.default_rng(3)
    base = rng.integers(-128, 113, size=(3, 1))
    Q = base + rng.integers(0, 16, size=(3, 128))
    q, s, a = w4a8.quantize_groups_u4(Q)
    assert np.all(s == 1)
    assert np.array_equal(w4a8.dequant_i8(q, s, a), Q)


def test_dequant_reconstruction_error_is_at_most_half_a_step():
    """Away from the int8 ceiling every weight comes back within s / 2 of its int8 value."""
    rng = np.random.default_rng(4)
    Q = rng.integers(-127, 100, size=(8, 512))
    q, s, a = w4a8.quantize_groups_u4(Q)
    back = w4a8.dequant_i8(q, s, a)
    step = np.repeat(s, 128, axis=1)
    assert np.all(np.abs(back - Q) * 2 <= step)
    assert back.min() >= -128 and back.max() <= 127


def test_first_level_int8_reaches_127_at_the_channel_maximum():
    W = np.array([[0.5, -2.0, 1.0, 0.0], [3.0, 3.0, -1.5, 0.25], [0.0, 0.0, 0.0, 0.0]])
    Q, s_w = w4a8.quantize_weights_int8(W)
    assert Q[0, 1] == -127 and Q[1, 0] == 127 and Q[1, 1] == 127
    assert np.all(Q[2] == 0) and s_w[2] == 1.0
    assert np.all(np.abs(Q) <= 127)
    assert np.allclose(Q * s_w[:, None], W, atol=float(s_w.max()) / 2 + 1e-7)


def test_activation_quantiser_closed_forms():
    """Per row: the element of largest magnitude maps to +-127, an all-zero row to zeros,
    every element to the nearest multiple of the row step (fp32 rounding aside)."""
    A = np.array([[1.0, -0.5, 0.25, 0.0], [0.0, 0.0, 0.0, 0.0], [-3.0, 1.5, 2.0, 3.0]],
                 dtype=np.float32)
    q, s = w4a8.quantize_activations(A)
    assert q[0, 0] == 127 and q[2, 0] == -127 and q[2, 3] == 127
    assert np.all(q[1] == 0) and s[1] == 1.0
    assert s[0] == np.float32(1.0) / np.float32(127.0)
    rng = np.random.default_rng(5)
    A = rng.standard_normal((4, 300)).astype(np.float16).astype(np.float32)
    q, s = w4a8.quantize_activations(A)
    assert np.all(np.abs(q * s[:, None].astype(np.float64) - A) <= s[:, None] * 0.5001)


def test_integer_gemm_against_python_integers():
    """The accumulation is exact: pure-Python integer dot products on small shapes."""
    rng = np.random.default_rng(6)
    A = rng.integers(-127, 128, size=(3, 256))
    Q = rng.integers(-128, 128, size=(5, 256))
    acc = w4a8.gemm_acc(A, Q)
    for m in range(3):
        for n in range(5):
            assert acc[m, n] == sum(int(x) * int(y) for x, y in zip(A[m], Q[n]))


def test_gemm_scaling_is_two_fp32_multiplies_in_order():
    """fp32(acc) * s_a then * s_w, each rounded to fp32: the largest int32-range sums
    and scales that do not commute bit for bit still follow that order."""
    acc = np.array([[16777217, -3]], dtype=np.int64)  # 2^24 + 1 rounds to 2^24 in fp32
    s_a = np.array([np.float32(0.1)], dtype=np.float32)
    s_w = np.array([np.float32(3.0), np.float32(1.0 / 3.0)], dtype=np.float32)
    y = w4a8.gemm_f32(acc, s_a, s_w)
    e00 = np.float32(np.float32(np.float32(16777216.0) * np.float32(0.1)) * np.float32(3.0))
    e01 = np.float32(np.float32(np.float32(-3.0) * np.float32(0.1)) * np.float32(1.0 / 3.0))
    assert y[0, 0] == e00 and y[0, 1] == e01


@pytest.mark.parametrize("planted", ["no_xor", "signed_a", "wrong_group"])
def test_planted_mistakes_in_the_dequant_are_caught(planted):
    """A dropped XOR, a minimum taken without the 128 offset, or groups broadcast with
    the wrong size all break the plain-value pin above."""
    rng = np.random.default_rng(7)
    Q = rng.integers(-120, 120, size=(2, 256))
    q, s, a = w4a8.quantize_groups_u4(Q)
    ref = np.repeat(s, 128, axis=1) * q + np.repeat(a - 128, 128, axis=1)
    if planted == "no_xor":
        u = (q * np.repeat(s, 128, axis=1) + np.repeat(a, 128, axis=1)) & 0xFF
        bad = np.where(u >= 128, u - 256, u)
    elif planted == "signed_a":
        bad = w4a8.dequant_i8(q, s, a - 128)
    else:
        bad = w4a8.congruence_dequant(q, np.tile(np.repeat(s, 64, axis=1), (1, 2)),
                                      np.tile(np.repeat(a, 64, axis=1), (1, 2)))
    assert np.array_equal(w4a8.dequant_i8(q, s, a), ref)
    assert not np.array_equal(bad, ref)


def test_whole_gemm_from_canonical_inputs_matches_brute_force():
    """gemm_codes on generator inputs against a pure-Python loop that reads each nibble
    by shifting and masking, applies q * s + (a - 128) and sums integers."""
    import synth_inputs as si
    c = si.make_w4a8_case(2, 16, 256, seed=11)
    A32 = np.asarray(c.A.view(np.float16), dtype=np.float32)
    A_i8, s_a = w4a8.quantize_activations(A32)
    y = w4a8.gemm_codes(A_i8, s_a, c.qweight, c.s_u8, c.a, c.s_w, c.N, c.K)
    for m in range(2):
        for n in range(16):
            acc = 0
            for k in range(c.K):
                q = (int(c.qweight[n, k // 8]) >> (4 * (k % 8))) & 0xF
                g = k // 128
                w = q * int(c.s_u8[n, g]) + int(c.a[n, g]) - 128
                acc += int(A_i8[m, k]) * w
            e = np.float32(np.float32(np.float32(acc) * s_a[m]) * c.s_w[n])
            assert y[m, n] == e
