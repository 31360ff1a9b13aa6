"""Pins for the oracle's IEEE-754 fp16 / bf16 decode and round-to-nearest-even encode.

They check the oracle against facts that do not come from its own code: numpy's
float16 conversions, torch's bfloat16 conversion, the bf16 = upper half of binary32
definition, and exhaustive enumeration of every 16-bit pattern and every midpoint.
"""
import numpy as np
import pytest
import torch

FP16, BF16 = 0, 1
ALL = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)


def _bf16_ref(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_f16_decode_exhaustive(orc):
    d = orc.decode(ALL, FP16)
    ref = ALL.view(np.float16).astype(np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(d[fin], ref[fin])
    assert np.array_equal(np.isnan(d), np.isnan(ref))
    assert np.array_equal(np.isinf(d) & (d > 0), np.isinf(ref) & (ref > 0))
    assert np.array_equal(np.signbit(d[fin]), np.signbit(ref[fin]))


def test_bf16_decode_exhaustive(orc):
    d = orc.decode(ALL, BF16)
    ref = _bf16_ref(ALL)
    fin = np.isfinite(ref)
    assert np.array_equal(d[fin], ref[fin])
    assert np.array_equal(np.isnan(d), np.isnan(ref))
    assert np.array_equal(np.signbit(d[fin]), np.signbit(ref[fin]))


@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_encode_roundtrip_every_finite_pattern(orc, dtype):
    d = orc.decode(ALL, dtype)
    fin = np.isfinite(d)
    e = orc.encode(d[fin], dtype)
    assert np.array_equal(e, ALL[fin])


@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_encode_midpoints_ties_to_even(orc, dtype):
    # Every pair of adjacent positive finite values: the exact midpoint goes to the one
    # with an even last bit; a hair either side goes to the nearer neighbour.
    pos = ALL[ALL < 0x8000]
    vals = orc.decode(pos, dtype)
    fin = np.isfinite(vals)
    lo_bits = pos[fin][:-1]
    hi_bits = pos[fin][1:]
    lo, hi = vals[fin][:-1], vals[fin][1:]
    mid = (lo + hi) / 2.0  # exact in fp64 (both have <= 11 significant bits)
    got = orc.encode(mid, dtype)
    want = np.where(lo_bits % 2 == 0, lo_bits, hi_bits)
    assert np.array_equal(got, want)
    eps = (hi - lo) * 2.0 ** -20
    assert np.array_equal(orc.encode(mid - eps, dtype), lo_bits)
    assert np.array_equal(orc.encode(mid + eps, dtype), hi_bits)
    # negative side is the mirror image
    assert np.array_equal(orc.encode(-mid, dtype), want | 0x8000)


def test_f16_encode_matches_numpy_on_random_doubles(orc):
    rng = np.random.default_rng(123)
    x = np.concatenate([
        rng.standard_normal(200_000),
        rng.standard_normal(50_000) * 1e-5,      # subnormal range
        rng.standard_normal(50_000) * 3e4,       # near overflow
        rng.uniform(-1, 1, 50_000) * 2.0 ** -25,  # below the smallest subnormal
    ])
    got = orc.encode(x, FP16)
    ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_encode_matches_torch_on_random_floats(orc):
    rng = np.random.default_rng(7)
    x32 = np.concatenate([
        rng.standard_normal(200_000).astype(np.float32),
        (rng.standard_normal(50_000) * 1e-39).astype(np.float32),
        (rng.standard_normal(50_000) * 1e38).astype(np.float32),
    ])
    got = orc.encode(x32.astype(np.float64), BF16)
    ref = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


def test_overflow_and_limits(orc):
    assert orc.encode(np.array([65504.0]), FP16)[0] == 0x7BFF
    assert orc.encode(np.array([65519.99]), FP16)[0] == 0x7BFF
    assert orc.encode(np.array([65520.0]), FP16)[0] == 0x7C00  # tie rounds to even = inf
    assert orc.encode(np.array([-1e9]), FP16)[0] == 0xFC00
    assert orc.encode(np.array([2.0 ** -24]), FP16)[0] == 0x0001
    assert orc.encode(np.array([2.0 ** -25]), FP16)[0] == 0x0000  # tie to even (zero)
    assert orc.encode(np.array([-0.0]), FP16)[0] == 0x8000


def test_ulp(orc):
    assert orc.ulp(0x3C00, FP16) == 2.0 ** -10   # 1.0
    assert orc.ulp(0x6400, FP16) == 1.0          # 1024
    assert orc.ulp(0x0001, FP16) == 2.0 ** -24   # subnormal spacing
    assert orc.ulp(0x3F80, BF16) == 2.0 ** -7    # 1.0
    assert orc.ulp(0x4300, BF16) == 1.0          # 128
