"""Pins of the MX block-scaled format oracle (oracle/mxfp.py) against what the formats'
definitions and independent library routines fix (CPU only)."""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import mxfp


def test_e2m1_codes_are_the_format_table():
    # the sixteen E2M1 values: +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}
    table = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert [mxfp.e2m1_value(c) for c in range(8)] == table
    assert [mxfp.e2m1_value(c + 8) for c in range(8)] == [-v for v in table]


@pytest.mark.skipif(not hasattr(torch, "float8_e4m3fn"), reason="no float8_e4m3fn in torch")
def test_e4m3_every_code_against_torch():
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    mine = np.array([mxfp.e4m3_value(c) for c in range(256)])
    assert np.array_equal(np.isnan(lib), np.isnan(mine))
    ok = ~np.isnan(lib)
    assert np.array_equal(lib[ok], mine[ok])
    assert np.nanmax(mine) == 448.0


@pytest.mark.skipif(not hasattr(torch, "float8_e8m0fnu"), reason="no float8_e8m0fnu in torch")
def test_e8m0_every_code_against_torch():
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).double().numpy()
    mine = np.array([mxfp.e8m0_value(c) for c in range(256)])
    assert np.array_equal(np.isnan(lib), np.isnan(mine))
    ok = ~np.isnan(lib)
    assert np.array_equal(lib[ok], mine[ok])


@pytest.mark.parametrize("fmt", [mxfp.E2M1, mxfp.E4M3])
def test_rounding_ties_to_even_and_saturation(fmt):
    vals = sorted({v for v in (mxfp._values(fmt)) if not math.isnan(v) and v >= 0})
    for lo, hi in zip(vals, vals[1:]):
        mid = (lo + hi) / 2
        c = mxfp.round_to_element(mid, fmt)
        v = mxfp._values(fmt)[c]
        assert v in (lo, hi)
        assert c & 1 == 0, (fmt, lo, hi, c)  # the even code wins the tie
        assert mxfp._values(fmt)[mxfp.round_to_element(lo + (hi - lo) / 4, fmt)] == lo
        assert mxfp._values(fmt)[mxfp.round_to_element(hi - (hi - lo) / 4, fmt)] == hi
        assert mxfp._values(fmt)[mxfp.round_to_element(-mid, fmt)] == -v
    top = vals[-1]
    assert mxfp._values(fmt)[mxfp.round_to_element(top * 10, fmt)] == top
    assert mxfp._values(fmt)[mxfp.round_to_element(-top * 10, fmt)] == -top


@pytest.mark.parametrize("fmt", [mxfp.E2M1, mxfp.E4M3])
def test_block_exponent_puts_the_block_max_in_the_top_binade(fmt):
    emax = {mxfp.E2M1: 2, mxfp.E4M3: 8}[fmt]
    rng = np.random.default_rng(0)
    for _ in range(200):
        amax = float(np.ldexp(rng.uniform(1.0, 2.0), int(rng.integers(-60, 60))))
        blk = rng.uniform(-amax, amax, mxfp.BLOCK)
        blk[int(rng.integers(0, mxfp.BLOCK))] = amax
        x = mxfp.block_exponent(blk, fmt)
        assert 2.0 ** (x + emax) <= amax < 2.0 ** (x + emax + 1)
    assert mxfp.block_exponent(np.zeros(mxfp.BLOCK), fmt) == -127
    # exact powers of two sit at the bottom of their binade
    blk = np.zeros(mxfp.BLOCK)
    blk[3] = 2.0 ** 10
    assert mxfp.block_exponent(blk, fmt) == 10 - emax


@pytest.mark.parametrize("fmt", [mxfp.E2M1, mxfp.E4M3])
def test_quantise_round_trip_of_representable_blocks(fmt):
    """Blocks made of format values times a power of two, with the format's largest value
    present, come back with the same scale and the same values."""
    rng = np.random.default_rng(1)
    vals = mxfp._values(fmt)
    good = [c for c in range(len(vals)) if not math.isnan(vals[c])]
    top = [c for c in good if vals[c] == np.nanmax(vals)][0]
    R, K = 3, 4 * mxfp.BLOCK
    codes = rng.choice(good, size=(R, K))
    codes[:, ::mxfp.BLOCK] = top
    x = rng.integers(-20, 20, size=(R, K // mxfp.BLOCK))
    V = vals[codes] * np.ldexp(1.0, np.repeat(x, mxfp.BLOCK, axis=1))
    qc, qe = mxfp.quantize_mx(V, fmt)
    assert np.array_equal(qe - 127, x)
    assert np.array_equal(mxfp.dequant_mx(qc, qe, fmt), V)


def test_planted_scale_error_is_caught():
    """A dequant that forgot the block scale (or used the wrong block) would fail the
    round trip above; here the scale of block 1 applied to block 0 is detected."""
    vals = mxfp._values(mxfp.E2M1)
    V = np.zeros((1, 2 * mxfp.BLOCK))
    V[0, :mxfp.BLOCK] = 6.0
    V[0, mxfp.BLOCK:] = 0.75
    qc, qe = mxfp.quantize_mx(V, mxfp.E2M1)
    assert qe[0, 0] != qe[0, 1]
    swapped = qe[:, ::-1].copy()
    assert not np.array_equal(mxfp.dequant_mx(qc, swapped, mxfp.E2M1), V)
    assert np.array_equal(mxfp.dequant_mx(qc, qe, mxfp.E2M1), V)
    assert vals[qc[0, 0]] * 2.0 ** (qe[0, 0] - 127) == 6.0


def test_gemm_against_fractions():
    rng = np.random.default_rng(2)
    M, N, K = 2, 3, 2 * mxfp.BLOCK
    a = rng.standard_normal((M, K)) * 3
    w = rng.standard_normal((N, K)) * 0.02
    ac, ae = mxfp.quantize_mx(a, mxfp.E4M3)
    wc, we = mxfp.quantize_mx(w, mxfp.E2M1)
    y, b = mxfp.gemm_mx(ac, ae, wc, we)
    av = [[Fraction(mxfp.e4m3_value(int(ac[m, k]))) * Fraction(2) ** int(ae[m, k // 32] - 127)
           for k in range(K)] for m in range(M)]
    wv = [[Fraction(mxfp.e2m1_value(int(wc[n, k]))) * Fraction(2) ** int(we[n, k // 32] - 127)
           for k in range(K)] for n in range(N)]
    for m in range(M):
        for n in range(N):
            exact = sum(av[m][k] * wv[n][k] for k in range(K))
            assert abs(Fraction(y[m, n]) - exact) <= Fraction(b[m, n]) * Fraction(2) ** -50
    # the quantised operands are close to the originals (a sanity bound on the reading)
    assert np.max(np.abs(mxfp.dequant_mx(wc, we, mxfp.E2M1) - w)) <= np.max(np.abs(w)) / 4


@pytest.mark.skipif(not hasattr(torch, "float8_e4m3fn"), reason="no float8_e4m3fn in torch")
def test_e4m3_rounding_against_torch():
    """In-range values (including every midpoint between neighbouring codes) round as the
    library's float -> float8_e4m3fn conversion rounds them."""
    vals = sorted({v for v in mxfp._values(mxfp.E4M3) if not math.isnan(v) and v >= 0})
    mids = [(a + b) / 2 for a, b in zip(vals, vals[1:])]
    rng = np.random.default_rng(4)
    xs = np.concatenate([mids, rng.uniform(-448, 448, 2000), rng.uniform(-0.02, 0.02, 2000)])
    xs = xs.astype(np.float32).astype(np.float64)  # values the library sees exactly
    lib = torch.from_numpy(xs.astype(np.float32)).to(torch.float8_e4m3fn).double().numpy()
    mine = np.array([mxfp._values(mxfp.E4M3)[mxfp.round_to_element(float(x), mxfp.E4M3)]
                     for x in xs])
    assert np.array_equal(np.abs(lib), np.abs(mine))


def test_unpack_e2m1_bytes_nibble_order():
    b = np.array([[0x21, 0xF0]], dtype=np.uint8)  # K 0 = 1, K 1 = 2, K 2 = 0, K 3 = 15
    assert mxfp.unpack_e2m1_bytes(b, 1, 4).tolist() == [[1, 2, 0, 15]]
