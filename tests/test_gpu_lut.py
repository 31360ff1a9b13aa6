"""GPU parity of the table unpack (W4A16_GEMM_DEQUANT_LUT): nibble -> value through a
16-entry shared-memory table, then the group's zero and scale with one rounding.  The
dequantised weights are the same bits as the default unpack, so the tensor-core results
must be bit-identical to the default path and within the oracle's bound."""
import numpy as np
import pytest
import torch

import synth_inputs as si
import weight_only_int4_tma_gb300 as w4
from gpu_util import assert_parity_full, repack_case, run_gemm, to_dev

pytestmark = pytest.mark.gpu

FP16, BF16 = 0, 1
LUT = w4.W4A16_GEMM_DEQUANT_LUT


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_only_int4_tma_gb300 import build
    build.build()
    torch.cuda.init()


CASES = [
    # M, N, K, group, dtype, asym
    (1, 512, 1024, 128, FP16, True),
    (2, 384, 768, 64, FP16, False),
    (8, 256, 1536, 32, BF16, True),
    (16, 640, 1024, 128, BF16, False),
    (24, 256, 512, 32, FP16, True),     # 32-row tile, ragged M
    (32, 384, 1024, 64, BF16, True),
    (5, 520, 960, 32, FP16, True),      # ragged N and K
]


@pytest.mark.parametrize("M,N,K,group,dtype,asym", CASES)
def test_lut_matches_default_bit_for_bit(M, N, K, group, dtype, asym):
    c = si.make_case(M, N, K, group, dtype, seed=M * 7 + group + dtype, asym=asym,
                     s_lo=-0.03, s_hi=0.05)
    packed = repack_case(c)
    A = to_dev(c.A)
    y_def = run_gemm(c, packed, A, kernel=w4.W4A16_KERNEL_TC)
    y_lut = run_gemm(c, packed, A, kernel=w4.W4A16_KERNEL_TC, flags=LUT)
    assert np.array_equal(y_lut, y_def), f"{np.sum(y_lut != y_def)} elements differ"
    assert_parity_full(c, y_lut)


@pytest.mark.parametrize("split", [1, 3, 8])
def test_lut_split_k(split):
    c = si.make_case(4, 512, 2048, 128, FP16, seed=11 + split)
    packed = repack_case(c)
    A = to_dev(c.A)
    y_def = run_gemm(c, packed, A, kernel=w4.W4A16_KERNEL_TC, split_k=split)
    y_lut = run_gemm(c, packed, A, kernel=w4.W4A16_KERNEL_TC, split_k=split, flags=LUT)
    assert np.array_equal(y_lut, y_def)
    assert_parity_full(c, y_lut)


def test_lut_full_range_scales_fp16():
    # scales from subnormal to large: the default path then mixes its two fp16 unpack
    # forms; the table path has one form and must still give the same bits
    c = si.make_case(3, 256, 512, 32, FP16, seed=9)
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 0x5000, size=c.scales.shape, dtype=np.uint16)
    sign = rng.integers(0, 2, size=c.scales.shape, dtype=np.uint16) << 15
    c.scales = (bits | sign).astype(np.uint16)
    packed = repack_case(c)
    A = to_dev(c.A)
    y_def = run_gemm(c, packed, A, kernel=w4.W4A16_KERNEL_TC)
    y_lut = run_gemm(c, packed, A, kernel=w4.W4A16_KERNEL_TC, flags=LUT)
    assert np.array_equal(y_lut, y_def)


def test_lut_plan_and_unsupported():
    # the heuristic would pick the GEMV for M = 1: the flag keeps the tensor-core kernel
    p = w4.w4a16_gemm_plan(1, 4096, 4096, 128, FP16, flags=LUT)
    assert p["kernel"] == w4.W4A16_KERNEL_TC and p["tile_m"] == 16
    assert p["flags"] & LUT
    for kw in (dict(kernel=w4.W4A16_KERNEL_SIMT), dict(tile_m=64)):
        with pytest.raises(w4.W4A16Error):
            w4.w4a16_gemm_plan(1, 4096, 4096, 128, FP16, flags=LUT, **kw)
    with pytest.raises(w4.W4A16Error):
        w4.w4a16_gemm_plan(64, 4096, 4096, 128, FP16, flags=LUT)  # heuristic: 64-row tile
