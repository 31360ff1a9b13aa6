"""GPU parity of the integer-operand variant (W4A16_GEMM_DEQUANT_INT): the MMA takes the
exact integers q - z and each 128-K block's fp32 partial is multiplied by its group scale.
The weights are not rounded to the activation dtype, so the reference is the oracle's
product with exact weights (q - z) * s, under the same acceptance bound as the default
path: |Y - Yd| <= 1e-3 * sum_k |A W| + 1 ulp."""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
import weight_only_int4_tma_gb300 as w4
from gpu_util import repack_case, run_gemm, to_dev

pytestmark = pytest.mark.gpu

FP16, BF16 = 0, 1
INT = w4.W4A16_GEMM_DEQUANT_INT


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_only_int4_tma_gb300 import build
    build.build()
    torch.cuda.init()


def _check_exact(c, Y):
    yd, bb, _ = oracle.gemm_exact_w(c.A, c.qweight, c.scales, c.qzeros, c.M, c.N, c.K,
                                    c.group, c.dtype, cscale=c.cscale)
    bad, first, worst = oracle.check(Y, yd, bb, c.dtype)
    assert bad == 0, f"{bad} elements outside the bound (first {first}, worst {worst:.3g})"
    return worst


CASES = [
    # M, N, K, dtype, asym
    (1, 512, 1024, FP16, True),
    (4, 384, 2048, BF16, True),
    (8, 640, 1536, FP16, False),
    (16, 256, 4096, BF16, False),
    (13, 520, 896, FP16, True),   # ragged N, K not a multiple of 256
]


@pytest.mark.parametrize("M,N,K,dtype,asym", CASES)
def test_intop_matches_exact_weight_oracle(M, N, K, dtype, asym):
    c = si.make_case(M, N, K, 128, dtype, seed=M + N + dtype, asym=asym, s_lo=-0.03,
                     s_hi=0.05)
    Y = run_gemm(c, repack_case(c), kernel=w4.W4A16_KERNEL_TC, flags=INT)
    _check_exact(c, Y)


@pytest.mark.parametrize("split", [1, 2, 3, 8])
def test_intop_split_k(split):
    c = si.make_case(6, 384, 2048, 128, FP16, seed=40 + split)
    Y = run_gemm(c, repack_case(c), kernel=w4.W4A16_KERNEL_TC, split_k=split, flags=INT)
    _check_exact(c, Y)


def test_intop_fp16_is_also_within_the_default_bound():
    """fp16 rounding of a weight moves it by at most 2^-11 relative, below the bound's
    1e-3, so the variant also passes against the default (rounded-weight) reference."""
    c = si.make_case(8, 512, 2048, 128, FP16, seed=77)
    Y = run_gemm(c, repack_case(c), kernel=w4.W4A16_KERNEL_TC, flags=INT)
    wd = oracle.dequant(c.qweight, c.scales, c.qzeros, c.N, c.K, c.group, c.dtype)
    yd, bb, _ = oracle.gemm(c.A, wd, c.M, c.N, c.K, c.dtype)
    bad, _, _ = oracle.check(Y, yd, bb, c.dtype)
    assert bad == 0


def test_intop_channel_scale_and_epilogue():
    c = si.make_case(5, 256, 1024, 128, BF16, seed=3, channel_scale=(0.25, 4.0))
    packed = repack_case(c)
    Y = run_gemm(c, packed, kernel=w4.W4A16_KERNEL_TC, flags=INT)
    _check_exact(c, Y)
    rng = np.random.default_rng(2)
    bias = oracle.encode(rng.normal(size=c.N), c.dtype)
    res = oracle.encode(rng.normal(size=(c.M, c.N)), c.dtype)
    yd, bb, _ = oracle.gemm_exact_w(c.A, c.qweight, c.scales, c.qzeros, c.M, c.N, c.K,
                                    c.group, c.dtype, cscale=c.cscale)
    out, bo, _ = oracle.epilogue(yd, bb, bias, res, oracle.ACT_SILU, c.M, c.N, c.dtype)
    Yt = torch.empty((c.M, c.N), dtype=torch.int16, device="cuda")
    w4.w4a16_gemm_epilogue(to_dev(c.A), packed, c.M, c.N, c.K, c.group, c.dtype,
                           to_dev(bias), to_dev(res), w4.W4A16_ACT_SILU, Yt,
                           kernel=w4.W4A16_KERNEL_TC, flags=INT)
    assert w4.w4a16_get_device_status() == 0
    bad, _, _ = oracle.check(Yt.cpu().numpy().view(np.uint16), out, bo, c.dtype)
    assert bad == 0


def test_intop_plan_and_unsupported():
    p = w4.w4a16_gemm_plan(1, 4096, 4096, 128, FP16, flags=INT)
    assert p["kernel"] == w4.W4A16_KERNEL_TC and p["tile_m"] == 16 and p["flags"] & INT
    for args, kw in (((1, 4096, 4096, 64, FP16), {}),                          # group 64
                     ((24, 4096, 4096, 128, FP16), {}),                        # 32-row tile
                     ((1, 4096, 4096, 128, FP16), dict(kernel=w4.W4A16_KERNEL_SIMT))):
        with pytest.raises(w4.W4A16Error) as e:
            w4.w4a16_gemm_plan(*args, flags=INT, **kw)
        assert e.value.status == w4.W4A16_ERR_UNSUPPORTED
    with pytest.raises(w4.W4A16Error) as e:
        w4.w4a16_gemm_plan(1, 4096, 4096, 128, FP16, flags=INT | w4.W4A16_GEMM_DEQUANT_LUT)
    assert e.value.status == w4.W4A16_ERR_INVALID_ARG
