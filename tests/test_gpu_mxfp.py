"""GPU parity of the MX block-scaled decode GEMM (include/mxfp.h: MXFP4 weights x MXFP8
activations, E8M0 block-32 scales, "量化开销对比" §5) against the MX oracle's fp64 product:
every element within |Y - Yd| <= 1e-3 * sum_k |a w| + 1 ulp of the output dtype (the
kernel's element products are exact; its fp32 sums are the only rounding)."""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from oracle import mxfp
import weight_only_int4_tma_gb300 as w4

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_only_int4_tma_gb300 import build
    build.build()
    assert w4.w4a16_get_device_status() == 0


def _run(c):
    nb = w4.mx_packed_bytes(c.N, c.K)
    packed = torch.empty(nb, dtype=torch.uint8, device="cuda")
    w4.mx_repack(torch.from_numpy(c.w_codes).cuda(), torch.from_numpy(c.w_scales).cuda(), c.N,
                 c.K, packed)
    Y = torch.empty((c.M, c.N), dtype=torch.int16, device="cuda")
    w4.mx_gemm(torch.from_numpy(c.a_codes).cuda(), torch.from_numpy(c.a_scales).cuda(), packed,
               c.M, c.N, c.K, c.dtype, Y)
    st = w4.w4a16_get_device_status()
    assert st == 0, w4.status_string(st)
    return packed, Y.cpu().numpy().view(np.uint16)


def _check(c, Y, n0=0, n1=None):
    n1 = c.N if n1 is None else n1
    wc = mxfp.unpack_e2m1_bytes(c.w_codes[n0:n1], n1 - n0, c.K)
    yd, b = mxfp.gemm_mx(c.a_codes, c.a_scales, wc, c.w_scales[n0:n1])
    bad, first, worst = oracle.check(np.ascontiguousarray(Y[:, n0:n1]), yd, b, c.dtype)
    assert bad == 0, f"{bad} elements outside the bound (first flat index {first}, worst {worst})"


CASES = [(1, 32, 128, si.FP16), (3, 40, 256, si.BF16), (8, 200, 512, si.FP16),
         (9, 96, 1024, si.BF16), (16, 4096, 4096, si.FP16), (16, 1000, 2048, si.BF16),
         (5, 8200, 384, si.FP16), (2, 64, 4096, si.BF16)]


@pytest.mark.parametrize("M,N,K,dt", CASES,
                         ids=[f"m{m}_n{n}_k{k}_{si.DTYPE_NAMES[d]}" for m, n, k, d in CASES])
def test_mx_gemm_against_oracle(M, N, K, dt):
    c = si.make_mx_case(M, N, K, dtype=dt, seed=M + N + K)
    _, Y = _run(c)
    _check(c, Y)


def test_mx_gemm_wide_scale_range():
    """Block scales far from 1 on both sides (their product stays inside fp32)."""
    c = si.make_mx_case(4, 128, 1024, dtype=si.BF16, seed=9, w_exp=(100, 112), a_exp=(138, 150))
    _, Y = _run(c)
    _check(c, Y)


@pytest.mark.parametrize("p", si.MX_WORKLOADS["mx_ffn70b_decode"],
                         ids=[si.mx_shape_tag(p) for p in si.MX_WORKLOADS["mx_ffn70b_decode"]])
def test_mx_gemm_ffn70b_stripes(p):
    c = si.make_mx_case(**p)
    _, Y = _run(c)
    N = c.N
    for n0, n1 in [(0, 64), (N // 2 - 24, N // 2 + 40), (N - 64, N)]:
        _check(c, Y, n0, n1)


def test_mx_header_check_and_limits():
    c = si.make_mx_case(4, 64, 512, seed=3)
    packed, _ = _run(c)
    Y = torch.full((c.M, c.N), 0x1234, dtype=torch.int16, device="cuda")
    w4.mx_gemm(torch.from_numpy(c.a_codes).cuda(), torch.from_numpy(c.a_scales).cuda(), packed,
               c.M, c.N, 384, c.dtype, Y)
    assert w4.w4a16_get_device_status() == w4.W4A16_ERR_FORMAT
    assert bool((Y == 0x1234).all())
    with pytest.raises(w4.W4A16Error):
        w4.mx_gemm(torch.from_numpy(c.a_codes).cuda(), torch.from_numpy(c.a_scales).cuda(),
                   packed, 17, c.N, c.K, c.dtype, Y)
