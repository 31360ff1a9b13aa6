"""GPU parity of the fused epilogue (bias / ReLU / SiLU / residual) against the oracle,
through w4a16_gemm_epilogue, on both kernels and both split-K paths.

Bound: |Y - out| <= 1e-3 * B' + 1 ulp of the output dtype, with out and
B' = L * sum_k |A W| * |c| + |bias| + |residual| from the oracle's epilogue (L = 1.1 for
SiLU, whose slope lies in [-0.1, 1.1]; 1 otherwise)."""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
import weight_only_int4_tma_gb300 as w4
from gpu_util import repack_case, to_dev, to_host_u16

pytestmark = pytest.mark.gpu

FP16, BF16 = 0, 1
NONE, RELU, SILU = w4.W4A16_ACT_NONE, w4.W4A16_ACT_RELU, w4.W4A16_ACT_SILU


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_only_int4_tma_gb300 import build
    build.build()
    assert w4.w4a16_get_device_status() == 0


def epilogue_inputs(c, seed, with_bias, with_res):
    rng = np.random.default_rng(seed)
    bias = oracle.encode(rng.normal(size=c.N), c.dtype) if with_bias else None
    res = oracle.encode(rng.normal(size=(c.M, c.N)), c.dtype) if with_res else None
    return bias, res


def run_epilogue(c, packed, bias, res, act, in_place=False, **ex):
    A = to_dev(c.A)
    b = to_dev(bias)
    if in_place:
        Y = to_dev(res)
        r = Y
    else:
        Y = torch.empty((c.M, c.N), dtype=torch.int16, device="cuda")
        r = to_dev(res)
    w4.w4a16_gemm_epilogue(A, packed, c.M, c.N, c.K, c.group, c.dtype, b, r, act, Y, **ex)
    st = w4.w4a16_get_device_status()
    assert st == 0, w4.status_string(st)
    return to_host_u16(Y)


def oracle_epilogue(c, bias, res, act):
    wd = oracle.dequant(c.qweight, c.scales, c.qzeros, c.N, c.K, c.group, c.dtype)
    yd, bb, _ = oracle.gemm(c.A, wd, c.M, c.N, c.K, c.dtype, cscale=c.cscale)
    out, bo, _ = oracle.epilogue(yd, bb, bias, res, act, c.M, c.N, c.dtype)
    return out, bo


def assert_epilogue_parity(c, Y, bias, res, act):
    out, bo = oracle_epilogue(c, bias, res, act)
    bad, first, worst = oracle.check(Y, out, bo, c.dtype)
    assert bad == 0, (bad, first, worst)


KERNELS = {
    "tc_split1": dict(kernel=w4.W4A16_KERNEL_TC, tile_m=16, split_k=1),
    "tc_split4": dict(kernel=w4.W4A16_KERNEL_TC, tile_m=16, split_k=4),
    "tc_tile128": dict(kernel=w4.W4A16_KERNEL_TC, tile_m=128),
    # one K slice: the larger tiles' staged, vectorised store path
    "tc_tile128_s1": dict(kernel=w4.W4A16_KERNEL_TC, tile_m=128, split_k=1),
    "tc_tile64_s1": dict(kernel=w4.W4A16_KERNEL_TC, tile_m=64, split_k=1),
    "gemv": dict(kernel=w4.W4A16_KERNEL_SIMT),
}


@pytest.mark.parametrize("kname", list(KERNELS))
@pytest.mark.parametrize("act", [NONE, RELU, SILU])
@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_bias_act_residual(kname, act, dtype):
    M = {"tc_tile128": 130, "tc_tile128_s1": 130, "tc_tile64_s1": 70, "gemv": 3}.get(kname, 11)
    c = si.make_case(M, 384, 1024, 64, dtype, seed=7 + act, channel_scale=(0.5, 2.0))
    packed = repack_case(c)
    bias, res = epilogue_inputs(c, seed=act, with_bias=True, with_res=True)
    Y = run_epilogue(c, packed, bias, res, act, **KERNELS[kname])
    assert_epilogue_parity(c, Y, bias, res, act)


@pytest.mark.parametrize("with_bias,with_res", [(True, False), (False, True), (False, False)])
@pytest.mark.parametrize("kname", ["tc_split4", "gemv"])
def test_optional_parts(kname, with_bias, with_res):
    c = si.make_case(2, 256, 512, 128, FP16, seed=3)
    packed = repack_case(c)
    bias, res = epilogue_inputs(c, seed=5, with_bias=with_bias, with_res=with_res)
    Y = run_epilogue(c, packed, bias, res, SILU, **KERNELS[kname])
    assert_epilogue_parity(c, Y, bias, res, SILU)


@pytest.mark.parametrize("kname", ["tc_split1", "tc_split4", "tc_tile128_s1", "gemv"])
def test_in_place_residual(kname):
    c = si.make_case(4, 256, 768, 128, BF16, seed=11)
    packed = repack_case(c)
    bias, res = epilogue_inputs(c, seed=9, with_bias=True, with_res=True)
    Y = run_epilogue(c, packed, bias, res, RELU, in_place=True, **KERNELS[kname])
    assert_epilogue_parity(c, Y, bias, res, RELU)


def test_identity_epilogue_is_the_plain_gemm():
    c = si.make_case(8, 512, 1024, 128, FP16, seed=2)
    packed = repack_case(c)
    A = to_dev(c.A)
    Y0 = torch.empty((c.M, c.N), dtype=torch.int16, device="cuda")
    Y1 = torch.empty_like(Y0)
    w4.w4a16_gemm(A, packed, c.M, c.N, c.K, c.group, c.dtype, Y0)
    w4.w4a16_gemm_epilogue(A, packed, c.M, c.N, c.K, c.group, c.dtype, None, None, NONE, Y1)
    assert w4.w4a16_get_device_status() == 0
    assert torch.equal(Y0, Y1)


def test_q_equals_z_gives_act_of_bias_plus_residual():
    c = si.make_case(5, 256, 512, 64, FP16, seed=4)
    c.qweight[:] = 0x99999999
    c.qzeros = np.full_like(c.qzeros, 0x99999999)
    packed = repack_case(c)
    bias, res = epilogue_inputs(c, seed=1, with_bias=True, with_res=True)
    for act in (NONE, RELU, SILU):
        Y = run_epilogue(c, packed, bias, res, act)
        assert_epilogue_parity(c, Y, bias, res, act)


def test_bad_activation_rejected():
    c = si.make_case(1, 256, 512, 128, FP16, seed=1)
    packed = repack_case(c)
    with pytest.raises(w4.W4A16Error) as e:
        run_epilogue(c, packed, None, None, 7)
    assert e.value.status == w4.W4A16_ERR_INVALID_ARG


@pytest.mark.parametrize("offset", [0, 1])
def test_staged_store_ragged_and_unaligned(offset):
    """Larger tiles with one K slice store through shared memory, 8 channels per 16-byte
    access; a ragged N and M, and a residual that is only 2-byte aligned (the scalar path
    then; Y itself must be 16-byte aligned), give the same results."""
    c = si.make_case(70, 520, 512, 128, FP16, seed=21 + offset)
    packed = repack_case(c)
    bias, res = epilogue_inputs(c, seed=4, with_bias=True, with_res=True)
    n = c.M * c.N
    rbuf = torch.zeros(n + 8, dtype=torch.int16, device="cuda")
    rbuf[offset:offset + n] = torch.from_numpy(res.view(np.int16).ravel()).cuda()
    Y = torch.empty((c.M, c.N), dtype=torch.int16, device="cuda")
    R = rbuf[offset:offset + n].view(c.M, c.N)
    w4.w4a16_gemm_epilogue(to_dev(c.A), packed, c.M, c.N, c.K, c.group, c.dtype,
                           to_dev(bias), R, SILU, Y, kernel=w4.W4A16_KERNEL_TC, tile_m=64,
                           split_k=1)
    assert w4.w4a16_get_device_status() == 0
    assert_epilogue_parity(c, Y.cpu().numpy().view(np.uint16), bias, res, SILU)
