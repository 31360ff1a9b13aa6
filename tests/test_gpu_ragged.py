"""GPU parity for shapes that are not multiples of 128 (padded to whole blocks by the
repack): bit-exact debug dequant, GEMM on both kernels (3-D and 2-D A boxes on the
tensor-core kernel, K tails inside a block, N tails inside a tile, split-K), and the fused
epilogue on a ragged N."""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
import weight_only_int4_tma_gb300 as w4
from gpu_util import assert_parity_full, repack_case, run_gemm, to_dev, to_host_u16

pytestmark = pytest.mark.gpu

FP16, BF16 = 0, 1


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_only_int4_tma_gb300 import build
    build.build()
    assert w4.w4a16_get_device_status() == 0


@pytest.mark.parametrize("N,K,g,dt", [(520, 4160, 64, FP16), (264, 96, 32, BF16),
                                      (8, 128, 128, FP16), (136, 4128, 32, FP16)])
def test_dequant_debug_ragged_bit_exact(N, K, g, dt):
    c = si.make_case(1, N, K, g, dt, seed=N + K)
    packed = repack_case(c)
    assert packed.numel() == w4.w4a16_packed_bytes(N, K, g, True)
    W = torch.full((N, K), 0x7777, dtype=torch.int16, device="cuda")
    w4.w4a16_dequant_debug(packed, N, K, g, dt, W)
    assert w4.w4a16_get_device_status() == 0
    wd = oracle.dequant(c.qweight, c.scales, c.qzeros, N, K, g, dt)
    assert np.array_equal(to_host_u16(W), wd)


RAGGED = [
    # (M, N, K, group, dtype, asym, extra launch options)
    (1, 520, 512, 128, FP16, True, {}),                      # GEMV, N tail
    (1, 136, 96, 32, BF16, True, {}),                        # GEMV, one partial block
    (1, 264, 4160, 64, FP16, True, dict(kernel=2, tile_m=32)),
    (5, 264, 4160, 64, FP16, True, {}),                      # tcgen05, K % 64 == 0: 3-D A box
    (3, 776, 4128, 32, FP16, True, {}),                      # K % 64 == 32: 2-D A boxes
    (7, 392, 1120, 32, BF16, False, dict(kernel=1, tile_m=16, split_k=3)),
    (40, 392, 1120, 32, FP16, True, {}),                     # 64-row tile, 2-D A boxes
    (130, 200, 640, 128, BF16, True, {}),                    # 128-row tiles, N tail
    (300, 456, 352, 32, FP16, False, dict(kernel=1, tile_m=256)),
    # split-K owners of larger tiles sum four channels per thread; slices of 44 / 28 /
    # 20 channels (split 3 / 5 / 7) with the last tile ending inside a slice or before it
    (64, 392, 2048, 64, FP16, True, dict(kernel=1, tile_m=64, split_k=3)),
    (100, 264, 2048, 128, BF16, True, dict(kernel=1, tile_m=128, split_k=5)),
    (64, 200, 1792, 32, FP16, False, dict(kernel=1, tile_m=64, split_k=7)),
    (128, 136, 4096, 128, FP16, True, dict(kernel=1, tile_m=128, split_k=2)),
]


@pytest.mark.parametrize("shape", RAGGED, ids=lambda s: "M{}_N{}_K{}_g{}_{}{}{}".format(
    s[0], s[1], s[2], s[3], "bf16" if s[4] else "fp16", "" if s[5] else "_sym",
    "_" + "_".join(f"{k}{v}" for k, v in s[6].items()) if s[6] else ""))
def test_gemm_ragged(shape):
    M, N, K, g, dt, asym, ex = shape
    c = si.make_case(M, N, K, g, dt, seed=M + N + K, asym=asym, channel_scale=(0.5, 2.0))
    packed = repack_case(c)
    assert_parity_full(c, run_gemm(c, packed, **ex))


@pytest.mark.parametrize("kernel", [w4.W4A16_KERNEL_TC, w4.W4A16_KERNEL_SIMT])
def test_epilogue_ragged_n(kernel):
    M, N, K, g = 2, 264, 640, 64
    c = si.make_case(M, N, K, g, FP16, seed=21)
    packed = repack_case(c)
    rng = np.random.default_rng(3)
    bias = oracle.encode(rng.normal(size=N), FP16)
    res = oracle.encode(rng.normal(size=(M, N)), FP16)
    A = to_dev(c.A)
    Y = torch.empty((M, N), dtype=torch.int16, device="cuda")
    w4.w4a16_gemm_epilogue(A, packed, M, N, K, g, FP16, to_dev(bias), to_dev(res),
                           w4.W4A16_ACT_SILU, Y, kernel=kernel)
    assert w4.w4a16_get_device_status() == 0
    wd = oracle.dequant(c.qweight, c.scales, c.qzeros, N, K, g, FP16)
    yd, bb, _ = oracle.gemm(c.A, wd, M, N, K, FP16)
    out, bo, _ = oracle.epilogue(yd, bb, bias, res, w4.W4A16_ACT_SILU, M, N, FP16)
    bad, first, worst = oracle.check(to_host_u16(Y), out, bo, FP16)
    assert bad == 0, (bad, first, worst)


@pytest.mark.parametrize("tile_m,split_k", [(64, 3), (128, 2)])
def test_epilogue_split_k_larger_tiles_ragged_n(tile_m, split_k):
    """Bias, SiLU, residual and the per-channel factor applied by the split-K owner of a
    larger tile (four channels per thread) on a ragged N, against the oracle's fused
    epilogue."""
    M, N, K, g = 70, 392, 2048, 64
    c = si.make_case(M, N, K, g, BF16, seed=tile_m + split_k, channel_scale=(0.5, 2.0))
    packed = repack_case(c)
    rng = np.random.default_rng(tile_m)
    bias = oracle.encode(rng.normal(size=N), BF16)
    res = oracle.encode(rng.normal(size=(M, N)), BF16)
    A = to_dev(c.A)
    Y = torch.empty((M, N), dtype=torch.int16, device="cuda")
    w4.w4a16_gemm_epilogue(A, packed, M, N, K, g, BF16, to_dev(bias), to_dev(res),
                           w4.W4A16_ACT_SILU, Y, kernel=w4.W4A16_KERNEL_TC, tile_m=tile_m,
                           split_k=split_k)
    assert w4.w4a16_get_device_status() == 0
    wd = oracle.dequant(c.qweight, c.scales, c.qzeros, N, K, g, BF16)
    yd, bb, _ = oracle.gemm(c.A, wd, M, N, K, BF16, cscale=c.cscale)
    out, bo, _ = oracle.epilogue(yd, bb, bias, res, w4.W4A16_ACT_SILU, M, N, BF16)
    bad, first, worst = oracle.check(to_host_u16(Y), out, bo, BF16)
    assert bad == 0, (bad, first, worst)


def test_output_past_n_is_untouched():
    """Y has exactly N columns: the padded channels of the last tile must not be stored."""
    M, N, K, g = 4, 136, 256, 128
    c = si.make_case(M, N, K, g, FP16, seed=5)
    packed = repack_case(c)
    A = to_dev(c.A)
    for kernel in (w4.W4A16_KERNEL_TC, w4.W4A16_KERNEL_SIMT):
        buf = torch.full((M * N + 4096,), 0x3C00, dtype=torch.int16, device="cuda")
        Y = buf[:M * N].view(M, N)
        w4.w4a16_gemm_ex(A, packed, M, N, K, g, FP16, Y, kernel=kernel)
        assert w4.w4a16_get_device_status() == 0
        assert bool((buf[M * N:] == 0x3C00).all())
