"""GPU parity of the tensor-core kernel's larger tiles, one test per tile instance the
launch choice can take: 64-row tiles two to an SM whose two warpgroups share every block
(with and without split-K), 64-row tiles alone on an SM (four warpgroups unpacking whole
blocks, two MMA issuers taking alternate blocks; with and without split-K), 128-row tiles
two to an SM (two warpgroups sharing every block),
128-row tiles alone on an SM (four warpgroups unpacking whole blocks, six TMEM W
buffers, each group owning every fourth slot of the weight ring; with and without
split-K), 256-row tiles with two and four warpgroups, ragged M, N and K, every group
size and both dtypes.  Every element of Y is compared with
the oracle's fp64 product (|Y - Yd| <= 1e-3 * sum_k |A W| + 1 ulp)."""
import pytest
import torch

import synth_inputs as si
import weight_only_int4_tma_gb300 as w4
from gpu_util import assert_parity_full, repack_case, run_gemm

pytestmark = pytest.mark.gpu

FP16, BF16 = 0, 1


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_only_int4_tma_gb300 import build
    build.build()
    assert w4.w4a16_get_device_status() == 0


CASES = [
    # (M, N, K, group, dtype, tile_m, split_k)
    (64, 1024, 2048, 128, FP16, 64, 1),
    (70, 520, 1152, 64, BF16, 64, 1),
    (64, 1024, 4096, 32, FP16, 64, 2),
    # 64-row tiles alone on an SM (enough tiles x K slices to fill the SMs one CTA each)
    (64, 8192, 1024, 128, FP16, 64, 2),
    (50, 8192, 1152, 64, BF16, 64, 2),   # 9 K blocks over 2 slices
    (40, 16000, 640, 64, BF16, 64, 1),   # 125 tiles, no split-K
    (64, 4096, 2048, 32, FP16, 64, 4),
    (128, 1024, 2048, 128, FP16, 128, 1),
    (200, 776, 1664, 64, BF16, 128, 1),
    (128, 1024, 4096, 128, FP16, 128, 2),
    (256, 2048, 2048, 32, BF16, 128, 1),
    (300, 13056, 256, 128, FP16, 128, 1),  # 306 tiles: two per SM, two warpgroups
    (256, 1024, 2048, 128, FP16, 256, 1),
    (300, 520, 1152, 64, BF16, 256, 1),
]


@pytest.mark.parametrize("M,N,K,group,dtype,tile_m,split_k", CASES,
                         ids=[f"M{c[0]}_N{c[1]}_K{c[2]}_g{c[3]}_{'bf16' if c[4] else 'fp16'}"
                              f"_t{c[5]}_s{c[6]}" for c in CASES])
def test_large_tile_instance(M, N, K, group, dtype, tile_m, split_k):
    c = si.make_case(M, N, K, group, dtype, seed=M + N + K + group, asym=(group != 32))
    plan = w4.w4a16_gemm_plan(M, N, K, group, dtype, kernel=w4.W4A16_KERNEL_TC,
                              tile_m=tile_m, split_k=split_k)
    assert plan["tile_m"] == tile_m and plan["split_k"] == split_k
    Y = run_gemm(c, repack_case(c), kernel=w4.W4A16_KERNEL_TC, tile_m=tile_m, split_k=split_k)
    assert_parity_full(c, Y)


@pytest.mark.parametrize("M,N,K,split_k,alone", [
    (64, 8192, 1024, 2, True), (50, 8192, 1152, 2, True), (40, 16000, 640, 1, True),
    (64, 4096, 2048, 4, True), (64, 1024, 2048, 1, False), (64, 1024, 4096, 2, False),
    (64, 11008, 4096, 0, False)])
def test_64_row_tile_arrangement(M, N, K, split_k, alone):
    """64-row tiles run alone on an SM (four whole-block warpgroups) where one CTA per SM
    fills at least 4/5 of the SMs, else two to an SM with two warpgroups sharing every
    block (here with 132 or more SMs: 64 or 125 tiles fill them, 8 or 86 do not)."""
    if torch.cuda.get_device_properties(0).multi_processor_count < 132:
        pytest.skip("arrangement thresholds assume a GPU with 132 or more SMs")
    p = w4.w4a16_gemm_plan(M, N, K, 128 if K % 128 == 0 else 64, FP16,
                           kernel=w4.W4A16_KERNEL_TC, tile_m=64, split_k=split_k)
    assert p["whole_blocks"] == alone and p["groups"] == (4 if alone else 2), p
    if alone:
        assert p["stages"] % 2 == 0 and p["w_stages"] % 4 == 0, p


@pytest.mark.parametrize("stages", [2, 3, 4, 6])
def test_64_row_whole_block_ring_depths(stages):
    """64-row tiles alone on an SM with A rings of 2, 4 and 6 stages beside a weight ring
    whose depth is a multiple of 4 (each group reads every fourth weight slot), K long
    enough that both rings wrap many times; an odd A ring (3) keeps the shared-block
    arrangement instead (the two issuers take alternate A stages)."""
    p = w4.w4a16_gemm_plan(64, 8192, 4096, 128, FP16, kernel=w4.W4A16_KERNEL_TC, tile_m=64,
                           split_k=2, stages=stages)
    assert p["stages"] == stages and p["whole_blocks"] == (stages % 2 == 0), p
    if stages % 2 == 0:
        assert p["w_stages"] % 4 == 0 and p["groups"] == 4, p
    c = si.make_case(64, 8192, 4096, 128, FP16, seed=100 + stages)
    Y = run_gemm(c, repack_case(c), kernel=w4.W4A16_KERNEL_TC, tile_m=64, split_k=2,
                 stages=stages)
    assert_parity_full(c, Y)


@pytest.mark.parametrize("stages", [2, 4])
def test_128_row_tile_ring_depths(stages):
    """Four whole-block warpgroups and two MMA issuers taking alternate blocks, with A
    rings of 2 and 4 stages beside a weight ring whose depth is a multiple of 4 (each
    group reads every fourth weight slot); K = 8192 makes both rings wrap many times at
    depths that differ from each other."""
    p = w4.w4a16_gemm_plan(128, 256, 8192, 128, FP16, kernel=w4.W4A16_KERNEL_TC, tile_m=128,
                           split_k=1, stages=stages)
    assert p["stages"] == stages and p["w_stages"] % 4 == 0 and p["w_stages"] >= 4
    c = si.make_case(128, 256, 8192, 128, FP16, seed=stages)
    Y = run_gemm(c, repack_case(c), kernel=w4.W4A16_KERNEL_TC, tile_m=128, split_k=1,
                 stages=stages)
    assert_parity_full(c, Y)


@pytest.mark.parametrize("tile_m,split_k,stages", [(64, 1, 2), (64, 2, 3), (128, 2, 2),
                                                   (256, 1, 2), (256, 1, 3), (32, 1, 2)])
def test_rings_of_different_depths_wrap(tile_m, split_k, stages):
    """The A ring (depth `stages`) and the weight ring (depth chosen by the library) are
    independent: long K so that both wrap many times, with and without split-K, against
    every element of the oracle's product."""
    M = min(tile_m, 100) if tile_m > 32 else 24
    p = w4.w4a16_gemm_plan(M, 256, 8192, 64, BF16, kernel=w4.W4A16_KERNEL_TC, tile_m=tile_m,
                           split_k=split_k, stages=stages)
    assert p["stages"] == stages and p["w_stages"] >= 2
    c = si.make_case(M, 256, 8192, 64, BF16, seed=tile_m + stages, asym=True)
    Y = run_gemm(c, repack_case(c), kernel=w4.W4A16_KERNEL_TC, tile_m=tile_m,
                 split_k=split_k, stages=stages)
    assert_parity_full(c, Y)


def test_128_row_tile_rejects_an_odd_a_ring():
    """The two issuers of 128-row whole-block tiles take every other A stage, so an odd
    A ring depth would give an A slot two waiting issuers; the host refuses it."""
    with pytest.raises(w4.W4A16Error) as e:
        w4.w4a16_gemm_plan(128, 512, 4096, 128, FP16, kernel=w4.W4A16_KERNEL_TC, tile_m=128,
                           split_k=1, stages=3)
    assert e.value.status == w4.W4A16_ERR_UNSUPPORTED


def test_128_row_tile_rejects_a_ring_that_does_not_fit():
    """A ring depth above what fits in shared memory is refused on the host; nothing
    runs."""
    with pytest.raises(w4.W4A16Error) as e:
        w4.w4a16_gemm_plan(128, 512, 4096, 128, FP16, kernel=w4.W4A16_KERNEL_TC, tile_m=128,
                           split_k=1, stages=8)
    assert e.value.status == w4.W4A16_ERR_UNSUPPORTED


@pytest.mark.parametrize("act,with_res", [(w4.W4A16_ACT_SILU, True), (w4.W4A16_ACT_SILU, False),
                                          (w4.W4A16_ACT_NONE, True), (w4.W4A16_ACT_RELU, True)])
@pytest.mark.parametrize("tile_m", [128, 256])
def test_large_tile_fused_epilogue(tile_m, act, with_res):
    """Larger tiles with a fused activation and / or residual take four warpgroups (the
    staged 16-byte store path, the next group's residual loaded ahead); every element
    against the oracle's fused epilogue, including an in-place residual (Y aliases it)."""
    import numpy as np
    import oracle
    from gpu_util import to_dev, to_host_u16
    c = si.make_case(300, 520, 1152, 64, FP16, seed=tile_m + act)
    packed = repack_case(c)
    rng = np.random.default_rng(act + tile_m)
    bias = oracle.encode(rng.normal(size=c.N), c.dtype)
    res = oracle.encode(rng.normal(size=(c.M, c.N)), c.dtype) if with_res else None
    Y = to_dev(res) if with_res else torch.empty((c.M, c.N), dtype=torch.int16, device="cuda")
    w4.w4a16_gemm_epilogue(to_dev(c.A), packed, c.M, c.N, c.K, c.group, c.dtype, to_dev(bias),
                           Y if with_res else None, act, Y, kernel=w4.W4A16_KERNEL_TC,
                           tile_m=tile_m, split_k=1)
    assert w4.w4a16_get_device_status() == 0
    wd = oracle.dequant(c.qweight, c.scales, c.qzeros, c.N, c.K, c.group, c.dtype)
    yd, bb, _ = oracle.gemm(c.A, wd, c.M, c.N, c.K, c.dtype)
    out, bo, _ = oracle.epilogue(yd, bb, bias, res, act, c.M, c.N, c.dtype)
    bad, first, worst = oracle.check(to_host_u16(Y), out, bo, c.dtype)
    assert bad == 0, (bad, first, worst)


@pytest.mark.parametrize("M,N,K,split_k", [(40, 16000, 640, 1), (64, 8192, 1024, 2)],
                         ids=["no_split_staged_store", "split2_owner_reduction"])
@pytest.mark.parametrize("act,with_res", [(w4.W4A16_ACT_SILU, True), (w4.W4A16_ACT_RELU, False)])
def test_64_row_tiles_alone_fused_epilogue(M, N, K, split_k, act, with_res):
    """64-row tiles alone on an SM (four whole-block groups, two issuers) with a fused
    bias, activation and in-place residual: through the staged 16-byte store without
    split-K and through the owner's reduction with it; every element against the
    oracle's fused epilogue."""
    import numpy as np
    import oracle
    from gpu_util import to_dev, to_host_u16
    c = si.make_case(M, N, K, 64, BF16, seed=M + split_k + act, asym=True)
    p = w4.w4a16_gemm_plan(M, N, K, 64, BF16, kernel=w4.W4A16_KERNEL_TC, tile_m=64,
                           split_k=split_k)
    if torch.cuda.get_device_properties(0).multi_processor_count >= 132:
        assert p["whole_blocks"] and p["groups"] == 4, p
    rng = np.random.default_rng(act + M)
    bias = oracle.encode(rng.normal(size=c.N), c.dtype)
    res = oracle.encode(rng.normal(size=(c.M, c.N)), c.dtype) if with_res else None
    Y = to_dev(res) if with_res else torch.empty((c.M, c.N), dtype=torch.int16, device="cuda")
    w4.w4a16_gemm_epilogue(to_dev(c.A), repack_case(c), c.M, c.N, c.K, c.group, c.dtype,
                           to_dev(bias), Y if with_res else None, act, Y,
                           kernel=w4.W4A16_KERNEL_TC, tile_m=64, split_k=split_k)
    assert w4.w4a16_get_device_status() == 0
    wd = oracle.dequant(c.qweight, c.scales, c.qzeros, c.N, c.K, c.group, c.dtype)
    yd, bb, _ = oracle.gemm(c.A, wd, c.M, c.N, c.K, c.dtype)
    out, bo, _ = oracle.epilogue(yd, bb, bias, res, act, c.M, c.N, c.dtype)
    bad, first, worst = oracle.check(to_host_u16(Y), out, bo, c.dtype)
    assert bad == 0, (bad, first, worst)
