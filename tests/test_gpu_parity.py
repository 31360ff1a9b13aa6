"""GPU parity: the CUDA library, called through its C ABI, against the oracle.

Bars: the debug dequant kernel is bit-exact with the oracle's Wd; every GEMM output
element satisfies |Y - Yd| <= 1e-3 * sum_k |A W| + 1 ulp of the output dtype.
"""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
import weight_only_int4_tma_gb300 as w4
from gpu_util import (assert_parity_full, assert_parity_sampled, oracle_full, repack_case,
                      run_gemm, to_dev, to_host_u16)

pytestmark = pytest.mark.gpu

FP16, BF16 = 0, 1


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_only_int4_tma_gb300 import build
    build.build()
    torch.cuda.init()
    assert w4.w4a16_get_device_status() == 0


# ---- failure path first: the bounded wait must return, and the context stay usable ----

def test_timeout_probe_reports_and_context_survives():
    w4.w4a16_debug_timeout_probe(2000)
    assert w4.w4a16_get_device_status() == w4.W4A16_ERR_DEVICE_TIMEOUT
    assert w4.w4a16_get_device_status() == 0  # cleared by the read
    x = torch.arange(10, device="cuda")
    assert int(x.sum().item()) == 45


def test_splitk_timeout_probe_reports_and_context_survives():
    """Split-K exchange failure path: cluster rank 0 of every tile pushes none of its
    partials, so the other ranks' bounded waits for them run out (20 ms).  The kernel
    reports the timeout, every rank leaves only after its peers stopped pushing into it,
    and the context stays usable: the same GEMM right after is correct."""
    c = si.make_case(4, 1024, 4096, 128, FP16, seed=3)
    packed = repack_case(c)
    plan = w4.w4a16_gemm_plan(c.M, c.N, c.K, c.group, c.dtype, kernel=w4.W4A16_KERNEL_TC,
                              tile_m=16)
    assert plan["split_k"] >= 2
    Y = torch.zeros((c.M, c.N), dtype=torch.int16, device="cuda")
    w4.w4a16_debug_splitk_timeout_probe(to_dev(c.A), packed, c.M, c.N, c.K, c.group, c.dtype,
                                        Y, 20000)
    assert w4.w4a16_get_device_status() == w4.W4A16_ERR_DEVICE_TIMEOUT
    assert w4.w4a16_get_device_status() == 0  # cleared by the read
    assert_parity_full(c, run_gemm(c, packed))


# ---- repack + debug dequant: bit-exact ----------------------------------------------

@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("asym", [True, False])
def test_dequant_debug_bitexact(dtype, group, asym):
    c = si.make_case(1, 384, 640, group, dtype, seed=group + dtype, asym=asym,
                     s_lo=-0.03, s_hi=0.05)
    packed = repack_case(c)
    W = torch.empty((c.N, c.K), dtype=torch.int16, device="cuda")
    w4.w4a16_dequant_debug(packed, c.N, c.K, c.group, c.dtype, W)
    assert w4.w4a16_get_device_status() == 0
    wd = oracle.dequant(c.qweight, c.scales, c.qzeros, c.N, c.K, c.group, c.dtype)
    got = to_host_u16(W)
    if not np.array_equal(got, wd):
        idx = np.argwhere(got != wd)[0]
        raise AssertionError(f"first mismatch at {tuple(idx)}: {got[tuple(idx)]:#06x} vs "
                             f"{wd[tuple(idx)]:#06x}; {np.sum(got != wd)} mismatches")


def test_dequant_debug_full_range_scales_fp16():
    # scales spanning subnormal to large fp16 values, all (q, z) combinations present
    c = si.make_case(1, 256, 256, 32, FP16, seed=5)
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 0x7800, size=c.scales.shape, dtype=np.uint16)  # finite, |s| < 32768
    sign = rng.integers(0, 2, size=c.scales.shape, dtype=np.uint16) << 15
    c.scales = (bits | sign).astype(np.uint16)
    packed = repack_case(c)
    W = torch.empty((c.N, c.K), dtype=torch.int16, device="cuda")
    w4.w4a16_dequant_debug(packed, c.N, c.K, c.group, c.dtype, W)
    wd = oracle.dequant(c.qweight, c.scales, c.qzeros, c.N, c.K, c.group, c.dtype)
    assert np.array_equal(to_host_u16(W), wd)


def test_format_mismatch_is_reported():
    c = si.make_case(1, 256, 512, 128, FP16, seed=1)
    packed = repack_case(c)
    W = torch.zeros((c.N, c.K), dtype=torch.int16, device="cuda")
    w4.w4a16_dequant_debug(packed, c.N, c.K, 64, c.dtype, W)  # wrong group
    assert w4.w4a16_get_device_status() == w4.W4A16_ERR_FORMAT
    assert int(W.abs().sum().item()) == 0
    Y = torch.zeros((4, c.N), dtype=torch.int16, device="cuda")
    A = torch.zeros((4, c.K), dtype=torch.int16, device="cuda")
    w4.w4a16_gemm(A, packed, 4, c.N, c.K, c.group, BF16, Y)  # wrong dtype
    assert w4.w4a16_get_device_status() == w4.W4A16_ERR_FORMAT
    w4.w4a16_gemm_ex(A, packed, 4, c.N, c.K, c.group, BF16, Y, kernel=w4.W4A16_KERNEL_SIMT)
    assert w4.w4a16_get_device_status() == w4.W4A16_ERR_FORMAT
    assert int(Y.abs().sum().item()) == 0


# ---- GEMM parity at sizes the oracle checks element by element ----------------------

SMALL = [
    # (M, N, K, group, dtype, asym)
    (1, 512, 512, 128, FP16, True),      # the tiny single-token case
    (5, 384, 1152, 64, FP16, True),      # ragged M, K blocks not divisible by the split
    (16, 256, 2048, 32, BF16, True),
    (17, 512, 1024, 128, BF16, False),   # one row past a 16-row tile
    (33, 256, 768, 128, FP16, True),
    (100, 384, 512, 64, FP16, False),
    (130, 256, 640, 128, BF16, True),    # two 128-row tiles, second ragged
    (300, 256, 384, 32, FP16, True),
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "M{}_N{}_K{}_g{}_{}{}".format(
    s[0], s[1], s[2], s[3], "bf16" if s[4] else "fp16", "" if s[5] else "_sym"))
def test_gemm_small_auto(shape):
    M, N, K, g, dt, asym = shape
    c = si.make_case(M, N, K, g, dt, seed=M + N, asym=asym)
    packed = repack_case(c)
    assert_parity_full(c, run_gemm(c, packed))


@pytest.mark.parametrize("tile_m", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("split_k", [1, 2, 3, 5, 8])
def test_gemm_tc_tilings(tile_m, split_k):
    M = {16: 13, 32: 30, 64: 64, 128: 129, 256: 200}[tile_m]
    c = si.make_case(M, 256, 1024, 128, FP16, seed=tile_m + split_k)
    packed = repack_case(c)
    if tile_m == 256 and split_k > 2:
        # the split-K receive area of a 256-row tile fits beside its rings for two
        # K slices only
        with pytest.raises(w4.W4A16Error) as e:
            run_gemm(c, packed, kernel=w4.W4A16_KERNEL_TC, tile_m=tile_m, split_k=split_k)
        assert e.value.status == w4.W4A16_ERR_UNSUPPORTED
        return
    Y = run_gemm(c, packed, kernel=w4.W4A16_KERNEL_TC, tile_m=tile_m, split_k=split_k)
    assert_parity_full(c, Y)


@pytest.mark.parametrize("flags", [0, w4.W4A16_GEMM_NO_PDL, w4.W4A16_GEMM_NO_WEIGHT_PREFETCH,
                                   w4.W4A16_GEMM_NO_PDL | w4.W4A16_GEMM_NO_WEIGHT_PREFETCH])
@pytest.mark.parametrize("split_k", [1, 4, 7])
def test_gemm_tc_launch_flags(flags, split_k):
    c = si.make_case(3, 384, 1792, 128, BF16, seed=flags + 10 * split_k)
    packed = repack_case(c)
    Y = run_gemm(c, packed, kernel=w4.W4A16_KERNEL_TC, split_k=split_k, flags=flags)
    assert_parity_full(c, Y)


@pytest.mark.parametrize("flags", [w4.W4A16_GEMM_NO_PDL, w4.W4A16_GEMM_NO_WEIGHT_PREFETCH])
@pytest.mark.parametrize("tile_m,split_k", [(64, 2), (128, 1), (256, 1)])
def test_gemm_tc_launch_flags_larger_tiles(flags, tile_m, split_k):
    """The larger tiles stream weights and A from two producer warps; without weight
    prefetch the weight producer starts only after the dependency wait, without PDL the
    launch waits for the previous kernel."""
    c = si.make_case(tile_m - 5, 384, 2048, 64, BF16, seed=flags + tile_m)
    packed = repack_case(c)
    Y = run_gemm(c, packed, kernel=w4.W4A16_KERNEL_TC, tile_m=tile_m, split_k=split_k,
                 flags=flags)
    assert_parity_full(c, Y)


def test_back_to_back_gemms_share_nothing():
    """Consecutive launches overlap under programmatic dependent launch: the second
    GEMM reads the first one's output as its A, so a missing dependency wait would
    show up as a mismatch."""
    c1 = si.make_case(4, 512, 512, 128, FP16, seed=31)
    c2 = si.make_case(4, 256, 512, 128, FP16, seed=32)
    p1, p2 = repack_case(c1), repack_case(c2)
    A = to_dev(c1.A)
    Y1 = torch.empty((4, 512), dtype=torch.int16, device="cuda")
    Y2 = torch.empty((4, 256), dtype=torch.int16, device="cuda")
    for _ in range(3):
        w4.w4a16_gemm(A, p1, 4, 512, 512, 128, FP16, Y1)
        w4.w4a16_gemm(Y1, p2, 4, 256, 512, 128, FP16, Y2)
    assert w4.w4a16_get_device_status() == 0
    c2.A = to_host_u16(Y1)
    assert_parity_full(c2, to_host_u16(Y2))


@pytest.mark.parametrize("stages", [2, 3, 5])
def test_gemm_tc_ring_depths(stages):
    c = si.make_case(8, 256, 2048, 64, BF16, seed=stages)
    packed = repack_case(c)
    Y = run_gemm(c, packed, kernel=w4.W4A16_KERNEL_TC, tile_m=16, split_k=2, stages=stages)
    assert_parity_full(c, Y)


@pytest.mark.parametrize("M", [1, 2, 3, 4, 7, 8])
@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_gemm_simt(M, dtype):
    c = si.make_case(M, 512, 1024, 128, dtype, seed=M)
    packed = repack_case(c)
    Y = run_gemm(c, packed, kernel=w4.W4A16_KERNEL_SIMT)
    assert_parity_full(c, Y)


# CUDA-core GEMV work split: units of 16 or 32 channels over a persistent grid (several
# units per CTA once N / rows exceeds the CTAs that fit), K blocks dealt to 8 or 16 slots
# (ragged and idle slots when K / 128 is not a multiple), 1, 2 or 4 groups per block.
SIMT_SPLITS = [
    # (M, N, K, group, dtype, asym, rows)
    (1, 8192, 1024, 128, FP16, True, 16),    # 512 units > resident CTAs: 2 per CTA
    (1, 12288, 640, 64, BF16, True, 32),     # 384 units; 5 blocks over 8 slots
    (2, 8192, 384, 32, FP16, False, 16),     # 3 blocks over 16 slots, symmetric
    (1, 256, 2944, 32, BF16, True, 16),      # 23 blocks: uneven slots, odd counts
    (3, 6016, 1152, 64, FP16, True, 32),     # 47 tiles' worth of rows, 9 blocks
]


@pytest.mark.parametrize("shape", SIMT_SPLITS, ids=lambda s: "M{}_N{}_K{}_g{}_{}{}_r{}".format(
    s[0], s[1], s[2], s[3], "bf16" if s[4] else "fp16", "" if s[5] else "_sym", s[6]))
def test_gemm_simt_work_split(shape):
    M, N, K, g, dt, asym, rows = shape
    c = si.make_case(M, N, K, g, dt, seed=N + K, asym=asym)
    packed = repack_case(c)
    Y = run_gemm(c, packed, kernel=w4.W4A16_KERNEL_SIMT, tile_m=rows)
    assert_parity_sampled(c, Y, count=6000, seed=rows)


def test_auto_routes_single_row():
    """M == 1 goes to the GEMV for matrices of up to 26 Mi weights (and one 128-channel
    tile per SM at most), otherwise to the tensor-core kernel; both routes agree with the
    oracle."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = lambda M, N, K: w4.w4a16_gemm_plan(M, N, K, 128, FP16)["kernel"]
    assert plan(1, 2048, 13312) == w4.W4A16_KERNEL_SIMT   # exactly 26 Mi weights
    assert plan(1, 2048, 13440) == w4.W4A16_KERNEL_TC
    assert plan(1, 4096, 4096) == w4.W4A16_KERNEL_SIMT
    assert plan(1, 11008, 4096) == w4.W4A16_KERNEL_TC
    assert plan(1, 128 * (sms + 1), 128) == w4.W4A16_KERNEL_TC  # more tiles than SMs
    assert plan(2, 256, 4096) == w4.W4A16_KERNEL_TC
    # between one and two decode tiles per SM: two K slices balance the SMs
    p = w4.w4a16_gemm_plan(8, 128 * (sms + 8), 8192, 128, BF16)
    assert (p["kernel"], p["tile_m"], p["split_k"]) == (w4.W4A16_KERNEL_TC, 16, 2)
    for N, K in ((4096, 4096), (2048, 13440)):  # one case on each route
        c = si.make_case(1, N, K, 128, FP16, seed=K)
        packed = repack_case(c)
        assert_parity_full(c, run_gemm(c, packed))
    with pytest.raises(w4.W4A16Error) as e:  # the GEMV has no ring depth or split to set
        c = si.make_case(1, 256, 512, 128, FP16, seed=1)
        run_gemm(c, repack_case(c), kernel=w4.W4A16_KERNEL_SIMT, stages=3)
    assert e.value.status == w4.W4A16_ERR_UNSUPPORTED


def test_heuristic_split_keeps_clusters_in_one_wave():
    """The split-K heuristic fills the SMs' two slots per SM, but a clustered launch stays
    within ~6/7 of them (clusters are placed whole within a GPC; above that the launch
    ran in two waves)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    slots = 2 * sms
    for tiles in (16, 24, 32, 40, 48, 56, 64, 86, 112):
        p = w4.w4a16_gemm_plan(16, 128 * tiles, 4096, 128, FP16)
        assert p["kernel"] == w4.W4A16_KERNEL_TC and p["tile_m"] == 16
        ctas = tiles * p["split_k"]
        assert p["split_k"] <= 8 and ctas <= slots
        if p["split_k"] > 2:
            assert ctas <= slots * 6 // 7, (tiles, p["split_k"])
        # and it is not needlessly small: one more K slice would break the bound
        if p["split_k"] < 8 and p["split_k"] > 2:
            assert tiles * (p["split_k"] + 1) > slots * 6 // 7


@pytest.mark.parametrize("kernel", [w4.W4A16_KERNEL_TC, w4.W4A16_KERNEL_SIMT])
def test_channel_scale(kernel):
    c = si.make_case(4, 256, 512, 128, BF16, seed=3, channel_scale=(0.25, 4.0))
    packed = repack_case(c)
    assert_parity_full(c, run_gemm(c, packed, kernel=kernel))


@pytest.mark.parametrize("kernel", [w4.W4A16_KERNEL_TC, w4.W4A16_KERNEL_SIMT])
def test_one_hot_rows_exact(kernel):
    """A one-hot row of A selects a dequantised weight column: exact on the GPU too."""
    N, K, g = 256, 512, 128
    c = si.make_case(8, N, K, g, FP16, seed=2)
    ks = [0, 1, 127, 128, 255, 300, 510, 511]
    A = np.zeros((8, K), dtype=np.uint16)
    for i, k in enumerate(ks):
        A[i, k] = 0x3C00
    c.A = A
    packed = repack_case(c)
    Y = run_gemm(c, packed, kernel=kernel)
    wd = oracle.dequant(c.qweight, c.scales, c.qzeros, N, K, g, FP16)
    for i, k in enumerate(ks):
        assert np.array_equal(Y[i], wd[:, k]), i


def test_q_equals_z_gives_zero():
    c = si.make_case(16, 256, 512, 64, FP16, seed=4)
    c.qweight[:] = 0x77777777
    c.qzeros = np.full_like(c.qzeros, 0x77777777)
    packed = repack_case(c)
    Y = run_gemm(c, packed)
    assert (oracle.decode(Y, FP16) == 0).all()


def test_empty_m_is_noop():
    c = si.make_case(1, 256, 512, 128, FP16, seed=6)
    packed = repack_case(c)
    Y = torch.full((1, 256), 7, dtype=torch.int16, device="cuda")
    A = to_dev(c.A)
    w4.w4a16_gemm(A, packed, 0, c.N, c.K, c.group, c.dtype, Y)
    assert w4.w4a16_get_device_status() == 0
    assert int(Y.sum().item()) == 7 * 256


def test_unsupported_shapes_rejected():
    A = torch.zeros((4, 512), dtype=torch.int16, device="cuda")
    Y = torch.zeros((4, 512), dtype=torch.int16, device="cuda")
    P = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(w4.W4A16Error) as e:
        w4.w4a16_gemm(A, P, 4, 500, 512, 128, FP16, Y)
    assert e.value.status == w4.W4A16_ERR_UNSUPPORTED
    with pytest.raises(w4.W4A16Error):
        w4.w4a16_gemm_ex(A, P, 16, 512, 512, 128, FP16, Y, kernel=w4.W4A16_KERNEL_SIMT)


def test_deterministic():
    c = si.make_case(8, 512, 4096, 128, FP16, seed=9)
    packed = repack_case(c)
    A = to_dev(c.A)
    y1 = run_gemm(c, packed, A_dev=A)
    y2 = run_gemm(c, packed, A_dev=A)
    assert np.array_equal(y1, y2)
