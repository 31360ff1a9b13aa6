"""GPU parity over seeded random launch configurations of the tensor-core kernel: tile
height, split-K, A ring depth, launch flags, group size, dtype, zeros, channel factor and
ragged N / K drawn together, so that ring depths, K slices and tile edges meet in
combinations the hand-written cases do not list, with and without a fused epilogue
(bias, activation, in-place residual).  A configuration the host refuses
(W4A16_ERR_UNSUPPORTED: its rings or receive area do not fit) is checked to be refused by
the plan as well and skipped; every other one is compared with the oracle on every
element."""
import numpy as np
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


def _configs(n=120, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        tile = int(rng.choice([16, 32, 64, 128, 256]))
        M = int(rng.integers(max(1, tile // 2 - 7), tile + 1)) if tile > 16 else int(rng.integers(1, 17))
        group = int(rng.choice([32, 64, 128]))
        K = group * int(rng.integers(1, max(2, 3072 // group)))
        N = 8 * int(rng.integers(1, 97))
        if M * N * K > 4e8:
            continue
        split = int(rng.choice([1, 1, 2, 3, 4, 8]))
        stages = int(rng.choice([0, 0, 2, 3, 4]))
        flags = int(rng.choice([0, 0, w4.W4A16_GEMM_NO_PDL, w4.W4A16_GEMM_NO_WEIGHT_PREFETCH]))
        epi = int(rng.choice([0, 0, 1, 2, 3]))  # none, bias + ReLU, bias + SiLU + residual, residual
        out.append(dict(M=M, N=N, K=K, group=group, dtype=int(rng.integers(0, 2)),
                        asym=bool(rng.integers(0, 2)), cscale=bool(rng.integers(0, 2)),
                        tile_m=tile, split_k=min(split, -(-K // 128)), stages=stages,
                        flags=flags, epi=epi, seed=int(rng.integers(0, 1 << 20))))
    return out


CONFIGS = _configs()


@pytest.mark.parametrize("cfg", CONFIGS, ids=[
    "M{M}_N{N}_K{K}_g{group}_{dt}_t{tile_m}_s{split_k}_a{stages}_f{flags}_e{epi}".format(
        dt="bf16" if c["dtype"] else "fp16", **c) for c in CONFIGS])
def test_random_launch_configuration(cfg):
    c = si.make_case(cfg["M"], cfg["N"], cfg["K"], cfg["group"], cfg["dtype"],
                     seed=cfg["seed"], asym=cfg["asym"],
                     channel_scale=(0.5, 2.0) if cfg["cscale"] else None)
    ex = dict(kernel=w4.W4A16_KERNEL_TC, tile_m=cfg["tile_m"], split_k=cfg["split_k"],
              stages=cfg["stages"], flags=cfg["flags"])
    try:
        plan = w4.w4a16_gemm_plan(c.M, c.N, c.K, c.group, c.dtype, **ex)
    except w4.W4A16Error as e:
        assert e.status == w4.W4A16_ERR_UNSUPPORTED
        with pytest.raises(w4.W4A16Error):
            run_gemm(c, repack_case(c), **ex)
        pytest.skip("refused by the host (rings or receive area do not fit)")
    assert plan["tile_m"] == cfg["tile_m"] and plan["split_k"] == cfg["split_k"]
    if cfg["stages"]:
        assert plan["stages"] == cfg["stages"]
    if cfg["epi"] == 0:
        assert_parity_full(c, run_gemm(c, repack_case(c), **ex))
        return
    # fused epilogue: y = act(v * c[n] + bias[n]) + residual[m, n], in place on the residual
    import oracle
    from gpu_util import to_dev, to_host_u16
    act = {1: w4.W4A16_ACT_RELU, 2: w4.W4A16_ACT_SILU, 3: w4.W4A16_ACT_NONE}[cfg["epi"]]
    rng = np.random.default_rng(cfg["seed"])
    bias = oracle.encode(rng.normal(size=c.N), c.dtype) if cfg["epi"] in (1, 2) else None
    res = oracle.encode(rng.normal(size=(c.M, c.N)), c.dtype) if cfg["epi"] in (2, 3) else None
    Y = to_dev(res) if res is not None else torch.empty((c.M, c.N), dtype=torch.int16,
                                                       device="cuda")
    w4.w4a16_gemm_epilogue(to_dev(c.A), repack_case(c), c.M, c.N, c.K, c.group, c.dtype,
                           to_dev(bias), Y if res is not None else None, act, Y, **ex)
    assert w4.w4a16_get_device_status() == 0
    wd = oracle.dequant(c.qweight, c.scales, c.qzeros, c.N, c.K, c.group, c.dtype)
    yd, bb, _ = oracle.gemm(c.A, wd, c.M, c.N, c.K, c.dtype, cscale=c.cscale)
    out, bo, _ = oracle.epilogue(yd, bb, bias, res, act, c.M, c.N, c.dtype)
    bad, first, worst = oracle.check(to_host_u16(Y), out, bo, c.dtype)
    assert bad == 0, (bad, first, worst)


def _simt_configs(n=40, seed=77):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        group = int(rng.choice([32, 64, 128]))
        out.append(dict(M=int(rng.integers(1, 9)), N=8 * int(rng.integers(1, 257)),
                        K=group * int(rng.integers(1, max(2, 4096 // group))), group=group,
                        dtype=int(rng.integers(0, 2)), asym=bool(rng.integers(0, 2)),
                        cscale=bool(rng.integers(0, 2)), rows=int(rng.choice([0, 16, 32])),
                        flags=int(rng.choice([0, w4.W4A16_GEMM_NO_PDL,
                                              w4.W4A16_GEMM_NO_WEIGHT_PREFETCH])),
                        seed=int(rng.integers(0, 1 << 20))))
    return out


SIMT = _simt_configs()


@pytest.mark.parametrize("cfg", SIMT, ids=[
    "M{M}_N{N}_K{K}_g{group}_{dt}_r{rows}_f{flags}".format(
        dt="bf16" if c["dtype"] else "fp16", **c) for c in SIMT])
def test_random_simt_configuration(cfg):
    """The CUDA-core GEMV (M <= 8) over random shapes, unit heights and flags."""
    c = si.make_case(cfg["M"], cfg["N"], cfg["K"], cfg["group"], cfg["dtype"],
                     seed=cfg["seed"], asym=cfg["asym"],
                     channel_scale=(0.5, 2.0) if cfg["cscale"] else None)
    ex = dict(kernel=w4.W4A16_KERNEL_SIMT, tile_m=cfg["rows"], flags=cfg["flags"])
    assert w4.w4a16_gemm_plan(c.M, c.N, c.K, c.group, c.dtype, **ex)["kernel"] == \
        w4.W4A16_KERNEL_SIMT
    assert_parity_full(c, run_gemm(c, repack_case(c), **ex))


def _alone64_configs(n=12, seed=404):
    """Shapes whose 64-row tiles run alone on an SM: 64 or more channel tiles, so that one
    CTA per SM (with the K slices that fit) fills most of a 152-SM GPU."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        group = int(rng.choice([32, 64, 128]))
        out.append(dict(M=int(rng.integers(33, 65)), N=128 * int(rng.integers(61, 76)) - 8 * int(rng.integers(0, 15)),
                        K=group * int(rng.integers(1, max(2, 1536 // group))), group=group,
                        dtype=int(rng.integers(0, 2)), asym=bool(rng.integers(0, 2)),
                        split_k=int(rng.choice([0, 2])), stages=int(rng.choice([0, 2, 4, 6])),
                        epi=int(rng.choice([0, 0, 2])), seed=int(rng.integers(0, 1 << 20))))
    return out


ALONE64 = _alone64_configs()


@pytest.mark.parametrize("cfg", ALONE64, ids=[
    "M{M}_N{N}_K{K}_g{group}_{dt}_s{split_k}_a{stages}_e{epi}".format(
        dt="bf16" if c["dtype"] else "fp16", **c) for c in ALONE64])
def test_random_64_row_tiles_alone(cfg):
    """64-row tiles with four whole-block warpgroups over random ragged shapes, K slices,
    A ring depths and (e2) a fused bias + SiLU + in-place residual."""
    c = si.make_case(cfg["M"], cfg["N"], cfg["K"], cfg["group"], cfg["dtype"],
                     seed=cfg["seed"], asym=cfg["asym"])
    split = min(cfg["split_k"], -(-c.K // 128)) if cfg["split_k"] else 0
    ex = dict(kernel=w4.W4A16_KERNEL_TC, tile_m=64, split_k=split, stages=cfg["stages"])
    try:
        w4.w4a16_gemm_plan(c.M, c.N, c.K, c.group, c.dtype, **ex)
    except w4.W4A16Error as e:
        assert e.status == w4.W4A16_ERR_UNSUPPORTED
        pytest.skip("refused by the host")
    if cfg["epi"] == 0:
        assert_parity_full(c, run_gemm(c, repack_case(c), **ex))
        return
    import oracle
    from gpu_util import to_dev, to_host_u16
    rng = np.random.default_rng(cfg["seed"])
    bias = oracle.encode(rng.normal(size=c.N), c.dtype)
    res = oracle.encode(rng.normal(size=(c.M, c.N)), c.dtype)
    Y = to_dev(res)
    w4.w4a16_gemm_epilogue(to_dev(c.A), repack_case(c), c.M, c.N, c.K, c.group, c.dtype,
                           to_dev(bias), Y, w4.W4A16_ACT_SILU, Y, **ex)
    assert w4.w4a16_get_device_status() == 0
    wd = oracle.dequant(c.qweight, c.scales, c.qzeros, c.N, c.K, c.group, c.dtype)
    yd, bb, _ = oracle.gemm(c.A, wd, c.M, c.N, c.K, c.dtype)
    out, bo, _ = oracle.epilogue(yd, bb, bias, res, w4.W4A16_ACT_SILU, c.M, c.N, c.dtype)
    bad, first, worst = oracle.check(to_host_u16(Y), out, bo, c.dtype)
    assert bad == 0, (bad, first, worst)
