"""Seeded synthetic inputs for the W4A16 GEMM (shared by tests, bench and smoke check).

This module only draws random numbers and lays them out in the canonical input format.
It holds none of the method's arithmetic (no unpacking, dequantisation or products), so
the oracle and the CUDA library can both be fed from it without sharing code.

Canonical input format (the user-facing layout, before the library's repack):
  A        activations, dtype bits uint16 [M, K], row-major.
  qweight  uint32 [N, K/8]; nibble j (bits 4j..4j+3) of word w in row n is q[n, 8w+j].
  scales   dtype bits uint16 [K/g, N].
  qzeros   uint32 [K/g, N/8]; nibble j of word w in group row gi is z[gi, 8w+j];
           None means symmetric weights, zero = 8.
  cscale   optional per-channel factor, dtype bits uint16 [N].

W4A8 canonical inputs (make_w4a8_case; groups of 128 along K):
  A        activations, dtype bits uint16 [M, K] (quantised to int8 by the library).
  qweight  uint32 [N, K/8], 4-bit codes in the same nibble order as above.
  s_u8     uint8 [N, K/128], the group's integer step, 1..16.
  a        uint8 [N, K/128], the group's offset, drawn in 0 .. 255 - 15 s_u8 (the range in
           which every code keeps its value inside a byte).
  s_w      float32 [N], the per-channel scale.

Recipe (one independent PCG64 stream per tensor, keyed by (seed, tensor id)):
  A ~ N(0, 1) drawn in float64; optional outlier columns (a fraction of K, chosen
  without replacement) are multiplied by a factor; then rounded to float32 and to the
  dtype (numpy for fp16, torch for bf16; both round to nearest even).
  q, z: uniform 32-bit words, i.e. eight independent uniform nibbles 0..15 per word.
  scales ~ U[lo, hi] in float64, rounded to the dtype the same way.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

FP16 = 0
BF16 = 1
DTYPE_NAMES = {FP16: "fp16", BF16: "bf16"}

_STREAM_A, _STREAM_Q, _STREAM_Z, _STREAM_S, _STREAM_OUT, _STREAM_C = 1, 2, 3, 4, 5, 6
_STREAM_STEP, _STREAM_OFF, _STREAM_SW = 7, 8, 9


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream])))


def to_dtype_bits(x: np.ndarray, dtype: int) -> np.ndarray:
    """float64 array -> fp16/bf16 bit patterns via the libraries' own RNE conversions."""
    if dtype == FP16:
        return np.ascontiguousarray(x.astype(np.float16).view(np.uint16))
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x.astype(np.float32))).to(torch.bfloat16)
    return np.ascontiguousarray(t.view(torch.int16).numpy().view(np.uint16))


@dataclass
class Case:
    M: int
    N: int
    K: int
    group: int
    dtype: int
    A: np.ndarray
    qweight: np.ndarray
    scales: np.ndarray
    qzeros: np.ndarray | None
    cscale: np.ndarray | None = None
    meta: dict = field(default_factory=dict)


def make_case(M: int, N: int, K: int, group: int, dtype: int = FP16, seed: int = 0, *,
              asym: bool = True, s_lo: float = 0.005, s_hi: float = 0.02,
              outlier_frac: float = 0.0, outlier_gain: float = 20.0,
              channel_scale: tuple[float, float] | None = None) -> Case:
    assert K % group == 0 and K % 8 == 0 and N % 8 == 0
    G = K // group
    a = _rng(seed, _STREAM_A).standard_normal((M, K))
    cols = np.zeros(0, dtype=np.int64)
    if outlier_frac > 0.0:
        n_out = int(round(outlier_frac * K))
        cols = np.sort(_rng(seed, _STREAM_OUT).choice(K, size=n_out, replace=False))
        a[:, cols] *= outlier_gain
    A = to_dtype_bits(a, dtype)
    qweight = _rng(seed, _STREAM_Q).integers(0, 1 << 32, size=(N, K // 8), dtype=np.uint32)
    qzeros = None
    if asym:
        qzeros = _rng(seed, _STREAM_Z).integers(0, 1 << 32, size=(G, N // 8), dtype=np.uint32)
    scales = to_dtype_bits(_rng(seed, _STREAM_S).uniform(s_lo, s_hi, size=(G, N)), dtype)
    cscale = None
    if channel_scale is not None:
        cscale = to_dtype_bits(_rng(seed, _STREAM_C).uniform(*channel_scale, size=N), dtype)
    return Case(M, N, K, group, dtype, A, qweight, scales, qzeros, cscale,
                meta={"seed": seed, "outlier_cols": cols})


@dataclass
class W4A8Case:
    M: int
    N: int
    K: int
    dtype: int
    A: np.ndarray
    qweight: np.ndarray
    s_u8: np.ndarray
    a: np.ndarray
    s_w: np.ndarray
    meta: dict = field(default_factory=dict)


def make_w4a8_case(M: int, N: int, K: int, dtype: int = FP16, seed: int = 0, *,
                   zero_rows: tuple = (), sw_lo: float = 5e-5, sw_hi: float = 2e-4,
                   steps: tuple[int, int] = (1, 16), outlier_frac: float = 0.0,
                   outlier_gain: float = 20.0) -> W4A8Case:
    """W4A8 inputs: A ~ N(0, 1) (rows listed in zero_rows all zero; optional outlier
    columns as in make_case), uniform 4-bit codes, per group a step uniform in `steps`
    and an offset uniform in 0 .. 255 - 15 step, per-channel scales ~ U[sw_lo, sw_hi] in
    float32."""
    assert K % 128 == 0 and N % 8 == 0
    G = K // 128
    a = _rng(seed, _STREAM_A).standard_normal((M, K))
    if outlier_frac > 0.0:
        n_out = int(round(outlier_frac * K))
        cols = np.sort(_rng(seed, _STREAM_OUT).choice(K, size=n_out, replace=False))
        a[:, cols] *= outlier_gain
    for m in zero_rows:
        a[m, :] = 0.0
    A = to_dtype_bits(a, dtype)
    qweight = _rng(seed, _STREAM_Q).integers(0, 1 << 32, size=(N, K // 8), dtype=np.uint32)
    s_u8 = _rng(seed, _STREAM_STEP).integers(steps[0], steps[1] + 1, size=(N, G)).astype(np.uint8)
    hi = 255 - 15 * s_u8.astype(np.int64)  # inclusive upper end of the offset
    off = np.floor(_rng(seed, _STREAM_OFF).uniform(size=(N, G)) * (hi + 1)).astype(np.int64)
    off = np.minimum(off, hi).astype(np.uint8)
    s_w = _rng(seed, _STREAM_SW).uniform(sw_lo, sw_hi, size=N).astype(np.float32)
    return W4A8Case(M, N, K, dtype, A, qweight, s_u8, off, s_w, meta={"seed": seed})


@dataclass
class MXCase:
    M: int
    N: int
    K: int
    dtype: int
    a_codes: np.ndarray   # uint8 [M, K] E4M3 codes
    a_scales: np.ndarray  # uint8 [M, K/32] E8M0 codes
    w_codes: np.ndarray   # uint8 [N, K/2], two E2M1 codes per byte (even K in the low nibble)
    w_scales: np.ndarray  # uint8 [N, K/32] E8M0 codes
    meta: dict = field(default_factory=dict)


def make_mx_case(M: int, N: int, K: int, dtype: int = FP16, seed: int = 0, *,
                 w_exp: tuple[int, int] = (119, 123), a_exp: tuple[int, int] = (122, 126)
                 ) -> MXCase:
    """MXFP4 weights and MXFP8 activations drawn directly as codes: uniform E2M1 codes,
    uniform E4M3 codes except the two NaN patterns, E8M0 scale codes uniform in the given
    inclusive ranges (2^-8..2^-4 for weights, 2^-5..2^-1 for activations by default)."""
    assert K % 128 == 0
    a_codes = _rng(seed, _STREAM_A).integers(0, 254, size=(M, K)).astype(np.uint8)
    a_codes[a_codes >= 0x7F] += 1  # skip 0x7F; 0xFF is never drawn (0..253 -> 0..254)
    a_scales = _rng(seed, _STREAM_S).integers(a_exp[0], a_exp[1] + 1, size=(M, K // 32)).astype(np.uint8)
    w_codes = _rng(seed, _STREAM_Q).integers(0, 256, size=(N, K // 2)).astype(np.uint8)
    w_scales = _rng(seed, _STREAM_STEP).integers(w_exp[0], w_exp[1] + 1, size=(N, K // 32)).astype(np.uint8)
    return MXCase(M, N, K, dtype, a_codes, a_scales, w_codes, w_scales, meta={"seed": seed})


def mx_algorithmic_bytes(M: int, N: int, K: int) -> int:
    """Bytes an MX decode GEMM moves at least once: E2M1 codes and weight scales, E4M3
    activations and their scales, and Y (16-bit)."""
    return K * N // 2 + (K // 32) * N + M * K + M * (K // 32) + 2 * M * N


# MX workloads (make_mx_case arguments): the 70B-shaped decode FFN shapes, M in {1, 8, 16}.
MX_WORKLOADS = {
    "mx_ffn70b_decode": [dict(M=m, N=n, K=k, dtype=BF16, seed=2)
                         for (k, n) in ((8192, 28672), (28672, 8192)) for m in (1, 8, 16)],
}


def mx_shape_tag(p: dict) -> str:
    return f"MX_M{p['M']}_N{p['N']}_K{p['K']}_{DTYPE_NAMES[p['dtype']]}"


def w4a8_algorithmic_bytes(M: int, N: int, K: int) -> int:
    """Bytes a W4A8 GEMM moves at least once: codes, steps and offsets, channel scales,
    int8 A with its row scales, and Y (16-bit)."""
    return K * N // 2 + 2 * (K // 128) * N + 4 * N + M * K + 4 * M + 2 * M * N


# ---- the workloads -------------------------------------------------------------------
# Each entry: name -> list of shapes; every shape is a dict of make_case arguments.

def _decode_sweep():
    out = []
    for n in (4096, 11008):
        for m in (1, 2, 4, 8, 16):
            out.append(dict(M=m, N=n, K=4096, group=128, dtype=FP16, seed=1, asym=True,
                            s_lo=0.005, s_hi=0.02))
    return out


def _ffn70b():
    out = []
    for (k, n) in ((8192, 28672), (28672, 8192)):
        for m in (1, 8, 32):
            out.append(dict(M=m, N=n, K=k, group=128, dtype=BF16, seed=2, asym=True,
                            s_lo=0.002, s_hi=0.01, outlier_frac=0.001, outlier_gain=20.0))
    return out


def _transition():
    out = []
    for g in (32, 64, 128):
        for m in (64, 128, 256):
            out.append(dict(M=m, N=8192, K=8192, group=g, dtype=FP16, seed=3, asym=False,
                            s_lo=0.005, s_hi=0.02))
    return out


WORKLOADS = {
    # tiny single-token GEMM, seed 0
    "tiny_m1_k512_n512_g128": [dict(M=1, N=512, K=512, group=128, dtype=FP16, seed=0,
                                    asym=True, s_lo=0.005, s_hi=0.02)],
    # decode sweep M in {1,2,4,8,16}, K=4096, N in {4096, 11008}
    "decode_k4096_n4096_n11008": _decode_sweep(),
    # 70B-shaped FFN decode, bf16 with 0.1% outlier columns x20
    "ffn70b_decode_bf16": _ffn70b(),
    # batch transition M in {64,128,256}, K=N=8192, g in {32,64,128}, symmetric
    "transition_k8192_n8192": _transition(),
    # prefill M=4096, K=4096, N=11008
    "prefill_m4096_k4096_n11008": [dict(M=4096, N=11008, K=4096, group=128, dtype=FP16,
                                        seed=4, asym=True, s_lo=0.005, s_hi=0.02)],
}


def _w4a8_ffn70b():
    return [dict(M=m, N=n, K=k, dtype=BF16, seed=2, outlier_frac=0.001, outlier_gain=20.0)
            for (k, n) in ((8192, 28672), (28672, 8192)) for m in (1, 8, 16)]


# W4A8 workloads (make_w4a8_case arguments): the 70B-shaped decode FFN shapes with bf16
# activations and 0.1% outlier columns x20, M in {1, 8, 16}.
W4A8_WORKLOADS = {
    "w4a8_ffn70b_decode_bf16": _w4a8_ffn70b(),
}


def w4a8_shape_tag(p: dict) -> str:
    return f"W4A8_M{p['M']}_N{p['N']}_K{p['K']}_{DTYPE_NAMES[p['dtype']]}"


def shape_tag(p: dict) -> str:
    return (f"M{p['M']}_N{p['N']}_K{p['K']}_g{p['group']}_{DTYPE_NAMES[p['dtype']]}"
            f"{'' if p.get('asym', True) else '_sym'}")


def algorithmic_bytes(M: int, N: int, K: int, group: int, asym: bool) -> int:
    """Bytes the GEMM must move at least once: packed weights, scales, zeros, A and Y."""
    G = K // group
    return K * N // 2 + G * N * 2 + (G * N // 2 if asym else 0) + 2 * M * K + 2 * M * N


def flops(M: int, N: int, K: int) -> int:
    return 2 * M * N * K
