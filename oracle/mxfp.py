"""MX block-scaled 4-bit / 8-bit formats (the pages' Blackwell "route A") -- TEST
INFRASTRUCTURE ONLY.

Source: "量化开销对比：各家方案的矩阵乘账本与省账手段", end of §3 and the MXFP4 / NVFP4 row
of the §5 overhead table (fp4 weights / fp8 activations, a native FP4 GEMM, the block-32
E8M0 exponent scale held by the hardware), and the glossary row (hardware-native block-
scaled 4-bit formats, block 32).  A plain CPU statement (numpy, fp64) of what such a GEMM
computes; only ``tests/`` may import it, and it shares no code with the CUDA library.

The pages give no more than the above; this module takes the plainest reading (each
listed in the design notes):
  * element formats: FP4 E2M1 for weights (1 sign bit, 2 exponent bits with bias 1, 1
    mantissa bit; no infinity or NaN; largest magnitude 6) and FP8 E4M3 for activations
    (bias 7, no infinity, S.1111.111 is NaN; largest magnitude 448);
  * block scale: E8M0, the value 2^(e - 127) (e = 255 is NaN), one per 32 consecutive
    values along K;
  * quantiser: per block, X = floor(log2(max |v|)) - emax with emax = 2 for E2M1 and 8
    for E4M3 (the exponent of the format's largest value), clamped to [-127, 127]; each
    element is the format value nearest to v / 2^X (ties to the even code), saturated to
    the largest magnitude; an all-zero block takes X = -127;
  * product: Y[m, n] = sum_k a[m, k] * w[n, k] of the decoded values (element times block
    scale), accumulated in fp64.
NVFP4's own layout (block 16 with an E4M3 scale) is not on the pages; the module follows
their block-32 E8M0 statement for both names.
"""
from __future__ import annotations

import math

import numpy as np

BLOCK = 32
E2M1, E4M3 = "e2m1", "e4m3"
_EMAX = {E2M1: 2, E4M3: 8}
_BITS = {E2M1: 4, E4M3: 8}


def e2m1_value(code: int) -> float:
    """FP4 E2M1 code (0..15) -> its value, from the bit fields."""
    s = (code >> 3) & 1
    e = (code >> 1) & 3
    m = code & 1
    mag = (m / 2.0) if e == 0 else (1.0 + m / 2.0) * 2.0 ** (e - 1)
    return -mag if s else mag


def e4m3_value(code: int) -> float:
    """FP8 E4M3 code (0..255) -> its value (NaN for S.1111.111), from the bit fields."""
    s = (code >> 7) & 1
    e = (code >> 3) & 15
    m = code & 7
    if e == 15 and m == 7:
        return math.nan
    mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -mag if s else mag


def e8m0_value(e: int) -> float:
    """E8M0 scale code (0..255) -> 2^(e - 127) (NaN for 255)."""
    return math.nan if e == 255 else math.ldexp(1.0, e - 127)


def _values(fmt: str) -> np.ndarray:
    dec = e2m1_value if fmt == E2M1 else e4m3_value
    return np.array([dec(c) for c in range(1 << _BITS[fmt])], dtype=np.float64)


def _max_value(fmt: str) -> float:
    v = _values(fmt)
    return float(np.nanmax(v))


def round_to_element(x: float, fmt: str) -> int:
    """The code whose value is nearest to x (ties to the even code, i.e. mantissa bit 0),
    saturated to the largest magnitude; +0 for zero."""
    vals = _values(fmt)
    sign = 1 if (x < 0 or (x == 0 and math.copysign(1.0, x) < 0)) else 0
    a = min(abs(x), _max_value(fmt))
    half = 1 << (_BITS[fmt] - 1)
    pos = [(vals[c], c) for c in range(half) if not math.isnan(vals[c])]
    best = None
    for v, c in pos:
        d = abs(v - a)
        if best is None or d < best[0] or (d == best[0] and (c & 1) == 0):
            best = (d, c)
    code = best[1]
    if code == 0:
        return 0
    return code | (half if sign else 0)


def block_exponent(block: np.ndarray, fmt: str) -> int:
    """X of one block: floor(log2(max |v|)) - emax, clamped to [-127, 127] (-127 if all
    values are zero)."""
    amax = float(np.max(np.abs(block)))
    if amax == 0.0:
        return -127
    x = math.floor(math.log2(amax)) - _EMAX[fmt]
    # log2 of a float can land a hair off an integer boundary: fix with exact ldexp tests
    while math.ldexp(1.0, x + _EMAX[fmt]) > amax:
        x -= 1
    while math.ldexp(1.0, x + _EMAX[fmt] + 1) <= amax:
        x += 1
    return max(-127, min(127, x))


def quantize_mx(V, fmt: str):
    """Rows of V (shape [R, K], K a multiple of 32) -> (codes [R, K] int64, scale codes
    [R, K/32] int64 with scale = 2^(code - 127))."""
    V = np.asarray(V, dtype=np.float64)
    R, K = V.shape
    assert K % BLOCK == 0
    codes = np.zeros((R, K), dtype=np.int64)
    exps = np.zeros((R, K // BLOCK), dtype=np.int64)
    for r in range(R):
        for b in range(K // BLOCK):
            blk = V[r, b * BLOCK:(b + 1) * BLOCK]
            x = block_exponent(blk, fmt)
            exps[r, b] = x + 127
            for j, v in enumerate(blk):
                codes[r, b * BLOCK + j] = round_to_element(math.ldexp(float(v), -x), fmt)
    return codes, exps


def dequant_mx(codes, exps, fmt: str) -> np.ndarray:
    """Decoded values: element value times its block's scale (exact in fp64)."""
    vals = _values(fmt)
    c = np.asarray(codes, dtype=np.int64)
    e = np.asarray(exps, dtype=np.int64)
    scale = np.ldexp(1.0, np.repeat(e, BLOCK, axis=1) - 127)
    return vals[c] * scale


def unpack_e2m1_bytes(w_bytes, N: int, K: int) -> np.ndarray:
    """Canonical weight bytes [N, K/2] (K value k in the low nibble of byte k/2 for even k,
    the high nibble for odd k) -> codes [N, K] int64."""
    b = np.asarray(w_bytes, dtype=np.int64).reshape(N, K // 2)
    out = np.empty((N, K), dtype=np.int64)
    out[:, 0::2] = b & 0xF
    out[:, 1::2] = b >> 4
    return out


def gemm_mx(a_codes, a_exps, w_codes, w_exps) -> np.ndarray:
    """Y[m, n] = sum_k a[m, k] w[n, k] of MXFP8 (E4M3) activations and MXFP4 (E2M1)
    weights, accumulated in fp64.  Also returns sum_k |a w| for a rounding bound."""
    A = dequant_mx(a_codes, a_exps, E4M3)
    W = dequant_mx(w_codes, w_exps, E2M1)
    return A @ W.T, np.abs(A) @ np.abs(W).T
