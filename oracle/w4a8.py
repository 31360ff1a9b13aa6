"""W4A8 (LiquidQuant) oracle -- TEST INFRASTRUCTURE ONLY.

A plain CPU statement (numpy, exact integer arithmetic, fp32 only where the method
rounds) of the W4A8 path of "W4A8量化计算优化：提升LLM推理效率的关键技术", §2.1
("LiquidQuant的数学魔术"): 4-bit weight codes are turned back into int8 by the congruence

    Q_i8 = (Q_u4 * s_u8 + a) XOR 0x80   (mod 256),   a = 128 + min(Q_i8),  s_u8 <= 16,

and multiplied with int8 activations; the group size is 128 (the page's deployment
example, §4.2 "--group-size 128").  Only ``tests/``, ``__graft_entry__.smoke()`` and the
bench's CPU legs may import it; it shares no code with the CUDA library.

Where the page is silent this module takes the plainest reading (each listed in the
design notes):
  * the int8 weights come from a symmetric per-channel quantisation (scale s_w[n] =
    max|W[n, :]| / 127, codes rint(W / s_w) clipped to [-127, 127]);
  * the second level is asymmetric per group of 128: s_u8 = ceil((max - min) / 15) clipped
    to [1, 16], Q_u4 = the nearest code (ties up) to (Q_i8 - min) / s_u8, clipped to
    [0, 15] and to the largest code whose value min + Q_u4 * s_u8 stays <= 127;
  * activations are quantised per row: s_a[m] = max|A[m, :]| / 127 in fp32 (1 for an
    all-zero row), codes rint(A / s_a) in fp32, clipped to [-127, 127];
  * Y[m, n] = fp32(sum_k A_i8 * Q_i8) * s_a[m] * s_w[n], two fp32 multiplies in that
    order, rounded once (to nearest even) to the output dtype.
"""
from __future__ import annotations

import numpy as np

GROUP = 128


def congruence_dequant(q_u4, s_u8, a):
    """The page's identity, computed as written: ((Q_u4 * s_u8 + a) mod 256) XOR 0x80,
    read as a two's-complement byte.  Arrays broadcast."""
    q = np.asarray(q_u4, dtype=np.int64)
    s = np.asarray(s_u8, dtype=np.int64)
    aa = np.asarray(a, dtype=np.int64)
    u = ((q * s + aa) & 0xFF) ^ 0x80
    return np.where(u >= 128, u - 256, u).astype(np.int64)


def quantize_weights_int8(W):
    """First level: symmetric per-channel int8.  W: [N, K] float.  Returns (Q_i8 [N, K]
    int64, s_w [N] float32)."""
    W32 = np.asarray(W, dtype=np.float32)
    amax = np.max(np.abs(W32), axis=1)
    s_w = np.where(amax > 0, amax / np.float32(127.0), np.float32(1.0)).astype(np.float32)
    q = np.rint(W32 / s_w[:, None]).astype(np.int64)
    return np.clip(q, -127, 127), s_w


def quantize_groups_u4(Q_i8, group=GROUP):
    """Second level: per (channel, group of `group` along K) unsigned 4-bit codes with an
    integer step s_u8 <= 16 and a = 128 + min.  Returns (Q_u4 [N, K], s_u8 [N, K/group],
    a [N, K/group]) as int64 arrays."""
    Q = np.asarray(Q_i8, dtype=np.int64)
    N, K = Q.shape
    assert K % group == 0
    G = Q.reshape(N, K // group, group)
    mn = G.min(axis=2)
    mx = G.max(axis=2)
    s = np.clip(-(-(mx - mn) // 15), 1, 16)  # ceil((max - min) / 15), in [1, 16]
    d = G - mn[:, :, None]                      # >= 0
    q = (2 * d + s[:, :, None]) // (2 * s[:, :, None])  # nearest code, ties up
    qmax = np.minimum(15, (127 - mn) // s)      # value min + q * s must stay <= 127
    q = np.clip(q, 0, qmax[:, :, None])
    return q.reshape(N, K), s, mn + 128


def dequant_i8(Q_u4, s_u8, a, group=GROUP):
    """Int8 weights of the codes, by the congruence, groups broadcast along K.
    Returns [N, K] int64."""
    Q = np.asarray(Q_u4, dtype=np.int64)
    N, K = Q.shape
    s = np.repeat(np.asarray(s_u8, dtype=np.int64), group, axis=1)
    aa = np.repeat(np.asarray(a, dtype=np.int64), group, axis=1)
    return congruence_dequant(Q, s, aa)


def quantize_activations(A):
    """Per-row int8 activations.  A: [M, K] values exactly representable in fp32 (fp16 /
    bf16 inputs).  Returns (A_i8 [M, K] int64, s_a [M] float32); every operation in fp32,
    division and rint rounding to nearest even."""
    A32 = np.asarray(A, dtype=np.float32)
    amax = np.max(np.abs(A32), axis=1)
    s_a = np.where(amax > 0, amax / np.float32(127.0), np.float32(1.0)).astype(np.float32)
    q = np.rint(A32 / s_a[:, None]).astype(np.int64)
    return np.clip(q, -127, 127), s_a


def gemm_acc(A_i8, Q_i8):
    """Exact integer products: acc[m, n] = sum_k A_i8[m, k] * Q_i8[n, k] (int64)."""
    return np.asarray(A_i8, dtype=np.int64) @ np.asarray(Q_i8, dtype=np.int64).T


def gemm_f32(acc, s_a, s_w):
    """fp32(acc) * s_a[m] * s_w[n], the two multiplies in that order, in fp32."""
    y = np.asarray(acc).astype(np.float32)  # int -> fp32 rounds to nearest even
    y = (y * np.asarray(s_a, dtype=np.float32)[:, None]).astype(np.float32)
    return (y * np.asarray(s_w, dtype=np.float32)[None, :]).astype(np.float32)


def gemm_codes(A_i8, s_a, qweight, s_u8, a, s_w, N: int, K: int):
    """The whole GEMM from canonical inputs: unpack the codes (the W4A16 oracle's nibble
    unpack: nibble j of word w is k = 8w + j), dequantise by the congruence, multiply
    exactly, scale in fp32.  Returns the fp32 result [M, N] (rounded to the output dtype
    by the caller with ``oracle.encode``)."""
    from . import unpack_q
    q = unpack_q(np.asarray(qweight), N, K).astype(np.int64)
    Q = dequant_i8(q, s_u8, a)
    return gemm_f32(gemm_acc(A_i8, Q), s_a, s_w)
