"""W4A16 oracle -- TEST INFRASTRUCTURE ONLY.

A plain CPU statement (C++17, fp64 accumulation) of what the fused W4A16 dequant-GEMM
computes: unpack -> dequantise with one round-to-nearest-even into the activation
dtype -> fp64 GEMM.  Only ``tests/``, ``__graft_entry__.smoke()`` and the bench's
CPU-baseline leg may import this package.  It shares no code with the CUDA library in
``weight_only_int4_tma_gb300`` and never imports it.

Sources (cited by page title and section):
  * "W4A16 GEMM 算子浅析：INT4 权重反量化的计算流水线", section "计算流水线的核心哲学"
    (W = (W_int4 - Zero) * Scale, FP16 x FP16 -> FP32) and section
    "Marlin 与 CUTLASS 中的寄存器解包黑魔法" (8 nibbles per uint32).
  * "量化开销对比：各家方案的矩阵乘账本与省账手段", §3 (route B), §6.2 (group scale applied
    to the weight operand inside the k loop), §6.4 (group sizes), §6.7 (per-channel scale
    in the epilogue).

Every function here is pinned by ``tests/test_oracle_*.py`` against facts that do not
come from this code: numpy's and torch's own fp16/bf16 conversions, exact rational
arithmetic (``fractions.Fraction``), closed forms and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4a16_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liboracle_w4a16.so")
_lock = threading.Lock()
_lib = None

FP16 = 0
BF16 = 1

# The acceptance bound: |Y - Yd| <= REL_TOL * sum_k |A W| + 1 ulp of the output dtype.
REL_TOL = 1e-3


def build(force: bool = False) -> str:
    """Compile the oracle shared library in place (g++, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f64, u16 = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_uint16
        lib.w4o_num_threads.restype = i32
        lib.w4o_decode.argtypes = [u16, i32]
        lib.w4o_decode.restype = f64
        lib.w4o_encode.argtypes = [f64, i32]
        lib.w4o_encode.restype = u16
        lib.w4o_ulp.argtypes = [u16, i32]
        lib.w4o_ulp.restype = f64
        lib.w4o_decode_array.argtypes = [P, i64, i32, P]
        lib.w4o_encode_array.argtypes = [P, i64, i32, P]
        lib.w4o_unpack_q.argtypes = [P, i32, i32, P]
        lib.w4o_unpack_q.restype = i32
        lib.w4o_unpack_z.argtypes = [P, i32, i32, P]
        lib.w4o_unpack_z.restype = i32
        lib.w4o_dequant.argtypes = [P, P, P, i32, i32, i32, i32, P]
        lib.w4o_dequant.restype = i32
        lib.w4o_gemm.argtypes = [P, P, P, i32, i32, i32, i32, P, P, P]
        lib.w4o_gemm.restype = i32
        lib.w4o_gemm_sampled.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32,
                                         P, P, i64, P, P, P]
        lib.w4o_gemm_sampled.restype = i32
        lib.w4o_gemm_exact_w.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, P, P, P]
        lib.w4o_gemm_exact_w.restype = i32
        lib.w4o_check.argtypes = [P, P, P, i64, i32, f64, P, P]
        lib.w4o_check.restype = i64
        lib.w4o_epilogue.argtypes = [P, P, P, P, i32, i32, i32, i32, P, P, P]
        lib.w4o_epilogue.restype = i32
        _lib = lib
        return lib


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a):
    return np.ascontiguousarray(a, dtype=np.uint16)


def _u32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.uint32)


def num_threads() -> int:
    return int(_load().w4o_num_threads())


# ---- IEEE-754 binary16 / bfloat16 ----------------------------------------------------

def decode(bits, dtype: int) -> np.ndarray:
    """fp16/bf16 bit patterns -> exact float64 values."""
    b = _u16(np.asarray(bits))
    out = np.empty(b.shape, dtype=np.float64)
    _load().w4o_decode_array(_ptr(b), b.size, dtype, _ptr(out))
    return out


def encode(x, dtype: int) -> np.ndarray:
    """float64 -> fp16/bf16 bit patterns, round to nearest, ties to even."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(a.shape, dtype=np.uint16)
    _load().w4o_encode_array(_ptr(a), a.size, dtype, _ptr(out))
    return out


def ulp(bits: int, dtype: int) -> float:
    return float(_load().w4o_ulp(int(bits), dtype))


# ---- unpack / dequant / gemm ---------------------------------------------------------

def unpack_q(qweight: np.ndarray, N: int, K: int) -> np.ndarray:
    qw = _u32(qweight)
    q = np.empty((N, K), dtype=np.uint8)
    rc = _load().w4o_unpack_q(_ptr(qw), N, K, _ptr(q))
    assert rc == 0
    return q


def unpack_z(qzeros, G: int, N: int) -> np.ndarray:
    qz = _u32(qzeros)
    z = np.empty((G, N), dtype=np.uint8)
    rc = _load().w4o_unpack_z(_ptr(qz), G, N, _ptr(z))
    assert rc == 0
    return z


def dequant(qweight, scales, qzeros, N: int, K: int, group: int, dtype: int) -> np.ndarray:
    """Wd[N, K] as dtype bit patterns: RNE((q - z) * s)."""
    qw, sc, qz = _u32(qweight), _u16(scales), _u32(qzeros)
    assert qw.size == N * K // 8 and sc.size == (K // group) * N
    assert qz is None or qz.size == (K // group) * N // 8
    wd = np.empty((N, K), dtype=np.uint16)
    rc = _load().w4o_dequant(_ptr(qw), _ptr(sc), _ptr(qz), N, K, group, dtype, _ptr(wd))
    assert rc == 0, rc
    return wd


def gemm(A, Wd, M: int, N: int, K: int, dtype: int, cscale=None):
    """Returns (Yd fp64 [M,N], Babs fp64 [M,N], Yref dtype bits [M,N])."""
    a, w = _u16(A), _u16(Wd)
    c = None if cscale is None else _u16(cscale)
    assert a.size == M * K and w.size == N * K
    yd = np.empty((M, N), dtype=np.float64)
    bb = np.empty((M, N), dtype=np.float64)
    yr = np.empty((M, N), dtype=np.uint16)
    rc = _load().w4o_gemm(_ptr(a), _ptr(w), _ptr(c), M, N, K, dtype, _ptr(yd), _ptr(bb),
                          _ptr(yr))
    assert rc == 0, rc
    return yd, bb, yr


def gemm_sampled(A, qweight, scales, qzeros, M: int, N: int, K: int, group: int, dtype: int,
                 idx_m, idx_n, cscale=None):
    """(Yd, Babs, Yref) at the listed (m, n) positions, dequantising on the fly."""
    a, qw, sc, qz = _u16(A), _u32(qweight), _u16(scales), _u32(qzeros)
    c = None if cscale is None else _u16(cscale)
    im = np.ascontiguousarray(idx_m, dtype=np.int64)
    inn = np.ascontiguousarray(idx_n, dtype=np.int64)
    cnt = im.size
    yd = np.empty(cnt, dtype=np.float64)
    bb = np.empty(cnt, dtype=np.float64)
    yr = np.empty(cnt, dtype=np.uint16)
    rc = _load().w4o_gemm_sampled(_ptr(a), _ptr(qw), _ptr(sc), _ptr(qz), _ptr(c), M, N, K,
                                  group, dtype, _ptr(im), _ptr(inn), cnt, _ptr(yd), _ptr(bb),
                                  _ptr(yr))
    assert rc == 0, rc
    return yd, bb, yr


def gemm_exact_w(A, qweight, scales, qzeros, M: int, N: int, K: int, group: int, dtype: int,
                 cscale=None):
    """(Yd, Babs, Yref) [M, N] of the product with unrounded weights (q - z) * s: what the
    integer-operand variant computes up to fp32 accumulation."""
    a, qw, sc, qz = _u16(A), _u32(qweight), _u16(scales), _u32(qzeros)
    c = None if cscale is None else _u16(cscale)
    yd = np.empty((M, N), dtype=np.float64)
    bb = np.empty((M, N), dtype=np.float64)
    yr = np.empty((M, N), dtype=np.uint16)
    rc = _load().w4o_gemm_exact_w(_ptr(a), _ptr(qw), _ptr(sc), _ptr(qz), _ptr(c), M, N, K,
                                  group, dtype, _ptr(yd), _ptr(bb), _ptr(yr))
    assert rc == 0, rc
    return yd, bb, yr


ACT_NONE, ACT_RELU, ACT_SILU = 0, 1, 2


def epilogue(Yd, Babs, bias, residual, act: int, M: int, N: int, dtype: int):
    """Fused epilogue on the GEMM's fp64 result: out = act(Yd + bias[n]) + residual[m, n].
    Returns (out fp64 [M,N], magnitude bound fp64 [M,N], RNE dtype bits [M,N])."""
    yd = np.ascontiguousarray(Yd, dtype=np.float64).reshape(M, N)
    bb = np.ascontiguousarray(Babs, dtype=np.float64).reshape(M, N)
    b = None if bias is None else _u16(bias)
    r = None if residual is None else _u16(residual)
    assert b is None or b.size == N
    assert r is None or r.size == M * N
    out = np.empty((M, N), dtype=np.float64)
    bo = np.empty((M, N), dtype=np.float64)
    yr = np.empty((M, N), dtype=np.uint16)
    rc = _load().w4o_epilogue(_ptr(yd), _ptr(bb), _ptr(b), _ptr(r), act, M, N, dtype,
                              _ptr(out), _ptr(bo), _ptr(yr))
    assert rc == 0, rc
    return out, bo, yr


def check(Y_bits, Yd, Babs, dtype: int, rel_tol: float = REL_TOL):
    """Returns (n_bad, first_bad_flat_index, worst_ratio) for |Y-Yd| <= tol*B + ulp."""
    y = _u16(Y_bits).ravel()
    yd = np.ascontiguousarray(Yd, dtype=np.float64).ravel()
    bb = np.ascontiguousarray(Babs, dtype=np.float64).ravel()
    assert y.size == yd.size == bb.size
    first = ctypes.c_int64(-1)
    worst = ctypes.c_double(0.0)
    bad = _load().w4o_check(_ptr(y), _ptr(yd), _ptr(bb), y.size, dtype, rel_tol,
                            ctypes.byref(first), ctypes.byref(worst))
    return int(bad), int(first.value), float(worst.value)
