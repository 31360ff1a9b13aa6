"""Python binding of the W4A16 GB300 library (libw4a16.so, C ABI in include/w4a16.h).

The functions here carry the C entry points' names and only marshal arguments: torch
CUDA tensors (or raw integer device addresses) become pointers, the current torch
stream becomes the cudaStream_t.  Every step of the computation runs in the library's
CUDA kernels.  There is no fallback: if the shared library is missing, importing the
binding's functions raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libw4a16.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "w4a16.h")
HEADERS = [HEADER, os.path.join(os.path.dirname(HERE), "include", "w4a8.h"),
           os.path.join(os.path.dirname(HERE), "include", "mxfp.h")]

W4A16_OK = 0
W4A16_ERR_INVALID_ARG = -1
W4A16_ERR_UNSUPPORTED = -2
W4A16_ERR_CUDA = -3
W4A16_ERR_DEVICE_TIMEOUT = -4
W4A16_ERR_FORMAT = -5

W4A16_FP16 = 0
W4A16_BF16 = 1

W4A16_KERNEL_AUTO = 0
W4A16_KERNEL_TC = 1
W4A16_KERNEL_SIMT = 2

W4A16_ACT_NONE = 0
W4A16_ACT_RELU = 1
W4A16_ACT_SILU = 2

W4A16_GEMM_NO_PDL = 1
W4A16_GEMM_NO_WEIGHT_PREFETCH = 2
W4A16_GEMM_DEQUANT_LUT = 4
W4A16_GEMM_DEQUANT_INT = 8

_lock = threading.Lock()
_lib = None


class W4A16Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


class GemmConfig(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int), ("split_k", ctypes.c_int), ("tile_m", ctypes.c_int),
                ("stages", ctypes.c_int), ("flags", ctypes.c_int),
                ("reserved", ctypes.c_int * 3)]


def lib() -> ctypes.CDLL:
    """Loads libw4a16.so (built by weight_only_int4_tma_gb300.build)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: run weight_only_int4_tma_gb300.build "
                                   "(or __graft_entry__.build()) first")
            L = ctypes.CDLL(LIB_PATH)
            P, I, U, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint, ctypes.c_size_t
            L.w4a16_abi_version.restype = I
            L.w4a16_status_string.argtypes = [I]
            L.w4a16_status_string.restype = ctypes.c_char_p
            L.w4a16_packed_bytes.argtypes = [I, I, I, I, I]
            L.w4a16_packed_bytes.restype = Z
            L.w4a16_repack.argtypes = [P, P, P, P, I, I, I, I, P, Z, P]
            L.w4a16_repack.restype = I
            L.w4a16_gemm.argtypes = [P, P, I, I, I, I, I, P, P]
            L.w4a16_gemm.restype = I
            L.w4a16_gemm_ex.argtypes = [P, P, I, I, I, I, I, P, ctypes.POINTER(GemmConfig), P]
            L.w4a16_gemm_ex.restype = I
            L.w4a16_gemm_epilogue.argtypes = [P, P, I, I, I, I, I, P, P, I, P,
                                              ctypes.POINTER(GemmConfig), P]
            L.w4a16_gemm_epilogue.restype = I
            L.w4a16_gemm_plan.argtypes = [I, I, I, I, I, ctypes.POINTER(GemmConfig),
                                          ctypes.POINTER(GemmConfig)]
            L.w4a16_gemm_plan.restype = I
            L.w4a16_dequant_debug.argtypes = [P, I, I, I, I, P, P]
            L.w4a16_dequant_debug.restype = I
            L.w4a16_get_device_status.argtypes = [P]
            L.w4a16_get_device_status.restype = I
            L.w4a16_debug_timeout_probe.argtypes = [U, P]
            L.w4a16_debug_timeout_probe.restype = I
            L.w4a16_debug_splitk_timeout_probe.argtypes = [P, P, I, I, I, I, I, P, U, P]
            L.w4a16_debug_splitk_timeout_probe.restype = I
            L.w4a8_packed_bytes.argtypes = [I, I]
            L.w4a8_packed_bytes.restype = Z
            L.w4a8_repack.argtypes = [P, P, P, P, I, I, P, Z, P]
            L.w4a8_repack.restype = I
            L.w4a8_quantize_act.argtypes = [P, I, I, I, P, P, P]
            L.w4a8_quantize_act.restype = I
            L.w4a8_gemm.argtypes = [P, P, P, I, I, I, I, P, P]
            L.w4a8_gemm.restype = I
            L.w4a8_dequant_debug.argtypes = [P, I, I, P, P]
            L.w4a8_dequant_debug.restype = I
            L.mx_packed_bytes.argtypes = [I, I]
            L.mx_packed_bytes.restype = Z
            L.mx_repack.argtypes = [P, P, I, I, P, Z, P]
            L.mx_repack.restype = I
            L.mx_gemm.argtypes = [P, P, P, I, I, I, I, P, P]
            L.mx_gemm.restype = I
            _lib = L
    return _lib


def header_functions() -> list[str]:
    """Names of the functions the public headers (include/w4a16.h, w4a8.h, mxfp.h) declare."""
    names = set()
    for h in HEADERS:
        src = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names.update(re.findall(r"\b((?:w4a16|w4a8|mx)_[a-z_0-9]+)\s*\(", src))
    return sorted(names)


def status_string(status: int) -> str:
    return lib().w4a16_status_string(int(status)).decode()


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, where: str) -> int:
    if rc != W4A16_OK:
        raise W4A16Error(rc, where)
    return rc


def w4a16_abi_version() -> int:
    return lib().w4a16_abi_version()


def w4a16_packed_bytes(N: int, K: int, group: int, has_zeros: bool,
                       has_channel_scale: bool = False) -> int:
    return int(lib().w4a16_packed_bytes(N, K, group, int(bool(has_zeros)),
                                        int(bool(has_channel_scale))))


def w4a16_repack(qweight, scales, qzeros, channel_scale, N: int, K: int, group: int,
                 dtype: int, packed, packed_bytes: int | None = None, stream=None) -> None:
    if packed_bytes is None:
        packed_bytes = packed.numel() * packed.element_size()
    _check(lib().w4a16_repack(_ptr(qweight), _ptr(scales), _ptr(qzeros), _ptr(channel_scale),
                              N, K, group, dtype, _ptr(packed), packed_bytes, _stream(stream)),
           "w4a16_repack")


def w4a16_gemm(A, packed, M: int, N: int, K: int, group: int, dtype: int, Y,
               stream=None) -> None:
    _check(lib().w4a16_gemm(_ptr(A), _ptr(packed), M, N, K, group, dtype, _ptr(Y),
                            _stream(stream)), "w4a16_gemm")


def w4a16_gemm_ex(A, packed, M: int, N: int, K: int, group: int, dtype: int, Y, *,
                  kernel: int = W4A16_KERNEL_AUTO, split_k: int = 0, tile_m: int = 0,
                  stages: int = 0, flags: int = 0, stream=None) -> None:
    cfg = GemmConfig(kernel, split_k, tile_m, stages, flags)
    _check(lib().w4a16_gemm_ex(_ptr(A), _ptr(packed), M, N, K, group, dtype, _ptr(Y),
                               ctypes.byref(cfg), _stream(stream)), "w4a16_gemm_ex")


def w4a16_gemm_epilogue(A, packed, M: int, N: int, K: int, group: int, dtype: int, bias,
                        residual, act: int, Y, *, kernel: int = W4A16_KERNEL_AUTO,
                        split_k: int = 0, tile_m: int = 0, stages: int = 0, flags: int = 0,
                        stream=None) -> None:
    cfg = GemmConfig(kernel, split_k, tile_m, stages, flags)
    _check(lib().w4a16_gemm_epilogue(_ptr(A), _ptr(packed), M, N, K, group, dtype, _ptr(bias),
                                     _ptr(residual), act, _ptr(Y), ctypes.byref(cfg),
                                     _stream(stream)), "w4a16_gemm_epilogue")


def w4a16_gemm_plan(M: int, N: int, K: int, group: int, dtype: int, *,
                    kernel: int = W4A16_KERNEL_AUTO, split_k: int = 0, tile_m: int = 0,
                    stages: int = 0, flags: int = 0) -> dict:
    """The resolved launch choice of w4a16_gemm_ex for these arguments (no launch)."""
    cfg = GemmConfig(kernel, split_k, tile_m, stages, flags)
    out = GemmConfig()
    _check(lib().w4a16_gemm_plan(M, N, K, group, dtype, ctypes.byref(cfg), ctypes.byref(out)),
           "w4a16_gemm_plan")
    return {"kernel": out.kernel, "split_k": out.split_k, "tile_m": out.tile_m,
            "stages": out.stages, "w_stages": out.reserved[0], "groups": out.reserved[1],
            "whole_blocks": bool(out.reserved[2]), "flags": out.flags}


def w4a16_dequant_debug(packed, N: int, K: int, group: int, dtype: int, W_out,
                        stream=None) -> None:
    _check(lib().w4a16_dequant_debug(_ptr(packed), N, K, group, dtype, _ptr(W_out),
                                     _stream(stream)), "w4a16_dequant_debug")


def w4a16_get_device_status(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device status word."""
    return int(lib().w4a16_get_device_status(_stream(stream)))


def w4a16_debug_timeout_probe(timeout_us: int, stream=None) -> None:
    _check(lib().w4a16_debug_timeout_probe(timeout_us, _stream(stream)),
           "w4a16_debug_timeout_probe")


def w4a16_debug_splitk_timeout_probe(A, packed, M: int, N: int, K: int, group: int,
                                     dtype: int, Y, timeout_us: int, stream=None) -> None:
    _check(lib().w4a16_debug_splitk_timeout_probe(_ptr(A), _ptr(packed), M, N, K, group, dtype,
                                                  _ptr(Y), timeout_us, _stream(stream)),
           "w4a16_debug_splitk_timeout_probe")


def w4a8_packed_bytes(N: int, K: int) -> int:
    return int(lib().w4a8_packed_bytes(N, K))


def w4a8_repack(qweight, s_u8, a, s_w, N: int, K: int, packed, packed_bytes: int | None = None,
                stream=None) -> None:
    if packed_bytes is None:
        packed_bytes = packed.numel() * packed.element_size()
    _check(lib().w4a8_repack(_ptr(qweight), _ptr(s_u8), _ptr(a), _ptr(s_w), N, K, _ptr(packed),
                             packed_bytes, _stream(stream)), "w4a8_repack")


def w4a8_quantize_act(A, M: int, K: int, dtype: int, A_i8, s_a, stream=None) -> None:
    _check(lib().w4a8_quantize_act(_ptr(A), M, K, dtype, _ptr(A_i8), _ptr(s_a),
                                   _stream(stream)), "w4a8_quantize_act")


def w4a8_gemm(A_i8, s_a, packed, M: int, N: int, K: int, dtype: int, Y, stream=None) -> None:
    _check(lib().w4a8_gemm(_ptr(A_i8), _ptr(s_a), _ptr(packed), M, N, K, dtype, _ptr(Y),
                           _stream(stream)), "w4a8_gemm")


def w4a8_dequant_debug(packed, N: int, K: int, W_out, stream=None) -> None:
    _check(lib().w4a8_dequant_debug(_ptr(packed), N, K, _ptr(W_out), _stream(stream)),
           "w4a8_dequant_debug")


def mx_packed_bytes(N: int, K: int) -> int:
    return int(lib().mx_packed_bytes(N, K))


def mx_repack(w_codes, w_scales, N: int, K: int, packed, packed_bytes: int | None = None,
              stream=None) -> None:
    if packed_bytes is None:
        packed_bytes = packed.numel() * packed.element_size()
    _check(lib().mx_repack(_ptr(w_codes), _ptr(w_scales), N, K, _ptr(packed), packed_bytes,
                           _stream(stream)), "mx_repack")


def mx_gemm(a_codes, a_scales, packed, M: int, N: int, K: int, dtype: int, Y,
            stream=None) -> None:
    _check(lib().mx_gemm(_ptr(a_codes), _ptr(a_scales), _ptr(packed), M, N, K, dtype, _ptr(Y),
                         _stream(stream)), "mx_gemm")


# ---- torch-friendly helpers (allocation + the calls above) ---------------------------

def repack(qweight, scales, qzeros, N: int, K: int, group: int, dtype: int,
           channel_scale=None, stream=None):
    """Allocates the packed blob on qweight's device and fills it; returns a uint8 tensor."""
    import torch
    nbytes = w4a16_packed_bytes(N, K, group, qzeros is not None, channel_scale is not None)
    if nbytes == 0:
        raise W4A16Error(W4A16_ERR_UNSUPPORTED, "w4a16_packed_bytes")
    packed = torch.empty(nbytes, dtype=torch.uint8, device=qweight.device)
    w4a16_repack(qweight, scales, qzeros, channel_scale, N, K, group, dtype, packed, nbytes,
                 stream)
    return packed


def gemm(A, packed, N: int, K: int, group: int, dtype: int, out=None, stream=None, **ex):
    """Y = A . W^T for a 2-D A on the GPU; returns Y (allocated unless `out` is given)."""
    import torch
    M = A.shape[0]
    Y = out if out is not None else torch.empty((M, N), dtype=A.dtype, device=A.device)
    if ex:
        w4a16_gemm_ex(A, packed, M, N, K, group, dtype, Y, stream=stream, **ex)
    else:
        w4a16_gemm(A, packed, M, N, K, group, dtype, Y, stream)
    return Y
