"""C-ABI library checks that need no GPU: it builds, loads, exports every function the
header declares, and rejects bad arguments on the host before launching anything."""
import ctypes

import pytest

import weight_only_int4_tma_gb300 as w4
from weight_only_int4_tma_gb300 import build as w4build


@pytest.fixture(scope="module")
def L():
    w4build.build()
    return w4.lib()


def test_exports_every_declared_function(L):
    names = w4.header_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), n


def test_abi_version(L):
    assert w4.w4a16_abi_version() == 1


def test_status_strings(L):
    for code in (0, -1, -2, -3, -4, -5):
        assert w4.status_string(code)
    assert w4.status_string(123) == "unknown status"


@pytest.mark.parametrize("N,K,g,z,c", [(512, 512, 128, 1, 0), (4096, 4096, 128, 1, 0),
                                       (8192, 8192, 32, 0, 0), (256, 384, 64, 1, 1)])
def test_packed_bytes_formula(L, N, K, g, z, c):
    want = 128 + K * N // 2 + (K // g) * N * 2 + (K // g) * N // 2 * z + 4 * N * c
    assert w4.w4a16_packed_bytes(N, K, g, z, c) == want


@pytest.mark.parametrize("N,K,g,z,c", [(520, 512, 128, 1, 0), (512, 64, 32, 1, 0),
                                       (264, 4160, 64, 0, 1), (8, 96, 32, 1, 1)])
def test_packed_bytes_padded(L, N, K, g, z, c):
    """Shapes that are not multiples of 128 occupy whole 128 x 128 blocks."""
    Np, Kp = -(-N // 128) * 128, -(-K // 128) * 128
    want = 128 + Kp * Np // 2 + (Kp // g) * Np * 2 + (Kp // g) * Np // 2 * z + 4 * N * c
    assert w4.w4a16_packed_bytes(N, K, g, z, c) == want


@pytest.mark.parametrize("N,K,g", [(100, 512, 128), (512, 500, 128), (512, 512, 16),
                                   (512, 512, 96), (0, 512, 128), (512, 80, 32)])
def test_packed_bytes_unsupported(L, N, K, g):
    assert w4.w4a16_packed_bytes(N, K, g, 1, 0) == 0


def test_repack_rejects_null_and_bad_shapes(L):
    rc = L.w4a16_repack(None, None, None, None, 512, 512, 128, 0, None, 0, None)
    assert rc == w4.W4A16_ERR_INVALID_ARG
    fake = 1 << 20  # never dereferenced: the shape check fails first
    assert L.w4a16_repack(fake, fake, None, None, 500, 512, 128, 0, fake, 1 << 30, None) \
        == w4.W4A16_ERR_UNSUPPORTED
    assert L.w4a16_repack(fake, fake, None, None, 512, 512, 128, 7, fake, 1 << 30, None) \
        == w4.W4A16_ERR_UNSUPPORTED
    # capacity smaller than the blob
    assert L.w4a16_repack(fake, fake, None, None, 512, 512, 128, 0, fake, 100, None) \
        == w4.W4A16_ERR_INVALID_ARG
    # misaligned qweight
    assert L.w4a16_repack(fake + 4, fake, None, None, 512, 512, 128, 0, fake, 1 << 30, None) \
        == w4.W4A16_ERR_INVALID_ARG


def test_gemm_host_validation(L):
    fake = 1 << 20
    # M == 0 is a no-op that succeeds without touching the device
    assert L.w4a16_gemm(None, None, 0, 512, 512, 128, 0, None, None) == w4.W4A16_OK
    assert L.w4a16_gemm(fake, fake, -1, 512, 512, 128, 0, fake, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_gemm(fake, fake, 4, 516, 512, 128, 0, fake, None) == w4.W4A16_ERR_UNSUPPORTED
    assert L.w4a16_gemm(fake, fake, 4, 512, 512, 48, 0, fake, None) == w4.W4A16_ERR_UNSUPPORTED
    assert L.w4a16_gemm(None, fake, 4, 512, 512, 128, 0, fake, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_gemm(fake + 2, fake, 4, 512, 512, 128, 0, fake, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_gemm(fake, fake, 4, 512, 512, 128, 0, fake + 8, None) == w4.W4A16_ERR_INVALID_ARG
    cfg = w4.GemmConfig(0, 0, 0, 0)
    cfg.reserved[0] = 0
    assert L.w4a16_dequant_debug(None, 512, 512, 128, 0, None, None) == w4.W4A16_ERR_INVALID_ARG


def test_timeout_probe_rejects_bad_limits(L):
    assert L.w4a16_debug_timeout_probe(0, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_debug_timeout_probe(2_000_000, None) == w4.W4A16_ERR_INVALID_ARG


# ---- W4A8 (include/w4a8.h) -------------------------------------------------------------

@pytest.mark.parametrize("N,K", [(32, 128), (4096, 4096), (28672, 8192), (40, 256), (8200, 384)])
def test_w4a8_packed_bytes_formula(L, N, K):
    Np = -(-N // 16) * 16
    assert w4.w4a8_packed_bytes(N, K) == 128 + (Np // 16) * (K // 128) * 1056 + 4 * Np


@pytest.mark.parametrize("N,K", [(0, 128), (32, 0), (32, 100), (32, 192), (32, 131072 + 128)])
def test_w4a8_packed_bytes_unsupported(L, N, K):
    assert w4.w4a8_packed_bytes(N, K) == 0


def test_w4a8_host_validation(L):
    fake = 1 << 20
    # repack: nulls, capacity, alignment, shape
    assert L.w4a8_repack(None, fake, fake, fake, 32, 128, fake, 1 << 20, None) \
        == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a8_repack(fake, fake, fake, fake, 32, 128, fake, 100, None) \
        == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a8_repack(fake + 4, fake, fake, fake, 32, 128, fake, 1 << 20, None) \
        == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a8_repack(fake, fake, fake, fake, 32, 192, fake, 1 << 20, None) \
        == w4.W4A16_ERR_UNSUPPORTED
    # quantize: M == 0 is a no-op; dtype, K and alignment are checked first
    assert L.w4a8_quantize_act(None, 0, 128, 0, None, None, None) == w4.W4A16_OK
    assert L.w4a8_quantize_act(fake, 2, 128, 5, fake, fake, None) == w4.W4A16_ERR_UNSUPPORTED
    assert L.w4a8_quantize_act(fake, 2, 100, 0, fake, fake, None) == w4.W4A16_ERR_UNSUPPORTED
    assert L.w4a8_quantize_act(fake + 8, 2, 128, 0, fake, fake, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a8_quantize_act(fake, 2, 128, 0, fake, fake + 2, None) == w4.W4A16_ERR_INVALID_ARG
    # gemm: M range, shape, pointers
    assert L.w4a8_gemm(None, None, None, 0, 32, 128, 0, None, None) == w4.W4A16_OK
    assert L.w4a8_gemm(fake, fake, fake, 17, 32, 128, 0, fake, None) == w4.W4A16_ERR_UNSUPPORTED
    assert L.w4a8_gemm(fake, fake, fake, -1, 32, 128, 0, fake, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a8_gemm(fake, fake, fake, 4, 32, 100, 0, fake, None) == w4.W4A16_ERR_UNSUPPORTED
    assert L.w4a8_gemm(fake, fake, fake, 4, 32, 128, 3, fake, None) == w4.W4A16_ERR_UNSUPPORTED
    assert L.w4a8_gemm(fake + 4, fake, fake, 4, 32, 128, 0, fake, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a8_gemm(fake, fake, fake, 4, 32, 128, 0, fake + 1, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a8_dequant_debug(None, 32, 128, fake, None) == w4.W4A16_ERR_INVALID_ARG


# ---- MX block-scaled decode GEMM (include/mxfp.h) ------------------------------------------

@pytest.mark.parametrize("N,K", [(16, 128), (40, 256), (28672, 8192)])
def test_mx_packed_bytes_formula(L, N, K):
    Np = -(-N // 16) * 16
    assert w4.mx_packed_bytes(N, K) == 128 + (Np // 16) * (K // 128) * 1088


def test_mx_host_validation(L):
    fake = 1 << 20
    assert w4.mx_packed_bytes(16, 100) == 0 and w4.mx_packed_bytes(0, 128) == 0
    assert L.mx_repack(None, fake, 16, 128, fake, 1 << 20, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.mx_repack(fake, fake, 16, 192, fake, 1 << 20, None) == w4.W4A16_ERR_UNSUPPORTED
    assert L.mx_repack(fake, fake, 16, 128, fake, 10, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.mx_gemm(None, None, None, 0, 16, 128, 0, None, None) == w4.W4A16_OK
    assert L.mx_gemm(fake, fake, fake, 17, 16, 128, 0, fake, None) == w4.W4A16_ERR_UNSUPPORTED
    assert L.mx_gemm(fake, fake, fake, 4, 16, 128, 2, fake, None) == w4.W4A16_ERR_UNSUPPORTED
    assert L.mx_gemm(fake + 4, fake, fake, 4, 16, 128, 0, fake, None) == w4.W4A16_ERR_INVALID_ARG
