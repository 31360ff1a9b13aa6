"""Helpers for the GPU parity tests: move a seeded case to the device, run the library
through its C ABI, and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import weight_only_int4_tma_gb300 as w4


def to_dev(a: np.ndarray | None, device="cuda"):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16))
    elif a.dtype == np.uint32:
        t = torch.from_numpy(a.view(np.int32))
    else:
        t = torch.from_numpy(a)
    return t.to(device)


def to_host_u16(t) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def repack_case(c, device="cuda"):
    qw, sc, qz = to_dev(c.qweight, device), to_dev(c.scales, device), to_dev(c.qzeros, device)
    cs = to_dev(c.cscale, device)
    packed = w4.repack(qw, sc, qz, c.N, c.K, c.group, c.dtype, channel_scale=cs)
    return packed


def run_gemm(c, packed, A_dev=None, **ex):
    A = A_dev if A_dev is not None else to_dev(c.A)
    Y = torch.empty((c.M, c.N), dtype=torch.int16, device=A.device)
    if ex:
        w4.w4a16_gemm_ex(A, packed, c.M, c.N, c.K, c.group, c.dtype, Y, **ex)
    else:
        w4.w4a16_gemm(A, packed, c.M, c.N, c.K, c.group, c.dtype, Y)
    st = w4.w4a16_get_device_status()
    assert st == 0, w4.status_string(st)
    return to_host_u16(Y)


def oracle_full(c):
    wd = oracle.dequant(c.qweight, c.scales, c.qzeros, c.N, c.K, c.group, c.dtype)
    yd, bb, yr = oracle.gemm(c.A, wd, c.M, c.N, c.K, c.dtype, cscale=c.cscale)
    return wd, yd, bb, yr


def assert_parity_full(c, Y):
    _, yd, bb, _ = oracle_full(c)
    bad, first, worst = oracle.check(Y, yd, bb, c.dtype)
    if bad:
        m, n = divmod(first, c.N)
        raise AssertionError(
            f"{bad} of {Y.size} elements outside the bound; first at (m={m}, n={n}): "
            f"gpu={oracle.decode(Y.ravel()[first:first+1], c.dtype)[0]!r} "
            f"ref={yd.ravel()[first]!r} B={bb.ravel()[first]!r}; worst ratio {worst:.3g}")
    return worst


def sample_positions(M, N, count, seed=0):
    rng = np.random.default_rng(seed)
    im = rng.integers(0, M, count)
    inn = rng.integers(0, N, count)
    # always include the corners and the last tile's tail
    im = np.concatenate([im, [0, M - 1, 0, M - 1]])
    inn = np.concatenate([inn, [0, 0, N - 1, N - 1]])
    return im, inn


def assert_parity_sampled(c, Y, count=4096, seed=0):
    im, inn = sample_positions(c.M, c.N, count, seed)
    yd, bb, _ = oracle.gemm_sampled(c.A, c.qweight, c.scales, c.qzeros, c.M, c.N, c.K,
                                    c.group, c.dtype, im, inn, cscale=c.cscale)
    got = Y[im, inn]
    bad, first, worst = oracle.check(got, yd, bb, c.dtype)
    if bad:
        raise AssertionError(f"{bad} of {got.size} sampled elements outside the bound; first "
                             f"at (m={im[first]}, n={inn[first]}) gpu="
                             f"{oracle.decode(got[first:first+1], c.dtype)[0]!r} "
                             f"ref={yd[first]!r}; worst {worst:.3g}")
    return worst
