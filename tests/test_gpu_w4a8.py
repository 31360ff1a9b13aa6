"""GPU parity of the W4A8 (LiquidQuant) path ("W4A8量化计算优化" §2.1-3.2) against the
W4A8 oracle, through the C ABI (include/w4a8.h).

Every result of this path is an exact integer or a fixed sequence of fp32 roundings, so
every comparison is bit for bit:
  * w4a8_dequant_debug: the int8 weights of the congruence, equal to oracle dequant_i8;
  * w4a8_quantize_act: the int8 activations and the fp32 row scales, equal to the
    oracle's per-row quantiser (fp32 division, ties to even);
  * w4a8_gemm: Y equal to RNE_dtype(fp32(exact int sum) * s_a * s_w) of the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from oracle import w4a8 as o8
import weight_only_int4_tma_gb300 as w4

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_only_int4_tma_gb300 import build
    build.build()


def _dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    elif a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a).cuda()


def _status_ok():
    st = w4.w4a16_get_device_status()
    assert st == 0, w4.status_string(st)


def _repack(c):
    nbytes = w4.w4a8_packed_bytes(c.N, c.K)
    assert nbytes > 0
    packed = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    w4.w4a8_repack(_dev(c.qweight), _dev(c.s_u8), _dev(c.a), _dev(c.s_w), c.N, c.K, packed)
    _status_ok()
    return packed


def _quantize(c, A=None):
    A = _dev(c.A) if A is None else A
    A_i8 = torch.empty((c.M, c.K), dtype=torch.int8, device="cuda")
    s_a = torch.empty(c.M, dtype=torch.float32, device="cuda")
    w4.w4a8_quantize_act(A, c.M, c.K, c.dtype, A_i8, s_a)
    return A_i8, s_a


def _gemm(c, packed, A_i8, s_a):
    Y = torch.empty((c.M, c.N), dtype=torch.int16, device="cuda")
    w4.w4a8_gemm(A_i8, s_a, packed, c.M, c.N, c.K, c.dtype, Y)
    _status_ok()
    return Y.cpu().numpy().view(np.uint16)


def _oracle_act(c):
    A32 = oracle.decode(c.A, c.dtype).astype(np.float32)
    return o8.quantize_activations(A32)


def _oracle_y(c, A_i8, s_a, n0=0, n1=None):
    """Expected Y bits for output channels n0..n1 (all rows)."""
    n1 = c.N if n1 is None else n1
    qw = np.ascontiguousarray(c.qweight[n0:n1])
    y = o8.gemm_codes(A_i8, s_a, qw, c.s_u8[n0:n1], c.a[n0:n1], c.s_w[n0:n1], n1 - n0, c.K)
    return oracle.encode(y.astype(np.float64), c.dtype)


def _assert_bits(got, want, what):
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        m, n = bad[0]
        raise AssertionError(f"{what}: {len(bad)} of {got.size} differ; first at (m={m}, n={n}) "
                             f"gpu=0x{int(got[m, n]):04x} oracle=0x{int(want[m, n]):04x}")


DEQUANT_SHAPES = [(32, 128), (40, 256), (200, 512), (4096, 1024), (1000, 4096)]


@pytest.mark.parametrize("N,K", DEQUANT_SHAPES, ids=[f"n{n}_k{k}" for n, k in DEQUANT_SHAPES])
def test_dequant_debug_bitexact(N, K):
    c = si.make_w4a8_case(1, N, K, seed=N + K)
    packed = _repack(c)
    W = torch.empty((N, K), dtype=torch.int8, device="cuda")
    w4.w4a8_dequant_debug(packed, N, K, W)
    _status_ok()
    q = oracle.unpack_q(c.qweight, N, K).astype(np.int64)
    want = o8.dequant_i8(q, c.s_u8, c.a)
    got = W.cpu().numpy().astype(np.int64)
    assert np.array_equal(got, want), int(np.count_nonzero(got != want))


def test_dequant_debug_quantiser_output():
    """Codes produced by the page's two-level quantiser (steps from 1 to 16, offsets that
    put the largest code right at 127) decode to exactly the quantiser's int8 values."""
    rng = np.random.default_rng(5)
    N, K = 96, 1024
    W = rng.standard_normal((N, K))
    W[:, rng.choice(K, 8, replace=False)] *= 12.0
    Q, s_w = o8.quantize_weights_int8(W)
    q, s, a = o8.quantize_groups_u4(Q)
    words = np.zeros((N, K // 8), dtype=np.uint32)
    for j in range(8):
        words |= (q[:, j::8].astype(np.uint32) << np.uint32(4 * j))
    c = si.W4A8Case(1, N, K, si.FP16, np.zeros((1, K), np.uint16), words, s.astype(np.uint8),
                    a.astype(np.uint8), s_w)
    packed = _repack(c)
    Wd = torch.empty((N, K), dtype=torch.int8, device="cuda")
    w4.w4a8_dequant_debug(packed, N, K, Wd)
    _status_ok()
    assert np.array_equal(Wd.cpu().numpy().astype(np.int64), o8.dequant_i8(q, s, a))


@pytest.mark.parametrize("dtype", [si.FP16, si.BF16], ids=["fp16", "bf16"])
@pytest.mark.parametrize("M,K", [(1, 128), (3, 4096), (16, 8192), (37, 28672), (2, 40960)])
def test_quantize_act_bitexact(M, K, dtype):
    c = si.make_w4a8_case(M, 32, K, dtype=dtype, seed=7 * M + K,
                          zero_rows=(1,) if M > 1 else ())
    A_i8, s_a = _quantize(c)
    _status_ok()
    want_q, want_s = _oracle_act(c)
    got_s = s_a.cpu().numpy()
    assert np.array_equal(got_s.view(np.uint32), want_s.view(np.uint32))
    assert np.array_equal(A_i8.cpu().numpy().astype(np.int64), want_q)


def test_quantize_act_outlier_columns_and_ties():
    """bf16 activations with 0.1 % of the columns scaled x20 (the 70B decode workload's
    outliers), and rows whose values sit exactly on .5 steps (ties go to even)."""
    M, K = 4, 8192
    c = si.make_w4a8_case(M, 32, K, dtype=si.BF16, seed=3)
    A = oracle.decode(c.A, si.BF16)
    cols = np.random.default_rng(3).choice(K, 8, replace=False)
    A[:, cols] *= 20.0
    # row 3: amax 127 and values k + 0.5 -> the quotient is exact, rint decides the tie
    A[3] = 0.0
    A[3, 0] = 127.0
    A[3, 1:64] = np.arange(63) + 0.5
    bits = si.to_dtype_bits(A, si.BF16)
    c.A = bits
    A_i8, s_a = _quantize(c)
    _status_ok()
    want_q, want_s = _oracle_act(c)
    assert np.array_equal(s_a.cpu().numpy().view(np.uint32), want_s.view(np.uint32))
    assert np.array_equal(A_i8.cpu().numpy().astype(np.int64), want_q)


GEMM_SHAPES = [
    # (M, N, K, dtype)
    (1, 32, 128, si.FP16), (2, 40, 256, si.FP16), (3, 200, 512, si.BF16),
    (4, 512, 1024, si.FP16), (5, 264, 2048, si.BF16), (8, 1024, 4096, si.FP16),
    (13, 96, 1152, si.BF16), (16, 4096, 4096, si.FP16), (16, 11008, 4096, si.FP16),
    (1, 11008, 4096, si.FP16), (7, 8200, 384, si.BF16),
]


@pytest.mark.parametrize("M,N,K,dtype", GEMM_SHAPES,
                         ids=[f"m{m}_n{n}_k{k}_{si.DTYPE_NAMES[d]}" for m, n, k, d in GEMM_SHAPES])
def test_gemm_every_element_bitexact(M, N, K, dtype):
    c = si.make_w4a8_case(M, N, K, dtype=dtype, seed=M * 1000 + N + K,
                          zero_rows=(M - 1,) if M > 2 else ())
    packed = _repack(c)
    A_i8, s_a = _quantize(c)
    Y = _gemm(c, packed, A_i8, s_a)
    qa, sa = _oracle_act(c)
    _assert_bits(Y, _oracle_y(c, qa, sa), "Y")


@pytest.mark.parametrize("M", [2, 16], ids=["dp4a_m2", "mma_m16"])
def test_gemm_extreme_codes(M):
    """Every group at its extremes: steps 16 with codes 15 (int8 127) and steps 1 with
    code 0 and offset 0 (int8 -128), against activations of +-127: the largest products
    the format allows, summed over K = 28672 (|sum| close to 2^29; on the tensor-core path
    each 128-K block's fp32 partial reaches 128 * 127 * 128, its largest exact case)."""
    N, K = 64, 28672
    G = K // 128
    qweight = np.full((N, K // 8), 0xFFFFFFFF, dtype=np.uint32)
    qweight[N // 2:] = 0
    s_u8 = np.full((N, G), 16, np.uint8)
    s_u8[N // 2:] = 1
    a = np.full((N, G), 15, np.uint8)   # 15 * 16 + 15 = 255 -> int8 127
    a[N // 2:] = 0                      # 0 * 1 + 0 = 0 -> int8 -128
    A = np.ones((M, K))
    A[1::2, ::2] = -1.0
    c = si.W4A8Case(M, N, K, si.FP16, si.to_dtype_bits(A, si.FP16), qweight, s_u8, a,
                    np.full(N, 1e-5, np.float32))
    packed = _repack(c)
    A_i8, s_a = _quantize(c)
    Y = _gemm(c, packed, A_i8, s_a)
    qa, sa = _oracle_act(c)
    _assert_bits(Y, _oracle_y(c, qa, sa), "Y")


@pytest.mark.parametrize("p", si.W4A8_WORKLOADS["w4a8_ffn70b_decode_bf16"],
                         ids=[si.w4a8_shape_tag(p) for p in
                              si.W4A8_WORKLOADS["w4a8_ffn70b_decode_bf16"]])
def test_gemm_ffn70b_workload(p):
    """The shapes the bench times (70B-shaped decode FFN, bf16 activations with 0.1 %
    outlier columns x20, M 1, 8, 16), through the same calls.  All rows of four stripes
    of output channels -- the first and last, and two that cross 16- and 32-channel CTA
    boundaries -- are compared bit for bit; the oracle's int64 product of the whole
    matrix would take minutes on the host."""
    c = si.make_w4a8_case(**p)
    N = c.N
    packed = _repack(c)
    A_i8, s_a = _quantize(c)
    Y = _gemm(c, packed, A_i8, s_a)
    qa, sa = _oracle_act(c)
    assert np.array_equal(A_i8.cpu().numpy().astype(np.int64), qa)
    for n0, n1 in [(0, 96), (N // 2 - 40, N // 2 + 56), (N // 3 - 8, N // 3 + 24), (N - 96, N)]:
        _assert_bits(Y[:, n0:n1], _oracle_y(c, qa, sa, n0, n1), f"Y[:, {n0}:{n1}]")


def test_gemm_twice_in_a_row_and_header_check():
    """Two launches back to back give identical bits; a blob repacked for another K is
    refused by the kernel's header check (W4A16_ERR_FORMAT, Y untouched)."""
    c = si.make_w4a8_case(4, 256, 1024, seed=9)
    packed = _repack(c)
    A_i8, s_a = _quantize(c)
    Y1 = _gemm(c, packed, A_i8, s_a)
    Y2 = _gemm(c, packed, A_i8, s_a)
    assert np.array_equal(Y1, Y2)
    Y = torch.full((c.M, c.N), 0x1234, dtype=torch.int16, device="cuda")
    w4.w4a8_gemm(A_i8, s_a, packed, c.M, c.N, 896, c.dtype, Y)
    assert w4.w4a16_get_device_status() == w4.W4A16_ERR_FORMAT
    assert bool((Y == 0x1234).all())


def test_repack_flags_codes_outside_a_byte():
    """An offset that pushes code 15 past 255 breaks the format's precondition: the repack
    records W4A16_ERR_INVALID_ARG in the device status word."""
    c = si.make_w4a8_case(1, 32, 128, seed=1)
    c.s_u8[:] = 16
    c.a[0, 0] = 100  # 15 * 16 + 100 > 255
    c.qweight[0, 0] = 0xF
    nbytes = w4.w4a8_packed_bytes(c.N, c.K)
    packed = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    w4.w4a8_repack(_dev(c.qweight), _dev(c.s_u8), _dev(c.a), _dev(c.s_w), c.N, c.K, packed)
    assert w4.w4a16_get_device_status() == w4.W4A16_ERR_INVALID_ARG


def _random_configs(n=40, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        M = int(rng.integers(1, 17))
        N = int(rng.integers(1, 400)) * 8
        K = int(rng.integers(1, 49)) * 128
        dt = int(rng.integers(0, 2))
        zero = (int(rng.integers(0, M)),) if M > 1 and rng.random() < 0.3 else ()
        steps = (1, int(rng.integers(1, 17)))
        out.append((M, N, K, dt, zero, steps, int(rng.integers(0, 1 << 30))))
    return out


@pytest.mark.parametrize("M,N,K,dt,zero,steps,seed", _random_configs(),
                         ids=[f"m{m}_n{n}_k{k}_{si.DTYPE_NAMES[d]}" for m, n, k, d, *_ in
                              _random_configs()])
def test_gemm_random_configs_bitexact(M, N, K, dt, zero, steps, seed):
    """Seeded random shapes (M 1..16, ragged N, K up to 6144), both dtypes, optional
    all-zero rows and narrower step ranges: every element bit for bit."""
    c = si.make_w4a8_case(M, N, K, dtype=dt, seed=seed, zero_rows=zero, steps=steps)
    packed = _repack(c)
    A_i8, s_a = _quantize(c)
    Y = _gemm(c, packed, A_i8, s_a)
    qa, sa = _oracle_act(c)
    assert np.array_equal(A_i8.cpu().numpy().astype(np.int64), qa)
    _assert_bits(Y, _oracle_y(c, qa, sa), "Y")
