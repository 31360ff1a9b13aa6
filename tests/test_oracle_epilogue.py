"""Pins of the oracle's fused epilogue (out = act(Yd + bias[n]) + residual[m, n]) against
closed forms and identities that do not restate its formula.

Source: "量化开销对比：各家方案的矩阵乘账本与省账手段" §6.2 (accumulator x scale ->
+ bias -> store) and §6.6 (scale + bias, + residual / activation, fused in one kernel)."""
import math

import numpy as np
import pytest

import oracle
import synth_inputs as si

FP16, BF16 = 0, 1


def enc(x, dtype):
    return oracle.encode(np.asarray(x, dtype=np.float64), dtype)


def dec(b, dtype):
    return oracle.decode(np.asarray(b, dtype=np.uint16), dtype)


@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_identity_epilogue_is_the_gemm(dtype):
    rng = np.random.default_rng(1)
    yd = rng.normal(size=(3, 5)) * 10
    bb = np.abs(yd) * 3
    out, bo, yr = oracle.epilogue(yd, bb, None, None, oracle.ACT_NONE, 3, 5, dtype)
    assert np.array_equal(out, yd) and np.array_equal(bo, bb)
    assert np.array_equal(yr, enc(yd, dtype))


@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_bias_and_residual_shift_exactly(dtype):
    """Small dyadic values: every sum is exact in fp64, so the shift is checkable exactly."""
    M, N = 4, 8
    yd = (np.arange(M * N, dtype=np.float64).reshape(M, N) - 13) / 8
    bias_v = (np.arange(N) - 3) / 4
    res_v = (np.arange(M * N).reshape(M, N) % 5 - 2) / 2
    out, _, _ = oracle.epilogue(yd, np.zeros_like(yd), enc(bias_v, dtype), enc(res_v, dtype),
                                oracle.ACT_NONE, M, N, dtype)
    assert np.array_equal(out, yd + bias_v[None, :] + res_v)


def test_relu_zeroes_negatives_exactly():
    yd = np.array([[-3.5, -0.0, 0.0, 2.25, -1e-30, 7.0]])
    out, _, _ = oracle.epilogue(yd, np.zeros_like(yd), None, None, oracle.ACT_RELU, 1, 6, FP16)
    assert list(out[0]) == [0.0, 0.0, 0.0, 2.25, 0.0, 7.0]


def test_silu_closed_forms():
    xs = np.array([[0.0, 40.0, -40.0, 1.0, -1.0, 2.5, -2.5, 0.125]])
    out, _, _ = oracle.epilogue(xs, np.zeros_like(xs), None, None, oracle.ACT_SILU, 1, 8, FP16)
    o = out[0]
    assert o[0] == 0.0
    assert o[1] == pytest.approx(40.0, rel=1e-15)                 # x sigma(x) -> x
    assert abs(o[2]) < 1e-15 and o[2] < 0                        # -> 0 from below
    # sigma(x) + sigma(-x) = 1  =>  silu(x) - silu(-x) = x
    for a, b, x in ((o[3], o[4], 1.0), (o[5], o[6], 2.5)):
        assert a - b == pytest.approx(x, rel=1e-15)
    # independent form: x sigma(x) = x/2 + (x/2) tanh(x/2) (cancels for large negative x,
    # so the absolute tolerance scales with |x|)
    for x, y in zip(xs[0], o):
        assert y == pytest.approx(x / 2 + x / 2 * math.tanh(x / 2), rel=1e-14,
                                  abs=1e-15 * abs(x) + 1e-300)
    # and the library logistic function
    from scipy.special import expit
    np.testing.assert_allclose(o, xs[0] * expit(xs[0]), rtol=1e-14, atol=0)


def test_silu_bound_constant_covers_the_slope():
    """The bound uses |silu'| <= 1.1: check the slope's range numerically."""
    x = np.linspace(-20, 20, 400001)
    s = 1 / (1 + np.exp(-x))
    d = s * (1 + x * (1 - s))
    assert d.max() < 1.1 and d.min() > -0.1


@pytest.mark.parametrize("act", [oracle.ACT_NONE, oracle.ACT_RELU, oracle.ACT_SILU])
def test_q_equals_z_gives_act_of_bias_plus_residual(act):
    """With q == z the GEMM is exactly 0, so the fused output is act(bias) + residual."""
    M, N, K, g = 2, 128, 256, 128
    c = si.make_case(M, N, K, g, FP16, seed=3)
    c.qweight[:] = 0x55555555
    c.qzeros = np.full_like(c.qzeros, 0x55555555)
    wd = oracle.dequant(c.qweight, c.scales, c.qzeros, N, K, g, FP16)
    yd, bb, _ = oracle.gemm(c.A, wd, M, N, K, FP16)
    assert not yd.any()
    rng = np.random.default_rng(7)
    bias = enc(rng.normal(size=N), FP16)
    res = enc(rng.normal(size=(M, N)), FP16)
    out, _, _ = oracle.epilogue(yd, bb, bias, res, act, M, N, FP16)
    b = dec(bias, FP16)
    from scipy.special import expit
    post = {oracle.ACT_NONE: b, oracle.ACT_RELU: np.maximum(b, 0),
            oracle.ACT_SILU: b * expit(b)}[act]
    np.testing.assert_allclose(out, post[None, :] + dec(res, FP16), rtol=1e-14, atol=1e-15)


def test_bound_adds_bias_and_residual_magnitudes():
    yd = np.array([[1.0, -2.0]])
    bb = np.array([[4.0, 8.0]])
    bias = enc([0.5, -0.25], FP16)
    res = enc([[-1.0, 2.0]], FP16)
    _, bo, _ = oracle.epilogue(yd, bb, bias, res, oracle.ACT_SILU, 1, 2, FP16)
    assert np.array_equal(bo[0], [1.1 * 4.0 + 0.5 + 1.0, 1.1 * 8.0 + 0.25 + 2.0])
