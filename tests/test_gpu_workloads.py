"""GPU parity on the full-size workloads, in the launch configuration the bench times
(automatic kernel choice): every element of Y of every shape of all five workloads is
checked against the oracle's fp64 product (|Y - Yd| <= 1e-3 * sum_k |A W| + 1 ulp).

The full oracle product of the largest shape (M 4096, K 4096, N 11008: 1.85e11 fp64
multiply-adds) takes tens of seconds on the host's cores; the sampled check stays as a
quick first test of each large shape, so a wrong kernel fails fast with a readable
position before the full comparison runs."""
import pytest
import torch

import synth_inputs as si
from gpu_util import assert_parity_full, assert_parity_sampled, repack_case, run_gemm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_only_int4_tma_gb300 import build
    build.build()


def _cases(name):
    return [pytest.param(p, id=si.shape_tag(p)) for p in si.WORKLOADS[name]]


def _sampled_then_full(p, count):
    c = si.make_case(**p)
    Y = run_gemm(c, repack_case(c))
    assert_parity_sampled(c, Y, count=count)
    assert_parity_full(c, Y)


@pytest.mark.parametrize("p", _cases("tiny_m1_k512_n512_g128"))
def test_tiny(p):
    c = si.make_case(**p)
    assert_parity_full(c, run_gemm(c, repack_case(c)))


@pytest.mark.parametrize("p", _cases("decode_k4096_n4096_n11008"))
def test_decode_sweep_every_element(p):
    c = si.make_case(**p)
    assert_parity_full(c, run_gemm(c, repack_case(c)))


@pytest.mark.parametrize("p", _cases("ffn70b_decode_bf16"))
def test_ffn70b_every_element(p):
    _sampled_then_full(p, 512)


@pytest.mark.parametrize("p", _cases("transition_k8192_n8192"))
def test_transition_every_element(p):
    _sampled_then_full(p, 512)


@pytest.mark.parametrize("p", _cases("prefill_m4096_k4096_n11008"))
def test_prefill_every_element(p):
    _sampled_then_full(p, 1024)
