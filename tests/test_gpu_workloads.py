"""GPU parity on the full-size workloads, in the launch configuration the bench times
(automatic kernel choice).  Decode sweep: every element; larger shapes: a sample of
positions the oracle computes one by one (corners and the last tile included)."""
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


@pytest.mark.parametrize("p", _cases("tiny_m1_k512_n512_g128"))
def test_tiny(p):
    c = si.make_case(**p)
    assert_parity_full(c, run_gemm(c, repack_case(c)))


@pytest.mark.parametrize("p", _cases("decode_k4096_n4096_n11008"))
def test_decode_sweep_every_element(p):
    c = si.make_case(**p)
    assert_parity_full(c, run_gemm(c, repack_case(c)))


@pytest.mark.parametrize("p", _cases("ffn70b_decode_bf16"))
def test_ffn70b_sampled(p):
    c = si.make_case(**p)
    assert_parity_sampled(c, run_gemm(c, repack_case(c)), count=3000)


@pytest.mark.parametrize("p", _cases("transition_k8192_n8192"))
def test_transition_sampled(p):
    c = si.make_case(**p)
    assert_parity_sampled(c, run_gemm(c, repack_case(c)), count=3000)


@pytest.mark.parametrize("p", _cases("prefill_m4096_k4096_n11008"))
def test_prefill_sampled(p):
    c = si.make_case(**p)
    assert_parity_sampled(c, run_gemm(c, repack_case(c)), count=6000)
