"""The seeded input generators (CPU): reproducible, and inside each format's domain."""
import numpy as np

import synth_inputs as si


def test_w4a8_offsets_keep_every_code_inside_a_byte():
    c = si.make_w4a8_case(3, 256, 1024, seed=4)
    s = c.s_u8.astype(np.int64)
    a = c.a.astype(np.int64)
    assert s.min() >= 1 and s.max() <= 16
    assert (15 * s + a).max() <= 255  # the format's precondition holds for any code


def test_w4a8_is_reproducible_and_seed_dependent():
    x, y = si.make_w4a8_case(2, 64, 256, seed=5), si.make_w4a8_case(2, 64, 256, seed=5)
    z = si.make_w4a8_case(2, 64, 256, seed=6)
    for f in ("A", "qweight", "s_u8", "a", "s_w"):
        assert np.array_equal(getattr(x, f), getattr(y, f))
    assert not np.array_equal(x.qweight, z.qweight)


def test_w4a8_outlier_columns_and_zero_rows():
    c = si.make_w4a8_case(4, 32, 8192, dtype=si.BF16, seed=2, outlier_frac=0.001,
                          zero_rows=(1,))
    assert not c.A[1].any()
    A = c.A.view(np.uint16).astype(np.uint32) << 16
    vals = np.abs(A.view(np.float32))
    col_max = vals[[0, 2, 3]].max(axis=0)
    assert (col_max > 8).sum() >= 5  # the x20 columns stand out of N(0, 1)


def test_mx_codes_are_never_nan_and_scales_in_range():
    c = si.make_mx_case(16, 64, 4096, seed=1)
    assert not np.isin(c.a_codes, [0x7F, 0xFF]).any()
    assert c.a_codes.min() == 0 and c.a_codes.max() == 254
    assert c.w_scales.min() >= 119 and c.w_scales.max() <= 123
    assert c.a_scales.min() >= 122 and c.a_scales.max() <= 126
    assert c.w_codes.shape == (64, 2048) and c.a_scales.shape == (16, 128)


def test_workload_shapes_fit_their_kernels():
    for p in si.W4A8_WORKLOADS["w4a8_ffn70b_decode_bf16"] + si.MX_WORKLOADS["mx_ffn70b_decode"]:
        assert p["M"] <= 16 and p["K"] % 128 == 0 and p["N"] % 16 == 0
