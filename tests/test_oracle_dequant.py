"""Pins for the oracle's unpack and dequant.

Unpack: hand-built words with one known nibble, brute force over every nibble value and
position, and a round trip through a packer written here in plain Python loops.
Dequant: q == z gives exactly zero; brute force over all (q, z) in 16 x 16 against the
libraries' own single rounding of the exact product; the group index is k // g.
"""
import os

import numpy as np
import pytest
import torch

import synth_inputs as si

FP16, BF16 = 0, 1
HERE = os.path.dirname(os.path.abspath(__file__))


def _pack_rows(q):
    """Plain packer: nibble j of word w holds column 8w + j."""
    R, C = q.shape
    out = np.zeros((R, C // 8), dtype=np.uint32)
    for r in range(R):
        for w in range(C // 8):
            v = 0
            for j in range(8):
                v |= int(q[r, 8 * w + j]) << (4 * j)
            out[r, w] = v
    return out


def _lib_round(x, dtype):
    """Single RNE of an exactly representable fp64/fp32 value, by numpy or torch."""
    if dtype == FP16:
        return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)
    t = torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_unpack_known_words(orc):
    qw = np.array([[0x76543210, 0xFEDCBA98]], dtype=np.uint32)
    q = orc.unpack_q(qw, 1, 16)
    assert q.tolist() == [list(range(16))]


def test_unpack_every_value_every_position(orc):
    for v in range(16):
        for j in range(8):
            qw = np.array([[v << (4 * j)]], dtype=np.uint32)
            q = orc.unpack_q(qw, 1, 8)[0]
            want = [0] * 8
            want[j] = v
            assert q.tolist() == want


def test_pack_unpack_roundtrip(orc):
    rng = np.random.default_rng(5)
    q = rng.integers(0, 16, size=(24, 64), dtype=np.uint8)
    assert np.array_equal(orc.unpack_q(_pack_rows(q), 24, 64), q)
    z = rng.integers(0, 16, size=(3, 40), dtype=np.uint8)
    assert np.array_equal(orc.unpack_z(_pack_rows(z), 3, 40), z)


def test_symmetric_zero_is_8(orc):
    z = orc.unpack_z(None, 2, 16)
    assert (z == 8).all()


def test_magic_bias_golden(orc):
    """The page's exponent-injection trick, read from the golden fixture."""
    rows = [ln.split() for ln in open(os.path.join(HERE, "golden", "magic_bias.txt"))
            if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 16
    for q, fb, fv, bb, bv in rows:
        q = int(q)
        assert int(fb, 16) == 0x6400 | q
        assert int(bb, 16) == 0x4300 | q
        assert orc.decode(np.array([int(fb, 16)]), FP16)[0] == float(fv) == 1024 + q
        assert orc.decode(np.array([int(bb, 16)]), BF16)[0] == float(bv) == 128 + q
        # independent decoders agree
        assert np.array([int(fb, 16)], np.uint16).view(np.float16)[0] == 1024 + q
        assert (np.array([int(bb, 16) << 16], np.uint32).view(np.float32)[0]) == 128 + q


def test_printed_mask_reading():
    """As printed on the page, x & 0x0F0F0F0F | 0x64006400 would put a second nibble in
    mantissa bits 8..11 of each half, so the per-half mask must be 0x000F000F."""
    x = 0x00000305  # nibbles: q0 = 5, q2 = 3 share the low 16-bit half
    lo_half = ((x & 0x0F0F0F0F) | 0x64006400) & 0xFFFF
    v = np.array([lo_half], np.uint16).view(np.float16)[0]
    assert v == 1024 + 256 * 3 + 5
    lo_half = ((x & 0x000F000F) | 0x64006400) & 0xFFFF
    assert np.array([lo_half], np.uint16).view(np.float16)[0] == 1024 + 5


def test_q_equals_z_gives_zero(orc):
    N, K, g = 16, 64, 32
    rng = np.random.default_rng(1)
    q = rng.integers(0, 16, size=(N, K), dtype=np.uint8)
    G = K // g
    z = np.zeros((G, N), dtype=np.uint8)
    # choose q constant within each (group, row) and equal to that group's zero
    for n in range(N):
        for gi in range(G):
            q[n, gi * g:(gi + 1) * g] = (n + 3 * gi) % 16
            z[gi, n] = (n + 3 * gi) % 16
    for dtype in (FP16, BF16):
        scales = si.to_dtype_bits(rng.uniform(0.005, 0.02, size=(G, N)), dtype)
        wd = orc.dequant(_pack_rows(q), scales, _pack_rows(z), N, K, g, dtype)
        assert (orc.decode(wd, dtype) == 0.0).all()


@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_dequant_bruteforce_all_q_z(orc, dtype):
    # One row per (z, s) combination, K = 16 columns holding q = 0..15 twice over 32.
    rng = np.random.default_rng(11 + dtype)
    svals = np.concatenate([rng.uniform(0.002, 0.02, 6), [1.0, 0.5, 3.75, 1e-3],
                            rng.uniform(-0.05, 0.05, 4)])
    sbits = si.to_dtype_bits(svals, dtype)
    K, g = 32, 32
    rows = []
    zs = []
    ss = []
    for z in range(16):
        for sb in sbits:
            rows.append(np.tile(np.arange(16, dtype=np.uint8), 2))
            zs.append(z)
            ss.append(sb)
    N = len(rows)
    q = np.stack(rows)
    z = np.array(zs, dtype=np.uint8)[None, :]
    s = np.array(ss, dtype=np.uint16)[None, :]
    wd = orc.dequant(_pack_rows(q), s, _pack_rows(z), N, K, g, dtype)
    sd = orc.decode(s[0], dtype)
    exact = (q.astype(np.float64) - z[0][:, None]) * sd[:, None]
    assert np.array_equal(wd, _lib_round(exact, dtype).reshape(N, K))


def test_group_index_is_k_over_g(orc):
    N, K = 8, 256
    for g in (32, 64, 128):
        G = K // g
        q = np.full((N, K), 9, dtype=np.uint8)
        z = np.full((G, N), 8, dtype=np.uint8)          # q - z = 1 everywhere
        s = np.array([[1.0 + gi + n / 16 for n in range(N)] for gi in range(G)])
        wd = orc.dequant(_pack_rows(q), si.to_dtype_bits(s, FP16), _pack_rows(z),
                         N, K, g, FP16)
        got = orc.decode(wd, FP16)
        for k in (0, g - 1, g, K - 1):
            assert np.array_equal(got[:, k], s[k // g])
