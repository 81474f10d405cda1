"""The FP8 E4M3 codec of the shared input generator, pinned to the format's
definition (OCP 8-bit floating point, E4M3: sign, 4 exponent bits with bias 7,
3 mantissa bits, subnormals at exponent 0, no infinities, S.1111.111 = NaN)."""

import numpy as np

from speculative_decoding_tree_mla_gb300 import workloads as W


def test_known_codes():
    codes = np.array([0x00, 0x01, 0x07, 0x08, 0x38, 0x39, 0x3F, 0x40, 0x7E, 0xB8, 0xC0, 0xFE],
                     dtype=np.uint8)
    want = [0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 1.125, 1.875, 2.0, 448.0, -1.0, -2.0,
            -448.0]
    assert W.fp8_e4m3_decode(codes).tolist() == want


def test_nan_codes():
    assert np.isnan(W.fp8_e4m3_decode(np.array([0x7F, 0xFF], dtype=np.uint8))).all()


def test_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = W.fp8_e4m3_decode(codes)
    back = W.fp8_e4m3_encode(vals)
    # +0 and -0 are distinct codes of the same value
    assert (back == codes).all()


def test_rounding_is_nearest_ties_to_even_and_saturates():
    x = np.array([1.0625, 1.1875, 1.06, 1.07, 500.0, -1e9, 2.0 ** -10, 3 * 2.0 ** -10],
                 dtype=np.float32)
    got = W.fp8_e4m3_decode(W.fp8_e4m3_encode(x)).tolist()
    # 1.0625 is halfway between 1.0 (even code 0x38) and 1.125 (0x39); 1.1875
    # between 1.125 (0x39) and 1.25 (0x3A, even); 2^-10 halfway between 0 and 2^-9
    assert got == [1.0, 1.25, 1.0, 1.125, 448.0, -448.0, 0.0, 2.0 ** -8]


def test_monotone_and_within_half_ulp():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(20000) * 20).astype(np.float32)
    v = W.fp8_e4m3_decode(W.fp8_e4m3_encode(x)).astype(np.float64)
    pos = np.sort(W.fp8_e4m3_decode(np.arange(0x7F, dtype=np.uint8)).astype(np.float64))
    a = np.abs(x.astype(np.float64))
    i = np.clip(np.searchsorted(pos, a), 1, len(pos) - 1)
    gap = pos[i] - pos[i - 1]
    assert (np.abs(np.abs(v) - a) <= gap / 2 + 1e-12).all()
