"""Pins of the oracle's q8_1 quantisation and MMQ path (CPU only)."""
from fractions import Fraction

import numpy as np
import pytest

from oracle import q4k as O
import synth


def test_integer_block_with_max_127_is_exact():
    rng = np.random.default_rng(1)
    x = rng.integers(-127, 128, (3, 64)).astype(np.float32)
    x[:, 0] = 127.0
    x[:, 40] = -127.0
    q, d8, s = O.quantize_q8_1(x)
    assert np.all(d8 == 1.0)
    assert np.array_equal(q.astype(np.float32), x)
    assert np.array_equal(s, x.reshape(3, 2, 32).sum(axis=2).astype(np.int32))


def test_ties_round_away_from_zero():
    x = np.zeros((1, 32), np.float32)
    x[0, :8] = [127, 2.5, -2.5, 0.5, -0.5, 1.5, -1.5, 126.5]
    q, d8, s = O.quantize_q8_1(x)
    assert d8[0, 0] == 1.0
    assert list(q[0, :8]) == [127, 3, -3, 1, -1, 2, -2, 127]
    assert s[0, 0] == 127 + 3 - 3 + 1 - 1 + 2 - 2 + 127


def test_zero_block_and_tiny_block():
    x = np.zeros((1, 64), np.float32)
    x[0, 32:] = np.float32(1e-44)      # amax/127 underflows to 0 in fp32
    q, d8, s = O.quantize_q8_1(x)
    assert np.all(q == 0) and np.all(d8 == 0) and np.all(s == 0)


def test_quantisation_error_bound_and_extremes():
    x = synth.activations(16, 1024, 21)
    q, d8, s = O.quantize_q8_1(x)
    xb = x.reshape(16, 32, 32).astype(np.float64)
    qb = q.reshape(16, 32, 32).astype(np.float64)
    d = d8.astype(np.float64)[:, :, None]
    # the division is rounded once, so allow a couple of ulps of x/d8
    assert np.all(np.abs(xb - d * qb) <= d * (0.5 + 1e-5))
    assert np.all(np.max(np.abs(qb), axis=2) == 127)    # the extreme maps to 127
    assert np.array_equal(s, qb.sum(axis=2).astype(np.int32))
    amax = np.max(np.abs(xb), axis=2)
    assert np.array_equal(d8, (amax.astype(np.float32) / np.float32(127)))


def test_power_of_two_scaling_invariance():
    x = synth.activations(4, 512, 22)
    q0, d0, s0 = O.quantize_q8_1(x)
    q1, d1, s1 = O.quantize_q8_1(x * np.float32(8.0))
    assert np.array_equal(q0, q1) and np.array_equal(s0, s1)
    assert np.array_equal(d1, d0 * np.float32(8.0))


def test_sign_symmetry():
    x = synth.activations(4, 512, 23)
    q0, d0, s0 = O.quantize_q8_1(x)
    q1, d1, s1 = O.quantize_q8_1(-x)
    assert np.array_equal(q1, -q0) and np.array_equal(d1, d0) and np.array_equal(s1, -s0)


def test_block_dots_brute_force():
    f = synth.q4k_fields(3, 256, 31)
    x = synth.activations(2, 256, 32)
    q8, _, _ = O.quantize_q8_1(x)
    p = O.block_dots(f["q"], q8)
    assert p.shape == (2, 3, 8)
    for t in range(2):
        for o in range(3):
            for b in range(8):
                acc = 0
                for i in range(32):
                    acc += int(f["q"][o, 32 * b + i]) * int(q8[t, 32 * b + i])
                assert p[t, o, b] == acc


def test_block_dot_extremes_fit_int32():
    q4 = np.full((1, 32), 15, np.uint8)
    q8 = np.full((1, 32), -127, np.int8)
    assert O.block_dots(q4, q8)[0, 0, 0] == -15 * 127 * 32


@pytest.mark.parametrize("rows,cols,n", [(5, 256, 3), (17, 768, 4)])
def test_mmq_equals_fp_path_on_dequantised_activations(rows, cols, n):
    f = synth.q4k_fields(rows, cols, rows + cols)
    x = synth.activations(n, cols, rows * cols)
    q8, d8, s = O.quantize_q8_1(x)
    y, norm = O.mmq(f, q8, d8, s)
    xhat = O.dequantize_q8_1(q8, d8)
    w = O.dequantize(f).astype(np.float64)
    y2 = xhat @ w.T
    # the fp path rounds w to fp32 once (2^-24 relative); otherwise equal
    assert np.all(np.abs(y - y2) <= 1e-6 * norm)


def test_mmq_all_zero_quants_leave_the_min_term():
    f = synth.q4k_fields(4, 512, 41)
    f["q"][:] = 0
    x = synth.activations(3, 512, 42)
    q8, d8, s = O.quantize_q8_1(x)
    y, _ = O.mmq(f, q8, d8, s)
    dmin = np.repeat(O.f16_bits_to_f64(f["dmin"]), 8, axis=1)
    dm = dmin * f["m"].astype(np.float64)
    u = d8.astype(np.float64) * s.astype(np.float64)
    np.testing.assert_allclose(y, -(u @ dm.T), rtol=1e-13, atol=1e-15)


def test_mmq_zero_activations():
    f = synth.q4k_fields(4, 256, 43)
    q8, d8, s = O.quantize_q8_1(np.zeros((2, 256), np.float32))
    y, norm = O.mmq(f, q8, d8, s)
    assert np.all(y == 0) and np.all(norm == 0)


def test_mmq_single_superblock_closed_form():
    # d = 1, dmin = 0.5, sc_j = j+1, m_j = 2, q_i = i mod 16; x = 127 for
    # every weight, so d8 = 1, q8 = 127, S = 32*127 per block and
    # y = 127 * 8384 (the fp closed form times 127).
    f = {"d": np.array([[1.0]], np.float16).view(np.uint16),
         "dmin": np.array([[0.5]], np.float16).view(np.uint16),
         "sc": np.arange(1, 9, dtype=np.uint8)[None, :],
         "m": np.full((1, 8), 2, np.uint8),
         "q": (np.arange(256) % 16).astype(np.uint8)[None, :]}
    q8, d8, s = O.quantize_q8_1(np.full((1, 256), 127, np.float32))
    y, _ = O.mmq(f, q8, d8, s)
    assert y[0, 0] == 127 * 8384


def _nearest_f32(v: Fraction) -> np.float32:
    """The float32 nearest to the rational v (ties to even), by exact search."""
    c = np.float32(float(v))
    best = c
    for cand in (np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))):
        dc, db = abs(Fraction(float(cand)) - v), abs(Fraction(float(best)) - v)
        if dc < db or (dc == db and (int(cand.view(np.uint32)) & 1) == 0):
            best = cand
    return best


def test_scale_divides_rather_than_multiplying_by_a_reciprocal():
    # amax = 932.5: d8 is the float32 nearest to 932.5/127.  x1 = 1.5*d8 and
    # x3 = 0.5*d8 are exact float32 values, so x/d8 is exactly 1.5 and 0.5
    # and rounds away from zero to 2 and 1.  Multiplying by the float32
    # reciprocal of d8 instead gives 1.4999999 and 0.49999997 (q = 1 and 0):
    # this block tells the two readings apart.
    d8_exact = _nearest_f32(Fraction(9325, 10) / 127)
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 932.5
    x[0, 1] = np.float32(float(Fraction(3, 2) * Fraction(float(d8_exact))))
    x[0, 2] = -x[0, 1]
    x[0, 3] = np.float32(float(Fraction(1, 2) * Fraction(float(d8_exact))))
    assert Fraction(float(x[0, 1])) == Fraction(3, 2) * Fraction(float(d8_exact))
    assert Fraction(float(x[0, 3])) == Fraction(1, 2) * Fraction(float(d8_exact))
    q, d8, s = O.quantize_q8_1(x)
    assert d8[0, 0] == d8_exact
    assert list(q[0, :4]) == [127, 2, -2, 1]
    assert s[0, 0] == 127 + 2 - 2 + 1
    # the reciprocal reading differs on exactly these elements
    recip = np.float32(1.0) / d8_exact
    assert np.float32(x[0, 1] * recip) < np.float32(1.5)
    assert np.float32(x[0, 3] * recip) < np.float32(0.5)
