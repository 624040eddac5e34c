"""Pins of the oracle's dequantisation and fp (decode GEMV) path (CPU only)."""
from fractions import Fraction

import numpy as np
import pytest

from oracle import q4k as O
import synth


def f16(v):
    return np.array(v, np.float16).view(np.uint16)


def test_single_superblock_closed_form():
    # d = 1, dmin = 0.5, sc_j = j+1, m_j = 2, q_i = i mod 16, x = 1:
    # each sub-block sums (j+1) * 2*(0+..+15) - 32 * 0.5*2 = 240(j+1) - 32,
    # so y = 240 * 36 - 256 = 8384.
    f = {"d": f16([[1.0]]), "dmin": f16([[0.5]]),
         "sc": np.arange(1, 9, dtype=np.uint8)[None, :],
         "m": np.full((1, 8), 2, np.uint8),
         "q": (np.arange(256) % 16).astype(np.uint8)[None, :]}
    y, norm = O.gemv(f, np.ones((1, 256), np.float32))
    assert y[0, 0] == 8384.0
    # |w| = |(j+1) q - 1|: the normaliser is a sum of those.
    expect = sum(abs((i // 32 + 1) * (i % 16) - 1) for i in range(256))
    assert norm[0, 0] == expect


def test_all_zero_quants_give_minus_dmin_m():
    f = synth.q4k_fields(5, 512, 3)
    f["q"][:] = 0
    w = O.dequantize(f)
    dmin = O.f16_bits_to_f64(f["dmin"])
    for o in range(5):
        for k in range(512):
            assert w[o, k] == -np.float32(dmin[o, k // 256]) * np.float32(f["m"][o, k // 32])
    x = synth.activations(2, 512, 4)
    y, _ = O.gemv(f, x)
    xs = x.astype(np.float64).reshape(2, 16, 32).sum(axis=2)        # [b][sub-block]
    dm = np.repeat(dmin, 8, axis=1) * f["m"].astype(np.float64)      # [o][sub-block]
    np.testing.assert_allclose(y, -(xs @ dm.T), rtol=1e-12, atol=1e-12)


def test_one_hot_activation_reads_out_a_column():
    f = synth.q4k_fields(7, 768, 5)
    w = O.dequantize(f)
    for k in (0, 31, 32, 255, 256, 500, 767):
        x = np.zeros((1, 768), np.float32)
        x[0, k] = 1.0
        y, _ = O.gemv(f, x)
        assert np.array_equal(y[0], w[:, k].astype(np.float64))


def test_linearity_in_activations():
    f = synth.q4k_fields(9, 1024, 6)
    x1 = synth.activations(3, 1024, 7)
    x2 = synth.activations(3, 1024, 8)
    y1, n1 = O.gemv(f, x1)
    y2, n2 = O.gemv(f, x2)
    y12, _ = O.gemv(f, (x1.astype(np.float64) + x2).astype(np.float32))
    # x1 + x2 is rounded to fp32 once: allow that rounding only.
    assert np.all(np.abs(y12 - (y1 + y2)) <= 1e-6 * (n1 + n2))


def decode_weight_from_bytes(block, i):
    """Exact rational weight i of one 144-byte superblock, decoded byte by
    byte with Python integers (independent of the oracle's array code)."""
    d = Fraction(float(np.array([block[0] | block[1] << 8], np.uint16).view(np.float16)[0]))
    dmin = Fraction(float(np.array([block[2] | block[3] << 8], np.uint16).view(np.float16)[0]))
    j = i // 32
    s = block[4:16]
    if j < 4:
        sc, m = s[j] & 63, s[j + 4] & 63
    else:
        sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4)
        m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4)
    byte = block[16 + 32 * (i // 64) + i % 32]
    q = (byte >> 4) if (i % 64) >= 32 else (byte & 15)
    return d * sc * q - dmin * m


@pytest.mark.parametrize("rows,cols", [(1, 256), (2, 512), (3, 768)])
def test_brute_force_exact_rationals(rows, cols):
    f = synth.q4k_fields(rows, cols, rows * 100 + cols)
    x = synth.activations(1, cols, 9)
    packed = O.pack_block144(f)
    y, norm = O.gemv(f, x)
    for o in range(rows):
        exact = Fraction(0)
        for k in range(cols):
            w = decode_weight_from_bytes([int(b) for b in packed[o, k // 256]], k % 256)
            exact += w * Fraction(float(x[0, k]))
        # the oracle rounds w to fp32 (2^-24 relative) and sums in fp64
        assert abs(float(exact) - y[0, o]) <= 1e-6 * norm[0, o]


def test_residual_is_added():
    f = synth.q4k_fields(4, 256, 10)
    x = synth.activations(2, 256, 11)
    r = synth.residual(2, 4, 12)
    y0, n0 = O.gemv(f, x)
    y1, n1 = O.gemv(f, x, r)
    assert np.array_equal(y1, y0 + r.astype(np.float64))
    assert np.array_equal(n1, n0 + np.abs(r.astype(np.float64)))


def test_tolerance_helper_rejects_a_planted_error():
    f = synth.q4k_fields(4, 256, 13)
    x = synth.activations(1, 256, 14)
    y, norm = O.gemv(f, x)
    ok, _ = O.within_tolerance(y.astype(np.float32), y, norm)
    assert ok
    bad = y.copy()
    bad[0, 2] += 2e-4 * norm[0, 2]
    ok, worst = O.within_tolerance(bad, y, norm)
    assert not ok and worst > 1.5


def test_magnitude_norm_hand_worked_cancellation():
    # one superblock, d = 1, dmin = 1; sub-block 0 has sc = 2, m = 6 and
    # q = 3 everywhere, so every weight is 2*3 - 1*6 = 0 (sum |w||x| = 0)
    # while each term has magnitude 6; the other sub-blocks have m = 0
    f = {"d": np.array([[0x3C00]], np.uint16), "dmin": np.array([[0x3C00]], np.uint16),
         "sc": np.array([[2, 1, 1, 1, 1, 1, 1, 1]], np.uint8),
         "m": np.array([[6, 0, 0, 0, 0, 0, 0, 0]], np.uint8),
         "q": np.full((1, 256), 3, np.uint8)}
    x = np.ones((1, 256), np.float32)
    x[0, :32] = np.arange(32, dtype=np.float32) - 10.5
    y, norm = O.gemv(f, x)
    mag = O.magnitude_norm(f, x)
    s0 = float(np.abs(x[0, :32]).astype(np.float64).sum())
    # sub-block 0: w = 0, |a| + |b| = 12; sub-blocks 1..7: w = a = 3, b = 0
    assert norm[0, 0] == 3.0 * 224
    assert mag[0, 0] == 12.0 * s0 + 3.0 * 224
    assert y[0, 0] == 3.0 * 224


def test_magnitude_norm_equals_norm_without_mins_and_bounds_it():
    f = synth.q4k_fields(7, 768, 91)
    x = synth.activations(3, 768, 92)
    mag = O.magnitude_norm(f, x)
    _, norm = O.gemv(f, x)
    assert np.all(norm <= mag * (1 + 2.0 ** -22))
    f0 = dict(f, m=np.zeros_like(f["m"]))
    _, norm0 = O.gemv(f0, x)
    assert np.array_equal(O.magnitude_norm(f0, x), norm0)
    r = synth.residual(3, 7, 93)
    assert np.allclose(O.magnitude_norm(f, x, r) - mag, np.abs(r.astype(np.float64)), rtol=0, atol=1e-12)
