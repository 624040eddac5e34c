"""Pins of the Q6_K oracle (CPU only).

The block layout is pinned by a hand-built superblock whose weights were
worked out by hand (tests/golden/q6k_block_example.txt): a swapped nibble,
a wrong 2-bit field of qh, a wrong half or quarter, an unsigned scale or a
dropped offset of 32 each change one of its listed weights."""
from pathlib import Path

import numpy as np

from oracle import q6k as O6
from oracle import q4k as O
import synth

GOLDEN = Path(__file__).parent / "golden" / "q6k_block_example.txt"


def _golden():
    blk = np.zeros(O6.Q6K_BYTES, np.uint8)
    weights = []
    mode = None
    for line in GOLDEN.read_text().splitlines():
        line = line.split("#")[0].strip()
        if not line:
            continue
        if line in ("bytes", "weights"):
            mode = line
            continue
        parts = line.split()
        if mode == "bytes":
            blk[int(parts[0])] = int(parts[1], 0)
        else:
            weights.append((int(parts[0]), int(parts[1]), float(parts[2])))
    return blk, weights


def test_hand_built_block_dequantises_to_the_hand_worked_weights():
    blk, weights = _golden()
    f = O6.unpack_q6k(blk.reshape(1, 1, -1))
    w = O6.dequantize_q6k(f)
    for k, q, wk in weights:
        assert f["q"][0, k] == q, k
        assert w[0, k] == wk, k


def test_every_unlisted_weight_is_minus_32_d_sc():
    blk, weights = _golden()
    w = O6.dequantize_q6k(O6.unpack_q6k(blk.reshape(1, 1, -1)))[0]
    listed = {k for k, _, _ in weights}
    sc = blk[192:208].view(np.int8).astype(np.float64)
    for k in range(256):
        if k not in listed:
            assert w[k] == 0.5 * sc[k // 16] * -32, k


def test_pack_writes_the_hand_built_bytes():
    blk, _ = _golden()
    f = O6.unpack_q6k(blk.reshape(1, 1, -1))
    assert np.array_equal(O6.pack_q6k(f).reshape(-1), blk)


def test_pack_unpack_round_trip_many_blocks():
    f = synth.q6k_fields(7, 1024, 11)
    g = O6.unpack_q6k(O6.pack_q6k(f))
    for key in ("d", "sc", "q"):
        assert np.array_equal(np.asarray(g[key]), np.asarray(f[key]).reshape(np.asarray(g[key]).shape)), key


def test_blocks_are_row_major_superblock_order():
    blk, weights = _golden()
    packed = np.zeros((2, 2, O6.Q6K_BYTES), np.uint8)
    packed[1, 1] = blk          # row 1, second superblock; d = 0 everywhere else
    w = O6.dequantize_q6k(O6.unpack_q6k(packed))
    assert not w[0].any() and not w[1, :256].any()
    for k, _, wk in weights:
        assert w[1, 256 + k] == wk


def test_gemv_of_the_hand_block_against_hand_sums():
    blk, _ = _golden()
    f = O6.unpack_q6k(blk.reshape(1, 1, -1))
    x = np.zeros((1, 256), np.float32)
    x[0, 0], x[0, 96], x[0, 225] = 2.0, 1.0, -2.0
    y, norm = O6.gemv_q6k(f, x)
    assert y[0, 0] == 2 * -33 + -1216 + -2 * -59.5          # = -1163
    assert norm[0, 0] == 66 + 1216 + 119
    r = np.array([[0.25]], np.float32)
    y2, norm2 = O6.gemv_q6k(f, x, r)
    assert y2[0, 0] == -1162.75 and norm2[0, 0] == 1401.25


def test_quants_of_32_give_zero_and_the_extremes_are_minus_32_and_31():
    f = synth.q6k_fields(3, 512, 12)
    f["q"][:] = 32
    assert not O6.dequantize_q6k(f).any()
    y, norm = O6.gemv_q6k(f, synth.activations(2, 512, 13))
    assert not y.any() and not norm.any()
    f["q"][:] = 0
    d = O.f16_bits_to_f64(f["d"])
    w0 = O6.dequantize_q6k(f)
    f["q"][:] = 63
    w63 = O6.dequantize_q6k(f)
    for o in range(3):
        for k in (0, 17, 300, 511):
            dsc = np.float32(d[o, k // 256]) * np.float32(f["sc"][o, k // 16])
            assert w0[o, k] == dsc * -32 and w63[o, k] == dsc * 31


def test_gemv_one_hot_columns_read_back_the_weights():
    f = synth.q6k_fields(5, 512, 14)
    w = O6.dequantize_q6k(f)
    for k in (0, 15, 16, 255, 256, 300, 511):
        x = np.zeros((1, 512), np.float32)
        x[0, k] = 1.0
        y, _ = O6.gemv_q6k(f, x)
        assert np.array_equal(y[0], w[:, k].astype(np.float64))


def test_gemv_is_brute_force_on_a_tiny_integer_case():
    # small integer weights and activations: every product and sum is exact
    # in fp64, so the GEMV must equal the integer triple loop over the fields
    rng = np.random.default_rng(15)
    f = {"d": np.full((2, 1), 0x3C00, np.uint16),                 # d = 1
         "sc": rng.integers(-4, 5, (2, 16)).astype(np.int8),
         "q": rng.integers(0, 64, (2, 256)).astype(np.uint8)}
    x = rng.integers(-3, 4, (3, 256)).astype(np.float32)
    y, _ = O6.gemv_q6k(f, x)
    for b in range(3):
        for o in range(2):
            s = 0
            for k in range(256):
                s += int(f["sc"][o, k // 16]) * (int(f["q"][o, k]) - 32) * int(x[b, k])
            assert y[b, o] == s


def test_q6k_block_dots_by_brute_force_and_extremes():
    rng = np.random.default_rng(16)
    q = rng.integers(0, 64, (3, 256)).astype(np.uint8)
    q8 = rng.integers(-127, 128, (2, 256)).astype(np.int8)
    P = O6.block_dots_q6k(q, q8)
    for t in range(2):
        for o in range(3):
            for g in range(16):
                assert P[t, o, g] == sum((int(q[o, 16 * g + i]) - 32) * int(q8[t, 16 * g + i]) for i in range(16))
    # extremes: q = 0 (-32) against +-127, and q = 63 (+31)
    q[:] = 0
    q8[:] = -127
    assert np.all(O6.block_dots_q6k(q, q8) == 16 * 32 * 127)
    q[:] = 63
    q8[:] = 127
    assert np.all(O6.block_dots_q6k(q, q8) == 16 * 31 * 127)


def test_q6k_mmq_equals_the_fp_path_on_the_dequantised_activations():
    """With x = d8 * q8 every MMQ term is the fp path's: the two agree to
    rounding (and exactly when the scales are powers of two)."""
    f = synth.q6k_fields(6, 768, 17)
    x = synth.activations(3, 768, 18)
    q8, d8, _ = O.quantize_q8_1(x)
    y, norm = O6.mmq_q6k(f, q8, d8)
    xh = O.dequantize_q8_1(q8, d8)                       # float64, exact
    w = O6.dequantize_q6k(f).astype(np.float64)
    y_fp, norm_fp = xh @ w.T, np.abs(xh) @ np.abs(w).T
    assert np.array_equal(norm, norm_fp)
    assert np.all(np.abs(y - y_fp) <= 1e-12 * norm)
    f["d"][:] = 0x3C00                                   # d = 1: every factor exact
    d8p = np.full_like(d8, 0.25)
    y2, _ = O6.mmq_q6k(f, q8, d8p)
    xh2 = O.dequantize_q8_1(q8, d8p)
    assert np.array_equal(y2, xh2 @ O6.dequantize_q6k(f).astype(np.float64).T)


def test_q6k_mmq_uses_the_scale_of_each_16_group_and_the_d8_of_its_32_block():
    """One nonzero q8 element at a time: y equals d * sc_(k/16) * d8_(k/32) * (q_k - 32) * q8_k,
    so a swapped scale group or block scale fails."""
    f = synth.q6k_fields(2, 256, 19)
    f["sc"] = np.arange(1, 17, dtype=np.int8)[None, :].repeat(2, axis=0)
    d8 = (np.arange(1, 9, dtype=np.float32) * 0.5)[None, :]
    d = O.f16_bits_to_f64(f["d"])
    for k in (0, 15, 16, 31, 32, 200, 255):
        q8 = np.zeros((1, 256), np.int8)
        q8[0, k] = 3
        y, _ = O6.mmq_q6k(f, q8, d8)
        for o in range(2):
            want = float(np.float32(np.float32(d[o, 0]) * np.float32(k // 16 + 1))) * float(d8[0, k // 32]) \
                * (int(f["q"][o, k]) - 32) * 3
            assert y[0, o] == want, (k, o)
