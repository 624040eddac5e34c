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
