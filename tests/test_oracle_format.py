"""Pins of the oracle's binary16 decoding and its Q4_K packing (CPU only)."""
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import q4k as O
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load_block_fixture():
    path = os.path.join(GOLDEN, "q4k_block144_example.txt")
    spec = {"bytes": {}, "w": {}}
    with open(path) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key in ("d", "dmin"):
                spec[key] = int(vals[0], 16)
            elif key in ("sc", "m"):
                spec[key] = [int(v) for v in vals]
            elif key == "q_rule":
                assert vals == ["i//16"]
                spec["q"] = [i // 16 for i in range(256)]
            elif key == "bytes":
                pos = int(vals[0])
                for tok in vals[1:]:
                    byte, _, rep = tok.partition("*")
                    for _ in range(int(rep or 1)):
                        spec["bytes"][pos] = int(byte, 16)
                        pos += 1
            elif key == "w":
                spec["w"][int(vals[0])] = Fraction(vals[1])
    return spec


def fixture_fields(spec):
    return {
        "d": np.array([[spec["d"]]], np.uint16),
        "dmin": np.array([[spec["dmin"]]], np.uint16),
        "sc": np.array([spec["sc"]], np.uint8),
        "m": np.array([spec["m"]], np.uint8),
        "q": np.array([spec["q"]], np.uint8),
    }


# --------------------------------------------------------------- binary16
def test_f16_decode_matches_numpy_for_every_bit_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    mine = O.f16_bits_to_f64(bits)
    lib = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], lib[~nan])


@pytest.mark.parametrize("bits,value", [
    (0x3C00, 1.0), (0xC000, -2.0), (0x0001, 2.0 ** -24), (0x03FF, 1023 * 2.0 ** -24),
    (0x0400, 2.0 ** -14), (0x7BFF, 65504.0), (0x3555, 1365 / 4096), (0x8000, -0.0),
    (0x7C00, np.inf), (0xFC00, -np.inf)])
def test_f16_decode_hand_values(bits, value):
    got = O.f16_bits_to_f64(np.array([bits], np.uint16))[0]
    assert got == value and np.signbit(got) == np.signbit(value)


# --------------------------------------------------------------- packing
def test_pack_matches_hand_packed_superblock():
    spec = load_block_fixture()
    packed = O.pack_block144(fixture_fields(spec))
    assert packed.shape == (1, 1, 144)
    assert len(spec["bytes"]) == 144
    expect = np.array([spec["bytes"][i] for i in range(144)], np.uint8)
    assert np.array_equal(packed[0, 0], expect)


def test_unpack_reads_hand_packed_superblock():
    spec = load_block_fixture()
    raw = np.array([spec["bytes"][i] for i in range(144)], np.uint8).reshape(1, 1, 144)
    back = O.unpack_block144(raw)
    f = fixture_fields(spec)
    for k in f:
        assert np.array_equal(back[k], f[k]), k


def test_dequantize_hand_worked_weights():
    spec = load_block_fixture()
    w = O.dequantize(fixture_fields(spec))
    for i, frac in spec["w"].items():
        assert Fraction(float(w[0, i])) == frac, i


def test_pack_roundtrip_every_scale_min_pair_at_every_position():
    # row r covers (a, b) = (r // 64, r % 64); sub-block j gets sc = a + j,
    # m = b + 3j (mod 64) so each j sees all 64 x 64 pairs exactly once.
    r = np.arange(4096)
    a, b = r // 64, r % 64
    j = np.arange(8)
    sc = ((a[:, None] + j[None, :]) % 64).astype(np.uint8)
    m = ((b[:, None] + 3 * j[None, :]) % 64).astype(np.uint8)
    rng = np.random.default_rng(7)
    f = {"d": rng.integers(0, 1 << 16, (4096, 1), dtype=np.uint16),
         "dmin": rng.integers(0, 1 << 16, (4096, 1), dtype=np.uint16),
         "sc": sc, "m": m,
         "q": rng.integers(0, 16, (4096, 256), dtype=np.uint8)}
    back = O.unpack_block144(O.pack_block144(f))
    for k in f:
        assert np.array_equal(back[k], f[k]), k


def test_pack_places_each_quant_in_its_own_nibble():
    # 256 rows, row i has a single nonzero quant (15) at weight i.
    q = np.zeros((256, 256), np.uint8)
    q[np.arange(256), np.arange(256)] = 15
    z16 = np.zeros((256, 1), np.uint16)
    z8 = np.zeros((256, 8), np.uint8)
    p = O.pack_block144({"d": z16, "dmin": z16, "sc": z8, "m": z8, "q": q})[:, 0, 16:]
    for i in range(256):
        nz = np.nonzero(p[i])[0]
        assert len(nz) == 1
        chunk, within = divmod(i, 64)
        half, lane = divmod(within, 32)
        assert nz[0] == 32 * chunk + lane
        assert p[i, nz[0]] == (0xF0 if half else 0x0F)


def test_pack_shape_and_size():
    f = synth.q4k_fields(3, 768, 11)
    p = O.pack_block144(f)
    assert p.shape == (3, 3, 144) and p.dtype == np.uint8
    assert p.nbytes == 3 * 768 * 9 // 16   # 4.5 bits per weight
