"""CPU oracle for the Q4_K weight matmul — TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously-correct numpy restatement of what the CUDA path
computes.  Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import it; the product path never does, and it shares
no code, table or helper with the CUDA library.

What the method computes (genie-ai-runtime, §2 "the roofline that dictates
strategy", §3 "The tensor-core kernel (Path E)", §4 Path C):

* a Q4_K weight matrix is a grid of 256-weight superblocks, each with an
  fp16 scale ``d`` and an fp16 min ``dmin``, and eight 32-weight sub-blocks
  with a 6-bit scale ``sc`` and a 6-bit min ``m``; a weight is
  ``w = d*sc*q - dmin*m`` for its 4-bit quant ``q``;
* decode (batch 1..B) is the fp GEMV ``y[b][o] = sum_k w[o][k] x[b][k]``
  (+ an optional residual, §4 Path C folds the residual add into the GEMV);
* prefill quantises activations to q8_1 (int8 blocks of 32 with an fp32
  scale and the block sum) and accumulates exact integer per-block dot
  products, then applies each block's scale and min (the MMQ form).

Readings where the pages are silent (each is listed in the design notes):

* the byte layout of a superblock is the common GGUF Q4_K layout
  (``pack_block144``);
* dequantisation is evaluated in fp32 as ``(d*sc)*q - (dmin*m)``;
* q8_1: ``d8 = amax/127`` (fp32 division), ``q = round(x/d8)`` with fp32
  division and ties away from zero, clamped to [-127, 127]; a block whose
  ``d8`` is zero quantises to all zeros;
* tolerance of the fp outputs: ``|y - y_ref| <= 1e-4 * sum_k |w||x|``; a
  kernel that applies a weight's scale term ``d*sc*q`` and its min term
  ``dmin*m`` as separate sums (the MMQ form does by definition) is also held
  to the bound with the magnitude normaliser
  ``sum_k (|d*sc*q| + |dmin*m|) |x|`` (``magnitude_norm``), which differs
  from ``sum |w||x|`` only where the two terms of a weight cancel.

Parity pins: every function here is pinned in ``tests/test_oracle_*.py``
against hand-worked values, closed forms, invariants or brute force.
"""
from __future__ import annotations

import numpy as np

QK_K = 256
QK_SUB = 32
BLOCK144_BYTES = 144


# --------------------------------------------------------------------------
# IEEE 754 binary16 -> float64, written from the format definition.
def f16_bits_to_f64(bits) -> np.ndarray:
    """Decode raw binary16 bits: 1 sign bit, 5 exponent bits (bias 15),
    10 fraction bits.  Exponent 0 is zero/subnormal (``f * 2**-24``),
    exponent 31 is infinity (f == 0) or NaN."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    sign = (b >> 15) & 1
    expo = (b >> 10) & 0x1F
    frac = b & 0x3FF
    normal = np.ldexp((1024 + frac).astype(np.float64), (expo - 25).astype(np.int64))
    sub = frac.astype(np.float64) * 2.0 ** -24
    mag = np.where(expo == 0, sub, normal)
    mag = np.where(expo == 31, np.where(frac == 0, np.inf, np.nan), mag)
    return np.where(sign == 1, -mag, mag)


# --------------------------------------------------------------------------
# Packing: fields -> 144-byte superblocks (GGUF Q4_K byte order).
def pack_block144(fields: dict) -> np.ndarray:
    """Pack the five field arrays into ``[rows][cols/256][144]`` bytes.

    Superblock bytes: 0-1 ``d`` (little-endian binary16), 2-3 ``dmin``,
    4-15 twelve scale bytes, 16-143 the 128 quant bytes.

    Scale bytes (sub-block j of the superblock):
      * j < 4: ``sc_j`` in the low 6 bits of byte j, ``m_j`` in the low
        6 bits of byte j+4;
      * j >= 4: low nibble of byte j+4 = low 4 bits of ``sc_j``, its high
        nibble = low 4 bits of ``m_j``; the top two bits of byte j-4 carry
        ``sc_j >> 4`` and the top two bits of byte j carry ``m_j >> 4``.

    Quant bytes: for the 64-weight chunk c (0..3) and l < 32, byte
    ``32c + l`` holds weight ``64c + l`` in its low nibble and weight
    ``64c + 32 + l`` in its high nibble.
    """
    q = np.asarray(fields["q"], np.uint8)
    rows, cols = q.shape
    nb = cols // QK_K
    out = np.zeros((rows, nb, BLOCK144_BYTES), np.uint8)
    d = np.asarray(fields["d"], np.uint16).reshape(rows, nb)
    dmin = np.asarray(fields["dmin"], np.uint16).reshape(rows, nb)
    out[:, :, 0] = d & 0xFF
    out[:, :, 1] = d >> 8
    out[:, :, 2] = dmin & 0xFF
    out[:, :, 3] = dmin >> 8
    sc = np.asarray(fields["sc"], np.uint8).reshape(rows, nb, 8)
    m = np.asarray(fields["m"], np.uint8).reshape(rows, nb, 8)
    for j in range(4):
        out[:, :, 4 + j] = (sc[:, :, j] & 63) | ((sc[:, :, j + 4] >> 4) << 6)
        out[:, :, 8 + j] = (m[:, :, j] & 63) | ((m[:, :, j + 4] >> 4) << 6)
        out[:, :, 12 + j] = (sc[:, :, j + 4] & 15) | ((m[:, :, j + 4] & 15) << 4)
    qb = q.reshape(rows, nb, 4, 2, 32)          # [.., chunk c, half, l]
    qs = qb[:, :, :, 0, :] | (qb[:, :, :, 1, :] << 4)
    out[:, :, 16:] = qs.reshape(rows, nb, 128)
    return out


def unpack_block144(packed: np.ndarray) -> dict:
    """Inverse of ``pack_block144`` (read back every field)."""
    p = np.asarray(packed, np.uint8)
    rows, nb, _ = p.shape
    d = p[:, :, 0].astype(np.uint16) | (p[:, :, 1].astype(np.uint16) << 8)
    dmin = p[:, :, 2].astype(np.uint16) | (p[:, :, 3].astype(np.uint16) << 8)
    s = p[:, :, 4:16]
    sc = np.zeros((rows, nb, 8), np.uint8)
    m = np.zeros((rows, nb, 8), np.uint8)
    for j in range(4):
        sc[:, :, j] = s[:, :, j] & 63
        m[:, :, j] = s[:, :, j + 4] & 63
        sc[:, :, j + 4] = (s[:, :, j + 8] & 15) | ((s[:, :, j] >> 6) << 4)
        m[:, :, j + 4] = (s[:, :, j + 8] >> 4) | ((s[:, :, j + 4] >> 6) << 4)
    qs = p[:, :, 16:].reshape(rows, nb, 4, 32)
    q = np.stack([qs & 15, qs >> 4], axis=3).reshape(rows, nb * QK_K)
    return {"d": d, "dmin": dmin, "sc": sc.reshape(rows, nb * 8),
            "m": m.reshape(rows, nb * 8), "q": q}


# --------------------------------------------------------------------------
# Dequantisation and the fp (decode GEMV) path.
def dequantize(fields: dict) -> np.ndarray:
    """``w[o][k] = (d*sc)*q - (dmin*m)`` evaluated with fp32 operations."""
    q = np.asarray(fields["q"], np.uint8)
    rows, cols = q.shape
    d = f16_bits_to_f64(fields["d"]).astype(np.float32)
    dmin = f16_bits_to_f64(fields["dmin"]).astype(np.float32)
    d_k = np.repeat(d.reshape(rows, -1), QK_K, axis=1)
    dmin_k = np.repeat(dmin.reshape(rows, -1), QK_K, axis=1)
    sc_k = np.repeat(np.asarray(fields["sc"]).reshape(rows, -1), QK_SUB, axis=1).astype(np.float32)
    m_k = np.repeat(np.asarray(fields["m"]).reshape(rows, -1), QK_SUB, axis=1).astype(np.float32)
    return (d_k * sc_k) * q.astype(np.float32) - (dmin_k * m_k)


def gemv(fields: dict, x: np.ndarray, residual: np.ndarray | None = None):
    """Reference decode GEMV.  ``x`` is ``[batch][cols]``.

    Returns ``(y_ref, norm)`` in float64, both ``[batch][rows]``:
    ``y_ref = sum_k w*x (+ residual)`` accumulated in fp64 and
    ``norm = sum_k |w||x| (+ |residual|)`` the tolerance normaliser.
    """
    w = dequantize(fields).astype(np.float64)
    x64 = np.atleast_2d(np.asarray(x, np.float32)).astype(np.float64)
    y = x64 @ w.T
    norm = np.abs(x64) @ np.abs(w).T
    if residual is not None:
        r = np.atleast_2d(np.asarray(residual, np.float32)).astype(np.float64)
        y = y + r
        norm = norm + np.abs(r)
    return y, norm


def weight_terms(fields: dict):
    """The two terms of every weight, ``a = (d*sc)*q`` and ``b = dmin*m``,
    each evaluated with the same fp32 operations as ``dequantize`` (so that
    ``w = a - b`` there)."""
    q = np.asarray(fields["q"], np.uint8)
    rows, cols = q.shape
    d = f16_bits_to_f64(fields["d"]).astype(np.float32)
    dmin = f16_bits_to_f64(fields["dmin"]).astype(np.float32)
    d_k = np.repeat(d.reshape(rows, -1), QK_K, axis=1)
    dmin_k = np.repeat(dmin.reshape(rows, -1), QK_K, axis=1)
    sc_k = np.repeat(np.asarray(fields["sc"]).reshape(rows, -1), QK_SUB, axis=1).astype(np.float32)
    m_k = np.repeat(np.asarray(fields["m"]).reshape(rows, -1), QK_SUB, axis=1).astype(np.float32)
    return (d_k * sc_k) * q.astype(np.float32), dmin_k * m_k


def magnitude_norm(fields: dict, x: np.ndarray, residual: np.ndarray | None = None):
    """``sum_k (|a_k| + |b_k|) |x_k|`` (+ ``|residual|``) in float64,
    ``[batch][rows]``, with ``a``, ``b`` the two terms of each weight
    (``weight_terms``); for the MMQ path ``x`` is ``dequantize_q8_1(q8, d8)``.  It is at least ``sum_k |w_k||x_k|`` (up to the fp32
    rounding of ``a - b``) and equal to it wherever ``b = 0``."""
    a, b = weight_terms(fields)
    mag = np.abs(a).astype(np.float64) + np.abs(b).astype(np.float64)
    x64 = np.atleast_2d(np.asarray(x)).astype(np.float64)    # float32 x, or the float64 d8*q8
    norm = np.abs(x64) @ mag.T
    if residual is not None:
        norm = norm + np.abs(np.atleast_2d(np.asarray(residual, np.float32)).astype(np.float64))
    return norm


# --------------------------------------------------------------------------
# q8_1 activation quantisation.
def round_half_away(v: np.ndarray) -> np.ndarray:
    """Round float32 values to integers, ties away from zero (C ``roundf``).
    Done in float64, where ``|v| + 0.5`` is exact for every float32 v that
    can round to a nonzero integer."""
    v64 = np.asarray(v, np.float32).astype(np.float64)
    return np.copysign(np.floor(np.abs(v64) + 0.5), v64)


def quantize_q8_1(x: np.ndarray):
    """q8_1 blocks of 32 along the last axis of ``x`` ``[n][cols]``.

    Per block: ``amax = max|x|``; ``d8 = amax / 127`` (fp32 division);
    ``q = clamp(round(x / d8), -127, 127)`` (fp32 division, ties away from
    zero); ``S = sum q``.  A block whose ``d8`` is 0 gives q = 0, S = 0.
    Returns ``(q int8 [n][cols], d8 float32 [n][cols/32], S int32 [n][cols/32])``.
    """
    x = np.atleast_2d(np.asarray(x, np.float32))
    n, cols = x.shape
    xb = x.reshape(n, cols // QK_SUB, QK_SUB)
    amax = np.max(np.abs(xb), axis=2)
    d8 = (amax / np.float32(127.0)).astype(np.float32)
    live = d8 != 0
    denom = np.where(live, d8, np.float32(1.0)).astype(np.float32)
    ratio = (xb / denom[:, :, None]).astype(np.float32)
    q = np.clip(round_half_away(ratio), -127, 127)
    q = np.where(live[:, :, None], q, 0).astype(np.int8)
    s = q.astype(np.int32).sum(axis=2, dtype=np.int32)
    return q.reshape(n, cols), d8, s


def dequantize_q8_1(q: np.ndarray, d8: np.ndarray) -> np.ndarray:
    """``x_hat = d8 * q`` in float64 (exact: 24-bit times 8-bit)."""
    n, cols = q.shape
    qb = q.reshape(n, cols // QK_SUB, QK_SUB).astype(np.float64)
    return (qb * d8.astype(np.float64)[:, :, None]).reshape(n, cols)


# --------------------------------------------------------------------------
# MMQ (prefill) path: exact per-block integer dots, then scales and mins.
def block_dots(q4: np.ndarray, q8: np.ndarray) -> np.ndarray:
    """``P[t][o][b] = sum_{i<32} q4[o][32b+i] * q8[t][32b+i]`` as exact int64."""
    rows, cols = q4.shape
    n = q8.shape[0]
    a = np.asarray(q4).reshape(rows, cols // QK_SUB, QK_SUB).astype(np.int64)
    b = np.asarray(q8).reshape(n, cols // QK_SUB, QK_SUB).astype(np.int64)
    return np.einsum("obi,tbi->tob", a, b)


def mmq(fields: dict, q8: np.ndarray, d8: np.ndarray, s: np.ndarray):
    """Reference prefill GEMM on q8_1 activations.

    ``y[t][o] = sum_b ( d*sc[o,b] * d8[t,b] * P[t,o,b]
                        - dmin*m[o,b] * d8[t,b] * S[t,b] )``
    with ``P`` the exact integer block dot (computed per block as a
    float64 matmul of integers, exact because every partial sum stays far
    below 2**53).  Returns ``(y_ref, norm)`` float64 ``[tokens][rows]`` with
    ``norm = sum_k |w[o][k]| |d8 q8[t][k]|``.
    """
    q4 = np.asarray(fields["q"], np.uint8)
    rows, cols = q4.shape
    n = q8.shape[0]
    nsub = cols // QK_SUB
    d = np.repeat(f16_bits_to_f64(fields["d"]).reshape(rows, -1), 8, axis=1)
    dmin = np.repeat(f16_bits_to_f64(fields["dmin"]).reshape(rows, -1), 8, axis=1)
    dsc = d * np.asarray(fields["sc"], np.float64).reshape(rows, nsub)
    dmm = dmin * np.asarray(fields["m"], np.float64).reshape(rows, nsub)
    d8_64 = d8.astype(np.float64)
    s64 = s.astype(np.float64)
    y = np.zeros((n, rows), np.float64)
    for b in range(nsub):
        a = q4[:, QK_SUB * b:QK_SUB * (b + 1)].astype(np.float64)
        t = q8[:, QK_SUB * b:QK_SUB * (b + 1)].astype(np.float64)
        p = t @ a.T                                    # exact integers
        y += d8_64[:, b:b + 1] * (p * dsc[None, :, b])
        y -= (d8_64[:, b] * s64[:, b])[:, None] * dmm[None, :, b]
    w = np.abs(dequantize(fields).astype(np.float64))
    norm = np.abs(dequantize_q8_1(q8, d8)) @ w.T
    return y, norm


# --------------------------------------------------------------------------
def within_tolerance(y, y_ref, norm, rel: float = 1e-4):
    """Elementwise acceptance: ``|y - y_ref| <= rel * norm`` (norm 0 needs y == 0).
    Returns (ok, worst ratio of error to allowed error)."""
    y = np.asarray(y, np.float64)
    err = np.abs(y - y_ref)
    allowed = rel * np.asarray(norm, np.float64)
    zero = allowed == 0
    bad_zero = np.any(err[zero] != 0) if np.any(zero) else False
    ratio = np.where(zero, 0.0, err / np.where(zero, 1.0, allowed))
    worst = float(np.max(ratio)) if ratio.size else 0.0
    return (not bad_zero) and worst <= 1.0, worst
