"""CPU oracle for the Q6_K weight matmul -- TEST INFRASTRUCTURE ONLY.

A plain, slow numpy restatement of what the Q6_K CUDA path computes.  Only
the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import it; the product path never does, and it shares no code with the
CUDA library.

What it computes.  Q6_K is the 6-bit K-quant that, mixed with Q4_K, makes
the Q4_K_M models the genie-ai-runtime page runs (§2 "Qwen3-4B Q4_K_M
weights"; its paused "Path G" is a Q6_K decode-side scale hoist and block
layout redesign).  The pages print no Q6_K layout; the reading here is the
common GGUF Q6_K block, restated in prose:

* a superblock holds 256 weights: one fp16 scale ``d``, sixteen int8 scales
  ``sc`` (one per 16 weights) and a 6-bit quant ``q`` (0..63) per weight;
  a weight is ``w = d * sc * (q - 32)``;
* 210 bytes: ``ql[128]`` (the low 4 bits of every quant), ``qh[64]`` (the
  high 2 bits), ``scales[16]`` (int8), ``d`` (little-endian binary16);
* for each half n (0, 1) of 128 weights and l < 32, with L = ql[64n..],
  H = qh[32n..]: weight 128n + l has low bits L[l] & 15 and high bits
  H[l] & 3; weight 128n + 32 + l: L[32 + l] & 15, (H[l] >> 2) & 3;
  weight 128n + 64 + l: L[l] >> 4, (H[l] >> 4) & 3; weight 128n + 96 + l:
  L[32 + l] >> 4, H[l] >> 6.

Readings where the pages are silent (listed in the design notes): the
dequantisation is evaluated in fp32 as ``(d * sc) * (q - 32)``; the GEMV
accumulates in fp64; the tolerance is ``|y - y_ref| <= 1e-4 * sum |w||x|``.
The MMQ form for q8_1 activations (the q8_1 block of 32 is the Q4_K path's,
``oracle.q4k.quantize_q8_1``) takes one exact integer dot per 16-weight scale
group, ``P = sum (q - 32) * q8``, and
``y = sum_g d * sc_g * d8_(g/2) * P_g`` (no min term: the offset of 32 is in
the integer dot).
Pinned in ``tests/test_oracle_q6k.py``.
"""
from __future__ import annotations

import numpy as np

from .q4k import f16_bits_to_f64

QK_K = 256
Q6K_BYTES = 210


def pack_q6k(fields: dict) -> np.ndarray:
    """``[rows][cols/256][210]`` bytes from ``d`` (uint16 binary16 bits,
    ``[rows][nb]``), ``sc`` (int8, ``[rows][cols/16]``) and ``q`` (uint8
    0..63, ``[rows][cols]``)."""
    q = np.asarray(fields["q"], np.uint8) & 63
    rows, cols = q.shape
    nb = cols // QK_K
    out = np.zeros((rows, nb, Q6K_BYTES), np.uint8)
    qb = q.reshape(rows, nb, 2, 4, 32)          # [.., half n, quarter, l]: weight 128n + 32*quarter + l
    lo = qb & 15
    hi = qb >> 4
    ql = np.zeros((rows, nb, 2, 64), np.uint8)
    ql[..., :32] = lo[..., 0, :] | (lo[..., 2, :] << 4)
    ql[..., 32:] = lo[..., 1, :] | (lo[..., 3, :] << 4)
    qh = hi[..., 0, :] | (hi[..., 1, :] << 2) | (hi[..., 2, :] << 4) | (hi[..., 3, :] << 6)
    out[:, :, 0:128] = ql.reshape(rows, nb, 128)
    out[:, :, 128:192] = qh.reshape(rows, nb, 64)
    out[:, :, 192:208] = np.asarray(fields["sc"], np.int8).reshape(rows, nb, 16).view(np.uint8)
    d = np.asarray(fields["d"], np.uint16).reshape(rows, nb)
    out[:, :, 208] = d & 0xFF
    out[:, :, 209] = d >> 8
    return out


def unpack_q6k(packed: np.ndarray) -> dict:
    """Inverse of ``pack_q6k``."""
    p = np.asarray(packed, np.uint8)
    rows, nb, _ = p.shape
    ql = p[:, :, 0:128].reshape(rows, nb, 2, 64)
    qh = p[:, :, 128:192].reshape(rows, nb, 2, 32)
    q = np.zeros((rows, nb, 2, 4, 32), np.uint8)
    q[..., 0, :] = (ql[..., :32] & 15) | ((qh & 3) << 4)
    q[..., 1, :] = (ql[..., 32:] & 15) | (((qh >> 2) & 3) << 4)
    q[..., 2, :] = (ql[..., :32] >> 4) | (((qh >> 4) & 3) << 4)
    q[..., 3, :] = (ql[..., 32:] >> 4) | ((qh >> 6) << 4)
    sc = p[:, :, 192:208].view(np.int8).reshape(rows, nb * 16)
    d = p[:, :, 208].astype(np.uint16) | (p[:, :, 209].astype(np.uint16) << 8)
    return {"d": d, "sc": sc.copy(), "q": q.reshape(rows, nb * QK_K)}


def dequantize_q6k(fields: dict) -> np.ndarray:
    """``w[o][k] = (d * sc) * (q - 32)`` evaluated with fp32 operations."""
    q = np.asarray(fields["q"], np.uint8).astype(np.int32)
    rows, cols = q.shape
    d = f16_bits_to_f64(fields["d"]).astype(np.float32)
    d_k = np.repeat(d.reshape(rows, -1), QK_K, axis=1)
    sc_k = np.repeat(np.asarray(fields["sc"], np.int8).reshape(rows, -1), 16, axis=1).astype(np.float32)
    return (d_k * sc_k) * (q - 32).astype(np.float32)


def gemv_q6k(fields: dict, x: np.ndarray, residual: np.ndarray | None = None):
    """Reference decode GEMV over Q6_K weights; ``(y_ref, norm)`` float64
    ``[batch][rows]``, ``norm = sum_k |w||x| (+ |residual|)``."""
    w = dequantize_q6k(fields).astype(np.float64)
    x64 = np.atleast_2d(np.asarray(x, np.float32)).astype(np.float64)
    y = x64 @ w.T
    norm = np.abs(x64) @ np.abs(w).T
    if residual is not None:
        r = np.atleast_2d(np.asarray(residual, np.float32)).astype(np.float64)
        y = y + r
        norm = norm + np.abs(r)
    return y, norm


def block_dots_q6k(q: np.ndarray, q8: np.ndarray) -> np.ndarray:
    """``P[t][o][g] = sum_{i<16} (q[o][16g+i] - 32) * q8[t][16g+i]``, exact int64."""
    q = np.asarray(q, np.int64) - 32
    rows, cols = q.shape
    n = np.asarray(q8).shape[0]
    a = q.reshape(rows, cols // 16, 16)
    b = np.asarray(q8).reshape(n, cols // 16, 16).astype(np.int64)
    return np.einsum("ogi,tgi->tog", a, b)


def mmq_q6k(fields: dict, q8: np.ndarray, d8: np.ndarray):
    """Reference MMQ product over Q6_K weights and q8_1 activations:
    ``y[t][o] = sum_g (d * sc_g)[o] * d8[t][g/2] * P[t][o][g]`` in float64
    (``d * sc`` in fp32, as the dequantisation forms it).  Returns
    ``(y_ref, norm)`` ``[tokens][rows]``, ``norm = sum_k |w||d8 q8|``."""
    q = np.asarray(fields["q"], np.uint8)
    rows, cols = q.shape
    P = block_dots_q6k(q, q8).astype(np.float64)                       # [t][o][g]
    d = f16_bits_to_f64(fields["d"]).astype(np.float32)                 # [o][nb]
    dsc = (np.repeat(d, 16, axis=1) * np.asarray(fields["sc"], np.int8).astype(np.float32)).astype(np.float64)
    d8g = np.repeat(np.asarray(d8, np.float32).astype(np.float64), 2, axis=1)   # [t][g]
    y = np.einsum("tog,og,tg->to", P, dsc, d8g)
    xh = (np.asarray(q8).reshape(q8.shape[0], cols // 32, 32).astype(np.float64)
          * np.asarray(d8, np.float32).astype(np.float64)[:, :, None]).reshape(q8.shape[0], cols)
    norm = np.abs(xh) @ np.abs(dequantize_q6k(fields).astype(np.float64)).T
    return y, norm

