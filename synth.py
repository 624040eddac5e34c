"""Seeded synthetic inputs for the Q4_K weight matmul.

This module only draws random numbers; it holds none of the method's
arithmetic (no packing, no dequantisation, no quantisation, no dot
products).  Both the CUDA path's tests and the CPU oracle take their inputs
from here, and nothing else is shared between them.

Distributions (one Q4_K weight matrix ``W[rows][cols]``, ``cols % 256 == 0``):

* ``d``, ``dmin``: ``|N(0, 0.01)|`` per 256-weight superblock, rounded to
  IEEE binary16 (round to nearest even) and returned as raw uint16 bits,
  shape ``[rows][cols/256]``;
* ``sc``, ``m``: uniform integers ``0..63`` per 32-weight sub-block,
  shape ``[rows][cols/32]``;
* ``q``: uniform integers ``0..15`` per weight, shape ``[rows][cols]``;
* activations: ``N(0, 1)`` float32, shape ``[n][cols]``.

Draw order inside one matrix is d, dmin, sc, m, q, all from one
``numpy.random.default_rng`` (PCG64) stream.  The workloads below are the
Qwen3-4B / Qwen3-8B projection shapes the genie-ai-runtime page runs
(§2 "Qwen3-4B Q4_K_M weights", §3 Path B/E prefill, §4 Path C decode);
weights and activations are synthetic, never trained.
"""
from __future__ import annotations

import numpy as np

QK_K = 256       # weights per Q4_K superblock
QK_SUB = 32      # weights per sub-block (one 6-bit scale and min each)


def _rng(seed):
    return np.random.default_rng(seed)


def draw_fields(rng: np.random.Generator, rows: int, cols: int) -> dict:
    """Draw the five Q4_K field arrays of one matrix from ``rng``."""
    if cols % QK_K:
        raise ValueError(f"cols={cols} is not a multiple of {QK_K}")
    nb = cols // QK_K
    d = np.abs(rng.normal(0.0, 0.01, (rows, nb))).astype(np.float16).view(np.uint16)
    dmin = np.abs(rng.normal(0.0, 0.01, (rows, nb))).astype(np.float16).view(np.uint16)
    sc = rng.integers(0, 64, (rows, cols // QK_SUB), dtype=np.uint8)
    m = rng.integers(0, 64, (rows, cols // QK_SUB), dtype=np.uint8)
    q = rng.integers(0, 16, (rows, cols), dtype=np.uint8)
    return {"d": d, "dmin": dmin, "sc": sc, "m": m, "q": q}


def draw_q6k_fields(rng: np.random.Generator, rows: int, cols: int) -> dict:
    """Q6_K fields of one matrix: ``d = |N(0, 0.01)|`` (binary16 bits,
    ``[rows][cols/256]``), ``sc`` uniform int8 -128..127 (``[rows][cols/16]``),
    ``q`` uniform 0..63 (``[rows][cols]``); drawn in that order."""
    if cols % QK_K:
        raise ValueError(f"cols={cols} is not a multiple of {QK_K}")
    d = np.abs(rng.normal(0.0, 0.01, (rows, cols // QK_K))).astype(np.float16).view(np.uint16)
    sc = rng.integers(-128, 128, (rows, cols // 16), dtype=np.int16).astype(np.int8)
    q = rng.integers(0, 64, (rows, cols), dtype=np.uint8)
    return {"d": d, "sc": sc, "q": q}


def q6k_fields(rows: int, cols: int, seed) -> dict:
    return draw_q6k_fields(_rng(seed), rows, cols)


def draw_activations(rng: np.random.Generator, n: int, cols: int) -> np.ndarray:
    return rng.standard_normal((n, cols), dtype=np.float32)


def q4k_fields(rows: int, cols: int, seed) -> dict:
    """Fields of one matrix from a fresh generator seeded with ``seed``."""
    return draw_fields(_rng(seed), rows, cols)


def activations(n: int, cols: int, seed) -> np.ndarray:
    """``n`` activation rows of width ``cols`` from a fresh generator."""
    return draw_activations(_rng(seed), n, cols)


def residual(n: int, rows: int, seed) -> np.ndarray:
    """A residual stream ``[n][rows]`` (N(0,1) float32) for the fused add."""
    return draw_activations(_rng(seed), n, rows)


def single_gemv_2048(seed: int = 0):
    """Single 2048x2048 GEMV, batch 1, one generator seeded 0: the five
    field arrays are drawn first, then x from the same stream."""
    rng = _rng(seed)
    f = draw_fields(rng, 2048, 2048)
    x = draw_activations(rng, 1, 2048)
    return f, x


# ---------------------------------------------------------------------------
# Workload shapes.  Each projection is (name, rows=out, cols=in, input name).
# q/k/v share the attention input, gate/up share the MLP input.
QWEN3_4B_LAYER = (
    ("q", 4096, 2560, "attn_in"),
    ("k", 1024, 2560, "attn_in"),
    ("v", 1024, 2560, "attn_in"),
    ("o", 2560, 4096, "o_in"),
    ("gate", 9728, 2560, "mlp_in"),
    ("up", 9728, 2560, "mlp_in"),
    ("down", 2560, 9728, "down_in"),
)
QWEN3_4B_INPUTS = (("attn_in", 2560), ("o_in", 4096), ("mlp_in", 2560), ("down_in", 9728))

QWEN3_8B_MLP = (
    ("gate", 12288, 4096, "mlp_in"),
    ("up", 12288, 4096, "mlp_in"),
    ("down", 4096, 12288, "down_in"),
)
QWEN3_8B_INPUTS = (("mlp_in", 4096), ("down_in", 12288))

# Workload tags used in seeds: one integer per workload family so that no
# two tensors anywhere share a stream.
WL_DECODE_4B = 1        # Qwen3-4B-shaped decode linear set (one layer)
WL_PREFILL_4B_512 = 2   # 512-token prefill: gate and down of Qwen3-4B
WL_STACK_4B = 3         # 36-layer Qwen3-4B-shaped stack
WL_PREFILL_8B_4096 = 4  # 4096-token prefill: Qwen3-8B MLP


def layer_seed(workload: int, layer: int, tensor: int):
    """Seed of tensor ``tensor`` of layer ``layer`` of a workload.

    Matrices take their index in the layer table (0..6); inputs take
    100 + their index in the input table; the residual stream 200 + index.
    """
    return [workload, layer, tensor]


def decode_layer(workload: int, layer: int, batch: int, shapes=QWEN3_4B_LAYER,
                 inputs=QWEN3_4B_INPUTS, with_fields: bool = True):
    """Fields of every projection of one layer plus its ``batch``-row inputs."""
    fields = {}
    if with_fields:
        for i, (name, rows, cols, _) in enumerate(shapes):
            fields[name] = q4k_fields(rows, cols, layer_seed(workload, layer, i))
    xs = {}
    for j, (name, cols) in enumerate(inputs):
        xs[name] = activations(batch, cols, layer_seed(workload, layer, 100 + j + 10 * batch))
    return fields, xs


def prefill_4b_512():
    """512-token prefill: X[512x2560] into gate 9728x2560, X_down[512x9728]
    into down 2560x9728 (both inputs N(0,1), quantised to q8_1 by the path)."""
    gate = q4k_fields(9728, 2560, layer_seed(WL_PREFILL_4B_512, 0, 4))
    down = q4k_fields(2560, 9728, layer_seed(WL_PREFILL_4B_512, 0, 6))
    x = activations(512, 2560, layer_seed(WL_PREFILL_4B_512, 0, 102))
    x_down = activations(512, 9728, layer_seed(WL_PREFILL_4B_512, 0, 103))
    return {"gate": gate, "down": down}, {"mlp_in": x, "down_in": x_down}


def prefill_8b_4096():
    """4096-token prefill of the Qwen3-8B MLP: gate/up 12288x4096, down
    4096x12288."""
    fields = {}
    for i, (name, rows, cols, _) in enumerate(QWEN3_8B_MLP):
        fields[name] = q4k_fields(rows, cols, layer_seed(WL_PREFILL_8B_4096, 0, i))
    xs = {}
    for j, (name, cols) in enumerate(QWEN3_8B_INPUTS):
        xs[name] = activations(4096, cols, layer_seed(WL_PREFILL_8B_4096, 0, 100 + j))
    return fields, xs
