"""GPU parity of the fp16-activation prefill GEMM (x_split_f16 +
q4k_gemm_f16) against the oracle's fp64 product with the fp32 activations.

The split keeps each scaled element to 2^-22 of itself and rounds elements
far below their row's largest in absolute terms, so each output must satisfy
    |y - y_ref| <= 1e-4 * (M + 2^-16 * max_k |x_k| * W1),
M = sum_k (|d sc q_k| + |dmin m_k|) |x_k| and W1 the same sum with |x_k| = 1
(the oracle's magnitude normaliser).  Shapes span several 128 x 128 tiles,
ragged token and row tails, superblock counts that are not a multiple of the
four that one block-sum copy holds, and the activation patterns where a
fixed-point or fp16 form of x is weakest."""
import numpy as np
import pytest
import torch

from oracle import q4k as O
import synth
from _gpu import pack_dev, slice_rows
from test_gpu_edges import CASES
import q4_weight_matmul_gb300 as q4k

pytestmark = pytest.mark.gpu
REL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    q4k.build()
    torch.cuda.init()


def f16_norm(f, x):
    m = O.magnitude_norm(f, x)
    w1 = O.magnitude_norm(f, np.ones((1, x.shape[1]), np.float32))
    amax = np.abs(np.asarray(x, np.float64)).max(axis=1, keepdims=True)
    return m + 2.0 ** -16 * amax * w1


def run(f, x):
    rows, cols = f["q"].shape
    w = pack_dev(f)
    xd = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    y = q4k.q4k_gemm_f16(w, rows, cols, *q4k.x_split_f16(xd))
    torch.cuda.synchronize()
    return y.cpu().numpy()


def check(y, f, x, what=""):
    y_ref, _ = O.gemv(f, x)
    ok, worst = O.within_tolerance(y, y_ref, f16_norm(f, x), REL)
    assert ok, f"{what}: worst error {worst:.3g} x the allowed error"


def test_split_properties():
    """s_t is a power of two putting max|x| in [2^14, 2^15); hi + lo keeps
    s_t x to 2^-22 (2^-25 absolute); the block sums are those of hi + lo."""
    rng = np.random.default_rng(900)
    cols = 1024
    x = rng.standard_normal((6, cols)).astype(np.float32)
    x[1] *= 2.0 ** -100
    x[2] *= 2.0 ** 100
    x[3] = 0.0
    x[4, :] = 1e-12
    x[4, 7] = 3.0
    x[5, ::2] = 0.0
    hi, lo, bs, inv = q4k.x_split_f16(torch.from_numpy(x).cuda())
    hi = hi.cpu().numpy().astype(np.float64)
    lo = lo.cpu().numpy().astype(np.float64)
    bs = bs.cpu().numpy().astype(np.float64)
    inv = inv.cpu().numpy().astype(np.float64)
    for t in range(6):
        s = 1.0 / inv[t]
        assert np.log2(s) == np.round(np.log2(s))
        X = x[t].astype(np.float64) * s
        if t != 3:
            assert 2.0 ** 14 <= np.abs(X).max() < 2.0 ** 15
        assert np.all(np.abs(hi[t] + lo[t] - X) <= 2.0 ** -22 * np.abs(X) + 2.0 ** -25)
        blocks = (hi[t] + lo[t]).reshape(-1, 32).sum(axis=1) * 2.0 ** -6
        got = (bs[t, :, :8] + bs[t, :, 8:]).reshape(-1)
        bound = 2.0 ** -20 * np.abs(hi[t] + lo[t]).reshape(-1, 32).sum(axis=1) * 2.0 ** -6 + 2.0 ** -24
        assert np.all(np.abs(got - blocks) <= bound)


@pytest.mark.parametrize("tokens,rows,cols", [
    (1, 9, 256), (5, 128, 768), (128, 128, 2560), (130, 300, 2560), (200, 77, 1024),
    (300, 260, 9728), (64, 1000, 512), (129, 129, 1280)])
def test_gemm_f16_parity(tokens, rows, cols):
    f = synth.q4k_fields(rows, cols, [910, rows, cols])
    x = synth.activations(tokens, cols, [911, tokens])
    check(run(f, x), f, x, f"{tokens}x{rows}x{cols}")


@pytest.mark.parametrize("name", sorted(CASES))
def test_gemm_f16_edge_activations(name):
    tokens, rows, cols = 133, 140, 1536
    f, x = CASES[name](rows, cols, tokens, 920)
    check(run(f, x), f, x, name)


def test_gemm_f16_prefill_512_sampled():
    """The Qwen3-4B gate projection at 512 tokens, sampled rows, every token."""
    rows, cols, tokens = 9728, 2560, 512
    f = synth.q4k_fields(rows, cols, 930)
    x = synth.activations(tokens, cols, 931)
    y = run(f, x)
    sample = np.sort(np.random.default_rng(932).choice(rows, 256, replace=False))
    fs = slice_rows(f, sample)
    check(y[:, sample], fs, x, "prefill 512")
    assert q4k.q4k_device_error() == 0


def test_gemm_f16_is_deterministic():
    rows, cols, tokens = 256, 2560, 256
    f = synth.q4k_fields(rows, cols, 940)
    w = pack_dev(f)
    xd = torch.from_numpy(synth.activations(tokens, cols, 941)).cuda()
    sp = q4k.x_split_f16(xd)
    a = q4k.q4k_gemm_f16(w, rows, cols, *sp)
    b = q4k.q4k_gemm_f16(w, rows, cols, *sp)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("form", ["int8", "h16", "f16"])
def test_gemm_writes_exactly_its_output(form):
    """Canary: the GEMM writes every element of y and nothing around it
    (ragged token and row tails: partial tiles at both edges)."""
    rows, cols, tokens, pad = 300, 768, 130, 4096
    f = synth.q4k_fields(rows, cols, 950)
    w = pack_dev(f)
    xd = torch.from_numpy(synth.activations(tokens, cols, 951)).cuda()
    buf = torch.full((pad + tokens * rows + pad,), float("nan"), device="cuda")
    y = buf[pad:pad + tokens * rows].view(tokens, rows)
    if form == "f16":
        q4k.q4k_gemm_f16(w, rows, cols, *q4k.x_split_f16(xd), y=y)
    elif form == "h16":
        q4k.q4k_gemm_h16(w, rows, cols, *q4k.q8_quantize_h16(xd), y=y)
    else:
        q4k.q4k_gemm(w, rows, cols, *q4k.q8_quantize(xd), y=y)
    torch.cuda.synchronize()
    assert torch.isnan(buf[:pad]).all() and torch.isnan(buf[pad + tokens * rows:]).all(), "wrote outside y"
    assert not torch.isnan(y).any(), "left part of y unwritten"
    assert q4k.q4k_device_error() == 0
