"""GPU parity at the full sizes of the larger workloads, on outputs the oracle
can compute one by one (sampled rows and tokens), in the launch form the
benchmark uses (QKV and gate/up fused into one GEMV launch each):

* the 36-layer Qwen3-4B-shaped decode stack at batch 1 and 4 (first, middle
  and last layer; every projection);
* its 2048-token prefill (one layer, all seven projections: q8_1 bit-exact
  on the whole input, GEMM on sampled rows and tokens);
* the 4096-token Qwen3-8B MLP prefill (gate/up 12288x4096, down 4096x12288).
"""
import numpy as np
import pytest
import torch

from oracle import q4k as O
import synth
from _gpu import pack_dev, slice_rows
import q4_weight_matmul_gb300 as q4k

pytestmark = pytest.mark.gpu
REL = 1e-4
STACK_LAYERS = 36


@pytest.fixture(scope="module", autouse=True)
def _built():
    q4k.build()
    torch.cuda.init()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def assert_close(y, y_ref, norm, what):
    ok, worst = O.within_tolerance(y, y_ref, norm, REL)
    assert ok, f"{what}: worst error {worst:.3g} x the allowed 1e-4*sum|w||x|"


SHAPES = {name: (rows, cols, inp) for name, rows, cols, inp in synth.QWEN3_4B_LAYER}
GROUPS = (("q", "k", "v"), ("o",), ("gate", "up"), ("down",))


@pytest.mark.parametrize("batch", [1, 4])
@pytest.mark.parametrize("layer", [0, STACK_LAYERS // 2, STACK_LAYERS - 1])
def test_decode_stack_layer(layer, batch):
    fields, xs = synth.decode_layer(synth.WL_STACK_4B, layer, batch)
    rng = np.random.default_rng(1000 + layer * 10 + batch)
    w = {name: pack_dev(fields[name]) for name in SHAPES}
    for names in GROUPS:
        rows = [SHAPES[n][0] for n in names]
        cols, inp = SHAPES[names[0]][1], SHAPES[names[0]][2]
        x = torch.from_numpy(xs[inp]).cuda()
        if len(names) == 1:
            ys = [q4k.q4k_gemv(w[names[0]], rows[0], cols, x)]
        else:
            ys = q4k.q4k_gemv_multi([w[n] for n in names], rows, cols, x)
        for name, y in zip(names, ys):
            y = host(y)
            sample = np.sort(rng.choice(SHAPES[name][0], 256, replace=False))
            y_ref, norm = O.gemv(slice_rows(fields[name], sample), xs[inp])
            assert_close(y[:, sample], y_ref, norm, f"layer {layer} batch {batch} {name}")


def check_prefill(fields, x, rows, cols, rng, what, n_rows=96, n_tok=8):
    w = pack_dev(fields)
    q, d8, s = q4k.q8_quantize(torch.from_numpy(x).cuda())
    rq, rd, rs = O.quantize_q8_1(x)
    assert np.array_equal(host(q), rq), f"{what}: q8 codes"
    assert np.array_equal(host(d8), rd), f"{what}: q8 scales"
    assert np.array_equal(host(s), rs), f"{what}: q8 sums"
    y = host(q4k.q4k_gemm(w, rows, cols, q, d8, s))
    # the binary16 form: same quants, and the tensor-copy GEMM on them
    qh, dh, sh = q4k.q8_quantize_h16(torch.from_numpy(x).cuda())
    assert np.array_equal(host(qh).astype(np.float32), rq.astype(np.float32)), f"{what}: h16 codes"
    yh = host(q4k.q4k_gemm_h16(w, rows, cols, qh, dh, sh))
    tokens = x.shape[0]
    # sampled rows on sampled tokens, and every row on a few tokens
    trow = np.sort(rng.choice(tokens, 64, replace=False))
    sample = np.sort(rng.choice(rows, n_rows, replace=False))
    y_ref, norm = O.mmq(slice_rows(fields, sample), rq[trow], rd[trow], rs[trow])
    assert_close(y[np.ix_(trow, sample)], y_ref, norm, f"{what} rows sample")
    assert_close(yh[np.ix_(trow, sample)], y_ref, norm, f"{what} rows sample (h16)")
    toks = np.sort(rng.choice(tokens, n_tok, replace=False))
    y_ref, norm = O.mmq(fields, rq[toks], rd[toks], rs[toks])
    assert_close(y[toks], y_ref, norm, f"{what} token sample")
    assert_close(yh[toks], y_ref, norm, f"{what} token sample (h16)")


def test_stack_prefill_2048_tokens():
    layer, tokens = 0, 2048
    fields, _ = synth.decode_layer(synth.WL_STACK_4B, layer, 1)
    xs = {name: synth.activations(tokens, cols, synth.layer_seed(synth.WL_STACK_4B, layer, 300 + j))
          for j, (name, cols) in enumerate(synth.QWEN3_4B_INPUTS)}
    rng = np.random.default_rng(2048)
    for name, (rows, cols, inp) in SHAPES.items():
        check_prefill(fields[name], xs[inp], rows, cols, rng, f"2048-token {name}")


def test_qwen3_8b_mlp_prefill_4096_tokens():
    fields, xs = synth.prefill_8b_4096()
    rng = np.random.default_rng(4096)
    for name, rows, cols, inp in synth.QWEN3_8B_MLP:
        check_prefill(fields[name], xs[inp], rows, cols, rng, f"4096-token {name}", n_rows=64, n_tok=4)
