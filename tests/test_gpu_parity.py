"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.  Integer stages are compared bit for bit; fp outputs must
satisfy |y - y_ref| <= 1e-4 * sum|w||x| element by element."""
import numpy as np
import pytest
import torch

from oracle import q4k as O
import synth
from _gpu import pack_dev, slice_rows, to_dev
import q4_weight_matmul_gb300 as q4k

pytestmark = pytest.mark.gpu
REL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    q4k.build()
    torch.cuda.init()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def assert_close(y, y_ref, norm, what=""):
    ok, worst = O.within_tolerance(y, y_ref, norm, REL)
    assert ok, f"{what}: worst error {worst:.3g} x the allowed 1e-4*sum|w||x|"


# ------------------------------------------------------------------ pack
@pytest.mark.parametrize("rows,cols", [(1, 256), (3, 768), (17, 2560), (64, 4096), (9728, 2560),
                                       (2560, 9728)])
def test_pack_bit_exact(rows, cols):
    f = synth.q4k_fields(rows, cols, [rows, cols])
    got = host(pack_dev(f)).reshape(rows, cols // 256, 144)
    assert np.array_equal(got, O.pack_block144(f))


def test_pack_ignores_bits_above_each_field():
    f = synth.q4k_fields(5, 512, 77)
    junk = dict(f)
    junk["sc"] = f["sc"] | 0xC0
    junk["m"] = f["m"] | 0x40
    junk["q"] = f["q"] | 0xF0
    assert np.array_equal(host(pack_dev(junk)), host(pack_dev(f)))


# ------------------------------------------------------------------ q8_1
def adversarial_activations():
    x = synth.activations(8, 512, 55)
    x[0, :32] = 0.0                                  # zero block
    x[1, :32] = np.arange(-16, 16) * 0.5             # exact ties after scaling
    x[1, 0] = -127 * 0.125
    x[2, :32] = 1e-44                                # d8 underflows to zero
    x[3, :32] = np.float32(3e38) * np.sign(np.arange(32) - 15.5)
    x[4, :32] = 2.5                                  # all equal
    x[5, 32:64] = -x[5, 32:64]
    x[6, :] *= np.float32(1e-30)
    return x


@pytest.mark.parametrize("case", ["adversarial", (1, 256), (5, 768), (512, 2560), (512, 9728)])
def test_q8_quantize_bit_exact(case):
    x = adversarial_activations() if case == "adversarial" else synth.activations(*case, 300)
    q, d8, s = q4k.q8_quantize(torch.from_numpy(x).cuda())
    rq, rd, rs = O.quantize_q8_1(x)
    assert np.array_equal(host(q), rq)
    assert np.array_equal(host(d8).view(np.uint32), rd.view(np.uint32))
    assert np.array_equal(host(s), rs)


# ------------------------------------------------------------------ GEMV
def run_gemv(f, x, r=None, w=None):
    rows, cols = f["q"].shape
    w = pack_dev(f) if w is None else w
    xd = torch.from_numpy(x).cuda()
    rd = None if r is None else torch.from_numpy(r).cuda()
    return host(q4k.q4k_gemv(w, rows, cols, xd, residual=rd))


@pytest.mark.parametrize("rows,cols,batch,res", [
    (1, 256, 1, False), (7, 768, 1, True), (8, 512, 2, False), (33, 2560, 1, False),
    (100, 1024, 3, True), (513, 4096, 4, False), (1024, 9728, 1, True), (257, 2560, 8, False),
    (3000, 256, 1, False)])
def test_gemv_parity(rows, cols, batch, res):
    f = synth.q4k_fields(rows, cols, [rows, cols, batch])
    x = synth.activations(batch, cols, [batch, cols])
    r = synth.residual(batch, rows, [7, rows]) if res else None
    y = run_gemv(f, x, r)
    y_ref, norm = O.gemv(f, x, r)
    assert_close(y, y_ref, norm, f"gemv {rows}x{cols} b{batch}")


def test_gemv_tall_matrix_sampled_rows():
    # many row blocks per SM and a long K: the kernel reduces in several passes
    rows, cols = 20000, 12288
    f = synth.q4k_fields(rows, cols, 4242)
    x = synth.activations(2, cols, 4243)
    y = run_gemv(f, x)
    rng = np.random.default_rng(9)
    sample = np.sort(rng.choice(rows, 384, replace=False))
    y_ref, norm = O.gemv(slice_rows(f, sample), x)
    assert_close(y[:, sample], y_ref, norm, "20000x12288 sampled")


def test_gemv_single_2048_seed0():
    f, x = synth.single_gemv_2048(0)
    y = run_gemv(f, x)
    y_ref, norm = O.gemv(f, x)
    assert_close(y, y_ref, norm, "2048x2048")


@pytest.mark.parametrize("batch", [1, 4])
def test_gemv_qwen3_4b_decode_set(batch):
    fields, xs = synth.decode_layer(synth.WL_DECODE_4B, 0, batch)
    for name, rows, cols, inp in synth.QWEN3_4B_LAYER:
        y = run_gemv(fields[name], xs[inp])
        y_ref, norm = O.gemv(fields[name], xs[inp])
        assert_close(y, y_ref, norm, name)


@pytest.mark.parametrize("batch", [1, 2])
def test_gemv_multi_qkv_and_gate_up(batch):
    fields, xs = synth.decode_layer(synth.WL_DECODE_4B, 1, batch)
    for names, inp in ((("q", "k", "v"), "attn_in"), (("gate", "up"), "mlp_in")):
        shapes = {n: (r, c) for n, r, c, _ in synth.QWEN3_4B_LAYER}
        cols = shapes[names[0]][1]
        ws = [pack_dev(fields[n]) for n in names]
        x = torch.from_numpy(xs[inp]).cuda()
        res = [torch.from_numpy(synth.residual(batch, shapes[n][0], [5, i])).cuda() for i, n in enumerate(names)]
        ys = q4k.q4k_gemv_multi(ws, [shapes[n][0] for n in names], cols, x, residuals=res)
        torch.cuda.synchronize()
        for n, y, r in zip(names, ys, res):
            y_ref, norm = O.gemv(fields[n], xs[inp], r.cpu().numpy())
            assert_close(y.cpu().numpy(), y_ref, norm, f"multi {n}")
        # the same fused call gives the same bits again
        again = q4k.q4k_gemv_multi(ws, [shapes[n][0] for n in names], cols, x, residuals=res)
        torch.cuda.synchronize()
        assert all(torch.equal(a, b) for a, b in zip(again, ys))


def test_gemv_multi_skips_empty_and_rejects_too_many():
    f = synth.q4k_fields(40, 512, 3)
    w = pack_dev(f)
    x = torch.from_numpy(synth.activations(1, 512, 4)).cuda()
    empty = torch.empty(0, dtype=torch.uint8, device="cuda")
    ys = q4k.q4k_gemv_multi([w, w], [40, 0], 512, x,
                            ys=[torch.empty((1, 40), device="cuda"), torch.empty((1, 0), device="cuda")])
    y_ref, norm = O.gemv(f, synth.activations(1, 512, 4))
    assert_close(host(ys[0]), y_ref, norm, "multi with an empty matrix")
    with pytest.raises(q4k.Q4KError):
        q4k.q4k_gemv_multi([w] * 5, [40] * 5, 512, x)


def test_gemv_is_deterministic():
    f = synth.q4k_fields(2560, 9728, 5)
    x = synth.activations(1, 9728, 6)
    w = pack_dev(f)
    assert np.array_equal(run_gemv(f, x, w=w), run_gemv(f, x, w=w))


def test_gemv_leaves_neighbouring_memory_alone():
    f = synth.q4k_fields(37, 512, 8)
    x = torch.from_numpy(synth.activations(2, 512, 9)).cuda()
    w = pack_dev(f)
    guard = torch.full((2 * 37 + 64,), 12345.0, device="cuda")
    y = guard[32:32 + 2 * 37].view(2, 37)
    q4k.q4k_gemv(w, 37, 512, x, y=y)
    g = host(guard)
    assert np.all(g[:32] == 12345.0) and np.all(g[32 + 74:] == 12345.0)


# ------------------------------------------------------------------ GEMM
def quantize_dev(x):
    q, d8, s = q4k.q8_quantize(torch.from_numpy(x).cuda())
    return q, d8, s


# token counts up to 32 run the q8_1 GEMV, the rest the tensor-core kernel
@pytest.mark.parametrize("tokens,rows,cols", [
    (1, 64, 256), (5, 70, 512), (15, 33, 768), (16, 128, 256), (40, 64, 256), (64, 128, 2560),
    (130, 200, 768), (33, 9, 4096), (200, 300, 1280), (129, 257, 512)])
def test_gemm_parity_and_block_dots(tokens, rows, cols):
    f = synth.q4k_fields(rows, cols, [tokens, rows, cols])
    x = synth.activations(tokens, cols, [cols, tokens])
    w = pack_dev(f)
    q, d8, s = quantize_dev(x)
    y = host(q4k.q4k_gemm(w, rows, cols, q, d8, s))
    rq, rd, rs = O.quantize_q8_1(x)
    y_ref, norm = O.mmq(f, rq, rd, rs)
    assert_close(y, y_ref, norm, f"gemm {tokens}x{rows}x{cols}")
    p = host(q4k.q4k_gemm_blockdots(w, rows, cols, q))
    assert np.array_equal(p, O.block_dots(f["q"], rq))


@pytest.mark.parametrize("case", ["adversarial", (3, 256), (512, 2560), (130, 9728)])
def test_q8_quantize_h16_matches_the_int8_form(case):
    """The binary16 quants hold exactly the int8 quants' values; d8 and the
    sums are the same bits (and so equal to the oracle's)."""
    x = adversarial_activations() if case == "adversarial" else synth.activations(*case, 301)
    xd = torch.from_numpy(x).cuda()
    q, d8, s = q4k.q8_quantize(xd)
    qh, dh, sh = q4k.q8_quantize_h16(xd)
    rq, rd, rs = O.quantize_q8_1(x)
    assert np.array_equal(host(qh).astype(np.float32), rq.astype(np.float32))
    assert np.array_equal(host(q), rq)
    assert np.array_equal(host(dh).view(np.uint32), rd.view(np.uint32))
    assert np.array_equal(host(sh), rs)


@pytest.mark.parametrize("tokens,rows,cols", [
    (1, 64, 256), (7, 70, 512), (16, 128, 256), (40, 64, 768), (64, 128, 2560),
    (130, 200, 768), (33, 9, 4096), (200, 300, 1280), (129, 257, 512), (256, 384, 3328)])
def test_gemm_h16_parity_and_block_dots(tokens, rows, cols):
    f = synth.q4k_fields(rows, cols, [tokens, rows, cols, 16])
    x = synth.activations(tokens, cols, [cols, tokens, 16])
    w = pack_dev(f)
    q, d8, s = q4k.q8_quantize_h16(torch.from_numpy(x).cuda())
    y = host(q4k.q4k_gemm_h16(w, rows, cols, q, d8, s))
    rq, rd, rs = O.quantize_q8_1(x)
    y_ref, norm = O.mmq(f, rq, rd, rs)
    assert_close(y, y_ref, norm, f"gemm_h16 {tokens}x{rows}x{cols}")
    p = host(q4k.q4k_gemm_blockdots_h16(w, rows, cols, q))
    assert np.array_equal(p, O.block_dots(f["q"], rq))


@pytest.mark.parametrize("tokens", [8, 48])
def test_gemm_h16_block_dots_at_the_extremes(tokens):
    rows, cols = 16, 512
    f = synth.q4k_fields(rows, cols, 90)
    f["q"][:8] = 15
    f["q"][8:, ::7] = 0
    x = np.full((tokens, cols), 1.0, np.float32)
    x[1:4:2] = -1.0
    x[4:, ::5] *= -1.0
    q, _, _ = q4k.q8_quantize_h16(torch.from_numpy(x).cuda())
    p = host(q4k.q4k_gemm_blockdots_h16(pack_dev(f), rows, cols, q))
    assert np.array_equal(p, O.block_dots(f["q"], O.quantize_q8_1(x)[0]))
    assert p.max() == 15 * 127 * 32 and p.min() == -15 * 127 * 32


def test_gemm_h16_equals_the_int8_entry_point():
    """Same MMQ form, same q8_1 values: both entry points agree within the
    bound of each against the oracle (they share no kernel code)."""
    rows, cols, tokens = 300, 2560, 200
    f = synth.q4k_fields(rows, cols, 3131)
    x = synth.activations(tokens, cols, 3132)
    w = pack_dev(f)
    xd = torch.from_numpy(x).cuda()
    y8 = host(q4k.q4k_gemm(w, rows, cols, *q4k.q8_quantize(xd)))
    yh = host(q4k.q4k_gemm_h16(w, rows, cols, *q4k.q8_quantize_h16(xd)))
    rq, rd, rs = O.quantize_q8_1(x)
    y_ref, norm = O.mmq(f, rq, rd, rs)
    assert_close(y8, y_ref, norm, "int8 entry")
    assert_close(yh, y_ref, norm, "h16 entry")
    assert_close(yh, y8.astype(np.float64), 2 * norm, "h16 vs int8")


@pytest.mark.parametrize("batch,rows,cols", [(1, 96, 256), (2, 100, 768), (4, 257, 2560), (8, 1000, 4096),
                                             (5, 33, 9728)])
def test_gemv_q8_parity(batch, rows, cols):
    """The few-token MMQ as a GEMV, with and without a residual."""
    f = synth.q4k_fields(rows, cols, [batch, rows, cols, 8])
    x = synth.activations(batch, cols, [cols, batch, 8])
    r = synth.residual(batch, rows, [rows, batch, 8])
    w = pack_dev(f)
    q, d8, s = quantize_dev(x)
    rq, rd, rs = O.quantize_q8_1(x)
    y_ref, norm = O.mmq(f, rq, rd, rs)
    y = host(q4k.q4k_gemv_q8(w, rows, cols, q, d8, s))
    assert_close(y, y_ref, norm, f"gemv_q8 {batch}x{rows}x{cols}")
    yr = host(q4k.q4k_gemv_q8(w, rows, cols, q, d8, s, residual=torch.from_numpy(r).cuda()))
    assert_close(yr, y_ref + r, norm + np.abs(r.astype(np.float64)), f"gemv_q8 {batch}x{rows}x{cols} + residual")


@pytest.mark.parametrize("tokens", [3, 8, 9, 32])
def test_few_token_gemm_runs_the_gemv_and_its_dots_are_exact(tokens):
    """q4k_gemm / q4k_gemm_h16 with up to 32 tokens go through the q8_1 GEMV
    (a launch per 8 tokens); outputs within the bound, block dots bit-exact."""
    rows, cols = 300, 2560
    f = synth.q4k_fields(rows, cols, [tokens, 31])
    x = synth.activations(tokens, cols, [tokens, 32])
    w = pack_dev(f)
    xd = torch.from_numpy(x).cuda()
    rq, rd, rs = O.quantize_q8_1(x)
    y_ref, norm = O.mmq(f, rq, rd, rs)
    q, d8, s = q4k.q8_quantize(xd)
    qh, dh, sh = q4k.q8_quantize_h16(xd)
    assert_close(host(q4k.q4k_gemm(w, rows, cols, q, d8, s)), y_ref, norm, "int8 entry")
    assert_close(host(q4k.q4k_gemm_h16(w, rows, cols, qh, dh, sh)), y_ref, norm, "h16 entry")
    dots = O.block_dots(f["q"], rq)
    assert np.array_equal(host(q4k.q4k_gemm_blockdots(w, rows, cols, q)), dots)
    assert np.array_equal(host(q4k.q4k_gemm_blockdots_h16(w, rows, cols, qh)), dots)


@pytest.mark.parametrize("tokens", [8, 48])
def test_gemm_block_dots_at_the_extremes(tokens):
    # rows 0-7 hold q = 15 everywhere and tokens 0-3 are all +1 or all -1, so
    # those block dots reach the extreme +-15*127*32; the rest are mixed.
    # (8 tokens run the q8_1 GEMV, 48 the tensor-core kernel.)
    rows, cols = 16, 512
    f = synth.q4k_fields(rows, cols, 90)
    f["q"][:8] = 15
    f["q"][8:, ::7] = 0
    x = np.full((tokens, cols), 1.0, np.float32)
    x[1:4:2] = -1.0
    x[4:, ::5] *= -1.0
    w = pack_dev(f)
    q, _, _ = quantize_dev(x)
    p = host(q4k.q4k_gemm_blockdots(w, rows, cols, q))
    assert np.array_equal(p, O.block_dots(f["q"], O.quantize_q8_1(x)[0]))
    assert p.max() == 15 * 127 * 32 and p.min() == -15 * 127 * 32


@pytest.mark.parametrize("form", ["int8", "h16"])
def test_gemm_prefill_512_sampled(form):
    fields, xs = synth.prefill_4b_512()
    rng = np.random.default_rng(123)
    for name, inp in (("gate", "mlp_in"), ("down", "down_in")):
        f, x = fields[name], xs[inp]
        rows, cols = f["q"].shape
        w = pack_dev(f)
        if form == "int8":
            q, d8, s = quantize_dev(x)
            y = host(q4k.q4k_gemm(w, rows, cols, q, d8, s))
        else:
            q, d8, s = q4k.q8_quantize_h16(torch.from_numpy(x).cuda())
            y = host(q4k.q4k_gemm_h16(w, rows, cols, q, d8, s))
        rq, rd, rs = O.quantize_q8_1(x)
        sample = np.sort(rng.choice(rows, 256, replace=False))
        y_ref, norm = O.mmq(slice_rows(f, sample), rq, rd, rs)
        assert_close(y[:, sample], y_ref, norm, f"{name} rows sample")
        toks = np.sort(rng.choice(512, 16, replace=False))
        y_ref, norm = O.mmq(f, rq[toks], rd[toks], rs[toks])
        assert_close(y[toks], y_ref, norm, f"{name} token sample")


# ------------------------------------------------------------------ unpack
@pytest.mark.parametrize("rows,cols", [(1, 256), (19, 768), (300, 2560)])
def test_unpack_inverts_the_gpu_pack(rows, cols):
    """Round trip on the GPU alone: the fields come back bit for bit
    (q4k_unpack does not share the packer's code path)."""
    f = synth.q4k_fields(rows, cols, [rows, cols, 5])
    got = q4k.q4k_unpack(pack_dev(f), rows, cols)
    torch.cuda.synchronize()
    for k in ("d", "dmin"):
        assert np.array_equal(got[k].cpu().numpy().view(np.uint16), f[k]), k
    for k in ("sc", "m", "q"):
        assert np.array_equal(got[k].cpu().numpy(), f[k]), k


def test_unpack_reads_the_oracles_bytes():
    """The GPU unpack of bytes packed by the oracle gives the oracle's fields,
    and those match the oracle's own unpack."""
    rows, cols = 40, 1024
    f = synth.q4k_fields(rows, cols, 606)
    packed = O.pack_block144(f)
    w = torch.from_numpy(packed.reshape(-1)).cuda()
    got = q4k.q4k_unpack(w, rows, cols)
    ref = O.unpack_block144(packed)
    torch.cuda.synchronize()
    for k in ("d", "dmin"):
        assert np.array_equal(got[k].cpu().numpy().view(np.uint16), ref[k]), k
    for k in ("sc", "m", "q"):
        assert np.array_equal(got[k].cpu().numpy(), ref[k]), k
