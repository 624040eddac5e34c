"""GPU parity of the Q6_K path: the device packer against the oracle's GGUF
bytes, the GPU-layout round trips, and q6k_gemv against the oracle's fp64
GEMV within |y - y_ref| <= 1e-4 * (sum_k |w||x| + |residual|), on shapes
that span several row blocks and stages with ragged tails, at the decode
batch sizes 1..8, and on the activation patterns where the fixed-point
staging of x is weakest (one large element per block with tiny others,
blocks of tiny or huge |x|, non-negative x)."""
import numpy as np
import pytest
import torch

from oracle import q4k as O
from oracle import q6k as O6
import synth
import q4_weight_matmul_gb300 as q4k

pytestmark = pytest.mark.gpu
REL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    q4k.build()
    torch.cuda.init()


def f16_bits(v):
    return np.asarray(v, np.float16).view(np.uint16)


def dev_fields(f):
    return (torch.from_numpy(np.ascontiguousarray(f["d"]).view(np.int16)).cuda(),
            torch.from_numpy(np.ascontiguousarray(f["sc"])).cuda(),
            torch.from_numpy(np.ascontiguousarray(f["q"])).cuda())


def pack_gpu(f):
    return q4k.q6k_pack(*dev_fields(f), layout=q4k.Q6K_GPU)


def check(y, f, x, residual=None, rows=None):
    sub = f if rows is None else {k: v[rows] for k, v in f.items()}
    if residual is not None and rows is not None:
        residual = residual[:, rows]
    y_ref, norm = O6.gemv_q6k(sub, x, residual)
    yy = y.cpu().numpy()
    if rows is not None:
        yy = yy[:, rows]
    ok, worst = O.within_tolerance(yy, y_ref, norm, REL)
    assert ok, f"{worst:.3g} x the allowed error"


# ------------------------------------------------------------------ packing
@pytest.mark.parametrize("rows,cols", [(1, 256), (37, 2560), (5, 9728)])
def test_device_gguf_pack_matches_the_oracle_bytes(rows, cols):
    f = synth.q6k_fields(rows, cols, [700, rows])
    w = q4k.q6k_pack(*dev_fields(f), layout=q4k.Q6K_GGUF)
    assert w.numel() == rows * cols // 256 * 210
    assert np.array_equal(w.cpu().numpy().reshape(rows, cols // 256, 210), O6.pack_q6k(f))


@pytest.mark.parametrize("rows,cols", [(1, 256), (37, 2560), (5, 9728)])
def test_gpu_layout_round_trips_and_repack_agrees(rows, cols):
    f = synth.q6k_fields(rows, cols, [701, rows])
    w = pack_gpu(f)
    row_bytes = (cols // 256 * 210 + 15) // 16 * 16
    assert w.numel() == rows * row_bytes == q4k.q6k_packed_bytes(rows, cols)
    back = q4k.q6k_unpack(w, rows, cols)
    assert np.array_equal(back["d"].cpu().numpy().view(np.uint16), f["d"])
    assert np.array_equal(back["sc"].cpu().numpy(), f["sc"])
    assert np.array_equal(back["q"].cpu().numpy(), f["q"])
    # padding bytes are zero
    pad = w.view(rows, row_bytes)[:, cols // 256 * 210:]
    assert not pad.any()
    # GGUF -> GPU equals packing the fields straight to the GPU layout, and back
    gguf = torch.from_numpy(O6.pack_q6k(f).reshape(-1)).cuda()
    w2 = q4k.q6k_repack(gguf, rows, cols)
    assert torch.equal(w2, w)
    g2 = q4k.q6k_repack(w, rows, cols, src_layout=q4k.Q6K_GPU, dst_layout=q4k.Q6K_GGUF)
    assert torch.equal(g2, gguf)
    back2 = q4k.q6k_unpack(gguf, rows, cols, layout=q4k.Q6K_GGUF)
    assert np.array_equal(back2["q"].cpu().numpy(), f["q"])


def test_repack_accepts_a_gguf_source_at_an_odd_block_offset():
    """GGUF blocks are 210 bytes, so a matrix inside a file image starts on
    a 2-byte boundary only; the converter reads it as such."""
    rows, cols = 9, 512
    f = synth.q6k_fields(rows, cols, 702)
    img = np.zeros(210 + rows * cols // 256 * 210, np.uint8)
    img[210:] = O6.pack_q6k(f).reshape(-1)
    gguf = torch.from_numpy(img).cuda()[210:]            # offset 210: 2-byte aligned, not 16
    assert gguf.data_ptr() % 16 != 0
    assert torch.equal(q4k.q6k_repack(gguf, rows, cols), pack_gpu(f))


# --------------------------------------------------------------------- GEMV
@pytest.mark.parametrize("rows,cols,batch", [
    (1000, 2560, 1), (1000, 2560, 2), (333, 2560, 3), (1024, 2560, 4),
    (300, 9728, 1), (300, 9728, 4), (77, 1024, 5), (64, 2560, 6), (45, 768, 7), (130, 2560, 8),
    (1, 256, 1), (31, 256, 8)])
def test_q6k_gemv_parity(rows, cols, batch):
    f = synth.q6k_fields(rows, cols, [710, rows, cols])
    x = synth.activations(batch, cols, [711, batch])
    y = q4k.q6k_gemv(pack_gpu(f), rows, cols, torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    check(y, f, x)


@pytest.mark.parametrize("batch", [1, 4])
def test_q6k_gemv_residual_and_in_place(batch):
    rows, cols = 2560, 9728
    f = synth.q6k_fields(rows, cols, 712)
    x = synth.activations(batch, cols, 713)
    r = synth.residual(batch, rows, 714)
    w = pack_gpu(f)
    xd = torch.from_numpy(x).cuda()
    y = q4k.q6k_gemv(w, rows, cols, xd, residual=torch.from_numpy(r).cuda())
    yi = torch.from_numpy(r).cuda()
    q4k.q6k_gemv(w, rows, cols, xd, residual=yi, y=yi)       # y aliases residual
    torch.cuda.synchronize()
    assert torch.equal(y, yi)
    sample = np.random.default_rng(715).choice(rows, 256, replace=False)
    check(y, f, x, r, rows=sample)


def test_q6k_gemv_is_deterministic_and_zero_quants_give_zero():
    rows, cols = 500, 2560
    f = synth.q6k_fields(rows, cols, 716)
    x = torch.from_numpy(synth.activations(2, cols, 717)).cuda()
    w = pack_gpu(f)
    a = q4k.q6k_gemv(w, rows, cols, x)
    b = q4k.q6k_gemv(w, rows, cols, x)
    assert torch.equal(a, b)
    f["q"][:] = 32
    z = q4k.q6k_gemv(pack_gpu(f), rows, cols, x)
    assert not z.any()


def test_q6k_gemv_full_size_output_head_sampled():
    """The Qwen3-4B output projection (151936 x 2560), batch 1, sampled rows."""
    rows, cols = 151936, 2560
    f = synth.q6k_fields(rows, cols, 718)
    x = synth.activations(1, cols, 719)
    y = q4k.q6k_gemv(pack_gpu(f), rows, cols, torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    rng = np.random.default_rng(720)
    sample = np.concatenate([rng.choice(rows, 512, replace=False), np.arange(rows - 40, rows)])
    check(y, f, x, rows=sample)


# ------------------------------------------------------- weak-staging inputs
def _q6_outlier(rows, cols, batch, small, seed):
    rng = np.random.default_rng(seed)
    f = synth.q6k_fields(rows, cols, [seed, 1])
    x = (rng.standard_normal((batch, cols)) * small).astype(np.float32)
    pos = rng.integers(0, 32, cols // 32)
    for j in range(cols // 32):
        x[:, 32 * j + pos[j]] = np.where(rng.random(batch) < 0.5, -1.0, 1.0) * (1 + rng.random(batch))
        f["q"][:, 32 * j + pos[j]] = 32              # w = 0 at the large element
    return f, x


def _q6_wide(rows, cols, batch, seed):
    rng = np.random.default_rng(seed)
    f = synth.q6k_fields(rows, cols, [seed, 11])
    mag = 2.0 ** rng.uniform(-12, -10, (batch, cols))
    x = (mag * np.where(rng.random((batch, cols)) < 0.5, -1.0, 1.0)).astype(np.float32)
    pos = rng.integers(0, 32, cols // 32)
    for j in range(cols // 32):
        x[:, 32 * j + pos[j]] = 1.0 + rng.random(batch)
    return f, x


def _q6_scaled(rows, cols, batch, seed, exp, d_lo, d_hi):
    rng = np.random.default_rng(seed)
    f = synth.q6k_fields(rows, cols, [seed, 2])
    f["d"] = f16_bits(rng.uniform(d_lo, d_hi, (rows, cols // 256)))
    x = (rng.standard_normal((batch, cols)) * 2.0 ** exp).astype(np.float32)
    return f, x


CASES = {
    "outlier_1e-3": lambda b: _q6_outlier(200, 2560, b, 1e-3, 730),
    "outlier_1e-6": lambda b: _q6_outlier(200, 2560, b, 1e-6, 731),
    "outlier_1e-12": lambda b: _q6_outlier(200, 2560, b, 1e-12, 732),
    "wide": lambda b: _q6_wide(200, 2560, b, 733),
    "tiny": lambda b: _q6_scaled(200, 2560, b, 734, -110, 2.0 ** 10, 2.0 ** 14),
    "huge": lambda b: _q6_scaled(200, 2560, b, 735, 95, 2.0 ** -14, 2.0 ** -10),
    "nonneg": lambda b: (synth.q6k_fields(200, 9728, 736),
                         np.abs(synth.activations(b, 9728, 737))),
}


@pytest.mark.parametrize("batch", [1, 3])
@pytest.mark.parametrize("name", sorted(CASES))
def test_q6k_gemv_weak_staging_inputs(name, batch):
    f, x = CASES[name](batch)
    rows, cols = f["q"].shape
    y = q4k.q6k_gemv(pack_gpu(f), rows, cols, torch.from_numpy(np.ascontiguousarray(x)).cuda())
    torch.cuda.synchronize()
    check(y, f, x)
    assert q4k.q4k_device_error() == 0


# --------------------------------------------------------- q8_1 activations
def _q8(x):
    q8, d8, s = O.quantize_q8_1(x)
    return (q8, d8, s), tuple(torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in (q8, d8, s))


@pytest.mark.parametrize("tokens", [1, 5, 8, 9, 17, 40])
def test_q6k_gemm_group_dots_are_exact(tokens):
    rows, cols = 77, 768
    f = synth.q6k_fields(rows, cols, [760, tokens])
    x = synth.activations(tokens, cols, [761, tokens])
    (q8, _, _), (q8d, _, _) = _q8(x)
    p = q4k.q6k_gemm_blockdots(pack_gpu(f), rows, cols, q8d)
    torch.cuda.synchronize()
    assert np.array_equal(p.cpu().numpy(), O6.block_dots_q6k(f["q"], q8))


def test_q6k_group_dots_at_the_extremes():
    """q = 0 and 63 (q - 32 = -32 and 31) against q8 = -127 and 127."""
    rows, cols = 40, 512
    f = synth.q6k_fields(rows, cols, 762)
    f["q"][: rows // 2] = 0
    f["q"][rows // 2:] = 63
    q8 = np.where(np.arange(cols) % 3 == 0, 127, -127).astype(np.int8)[None, :].repeat(3, axis=0)
    p = q4k.q6k_gemm_blockdots(pack_gpu(f), rows, cols, torch.from_numpy(q8).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(p.cpu().numpy(), O6.block_dots_q6k(f["q"], q8))


@pytest.mark.parametrize("tokens,rows,cols", [(1, 1000, 2560), (4, 333, 2560), (8, 300, 9728),
                                              (9, 130, 1024), (33, 2560, 9728), (40, 64, 256)])
def test_q6k_gemm_parity(tokens, rows, cols):
    f = synth.q6k_fields(rows, cols, [763, rows, tokens])
    x = synth.activations(tokens, cols, [764, tokens])
    (q8, d8, _), (q8d, d8d, sd) = _q8(x)
    y = q4k.q6k_gemm(pack_gpu(f), rows, cols, q8d, d8d, sd)
    torch.cuda.synchronize()
    ok, worst = O.within_tolerance(y.cpu().numpy(), *O6.mmq_q6k(f, q8, d8), REL)
    assert ok, f"{worst:.3g} x the allowed error"


@pytest.mark.parametrize("batch", [1, 3, 8])
def test_q6k_gemv_q8_with_residual_and_without_sums(batch):
    rows, cols = 2560, 9728
    f = synth.q6k_fields(rows, cols, [765, batch])
    x = synth.activations(batch, cols, [766, batch])
    r = synth.residual(batch, rows, [767, batch])
    (q8, d8, _), (q8d, d8d, _) = _q8(x)
    y = q4k.q6k_gemv_q8(pack_gpu(f), rows, cols, q8d, d8d, None, residual=torch.from_numpy(r).cuda())
    torch.cuda.synchronize()
    y_ref, norm = O6.mmq_q6k(f, q8, d8)
    ok, worst = O.within_tolerance(y.cpu().numpy(), y_ref + r, norm + np.abs(r), REL)
    assert ok, f"{worst:.3g} x the allowed error"
    assert q4k.q4k_device_error() == 0



# ------------------------------------------------ fp16-activation tensor-core GEMM
def _f16_norm(f, x):
    w = np.abs(O6.dequantize_q6k(f).astype(np.float64))
    x64 = np.abs(np.asarray(x, np.float64))
    return x64 @ w.T + 2.0 ** -16 * x64.max(axis=1, keepdims=True) * w.sum(axis=1)[None, :]


@pytest.mark.parametrize("tokens,rows,cols", [
    (1, 9, 256), (5, 128, 768), (128, 128, 2560), (130, 300, 2560), (200, 77, 1024),
    (300, 260, 9728), (64, 1000, 512), (129, 129, 2304)])
def test_q6k_gemm_f16_parity(tokens, rows, cols):
    f = synth.q6k_fields(rows, cols, [770, rows, cols])
    x = synth.activations(tokens, cols, [771, tokens])
    y = q4k.q6k_gemm_f16(pack_gpu(f), rows, cols, *q4k.x_split_f16(torch.from_numpy(x).cuda()))
    torch.cuda.synchronize()
    y_ref, _ = O6.gemv_q6k(f, x)
    ok, worst = O.within_tolerance(y.cpu().numpy(), y_ref, _f16_norm(f, x), REL)
    assert ok, f"{worst:.3g} x the allowed error"


def test_q6k_gemm_f16_extreme_weights():
    """sc = -128 / 127 with q = 0 / 63: |sc (q - 32)| above 2048, where the
    weight operand needs its low part."""
    rows, cols, tokens = 64, 1024, 40
    f = synth.q6k_fields(rows, cols, 772)
    f["sc"][: rows // 2] = -128
    f["sc"][rows // 2:] = 127
    f["q"][:, ::2] = 0
    f["q"][:, 1::2] = 63
    x = synth.activations(tokens, cols, 773)
    y = q4k.q6k_gemm_f16(pack_gpu(f), rows, cols, *q4k.x_split_f16(torch.from_numpy(x).cuda()))
    torch.cuda.synchronize()
    y_ref, _ = O6.gemv_q6k(f, x)
    ok, worst = O.within_tolerance(y.cpu().numpy(), y_ref, _f16_norm(f, x), REL)
    assert ok, f"{worst:.3g} x the allowed error"


@pytest.mark.parametrize("name", sorted(CASES))
def test_q6k_gemm_f16_weak_staging_inputs(name):
    f, x = CASES[name](3)
    rows, cols = f["q"].shape
    x = np.ascontiguousarray(np.tile(x, (45, 1)))     # 135 tokens: two token tiles
    y = q4k.q6k_gemm_f16(pack_gpu(f), rows, cols, *q4k.x_split_f16(torch.from_numpy(x).cuda()))
    torch.cuda.synchronize()
    y_ref, _ = O6.gemv_q6k(f, x)
    ok, worst = O.within_tolerance(y.cpu().numpy(), y_ref, _f16_norm(f, x), REL)
    assert ok, f"{name}: {worst:.3g} x the allowed error"
    assert q4k.q4k_device_error() == 0


def test_q6k_gemm_f16_canary_and_determinism():
    rows, cols, tokens, pad = 300, 768, 130, 4096
    f = synth.q6k_fields(rows, cols, 774)
    w = pack_gpu(f)
    sp = q4k.x_split_f16(torch.from_numpy(synth.activations(tokens, cols, 775)).cuda())
    buf = torch.full((pad + tokens * rows + pad,), float("nan"), device="cuda")
    y = buf[pad:pad + tokens * rows].view(tokens, rows)
    q4k.q6k_gemm_f16(w, rows, cols, *sp, y=y)
    y2 = q4k.q6k_gemm_f16(w, rows, cols, *sp)
    torch.cuda.synchronize()
    assert torch.isnan(buf[:pad]).all() and torch.isnan(buf[pad + tokens * rows:]).all()
    assert not torch.isnan(y).any()
    assert torch.equal(y, y2)
