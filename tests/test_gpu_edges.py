"""GPU parity on the activation patterns where a fixed-point staging of x is
weakest, through every GEMV entry point and the GEMM: one large element per
32-wide block with the rest 10^-3, 10^-6 or 10^-12 of it (on rows whose weight at
the large element is zero, so the small ones carry the whole result), blocks
whose largest |x| is below 2^-104 or above 2^100, non-negative x, and weights
whose scale and min terms cancel.  Each output must satisfy
|y - y_ref| <= 1e-4 * sum_k |w||x| (the cancelling weights: the magnitude
normaliser sum_k (|d sc q| + |dmin m|) |x|)."""
import numpy as np
import pytest
import torch

from oracle import q4k as O
import synth
from _gpu import pack_dev
import q4_weight_matmul_gb300 as q4k

pytestmark = pytest.mark.gpu
REL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    q4k.build()
    torch.cuda.init()


def f16_bits(v):
    return np.asarray(v, np.float16).view(np.uint16)


def outlier_case(rows, cols, batch, small, seed):
    """x: per 32-block one element of magnitude ~1 (random position), the
    rest `small` * N(0,1); weights zero at every large element (q = 0 there
    and m = 0 for the sub-block)."""
    rng = np.random.default_rng(seed)
    f = synth.q4k_fields(rows, cols, [seed, 1])
    nsub = cols // 32
    x = (rng.standard_normal((batch, cols)) * small).astype(np.float32)
    pos = rng.integers(0, 32, nsub)
    for j in range(nsub):
        x[:, 32 * j + pos[j]] = np.where(rng.random(batch) < 0.5, -1.0, 1.0) * (1 + rng.random(batch))
        f["q"][:, 32 * j + pos[j]] = 0
    f["m"][:, :] = 0
    return f, x


def wide_case(rows, cols, batch, seed):
    """per 32-block one element ~1 and the rest between 2^-12 and 2^-10 of
    it: every block needs the fourth digit plane (tier 2), none the fp32 path"""
    rng = np.random.default_rng(seed)
    f = synth.q4k_fields(rows, cols, [seed, 11])
    mag = 2.0 ** rng.uniform(-12, -10, (batch, cols))
    x = (mag * np.where(rng.random((batch, cols)) < 0.5, -1.0, 1.0)).astype(np.float32)
    pos = rng.integers(0, 32, cols // 32)
    for j in range(cols // 32):
        x[:, 32 * j + pos[j]] = 1.0 + rng.random(batch)
    return f, x


def tiny_case(rows, cols, batch, seed, exp=-110):
    """every |x| ~ 2^exp (below the fixed-point range), d large enough that
    the products stay far above the fp32 underflow"""
    rng = np.random.default_rng(seed)
    f = synth.q4k_fields(rows, cols, [seed, 2])
    nb = cols // 256
    f["d"] = f16_bits(rng.uniform(2.0 ** 10, 2.0 ** 14, (rows, nb)))
    f["dmin"] = f16_bits(rng.uniform(2.0 ** 8, 2.0 ** 12, (rows, nb)))
    x = (rng.standard_normal((batch, cols)) * 2.0 ** exp).astype(np.float32)
    return f, x


def mixed_tiny_case(rows, cols, batch, seed):
    """alternate superblocks of tiny (2^-110) and ordinary x, with the
    weights of the ordinary ones zero: the tiny blocks carry the result"""
    f, x = tiny_case(rows, cols, batch, seed)
    rng = np.random.default_rng([seed, 3])
    for sb in range(0, cols // 256, 2):
        x[:, 256 * sb:256 * (sb + 1)] = rng.standard_normal((batch, 256)).astype(np.float32)
        f["q"][:, 256 * sb:256 * (sb + 1)] = 0
        f["m"][:, 8 * sb:8 * (sb + 1)] = 0
    return f, x


def huge_case(rows, cols, batch, seed):
    """|x| ~ 2^100 (above the fixed-point range) with small d, dmin"""
    rng = np.random.default_rng(seed)
    f = synth.q4k_fields(rows, cols, [seed, 4])
    nb = cols // 256
    f["d"] = f16_bits(rng.uniform(2.0 ** -14, 2.0 ** -12, (rows, nb)))
    f["dmin"] = f16_bits(rng.uniform(2.0 ** -14, 2.0 ** -12, (rows, nb)))
    x = (rng.standard_normal((batch, cols)) * 2.0 ** 100).astype(np.float32)
    return f, x


def nonneg_case(rows, cols, batch, seed):
    f = synth.q4k_fields(rows, cols, [seed, 5])
    x = np.abs(synth.activations(batch, cols, [seed, 6]))
    return f, x


def cancel_case(rows, cols, batch, seed):
    """weights whose terms cancel: sc*q*d ~ m*dmin in every sub-block"""
    rng = np.random.default_rng(seed)
    f = synth.q4k_fields(rows, cols, [seed, 7])
    nb = cols // 256
    d = rng.uniform(0.005, 0.01, (rows, nb)).astype(np.float16)
    f["d"] = d.view(np.uint16)
    f["dmin"] = d.view(np.uint16)                       # dmin = d
    f["sc"] = rng.integers(20, 40, (rows, cols // 32)).astype(np.uint8)
    f["q"] = rng.integers(1, 3, (rows, cols)).astype(np.uint8)
    f["m"] = (f["sc"].astype(np.int32) * 3 // 2).astype(np.uint8)   # sc*q - m ~ 0 for q = 1.5
    x = synth.activations(batch, cols, [seed, 8])
    return f, x


CASES = {
    "outlier_1e-3": lambda r, c, b, s: outlier_case(r, c, b, 1e-3, s),
    "outlier_1e-6": lambda r, c, b, s: outlier_case(r, c, b, 1e-6, s),
    "outlier_1e-12": lambda r, c, b, s: outlier_case(r, c, b, 1e-12, s),
    "wide": wide_case,
    "tiny": tiny_case,
    "mixed_tiny": mixed_tiny_case,
    "huge": huge_case,
    "nonneg": nonneg_case,
    "cancel": cancel_case,
}


def reference(name, f, x, r=None):
    y_ref, norm = O.gemv(f, x, r)
    if name == "cancel":
        norm = O.magnitude_norm(f, x, r)
    return y_ref, norm


def check(name, y, y_ref, norm, what):
    ok, worst = O.within_tolerance(y, y_ref, norm, REL)
    assert ok, f"{name} {what}: worst error {worst:.3g} x the allowed error"


@pytest.mark.parametrize("batch", [1, 3])
@pytest.mark.parametrize("name", list(CASES))
def test_gemv_edge_activations(name, batch):
    rows, cols = 100, 1536
    f, x = CASES[name](rows, cols, batch, 40 + batch)
    w = pack_dev(f)
    xd = torch.from_numpy(x).cuda()
    y = q4k.q4k_gemv(w, rows, cols, xd)
    torch.cuda.synchronize()
    check(name, y.cpu().numpy(), *reference(name, f, x), "q4k_gemv")


@pytest.mark.parametrize("name", list(CASES))
def test_gemv_multi_edge_activations(name):
    cols, batch = 1024, 2
    f, x = CASES[name](96 + 40, cols, batch, 60)
    parts = [{k: np.ascontiguousarray(v[:96]) for k, v in f.items()},
             {k: np.ascontiguousarray(v[96:]) for k, v in f.items()}]
    ws = [pack_dev(p) for p in parts]
    ys = q4k.q4k_gemv_multi(ws, [96, 40], cols, torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    for p, y in zip(parts, ys):
        check(name, y.cpu().numpy(), *reference(name, p, x), "q4k_gemv_multi")


@pytest.mark.parametrize("batch", [1, 4])
def test_gemv_seq_edge_activations(batch):
    """one job list holding every case; each case is two jobs, the second
    waiting for the first and reading the case's x again, plus a residual"""
    cols = 768
    jobs, checks = [], []
    for i, name in enumerate(CASES):
        rows = 64 + 24 * i
        f, x = CASES[name](rows, cols, batch, 80 + i)
        w = pack_dev(f)
        xd = torch.from_numpy(x).cuda()
        r = synth.residual(batch, rows, [81, i])
        rd = torch.from_numpy(r).cuda()
        y1 = torch.full((batch, rows), float("nan"), device="cuda")
        y2 = torch.full((batch, rows), float("nan"), device="cuda")
        jobs.append({"w": w, "rows": rows, "cols": cols, "x": xd, "y": y1})
        jobs.append({"w": w, "rows": rows, "cols": cols, "x": xd, "residual": rd, "y": y2, "wait": True})
        checks.append((name, f, x, r, y1, y2))
    q4k.q4k_gemv_seq(jobs, batch)
    torch.cuda.synchronize()
    for name, f, x, r, y1, y2 in checks:
        check(name, y1.cpu().numpy(), *reference(name, f, x), "q4k_gemv_seq")
        check(name, y2.cpu().numpy(), *reference(name, f, x, r), "q4k_gemv_seq (residual)")
    assert q4k.q4k_device_error() == 0


@pytest.mark.parametrize("batch", [1, 4])
def test_more_tier2_blocks_than_the_pool_holds(batch):
    """4 x 4096 / 32 = 512 tier-2 sub-blocks per staging against 256 pool
    slots: the rest take the fp32 path; both GEMV kernels stay exact"""
    rows, cols = 70, 4096
    f, x = wide_case(rows, cols, batch, 71)
    w = pack_dev(f)
    xd = torch.from_numpy(x).cuda()
    y = q4k.q4k_gemv(w, rows, cols, xd)
    y2 = torch.empty((batch, rows), device="cuda")
    q4k.q4k_gemv_seq([{"w": w, "rows": rows, "cols": cols, "x": xd, "y": y2}], batch)
    torch.cuda.synchronize()
    ref = reference("wide", f, x)
    check("wide", y.cpu().numpy(), *ref, "q4k_gemv")
    check("wide", y2.cpu().numpy(), *ref, "q4k_gemv_seq")


@pytest.mark.parametrize("tokens", [7, 48, 200])
def test_gemm_nonnegative_activations(tokens):
    """x >= 0 makes every block sum S = sum q8 large and positive, so the
    min term is as large as it gets against sum |w||x|"""
    rows, cols = 300, 2560
    f = synth.q4k_fields(rows, cols, [tokens, 9])
    x = np.abs(synth.activations(tokens, cols, [tokens, 10]))
    q, d8, s = q4k.q8_quantize(torch.from_numpy(x).cuda())
    y = q4k.q4k_gemm(pack_dev(f), rows, cols, q, d8, s)
    torch.cuda.synchronize()
    rq, rd, rs = O.quantize_q8_1(x)
    ok, worst = O.within_tolerance(y.cpu().numpy(), *O.mmq(f, rq, rd, rs), REL)
    assert ok, f"worst error {worst:.3g} x the allowed error"
