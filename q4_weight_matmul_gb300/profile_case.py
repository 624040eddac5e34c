"""Run one library kernel on a small synthetic case, for profiler captures.

    python -m q4_weight_matmul_gb300.profile_case gemv --rows 9728 --cols 2560 --batch 1 --reps 5
    python -m q4_weight_matmul_gb300.profile_case gemm --rows 9728 --cols 2560 --tokens 512
    python -m q4_weight_matmul_gb300.profile_case gemm_h16 --rows 9728 --cols 2560 --tokens 512
    python -m q4_weight_matmul_gb300.profile_case q8 --tokens 512 --cols 9728
    python -m q4_weight_matmul_gb300.profile_case pack --rows 9728 --cols 2560
    python -m q4_weight_matmul_gb300.profile_case seq --layers 13 --batch 1 --reps 3
    python -m q4_weight_matmul_gb300.profile_case q6k_gemv --rows 151936 --cols 2560 --batch 1 --reps 3
    python -m q4_weight_matmul_gb300.profile_case gemm_f16 --rows 9728 --cols 2560 --tokens 512
    python -m q4_weight_matmul_gb300.profile_case q6k_gemm_f16 --rows 2560 --cols 9728 --tokens 512

``seq`` runs --layers Qwen3-4B-shaped decode linear sets (q, k, v, o, gate,
up, down; independent inputs) as one q4k_gemv_seq launch per rep, as the
benchmark does (13 sets per launch).

Inputs are uniformly random bytes / N(0,1) floats (valid Q4_K fields), made on
the device; nothing is checked here (the tests do that).  Weights are spread
over enough copies that consecutive launches miss L2.
"""
from __future__ import annotations

import argparse
import math

import torch

import q4_weight_matmul_gb300 as q4k


def rand_fields(rows, cols, dev, gen):
    nb = cols // 256
    d = (torch.rand((rows, nb), generator=gen, device=dev) * 0.02).half().view(torch.int16)
    dmin = (torch.rand((rows, nb), generator=gen, device=dev) * 0.02).half().view(torch.int16)
    sc = torch.randint(0, 64, (rows, cols // 32), generator=gen, device=dev, dtype=torch.uint8)
    m = torch.randint(0, 64, (rows, cols // 32), generator=gen, device=dev, dtype=torch.uint8)
    q = torch.randint(0, 16, (rows, cols), generator=gen, device=dev, dtype=torch.uint8)
    return d, dmin, sc, m, q


QWEN3_4B_LAYER = (("q", 4096, 2560, 0), ("k", 1024, 2560, 0), ("v", 1024, 2560, 0), ("o", 2560, 4096, 1),
                  ("gate", 9728, 2560, 2), ("up", 9728, 2560, 2), ("down", 2560, 9728, 3))


def run_seq(a, dev, gen):
    xs = [torch.randn((a.batch, c), device=dev, generator=gen) for c in (2560, 4096, 2560, 9728)]
    jobs = []
    for _ in range(a.layers):
        for name, rows, cols, inp in QWEN3_4B_LAYER:
            w = q4k.q4k_pack(*rand_fields(rows, cols, dev, gen))
            jobs.append({"w": w, "rows": rows, "cols": cols, "x": xs[inp],
                         "y": torch.empty((a.batch, rows), device=dev)})
    seq = q4k.GemvSeq(jobs, a.batch)
    for _ in range(a.reps):
        seq()
    torch.cuda.synchronize()
    if q4k.q4k_device_error() != 0:
        raise RuntimeError("a kernel gave up a bounded wait")
    print("profile case done: seq", a.layers, "layers, batch", a.batch, a.reps, "reps")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("kernel", choices=["gemv", "gemm", "gemm_h16", "gemm_f16", "q8", "pack", "seq", "q6k_gemv",
                                       "q6k_gemm_f16"])
    ap.add_argument("--layers", type=int, default=13)
    ap.add_argument("--rows", type=int, default=9728)
    ap.add_argument("--cols", type=int, default=2560)
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--tokens", type=int, default=512)
    ap.add_argument("--reps", type=int, default=5)
    a = ap.parse_args()
    q4k.build()
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    if a.kernel == "seq":
        run_seq(a, dev, gen)
        return
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 * 2 ** 20)
    if a.kernel in ("q6k_gemv", "q6k_gemm_f16"):
        d = (torch.rand((a.rows, a.cols // 256), generator=gen, device=dev) * 0.02).half().view(torch.int16)
        sc = torch.randint(-128, 128, (a.rows, a.cols // 16), generator=gen, device=dev,
                           dtype=torch.int16).to(torch.int8)
        q = torch.randint(0, 64, (a.rows, a.cols), generator=gen, device=dev, dtype=torch.uint8)
        w0 = q4k.q6k_pack(d, sc, q)
        n = max(1, math.ceil(2 * l2 / w0.numel()))
        ws = [w0] + [w0.clone() for _ in range(n - 1)]
        if a.kernel == "q6k_gemv":
            x = torch.randn((a.batch, a.cols), device=dev, generator=gen)
            y = torch.empty((a.batch, a.rows), device=dev)
            for i in range(a.reps):
                q4k.q6k_gemv(ws[i % n], a.rows, a.cols, x, y=y)
        else:
            sp = q4k.x_split_f16(torch.randn((a.tokens, a.cols), device=dev, generator=gen))
            y = torch.empty((a.tokens, a.rows), device=dev)
            for i in range(a.reps):
                q4k.q6k_gemm_f16(ws[i % n], a.rows, a.cols, *sp, y=y)
        torch.cuda.synchronize()
        print("profile case done:", a.kernel, a.rows, a.cols, a.batch, a.reps)
        return
    f = rand_fields(a.rows, a.cols, dev, gen)
    w0 = q4k.q4k_pack(*f)
    n = max(1, math.ceil(2 * l2 / w0.numel())) if a.kernel in ("gemv", "gemm", "gemm_h16", "gemm_f16") else 1
    ws = [w0] + [w0.clone() for _ in range(n - 1)]
    if a.kernel == "gemv":
        x = torch.randn((a.batch, a.cols), device=dev, generator=gen)
        y = torch.empty((a.batch, a.rows), device=dev)
        for i in range(a.reps):
            q4k.q4k_gemv(ws[i % n], a.rows, a.cols, x, y=y)
    elif a.kernel == "gemm":
        x = torch.randn((a.tokens, a.cols), device=dev, generator=gen)
        q, d8, s = q4k.q8_quantize(x)
        y = torch.empty((a.tokens, a.rows), device=dev)
        for i in range(a.reps):
            q4k.q4k_gemm(ws[i % n], a.rows, a.cols, q, d8, s, y=y)
    elif a.kernel == "gemm_h16":
        x = torch.randn((a.tokens, a.cols), device=dev, generator=gen)
        q, d8, s = q4k.q8_quantize_h16(x)
        y = torch.empty((a.tokens, a.rows), device=dev)
        for i in range(a.reps):
            q4k.q4k_gemm_h16(ws[i % n], a.rows, a.cols, q, d8, s, y=y)
    elif a.kernel == "gemm_f16":
        x = torch.randn((a.tokens, a.cols), device=dev, generator=gen)
        sp = q4k.x_split_f16(x)
        y = torch.empty((a.tokens, a.rows), device=dev)
        for i in range(a.reps):
            q4k.q4k_gemm_f16(ws[i % n], a.rows, a.cols, *sp, y=y)
    elif a.kernel == "q8":
        x = torch.randn((a.tokens, a.cols), device=dev, generator=gen)
        out = q4k.q8_quantize(x)
        for _ in range(a.reps):
            q4k.q8_quantize(x, *out)
    else:
        for _ in range(a.reps):
            q4k.q4k_pack(*f, out=w0)
    torch.cuda.synchronize()
    print("profile case done:", a.kernel, a.rows, a.cols, a.batch, a.tokens, a.reps)


if __name__ == "__main__":
    main()
