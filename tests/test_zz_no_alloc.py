"""q4k_gemv_seq_static: the GEMV job-list entry point that allocates nothing,
for callers that cannot allocate device memory (its scratch is a fixed array
inside the library).  Its results must match q4k_gemv_seq's, with the
caller-provided workspace, within the tolerance every GEMV test uses
(1e-4 * sum|w||x| + |residual| per element), on two calls in a row.  This file
runs last so that a failure here leaves every other test already run."""
import ctypes

import numpy as np
import pytest
import torch

from oracle import q4k as O
import synth
from _gpu import pack_dev
import q4_weight_matmul_gb300 as q4k

REL = 1e-4
SHAPES = {name: (rows, cols, inp) for name, rows, cols, inp in synth.QWEN3_4B_LAYER}
GROUPS = (("q", "k", "v"), ("o",), ("gate", "up"), ("down",))


def test_no_alloc_entry_validates_before_any_launch():
    lib = ctypes.CDLL(q4k.build())
    for name, (res, args) in q4k.SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    jobs = (q4k.GemvJob * 1)()
    jobs[0].w, jobs[0].rows, jobs[0].cols, jobs[0].x, jobs[0].y = 0x10000, 8, 300, 0x10000, 0x10000
    assert lib.q4k_gemv_seq_static(jobs, 1, 0, 1, None) == 1          # cols not a multiple of 256
    jobs[0].cols = 256
    assert lib.q4k_gemv_seq_static(jobs, 1, 0, 9, None) == 3          # batch above 8
    assert lib.q4k_gemv_seq_static(None, 1, 0, 1, None) == 1          # no job list
    assert lib.q4k_gemv_seq_static(jobs, 1, 0, 0, None) == 0          # nothing to do


@pytest.mark.gpu
def test_no_alloc_entry_matches_workspace_entry():
    q4k.build()
    batch = 2
    fields, xs = synth.decode_layer(synth.WL_DECODE_4B, 5, batch)
    w = {n: pack_dev(fields[n]) for n in SHAPES}
    xd = {k: torch.from_numpy(v).cuda() for k, v in xs.items()}
    r_down = torch.from_numpy(synth.residual(batch, 2560, [13, batch])).cuda()

    def jobs(ys):
        out = []
        for gi, names in enumerate(GROUPS):
            for k, n in enumerate(names):
                rows, cols, inp = SHAPES[n]
                j = {"w": w[n], "rows": rows, "cols": cols, "x": xd[inp], "y": ys[n], "wait": gi > 0 and k == 0}
                if n == "down":
                    j["residual"] = r_down
                out.append(j)
        return out

    ys_ref = {n: torch.empty((batch, SHAPES[n][0]), device="cuda") for n in SHAPES}
    q4k.q4k_gemv_seq(jobs(ys_ref), batch)
    torch.cuda.synchronize()
    ref = {n: y.cpu().numpy() for n, y in ys_ref.items()}
    norms = {n: O.gemv(fields[n], xs[SHAPES[n][2]], r_down.cpu().numpy() if n == "down" else None)[1]
             for n in SHAPES}
    for call in range(2):
        ys = {n: torch.full((batch, SHAPES[n][0]), float("nan"), device="cuda") for n in SHAPES}
        q4k.q4k_gemv_seq_static(jobs(ys), batch)
        torch.cuda.synchronize()
        for n in SHAPES:
            ok, worst = O.within_tolerance(ys[n].cpu().numpy(), ref[n], norms[n], REL)
            assert ok, f"call {call}, {n}: {worst:.3g} x the allowed error"
    assert q4k.q4k_device_error() == 0
