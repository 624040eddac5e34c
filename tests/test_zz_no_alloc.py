"""q4k_gemv_seq_static: the GEMV job-list entry point that allocates nothing.

Some callers of this library cannot allocate device memory when they call
it: a serving process that reserves all of its device memory at start-up
and may not allocate afterwards, a plug-in running inside a host program
whose allocator it must not touch, or plain C code with no allocator at
all.  For them the job list runs on a fixed scratch array inside the
library instead of a caller-provided workspace.

Both entry points run the same kernel on the same plan, so the results must
be the same bits as q4k_gemv_seq's with a workspace -- on two calls in a
row, on a list long enough to take two launches from one clear of the
array, and after a kernel has given up a bounded wait -- and within the
oracle's 1e-4 * sum|w||x| (+|residual|) bound.  This file runs last, so a
failure here leaves every other test already run."""
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


def _layer():
    batch = 2
    fields, xs = synth.decode_layer(synth.WL_DECODE_4B, 5, batch)
    w = {n: pack_dev(fields[n]) for n in SHAPES}
    xd = {k: torch.from_numpy(v).cuda() for k, v in xs.items()}
    r_down = synth.residual(batch, 2560, [13, batch])

    def jobs(ys):
        out = []
        for gi, names in enumerate(GROUPS):
            for k, n in enumerate(names):
                rows, cols, inp = SHAPES[n]
                j = {"w": w[n], "rows": rows, "cols": cols, "x": xd[inp], "y": ys[n],
                     "wait": gi > 0 and k == 0}
                if n == "down":
                    j["residual"] = torch.from_numpy(r_down).cuda()
                out.append(j)
        return out

    ref = {n: O.gemv(fields[n], xs[SHAPES[n][2]], r_down if n == "down" else None) for n in SHAPES}
    return batch, jobs, ref


@pytest.mark.gpu
def test_no_alloc_entry_matches_workspace_entry():
    q4k.build()
    batch, jobs, ref = _layer()
    ys_ws = {n: torch.empty((batch, SHAPES[n][0]), device="cuda") for n in SHAPES}
    q4k.q4k_gemv_seq(jobs(ys_ws), batch)
    torch.cuda.synchronize()
    for call in range(2):
        ys = {n: torch.full((batch, SHAPES[n][0]), float("nan"), device="cuda") for n in SHAPES}
        q4k.q4k_gemv_seq_static(jobs(ys), batch)
        torch.cuda.synchronize()
        for n in SHAPES:
            assert torch.equal(ys[n], ys_ws[n]), f"call {call}, {n}: bits differ from q4k_gemv_seq"
            ok, worst = O.within_tolerance(ys[n].cpu().numpy(), *ref[n], REL)
            assert ok, f"call {call}, {n}: {worst:.3g} x the allowed error"
    assert q4k.q4k_device_error() == 0


@pytest.mark.gpu
def test_no_alloc_entry_on_a_list_of_two_launches():
    """98 jobs: the list takes two launches that share the array after one
    clear; the second launch starts from the counters the first left."""
    q4k.build()
    cols, batch = 512, 1
    shapes = [(32 + 16 * (i % 7), cols) for i in range(98)]
    fields = [synth.q4k_fields(r, c, [950, i]) for i, (r, c) in enumerate(shapes)]
    x = synth.activations(batch, cols, 951)
    xd = torch.from_numpy(x).cuda()
    ws = [pack_dev(f) for f in fields]

    def jobs(ys):
        return [{"w": w, "rows": r, "cols": c, "x": xd, "y": y, "wait": i == 97}
                for i, (w, (r, c), y) in enumerate(zip(ws, shapes, ys))]

    ys_ws = [torch.empty((batch, r), device="cuda") for r, _ in shapes]
    q4k.q4k_gemv_seq(jobs(ys_ws), batch)
    for call in range(2):
        ys = [torch.full((batch, r), float("nan"), device="cuda") for r, _ in shapes]
        q4k.q4k_gemv_seq_static(jobs(ys), batch)
        torch.cuda.synchronize()
        for i in range(98):
            assert torch.equal(ys[i], ys_ws[i]), f"call {call}, job {i}: bits differ"
        for i in (0, 50, 95, 96, 97):
            ok, worst = O.within_tolerance(ys[i].cpu().numpy(), *O.gemv(fields[i], x), REL)
            assert ok, f"call {call}, job {i}: {worst:.3g} x the allowed error"
    assert q4k.q4k_device_error() == 0


@pytest.mark.gpu
def test_no_alloc_entry_after_a_kernel_gave_up_a_wait():
    """The bounded-wait self-test sets the device error word; the next call
    on the shared array still computes the same bits, and the error is
    reported once."""
    q4k.build()
    batch, jobs, ref = _layer()
    ys_ws = {n: torch.empty((batch, SHAPES[n][0]), device="cuda") for n in SHAPES}
    q4k.q4k_gemv_seq(jobs(ys_ws), batch)
    torch.cuda.synchronize()
    q4k.q4k_selftest_wait_timeout()
    ys = {n: torch.full((batch, SHAPES[n][0]), float("nan"), device="cuda") for n in SHAPES}
    q4k.q4k_gemv_seq_static(jobs(ys), batch)
    assert q4k.q4k_device_error() == 5            # the self-test's timeout, reported once
    for n in SHAPES:
        assert torch.equal(ys[n], ys_ws[n]), n
    ys2 = {n: torch.full((batch, SHAPES[n][0]), float("nan"), device="cuda") for n in SHAPES}
    q4k.q4k_gemv_seq_static(jobs(ys2), batch)
    assert q4k.q4k_device_error() == 0
    for n in SHAPES:
        assert torch.equal(ys2[n], ys_ws[n]), n
