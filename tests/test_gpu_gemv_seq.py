"""GPU parity of q4k_gemv_seq (one persistent launch over an ordered GEMV job
list) against the CPU oracle, through the C ABI.  Every fp output must satisfy
|y - y_ref| <= 1e-4 * sum|w||x| (+|residual|) element by element; a job that
consumes an earlier job's output gets the bound propagated through its own
weights (see test_dependent_chain)."""
import numpy as np
import pytest
import torch

from oracle import q4k as O
import synth
from _gpu import pack_dev, slice_rows
import q4_weight_matmul_gb300 as q4k

pytestmark = pytest.mark.gpu
REL = 1e-4
SHAPES = {name: (rows, cols, inp) for name, rows, cols, inp in synth.QWEN3_4B_LAYER}
GROUPS = (("q", "k", "v"), ("o",), ("gate", "up"), ("down",))
SLACK = 1.001


@pytest.fixture(scope="module", autouse=True)
def _built():
    q4k.build()
    torch.cuda.init()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def assert_close(y, y_ref, norm, what):
    ok, worst = O.within_tolerance(y, y_ref, norm, REL)
    assert ok, f"{what}: worst error {worst:.3g} x the allowed 1e-4*sum|w||x|"


def layer_jobs(w, xs_dev, ys, batch, residuals=None):
    """The decode layer as a job list: QKV | o | gate, up | down, each group
    waiting for the previous one (as in an engine, where each group's input
    is computed from the previous group's output)."""
    jobs = []
    for gi, names in enumerate(GROUPS):
        for k, n in enumerate(names):
            rows, cols, inp = SHAPES[n]
            j = {"w": w[n], "rows": rows, "cols": cols, "x": xs_dev[inp], "y": ys[n],
                 "wait": gi > 0 and k == 0}
            if residuals and n in residuals:
                j["residual"] = residuals[n]
            jobs.append(j)
    return jobs


@pytest.mark.parametrize("batch", [1, 4])
def test_decode_layer(batch):
    fields, xs = synth.decode_layer(synth.WL_DECODE_4B, 2, batch)
    w = {n: pack_dev(fields[n]) for n in SHAPES}
    xd = {k: dev(v) for k, v in xs.items()}
    ys = {n: torch.empty((batch, SHAPES[n][0]), device="cuda") for n in SHAPES}
    # o and down fold the residual add in; down writes in place over its residual
    r_o = synth.residual(batch, 2560, [11, batch])
    r_down = synth.residual(batch, 2560, [12, batch])
    ys["down"].copy_(dev(r_down))
    res = {"o": dev(r_o), "down": ys["down"]}
    q4k.q4k_gemv_seq(layer_jobs(w, xd, ys, batch, res), batch)
    for n in SHAPES:
        rows, cols, inp = SHAPES[n]
        r = {"o": r_o, "down": r_down}.get(n)
        y_ref, norm = O.gemv(fields[n], xs[inp], r)
        assert_close(host(ys[n]), y_ref, norm, f"layer {n} b{batch}")


def test_dependent_chain():
    """y_a = W_a x; y_b = W_b y_a + y_a (waits); y_c = W_c y_b (waits).  The
    oracle runs the same chain in fp64 on its own intermediates (rounded to
    fp32 as the device stores them).  A dependent output may differ by its own
    GEMV error plus the error of its input carried through the linear map,
    sum|w| * 1e-4 * norm(input); SLACK covers the second-order terms and the
    fp32 rounding of the intermediates."""
    fa = synth.q4k_fields(2560, 2560, 501)
    fb = synth.q4k_fields(2560, 2560, 502)
    fc = synth.q4k_fields(1024, 2560, 503)
    x = synth.activations(2, 2560, 504)
    wa, wb, wc = pack_dev(fa), pack_dev(fb), pack_dev(fc)
    ya, yb, yc = (torch.empty((2, r), device="cuda") for r in (2560, 2560, 1024))
    xd = dev(x)
    jobs = [{"w": wa, "rows": 2560, "cols": 2560, "x": xd, "y": ya},
            {"w": wb, "rows": 2560, "cols": 2560, "x": ya, "residual": ya, "y": yb, "wait": True},
            {"w": wc, "rows": 1024, "cols": 2560, "x": yb, "y": yc, "wait": True}]
    q4k.q4k_gemv_seq(jobs, 2)
    a_ref, a_norm = O.gemv(fa, x)
    assert_close(host(ya), a_ref, a_norm, "chain a")
    a32 = a_ref.astype(np.float32)
    b_ref, _ = O.gemv(fb, a32, a32)
    # y_b - b_ref = W_b e_a + e_a + (y_b's own GEMV error), |e_a| <= REL*a_norm
    # and the own error <= REL*(sum|W_b||y_a| + |y_a|): with the common REL
    # factored out, the normaliser is sum|W_b|(|a| + a_norm) + |a| + a_norm
    _, b_norm = O.gemv(fb, (np.abs(a_ref) + a_norm).astype(np.float32))
    b_norm = b_norm + np.abs(a_ref) + a_norm
    assert_close(host(yb), b_ref, b_norm * SLACK, "chain b")
    b32 = b_ref.astype(np.float32)
    c_ref, _ = O.gemv(fc, b32)
    _, c_norm = O.gemv(fc, (np.abs(b_ref) + b_norm).astype(np.float32))
    assert_close(host(yc), c_ref, c_norm * SLACK, "chain c")


@pytest.mark.parametrize("batch", [1, 3, 8])
def test_ragged_mixed_list(batch):
    """Rows that are not multiples of any row block, matrices too small to
    give every SM a row block, segments without a wait that change x, a job
    list that starts with a wait, and jobs with zero rows."""
    specs = [  # rows, cols, input index, wait
        (37, 512, 0, True), (1, 512, 0, False), (300, 768, 1, False), (0, 768, 1, False),
        (1500, 256, 2, False), (777, 4096, 3, True), (4100, 1024, 4, False), (96, 1024, 4, False),
        (0, 256, 2, True), (2048, 2048, 5, False)]
    cols_of = {}
    for _, cols, i, _ in specs:
        cols_of[i] = cols
    xs = {i: synth.activations(batch, c, [31, i, batch]) for i, c in cols_of.items()}
    xd = {i: dev(v) for i, v in xs.items()}
    jobs, refs = [], []
    for k, (rows, cols, i, wait) in enumerate(specs):
        f = synth.q4k_fields(max(rows, 1), cols, [32, k])
        w = pack_dev(f) if rows else torch.empty(0, dtype=torch.uint8, device="cuda")
        y = torch.full((batch, rows), np.nan, device="cuda")
        jobs.append({"w": w, "rows": rows, "cols": cols, "x": xd[i], "y": y, "wait": wait})
        refs.append((f, xs[i], y))
    q4k.q4k_gemv_seq(jobs, batch)
    for k, (f, x, y) in enumerate(refs):
        if specs[k][0] == 0:
            continue
        y_ref, norm = O.gemv(f, x)
        assert_close(host(y), y_ref, norm, f"job {k} {specs[k][:2]} b{batch}")


def test_tall_matrix_many_passes_sampled():
    # far more units per CTA than one pass of partial sums holds: row blocks
    # are carried from pass to pass
    rows, cols = 20000, 12288
    f = synth.q4k_fields(rows, cols, 4242)
    x = synth.activations(2, cols, 4243)
    y = torch.empty((2, rows), device="cuda")
    q4k.q4k_gemv_seq([{"w": pack_dev(f), "rows": rows, "cols": cols, "x": dev(x), "y": y}], 2)
    rng = np.random.default_rng(9)
    sample = np.sort(rng.choice(rows, 384, replace=False))
    y_ref, norm = O.gemv(slice_rows(f, sample), x)
    assert_close(host(y)[:, sample], y_ref, norm, "20000x12288 sampled")


def test_deterministic_graph_capture_and_clean_workspace():
    fields, xs = synth.decode_layer(synth.WL_DECODE_4B, 3, 1)
    w = {n: pack_dev(fields[n]) for n in SHAPES}
    xd = {k: dev(v) for k, v in xs.items()}
    ys = {n: torch.empty((1, SHAPES[n][0]), device="cuda") for n in SHAPES}
    seq = q4k.GemvSeq(layer_jobs(w, xd, ys, 1), 1)
    seq()
    first = {n: host(y).copy() for n, y in ys.items()}
    # the arrival counters (first 256 bytes) are reset by the launch itself
    assert int(torch.count_nonzero(seq.workspace[:256])) == 0, "counters not reset"
    for y in ys.values():
        y.zero_()
    seq()
    assert all(np.array_equal(host(ys[n]), first[n]) for n in SHAPES), "not deterministic"
    # the same launch replayed from a CUDA graph (as a decode engine does)
    for y in ys.values():
        y.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            seq(stream=s)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    g.replay()
    assert all(np.array_equal(host(ys[n]), first[n]) for n in SHAPES), "graph replay differs"
    assert int(torch.count_nonzero(seq.workspace[:256])) == 0
    assert q4k.q4k_device_error() == 0


def test_large_epoch_writes_every_row_and_is_deterministic():
    """13 independent decode sets in one launch (the bench's launch size):
    every output row is written (NaN canaries), sampled rows of every set
    match the oracle, and repeated launches give the same bits."""
    n_sets = 13
    fields, xs = synth.decode_layer(synth.WL_DECODE_4B, 4, 1)
    w = {n: pack_dev(fields[n]) for n in SHAPES}
    xd = {k: dev(v) for k, v in xs.items()}
    ys = [{n: torch.full((1, SHAPES[n][0]), float("nan"), device="cuda") for n in SHAPES} for _ in range(n_sets)]
    jobs = []
    for i in range(n_sets):
        for n in SHAPES:
            rows, cols, inp = SHAPES[n]
            jobs.append({"w": w[n], "rows": rows, "cols": cols, "x": xd[inp], "y": ys[i][n]})
    seq = q4k.GemvSeq(jobs, 1)
    seq()
    first = [{n: host(y).copy() for n, y in yset.items()} for yset in ys]
    for i in range(n_sets):
        for n in SHAPES:
            assert not np.isnan(first[i][n]).any(), f"set {i} {n}: rows left unwritten"
    rows = np.random.default_rng(44).choice(1024, 16, replace=False)
    for n in SHAPES:
        y_ref, norm = O.gemv(slice_rows(fields[n], rows), xs[SHAPES[n][2]])
        for i in range(n_sets):
            assert_close(first[i][n][:, rows], y_ref, norm, f"set {i} {n}")
    for rep in range(3):
        for yset in ys:
            for y in yset.values():
                y.fill_(float("nan"))
        seq()
        for i in range(n_sets):
            assert all(np.array_equal(host(ys[i][n]), first[i][n]) for n in SHAPES), f"rep {rep}: bits differ"
    assert int(torch.count_nonzero(seq.workspace[:256])) == 0, "counters not reset"
    assert q4k.q4k_device_error() == 0


@pytest.mark.parametrize("batch", [1, 4])
def test_36_layer_stack_in_one_launch(batch):
    """The 36-layer Qwen3-4B-shaped decode stack as ONE launch of 252 jobs
    (144 dependent groups).  Layers 0, 17 and 35 carry their own seeded
    weights and are checked on sampled rows; the other layers stream copies
    of layer 0's weights with their own inputs and outputs."""
    layers = 36
    checked = (0, 17, 35)
    data = {L: synth.decode_layer(synth.WL_STACK_4B, L, batch) for L in checked}
    packed = {L: {n: pack_dev(data[L][0][n]) for n in SHAPES} for L in checked}
    jobs, outs = [], {}
    for L in range(layers):
        _, xs = data[L] if L in data else synth.decode_layer(synth.WL_STACK_4B, L, batch, with_fields=False)
        xd = {k: dev(v) for k, v in xs.items()}
        ys = {n: torch.empty((batch, SHAPES[n][0]), device="cuda") for n in SHAPES}
        w = packed.get(L, packed[0])
        lj = layer_jobs(w, xd, ys, batch)
        lj[0]["wait"] = L > 0
        jobs += lj
        if L in checked:
            outs[L] = ys
    assert len(jobs) == 252
    q4k.q4k_gemv_seq(jobs, batch)
    rng = np.random.default_rng(77 + batch)
    for L in checked:
        fields, xs = data[L]
        for n in SHAPES:
            rows, cols, inp = SHAPES[n]
            sample = np.sort(rng.choice(rows, 128, replace=False))
            y_ref, norm = O.gemv(slice_rows(fields[n], sample), xs[inp])
            assert_close(host(outs[L][n])[:, sample], y_ref, norm, f"stack layer {L} {n} b{batch}")
    assert q4k.q4k_device_error() == 0


def test_plan_once_launch_many_with_new_inputs():
    """q4k_gemv_seq_plan then q4k_gemv_seq_launch three times, the inputs
    rewritten in place between launches (same buffers, new values), over a
    list of 100 jobs (two launches per plan): each launch matches the oracle."""
    cols, batch = 512, 1
    shapes = [(64 + 8 * (i % 5), cols) for i in range(100)]
    fields = [synth.q4k_fields(r, c, [900, i]) for i, (r, c) in enumerate(shapes)]
    ws = [pack_dev(f) for f in fields]
    xd = torch.empty((batch, cols), device="cuda")
    ys = [torch.empty((batch, r), device="cuda") for r, _ in shapes]
    jobs = [{"w": w, "rows": r, "cols": c, "x": xd, "y": y} for w, (r, c), y in zip(ws, shapes, ys)]
    seq = q4k.GemvSeq(jobs, batch)
    for rep in range(3):
        x = synth.activations(batch, cols, [901, rep])
        xd.copy_(torch.from_numpy(x))
        seq()
        torch.cuda.synchronize()
        for i in (0, 37, 95, 96, 99):
            y_ref, norm = O.gemv(fields[i], x)
            ok, worst = O.within_tolerance(ys[i].cpu().numpy(), y_ref, norm, REL)
            assert ok, f"rep {rep} job {i}: {worst:.3g}"
    assert q4k.q4k_device_error() == 0


def test_plan_and_one_shot_call_give_the_same_bits():
    batch = 2
    fields, xs = synth.decode_layer(synth.WL_DECODE_4B, 11, batch)
    w = {n: pack_dev(fields[n]) for n in SHAPES}
    xd = {k: dev(v) for k, v in xs.items()}
    y1 = {n: torch.empty((batch, SHAPES[n][0]), device="cuda") for n in SHAPES}
    y2 = {n: torch.empty((batch, SHAPES[n][0]), device="cuda") for n in SHAPES}
    q4k.q4k_gemv_seq(layer_jobs(w, xd, y1, batch), batch)
    q4k.GemvSeq(layer_jobs(w, xd, y2, batch), batch)()
    torch.cuda.synchronize()
    for n in SHAPES:
        assert torch.equal(y1[n], y2[n]), n


def test_host_buffer_step_matches_device_launch():
    """q4k_gemv_seq_launch_host: inputs copied from one pinned host buffer,
    outputs copied back into another, three steps with new host values;
    each step gives the bits of the device-buffer launch on the same values
    and matches the oracle on sampled rows."""
    batch = 1
    fields, xs = synth.decode_layer(synth.WL_DECODE_4B, 12, batch)
    w = {n: pack_dev(fields[n]) for n in SHAPES}
    in_off, off = {}, 0
    for k, v in xs.items():
        in_off[k] = (off, v.shape)
        off += v.size
    x_host = torch.empty(off, dtype=torch.float32).pin_memory()
    x_dev = torch.empty(off, device="cuda")
    xv = {k: x_dev[o:o + int(np.prod(shp))].view(shp) for k, (o, shp) in in_off.items()}
    y_off, off = {}, 0
    for n in SHAPES:
        y_off[n] = off
        off += batch * SHAPES[n][0]
    y_dev = torch.empty(off, device="cuda")
    y_host = torch.full((off,), float("nan"), dtype=torch.float32).pin_memory()
    yv = {n: y_dev[o:o + batch * SHAPES[n][0]].view(batch, SHAPES[n][0]) for n, o in y_off.items()}
    seq = q4k.GemvSeq(layer_jobs(w, xv, yv, batch), batch)
    xd = {k: torch.empty(v.shape, device="cuda") for k, v in xs.items()}
    y2 = {n: torch.empty((batch, SHAPES[n][0]), device="cuda") for n in SHAPES}
    ref = q4k.GemvSeq(layer_jobs(w, xd, y2, batch), batch)
    rows = np.random.default_rng(13).choice(1024, 24, replace=False)
    for step in range(3):
        x_np = {k: synth.activations(batch, v.shape[1], [14, step, i]) for i, (k, v) in enumerate(xs.items())}
        for k, (o, _) in in_off.items():
            x_host[o:o + x_np[k].size] = torch.from_numpy(x_np[k].reshape(-1))
            xd[k].copy_(torch.from_numpy(x_np[k]))
        seq.launch_host(x_host, x_dev, y_host, y_dev)
        ref()
        torch.cuda.synchronize()
        for n in SHAPES:
            o, r = y_off[n], SHAPES[n][0]
            got = y_host[o:o + batch * r].view(batch, r)
            assert torch.equal(got, y2[n].cpu()), f"step {step} {n}: bits differ from the device launch"
            y_ref, norm = O.gemv(slice_rows(fields[n], rows), x_np[SHAPES[n][2]])
            assert_close(got.numpy()[:, rows], y_ref, norm, f"step {step} {n}")
    # the same step through buffers bound once (bind_host, step)
    first = y_host.clone()
    y_host.fill_(float("nan"))
    seq.bind_host(x_host, x_dev, y_host, y_dev)
    seq.step()
    torch.cuda.synchronize()
    assert torch.equal(y_host, first), "bound step: bits differ"
    assert q4k.q4k_device_error() == 0


# ------------------------------------------------------- Q4_K_M job lists
Q6K_IN_LAYER = ("v", "down")     # the Q6_K matrices of a Q4_K_M layer (half the layers)


def q6_pack(f):
    return q4k.q6k_pack(dev(np.ascontiguousarray(f["d"]).view(np.int16)), dev(f["sc"]), dev(f["q"]))


def q4km_layer(seed, batch):
    """A Q4_K_M-style decode layer: q, k, o, gate, up in Q4_K; v, down in Q6_K."""
    from oracle import q6k as O6
    fields, xs = synth.decode_layer(synth.WL_DECODE_4B, seed, batch)
    w, ref_f = {}, {}
    for n, (rows, cols, _) in SHAPES.items():
        if n in Q6K_IN_LAYER:
            f6 = synth.q6k_fields(rows, cols, [790, seed, rows])
            w[n], ref_f[n] = q6_pack(f6), ("q6", f6)
        else:
            w[n], ref_f[n] = pack_dev(fields[n]), ("q4", fields[n])

    def ref(n, x, r=None):
        kind, f = ref_f[n]
        return O6.gemv_q6k(f, x, r) if kind == "q6" else O.gemv(f, x, r)
    return w, xs, ref


def q4km_jobs(w, xs_dev, ys, residuals=None):
    jobs = layer_jobs(w, xs_dev, ys, None, residuals)
    for j, (n, _) in zip(jobs, [(n, 0) for names in GROUPS for n in names]):
        if n in Q6K_IN_LAYER:
            j["format"] = 1
    return jobs


@pytest.mark.parametrize("batch", [1, 4])
def test_q4km_layer_mixed_formats(batch):
    """q, k (Q4_K) and v (Q6_K) read the same x: two segments, one staging;
    down (Q6_K) waits and adds the residual."""
    w, xs, ref = q4km_layer(3, batch)
    xs_dev = {k: dev(v) for k, v in xs.items()}
    ys = {n: torch.full((batch, SHAPES[n][0]), float("nan"), device="cuda") for n in SHAPES}
    r = synth.residual(batch, SHAPES["down"][0], [791, batch])
    q4k.q4k_gemv_seq(q4km_jobs(w, xs_dev, ys, {"down": dev(r)}), batch)
    for n, (rows, cols, inp) in SHAPES.items():
        assert_close(host(ys[n]), *ref(n, xs[inp], r if n == "down" else None), f"{n} (batch {batch})")
    assert q4k.q4k_device_error() == 0


def test_q4km_stack_across_launches_and_entry_points():
    """Six Q4_K_M layers (42 jobs, 12 of them Q6_K) as one list through the
    one-shot call, the prepared plan and the allocation-free entry: the same
    bits from all three, within the bound.  A list of 60 Q6_K jobs takes two
    launches (48 Q6_K jobs a launch)."""
    batch = 1
    layers = [q4km_layer(10 + i, batch) for i in range(6)]
    jobs, checks = [], []
    for w, xs, ref in layers:
        xs_dev = {k: dev(v) for k, v in xs.items()}
        ys = {n: torch.full((batch, SHAPES[n][0]), float("nan"), device="cuda") for n in SHAPES}
        jobs += q4km_jobs(w, xs_dev, ys)
        checks.append((xs, ref, ys))
    q4k.q4k_gemv_seq(jobs, batch)
    first = {id(c): {n: host(c[2][n]).copy() for n in SHAPES} for c in checks}
    for xs, ref, ys in checks:
        for n, (rows, cols, inp) in SHAPES.items():
            assert_close(host(ys[n]), *ref(n, xs[inp]), n)
    seq = q4k.GemvSeq(jobs, batch)
    seq()
    for c in checks:
        for n in SHAPES:
            assert np.array_equal(host(c[2][n]), first[id(c)][n]), f"plan: {n}"
    q4k.q4k_gemv_seq_static(jobs, batch)
    for c in checks:
        for n in SHAPES:
            assert np.array_equal(host(c[2][n]), first[id(c)][n]), f"static: {n}"
    # 60 Q6_K jobs (small): two launches
    from oracle import q6k as O6
    cols = 512
    x = synth.activations(batch, cols, 792)
    xd = dev(x)
    fs = [synth.q6k_fields(40 + (i % 5) * 16, cols, [793, i]) for i in range(60)]
    ys6 = [torch.full((batch, f["q"].shape[0]), float("nan"), device="cuda") for f in fs]
    jobs6 = [{"w": q6_pack(f), "rows": f["q"].shape[0], "cols": cols, "x": xd, "y": y, "format": 1,
              "wait": i == 50} for i, (f, y) in enumerate(zip(fs, ys6))]
    q4k.q4k_gemv_seq(jobs6, batch)
    for i in (0, 47, 48, 50, 59):
        assert_close(host(ys6[i]), *O6.gemv_q6k(fs[i], x), f"q6k job {i}")
    assert q4k.q4k_device_error() == 0
