#!/usr/bin/env python
"""Benchmark of the Q4_K weight matmul on GB300.

Headline: decode GEMV HBM GB/s at batch 1 over the Qwen3-4B-shaped decode
linear set (q 4096x2560, k/v 1024x2560, o 2560x4096, gate/up 9728x2560,
down 2560x9728; synthetic Q4_K weights, independent N(0,1) activations).  One
step runs the seven GEMVs of one set; consecutive steps read different
copies of the layer so that no step finds its weights in L2, and 13 steps
share one persistent q4k_gemv_seq launch.  Beside it: the same layer in
engine order (each group waits for the previous one), and the 36-layer stack
per decode token at batch 1 and 4.

Second leg (same JSON line, key "prefill"): q8_1 quantisation plus the MMQ
GEMM of the 512-token Qwen3-4B prefill (gate 9728x2560, down 2560x9728).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own replica of the workload (the
GEMV does not shard across GPUs here); value = bytes of all ranks / the
slowest rank's time.  ``--impl reference`` times the CPU oracle instead, on
rank 0 only, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "Q4_K GEMV HBM GB/s (batch 1, % of peak); prefill GEMM int8 TOPS & tok/s"
WORKLOAD = ("Qwen3-4B-shaped decode linear set, batch 1: q 4096x2560, k/v 1024x2560, "
            "o 2560x4096, gate/up 9728x2560, down 2560x9728 (Q4_K)")
PREFILL_WORKLOAD = "512-token prefill: q8_1 X[512x2560] x gate 9728x2560, X_down[512x9728] x down 2560x9728"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
BYTES_PER_WEIGHT = 144.0 / 256.0
STEPS_PER_LAUNCH = 13          # 91 GEMV jobs per q4k_gemv_seq launch (at most 96)


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# --------------------------------------------------------------------- peaks
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return p, "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS}, "fallback"


def code_digest(path: str) -> str:
    """First 16 hex digits of the SHA-256 of a C/C++/CUDA source with its
    comments and all white space removed: it changes when the code does,
    not when a comment does."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    text = re.sub(r"\s+", "", text)
    return hashlib.sha256(text.encode()).hexdigest()[:16]


def profile_traffic(kernel_tag: str, source: str):
    """DRAM bytes per launch recorded from an ncu capture in profiles/, valid
    only while the kernel's code is unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}_traffic.txt")
    try:
        text = open(path).read()
    except OSError:
        return None
    digest = code_digest(os.path.join(ROOT, "q4_weight_matmul_gb300", "csrc", source))
    m_hash = re.search(r"source_sha256_16:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_hash or not m_bytes or m_hash.group(1) != digest:
        return None
    return float(m_bytes.group(1))


# --------------------------------------------------------------------- ranks
def reduce_max(value: float, device=None) -> float:
    """Largest ``value`` over the ranks of the default process group (the
    value itself when no group is initialised or it has one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_step: float, steps: int, world: int, max_ms: float) -> float:
    """Whole-job GB/s: every rank streams ``bytes_per_step`` per step (weak
    scaling, independent replicas) and the job takes the slowest rank's time."""
    return bytes_per_step * steps * world / (max_ms * 1e-3) / 1e9


# --------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 9:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        rows = self.rows
        if self.uuid:
            mine = [r for r in rows if self.uuid in r[0] or r[0] in self.uuid]
            rows = mine or rows
        if not rows:
            return None
        uuids = {r[0] for r in rows}
        if len(uuids) > 1:
            rows = [r for r in rows if r[0] == sorted(uuids)[0]]
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------------- oracle (CPU)
_DECODE_CACHE = {}


def decode_inputs():
    if "layer" not in _DECODE_CACHE:
        _DECODE_CACHE["layer"] = synth.decode_layer(synth.WL_DECODE_4B, 0, 1)
    return _DECODE_CACHE["layer"]


def oracle_decode_sample(budget_s: float, seed_rows: int = 0):
    """Time the oracle GEMV on row samples of the seven decode matrices until
    ``budget_s`` of CPU time is spent.  Returns (GB/s, seconds, description)."""
    from oracle import q4k as O
    fields, xs = decode_inputs()
    rng = np.random.default_rng(seed_rows)
    done_bytes = 0.0
    spent = 0.0
    passes = 0
    per = 64
    while spent < budget_s:
        for name, rows, cols, inp in synth.QWEN3_4B_LAYER:
            sel = np.sort(rng.choice(rows, per, replace=False))
            f = {k: v[sel] for k, v in fields[name].items()}
            t0 = time.perf_counter()
            O.gemv(f, xs[inp])
            spent += time.perf_counter() - t0
            done_bytes += per * cols * BYTES_PER_WEIGHT + cols * 4 + per * 4
        passes += 1
    desc = f"oracle GEMV on {passes} passes of {per} random rows of each of the 7 decode matrices"
    return done_bytes / spent / 1e9, spent, desc


def cpu_threads() -> int:
    try:
        import threadpoolctl  # noqa: F401
        from threadpoolctl import threadpool_info
        n = max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
        return int(n)
    except Exception:
        return os.cpu_count() or 1


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    # each step: a bounded oracle sample of the decode set (~1 s)
    vals = []
    total_bytes = 0.0
    total_s = 0.0
    for i in range(args.warmup + args.steps):
        gbs, spent, desc = oracle_decode_sample(1.0, seed_rows=i)
        if i >= args.warmup:
            vals.append(gbs)
            total_bytes += gbs * spent
            total_s += spent
    value = total_bytes / total_s
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": 1, "sample": desc},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cpu_threads(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------- GPU arm
def run_ours(args, rank, world):
    import torch
    import q4_weight_matmul_gb300 as q4k

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    q4k.build()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20)
    uuid = str(getattr(props, "uuid", "") or "") or None
    peaks, peak_kind = measured_peaks()
    stream = torch.cuda.current_stream()

    # ---------------- weights: pack once, then rotate copies to defeat L2
    fields, xs_np = decode_inputs()
    t_pack0 = time.perf_counter()
    packed = {}
    pack_bytes = 0
    pack_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    dev_fields = {}
    for name, rows, cols, _ in synth.QWEN3_4B_LAYER:
        f = fields[name]
        dev_fields[name] = {k: torch.from_numpy(v.view(np.int16) if v.dtype == np.uint16 else v).to(dev)
                            for k, v in f.items()}
    torch.cuda.synchronize()
    pack_ev[0].record()
    for name, rows, cols, _ in synth.QWEN3_4B_LAYER:
        d = dev_fields[name]
        packed[name] = q4k.q4k_pack(d["d"], d["dmin"], d["sc"], d["m"], d["q"])
        pack_bytes += sum(t.numel() * t.element_size() for t in d.values()) + packed[name].numel()
    pack_ev[1].record()
    torch.cuda.synchronize()
    pack_ms = pack_ev[0].elapsed_time(pack_ev[1])
    del dev_fields
    layer_bytes = sum(p.numel() for p in packed.values())
    n_copies = max(2, math.ceil(4 * l2 / layer_bytes))
    copies = [packed] + [{k: v.clone() for k, v in packed.items()} for _ in range(n_copies - 1)]
    xs = {k: torch.from_numpy(v).to(dev) for k, v in xs_np.items()}
    ys = {name: torch.empty((1, rows), dtype=torch.float32, device=dev)
          for name, rows, _, _ in synth.QWEN3_4B_LAYER}
    log(f"[bench] rank {rank}: {n_copies} layer copies x {layer_bytes / 1e6:.1f} MB, pack {pack_ms:.2f} ms "
        f"(setup {time.perf_counter() - t_pack0:.1f}s)")

    step_bytes = 0.0
    for name, rows, cols, _ in synth.QWEN3_4B_LAYER:
        step_bytes += rows * cols * BYTES_PER_WEIGHT + cols * 4 + rows * 4

    shape = {name: (rows, cols, inp) for name, rows, cols, inp in synth.QWEN3_4B_LAYER}
    # engine order: one launch per input group (QKV triple, o, gate/up pair, down)
    launch_groups = (("q", "k", "v"), ("o",), ("gate", "up"), ("down",))

    def layer_jobs(layer, wait_groups):
        jobs = []
        for gi, names in enumerate(launch_groups):
            for k, n in enumerate(names):
                rows, cols, inp = shape[n]
                jobs.append({"w": layer[n], "rows": rows, "cols": cols, "x": xs[inp], "y": ys[n],
                             "wait": wait_groups and gi > 0 and k == 0})
        return jobs

    # Headline: each step is one pass over the seven matrices of the decode
    # linear set, each with its own input (the workload's N(0,1) inputs are
    # independent); steps go to q4k_gemv_seq in launches of STEPS_PER_LAUNCH
    # sets, rotating over the layer copies so that no step finds its weights
    # in L2.  One persistent launch streams all their weights.
    ws_seq = None

    def seq_calls(first, count, per_launch=STEPS_PER_LAUNCH, wait_groups=False):
        nonlocal ws_seq
        calls = []
        for c0 in range(first, first + count, per_launch):
            jobs = []
            for i in range(c0, min(first + count, c0 + per_launch)):
                jobs += layer_jobs(copies[i % n_copies], wait_groups)
            seq = q4k.GemvSeq(jobs, 1, workspace=ws_seq)
            ws_seq = seq.workspace if ws_seq is None or seq.workspace.numel() > ws_seq.numel() else ws_seq
            calls.append(seq)
        return calls

    def graph_of(calls):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for c in calls:
                c()
        return g

    def time_graph(g):
        g.replay()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        t0.record()
        g.replay()
        t1.record()
        barrier()
        return t0.elapsed_time(t1)

    warm_calls = seq_calls(0, args.warmup)
    timed_calls = seq_calls(args.warmup, args.steps)
    n_launch_total = len(timed_calls)
    for c in warm_calls:
        c()
    torch.cuda.synchronize()
    warm_graph = graph_of(warm_calls)
    timed_graph = graph_of(timed_calls)
    warm_graph.replay()
    sampler = ClockSampler(uuid)
    sampler.start()
    time.sleep(0.3)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    start.record()
    timed_graph.replay()
    stop.record()
    barrier()
    elapsed_ms = start.elapsed_time(stop)
    # keep the same replays running long enough to sample clocks under load
    t_end = time.perf_counter() + 2.0
    while time.perf_counter() < t_end:
        for _ in range(10):
            timed_graph.replay()
        torch.cuda.synchronize()
    clocks = sampler.stop()
    if q4k.q4k_device_error() != 0:
        raise RuntimeError("a GEMV kernel gave up a bounded wait during the timed region")

    # ---------------- decode in engine order (each group reads the previous
    # group's output): the 4-launch path and one q4k_gemv_seq per layer with waits
    def decode_step_4launch(i):
        layer = copies[i % n_copies]
        for names in launch_groups:
            rows = [shape[n][0] for n in names]
            cols, inp = shape[names[0]][1], shape[names[0]][2]
            if len(names) == 1:
                q4k.q4k_gemv(layer[names[0]], rows[0], cols, xs[inp], y=ys[names[0]])
            else:
                q4k.q4k_gemv_multi([layer[n] for n in names], rows, cols, xs[inp], ys=[ys[n] for n in names])

    g4 = torch.cuda.CUDAGraph()
    for i in range(3):
        decode_step_4launch(i)
    torch.cuda.synchronize()
    with torch.cuda.graph(g4):
        for i in range(args.steps):
            decode_step_4launch(i)
    ms_4launch = time_graph(g4)
    chain_calls = seq_calls(0, args.steps, per_launch=1, wait_groups=True)
    for c in chain_calls[:3]:
        c()
    ms_chain = time_graph(graph_of(chain_calls))

    # ---------------- 36-layer Qwen3-4B-shaped stack, one decode token per step
    stack = {}
    for sb in (1, 4):
        xs_b = {name: torch.from_numpy(synth.activations(sb, cols, synth.layer_seed(synth.WL_STACK_4B, 0, 100 + j)))
                .to(dev) for j, (name, cols) in enumerate(synth.QWEN3_4B_INPUTS)}
        ys_b = {n: torch.empty((sb, shape[n][0]), device=dev) for n in shape}
        jobs = []
        for L in range(36):
            layer = copies[L % n_copies]
            for n in shape:
                rows, cols, inp = shape[n]
                jobs.append({"w": layer[n], "rows": rows, "cols": cols, "x": xs_b[inp], "y": ys_b[n]})
        tok = q4k.GemvSeq(jobs, sb)
        tok()
        torch.cuda.synchronize()
        n_tok = 10
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(n_tok):
                tok()
        ms = time_graph(g)
        stack[f"batch{sb}"] = {"tokens_per_s": sb * n_tok / (ms * 1e-3),
                               "GB/s": 36 * layer_bytes * n_tok / (ms * 1e-3) / 1e9,
                               "ms_per_token_step": ms / n_tok}

    # ---------------- e2e: public API with host buffers, copies in the region
    inputs_host = {k: torch.from_numpy(v).pin_memory() for k, v in xs_np.items()}
    outputs_host = {name: torch.empty((1, rows), dtype=torch.float32).pin_memory()
                    for name, rows, _, _ in synth.QWEN3_4B_LAYER}
    h2d = sum(t.numel() * 4 for t in inputs_host.values())
    d2h = sum(t.numel() * 4 for t in outputs_host.values())
    e2e_calls = seq_calls(0, args.warmup + args.steps, per_launch=1)

    def e2e_step(i):
        for k_, t in inputs_host.items():
            xs[k_].copy_(t, non_blocking=True)
        e2e_calls[i]()   # one q4k_gemv_seq call per step through the public API
        for name, t in outputs_host.items():
            t.copy_(ys[name], non_blocking=True)

    for i in range(args.warmup):
        e2e_step(i)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.steps):
        e2e_step(args.warmup + i)
    e1.record()
    barrier()
    e2e_ms = e0.elapsed_time(e1)

    # ---------------- prefill leg: q8_1 + MMQ GEMM, 512 tokens
    pf, pxs = synth.prefill_4b_512()
    pw = {}
    for name in ("gate", "down"):
        d = {k: torch.from_numpy(v.view(np.int16) if v.dtype == np.uint16 else v).to(dev)
             for k, v in pf[name].items()}
        pw[name] = q4k.q4k_pack(d["d"], d["dmin"], d["sc"], d["m"], d["q"])
    px = {k: torch.from_numpy(v).to(dev) for k, v in pxs.items()}
    pbytes = sum(v.numel() for v in pw.values()) + sum(v.numel() * 4 for v in px.values())
    p_copies = max(2, math.ceil(4 * l2 / pbytes))
    prefill_sets = [(pw, px)] + [({k: v.clone() for k, v in pw.items()}, {k: v.clone() for k, v in px.items()})
                                 for _ in range(p_copies - 1)]
    T = 512
    pq = {"mlp_in": q4k.q8_quantize(px["mlp_in"]), "down_in": q4k.q8_quantize(px["down_in"])}
    py = {"gate": torch.empty((T, 9728), device=dev), "down": torch.empty((T, 2560), device=dev)}
    shapes = {"gate": (9728, 2560, "mlp_in"), "down": (2560, 9728, "down_in")}

    def prefill_step(i):
        wset, xset = prefill_sets[i % p_copies]
        for name in ("gate", "down"):
            rows, cols, inp = shapes[name]
            q, d8, s = pq[inp]
            q4k.q8_quantize(xset[inp], q, d8, s)
            q4k.q4k_gemm(wset[name], rows, cols, q, d8, s, y=py[name])

    def gemm_only(i):
        wset, _ = prefill_sets[i % p_copies]
        for name in ("gate", "down"):
            rows, cols, inp = shapes[name]
            q, d8, s = pq[inp]
            q4k.q4k_gemm(wset[name], rows, cols, q, d8, s, y=py[name])

    for i in range(args.warmup):
        prefill_step(i)
    torch.cuda.synchronize()

    def capture_fn(fn, first, count):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(first, first + count):
                fn(i)
        return g

    pwarm = capture_fn(prefill_step, 0, args.warmup)
    ptimed = capture_fn(prefill_step, args.warmup, args.steps)
    gwarm = capture_fn(gemm_only, 0, args.warmup)
    gtimed = capture_fn(gemm_only, args.warmup, args.steps)
    pwarm.replay()
    barrier()
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record()
    ptimed.replay()
    p1.record()
    barrier()
    prefill_ms = p0.elapsed_time(p1)
    # the GEMM launches alone (same inputs), for the GEMM's own roofline
    gwarm.replay()
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record()
    gtimed.replay()
    g1.record()
    torch.cuda.synchronize()
    gemm_ms = g0.elapsed_time(g1)
    gemm_ops = 2.0 * T * (9728 * 2560 + 2560 * 9728)
    # tensor-core rate probes on this GPU: the int8 rate of the warp-level
    # MMA (mma.sync m16n8k32 s8) and the fp16 rate of tcgen05.mma kind::f16
    from q4_weight_matmul_gb300 import peaks as tc_peaks
    int8_peak = tc_peaks.mma_s8_tops(iters=20000)
    f16_peak = tc_peaks.tc_f16_tflops(groups=2048)

    # ---------------- reduce over ranks (max time), sum of work
    def max_over_ranks(v):
        return reduce_max(v, dev if dist is not None else None)

    elapsed_ms = max_over_ranks(elapsed_ms)
    e2e_ms = max_over_ranks(e2e_ms)
    prefill_ms = max_over_ranks(prefill_ms)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    value = job_throughput(step_bytes, args.steps, world, elapsed_ms)
    e2e_value = job_throughput(step_bytes, args.steps, world, e2e_ms)
    # the timed region holds nothing but this kernel's launches: its average
    # launch duration is the region over the launches, and each launch
    # processes STEPS_PER_LAUNCH steps' algorithmic bytes
    achieved = step_bytes * args.steps / (elapsed_ms * 1e-3) / 1e9
    peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    traffic = profile_traffic("gemv_seq", "gemv_seq.cu")
    bf16 = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
    gemm_tops = gemm_ops * args.steps / (gemm_ms * 1e-3) / 1e12

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        gbs, spent, desc = oracle_decode_sample(args.cpu_seconds)
        cpu = {"value": gbs, "unit": "GB/s", "cores": cpu_threads(), "kind": "oracle", "sample": desc,
               "seconds": round(spent, 2)}

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": 1, "parallelism": "replicas" if world > 1 else "single",
                   "timing": f"one CUDA graph of exactly `steps` steps; each step is the seven GEMVs of the "
                             f"decode linear set (independent N(0,1) inputs), {STEPS_PER_LAUNCH} steps per "
                             f"q4k_gemv_seq launch",
                   "l2": f"inputs larger than L2: {n_copies} rotating layer copies "
                         f"({n_copies * layer_bytes / 1e6:.0f} MB, L2 {l2 / 1e6:.0f} MB)",
                   "launches": n_launch_total},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "peak_kind": f"{peak_kind} hbm_gbs",
                     "kernel": "gemv_seq_kernel<1>",
                     "duration": "CUDA events on the launching stream around the timed region (one graph "
                                 "of the launches of this kernel, nothing else), divided by its launches; "
                                 "algorithmic bytes per launch = the steps it holds x bytes per step"},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": n_launch_total,
        "clocks": clocks,
        "decode_engine_order": {
            "note": "each input group reads the previous group's output (QKV | o | gate,up | down)",
            "4_launches_per_layer": {"us_per_layer": 1e3 * ms_4launch / args.steps,
                                     "GB/s": step_bytes * args.steps / (ms_4launch * 1e-3) / 1e9},
            "gemv_seq_one_launch_per_layer_with_waits": {
                "us_per_layer": 1e3 * ms_chain / args.steps,
                "GB/s": step_bytes * args.steps / (ms_chain * 1e-3) / 1e9}},
        "decode_stack_36_layers": stack,
        "cpu_baseline": cpu,
        "pack": {"ms": pack_ms, "GB/s": pack_bytes / (pack_ms * 1e-3) / 1e9, "note": "one-off, 7 matrices"},
        "prefill": {
            "workload": PREFILL_WORKLOAD, "tokens": T,
            "ms_per_step": prefill_ms / args.steps,
            "tok_s": T * args.steps * world / (prefill_ms * 1e-3),
            "int_tops": gemm_ops * args.steps * world / (prefill_ms * 1e-3) / 1e12,
            "gemm_tops": gemm_tops,
            # the GEMM's MMAs are tcgen05 kind::f16 (exact small integers in
            # fp16), so its own-dtype peak is the dense fp16 = bf16 rate
            "roofline": {"bound": "tensor", "achieved": gemm_tops, "unit": "TOPS", "peak": bf16,
                         "frac": gemm_tops / bf16, "peak_kind": f"{peak_kind} bf16_tflops (fp16 rate)",
                         "int8_peak_mma_sync_s8": int8_peak, "frac_of_int8_peak": gemm_tops / int8_peak,
                         "tcgen05_f16_probe_tflops": f16_peak},
            "gpu_launches": 4 * args.steps,
            "timing": "one CUDA graph of exactly `steps` steps (q8_1 + GEMM for gate and down); "
                      "gemm_tops from a graph of the GEMM launches alone",
            "l2": f"{p_copies} rotating weight+input copies",
        },
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    return run_ours(args, rank, world)


if __name__ == "__main__":
    sys.exit(main())
