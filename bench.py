#!/usr/bin/env python
"""Benchmark of the Q4_K weight matmul on GB300.

Headline: decode GEMV HBM GB/s at batch 1 over the Qwen3-4B-shaped decode
linear set (q 4096x2560, k/v 1024x2560, o 2560x4096, gate/up 9728x2560,
down 2560x9728; synthetic Q4_K weights, independent N(0,1) activations).  One
step runs the seven GEMVs of one set; consecutive steps read different
copies of the layer so that no step finds its weights in L2, and the steps
are split evenly over persistent q4k_gemv_seq launches of at most 13 sets.
The timed unit is one CUDA-graph replay of exactly `steps` steps; the graph
is replayed back to back for about a second while nvidia-smi samples the
clocks, and the value comes from the median replay.

Beside it (same JSON line): the decode layer and the 36-layer decode token
in engine order (each input group waits for the previous group's output),
the 36-layer stack as independent jobs, batch 4, the single 2048x2048 GEMV
(L2-resident latency), the public API end to end with host buffers, and
the prefill GEMMs: 512 tokens (gate + down), the 2048-token 36-layer stack,
the 4096-token Qwen3-8B MLP, and 8..64-token short prompts.  The oracle is
timed on the host cores (one core and all cores) as the CPU baseline.

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
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
NOMINAL_HBM_GBS = 8000.0
BYTES_PER_WEIGHT = 144.0 / 256.0
MAX_SETS_PER_LAUNCH = 13       # 91 GEMV jobs per q4k_gemv_seq launch (at most 96)
REPLAY_SECONDS = 1.0           # back-to-back replays of each headline graph
MIN_REPLAYS = 20


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


def kernel_digest(sources) -> str:
    """Digest over several sources (a kernel and the headers it includes)."""
    csrc = os.path.join(ROOT, "q4_weight_matmul_gb300", "csrc")
    return hashlib.sha256("".join(code_digest(os.path.join(csrc, s)) for s in sources).encode()).hexdigest()[:16]


def profile_traffic(kernel_tag: str, source):
    """DRAM bytes per launch recorded from an ncu capture in profiles/, valid
    only while the kernel's code is unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}_traffic.txt")
    try:
        text = open(path).read()
    except OSError:
        return None
    sources = [source] if isinstance(source, str) else list(source)
    digest = code_digest(os.path.join(ROOT, "q4_weight_matmul_gb300", "csrc", sources[0])) \
        if len(sources) == 1 else kernel_digest(sources)
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


def even_split(count: int, max_per: int) -> list[int]:
    """``count`` items in the fewest groups of at most ``max_per``, sizes
    differing by at most one (no short tail group)."""
    if count <= 0:
        return []
    n = -(-count // max_per)
    return [count // n + (1 if i < count % n else 0) for i in range(n)]


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
        self.t_on = self.t_off = None

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
                self.rows.append((time.perf_counter(), parts))

    def mark(self, on: bool):
        """Bracket the timed region: only samples inside it are kept."""
        if on:
            self.t_on = time.perf_counter()
        else:
            self.t_off = time.perf_counter()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        rows = [r for t, r in self.rows
                if (self.t_on is None or t >= self.t_on) and (self.t_off is None or t <= self.t_off + 0.1)]
        rows = rows or [r for _, r in self.rows]
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


def oracle_decode_sample(budget_s: float, seed_rows: int = 0, per: int = 64):
    """Time the oracle GEMV on row samples of the seven decode matrices until
    ``budget_s`` of wall time is spent.  Returns (GB/s, seconds, description)."""
    from oracle import q4k as O
    fields, xs = decode_inputs()
    rng = np.random.default_rng(seed_rows)
    done_bytes = 0.0
    spent = 0.0
    passes = 0
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


def oracle_gemm_sample(budget_s: float, rows_per: int = 48):
    """Time the oracle MMQ (q8_1 quantisation + block dots + scales) on row
    samples of the 512-token prefill (gate 9728x2560 and down 2560x9728, all
    512 tokens).  Returns (integer TOPS, tok/s over the full problem, seconds,
    description)."""
    from oracle import q4k as O
    pf, pxs = synth.prefill_4b_512()
    rng = np.random.default_rng(7)
    shapes = (("gate", 9728, 2560, "mlp_in"), ("down", 2560, 9728, "down_in"))
    quant = {inp: O.quantize_q8_1(pxs[inp]) for _, _, _, inp in shapes}
    spent, ops, rows_done, passes = 0.0, 0.0, 0, 0
    while spent < budget_s:
        for name, rows, cols, inp in shapes:
            sel = np.sort(rng.choice(rows, rows_per, replace=False))
            f = {k: v[sel] for k, v in pf[name].items()}
            q, d8, s = quant[inp]
            t0 = time.perf_counter()
            O.mmq(f, q, d8, s)
            spent += time.perf_counter() - t0
            ops += 2.0 * 512 * rows_per * cols
        passes += 1
    full_ops = 2.0 * 512 * (9728 * 2560 + 2560 * 9728)
    tops = ops / spent / 1e12
    desc = (f"oracle MMQ on {passes} passes of {rows_per} random rows of gate and of down, all 512 tokens "
            f"(q8_1 of the inputs computed once, outside the timing)")
    return tops, 512 * tops * 1e12 / full_ops, spent, desc


def cpu_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def single_core_decode(budget_s: float):
    """The oracle GEMV sample in a child process pinned to one core with one
    BLAS thread (a fresh interpreter, so the limits apply from its start)."""
    code = ("import json,os,sys; sys.path.insert(0, %r); os.sched_setaffinity(0, {min(os.sched_getaffinity(0))});"
            "import bench; g,s,d = bench.oracle_decode_sample(%r); print(json.dumps([g,s,d]))" % (ROOT, budget_s))
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    try:
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                           timeout=budget_s * 10 + 120)
        g, s, d = json.loads(r.stdout.strip().splitlines()[-1])
        return {"value": g, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": d, "seconds": round(s, 2)}
    except Exception as e:  # noqa: BLE001 - the baseline is reported, never required
        return {"value": None, "error": f"{type(e).__name__}: {e}"[:200]}


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    # each step: a bounded oracle sample of the decode set (~1 s)
    total_bytes = 0.0
    total_s = 0.0
    desc = ""
    for i in range(args.warmup + args.steps):
        gbs, spent, desc = oracle_decode_sample(1.0, seed_rows=i)
        if i >= args.warmup:
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
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    bf16 = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS))

    def ev():
        return torch.cuda.Event(enable_timing=True)

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        return g

    def time_graph(g, reps=5):
        """Median over `reps` back-to-back replays (one warm replay first)."""
        g.replay()
        barrier()
        evs = [(ev(), ev()) for _ in range(reps)]
        for a, b in evs:
            a.record()
            g.replay()
            b.record()
        barrier()
        return statistics.median(a.elapsed_time(b) for a, b in evs)

    # ---------------- weights: pack once, then rotate copies to defeat L2
    fields, xs_np = decode_inputs()
    t_pack0 = time.perf_counter()
    packed = {}
    pack_bytes = 0
    dev_fields = {}
    for name, rows, cols, _ in synth.QWEN3_4B_LAYER:
        f = fields[name]
        dev_fields[name] = {k: torch.from_numpy(v.view(np.int16) if v.dtype == np.uint16 else v).to(dev)
                            for k, v in f.items()}
    torch.cuda.synchronize()
    p0, p1 = ev(), ev()
    p0.record()
    for name, rows, cols, _ in synth.QWEN3_4B_LAYER:
        d = dev_fields[name]
        packed[name] = q4k.q4k_pack(d["d"], d["dmin"], d["sc"], d["m"], d["q"])
        pack_bytes += sum(t.numel() * t.element_size() for t in d.values()) + packed[name].numel()
    p1.record()
    torch.cuda.synchronize()
    pack_ms = p0.elapsed_time(p1)
    del dev_fields
    layer_bytes = sum(p.numel() for p in packed.values())
    n_copies = max(2, math.ceil(4 * l2 / layer_bytes))
    copies = [packed] + [{k: v.clone() for k, v in packed.items()} for _ in range(n_copies - 1)]
    xs = {k: torch.from_numpy(v).to(dev) for k, v in xs_np.items()}
    ys = {name: torch.empty((1, rows), dtype=torch.float32, device=dev)
          for name, rows, _, _ in synth.QWEN3_4B_LAYER}
    log(f"[bench] rank {rank}: {n_copies} layer copies x {layer_bytes / 1e6:.1f} MB, pack {pack_ms:.2f} ms "
        f"(setup {time.perf_counter() - t_pack0:.1f}s)")

    def set_bytes(batch):
        return sum(rows * cols * BYTES_PER_WEIGHT + batch * (cols + rows) * 4
                   for _, rows, cols, _ in synth.QWEN3_4B_LAYER)

    step_bytes = set_bytes(1)
    shape = {name: (rows, cols, inp) for name, rows, cols, inp in synth.QWEN3_4B_LAYER}
    # engine order: one group per input (QKV triple, o, gate/up pair, down)
    launch_groups = (("q", "k", "v"), ("o",), ("gate", "up"), ("down",))

    def layer_jobs(layer, wait_groups, xs_=None, ys_=None):
        xs_ = xs if xs_ is None else xs_
        ys_ = ys if ys_ is None else ys_
        jobs = []
        for gi, names in enumerate(launch_groups):
            for k, n in enumerate(names):
                rows, cols, inp = shape[n]
                jobs.append({"w": layer[n], "rows": rows, "cols": cols, "x": xs_[inp], "y": ys_[n],
                             "wait": wait_groups and gi > 0 and k == 0})
        return jobs

    ws_seq = {}   # one workspace per batch, shared by the lists of that batch (never run concurrently)

    def gemv_seq(jobs, batch=1):
        try:
            seq = q4k.GemvSeq(jobs, batch, workspace=ws_seq.get(batch))
        except ValueError:                      # the shared workspace is too small for this list
            seq = q4k.GemvSeq(jobs, batch)
        if batch not in ws_seq or seq.workspace.numel() > ws_seq[batch].numel():
            ws_seq[batch] = seq.workspace
        return seq

    def seq_calls(first, count, max_per=MAX_SETS_PER_LAUNCH, wait_groups=False, xs_=None, ys_=None):
        calls, i = [], first
        for n in even_split(count, max_per):
            jobs = []
            for k in range(i, i + n):
                jobs += layer_jobs(copies[k % n_copies], wait_groups, xs_, ys_)
            calls.append(gemv_seq(jobs))
            i += n
        return calls

    # ---------------- headline: `steps` decode sets per replay
    warm_calls = seq_calls(0, args.warmup)
    timed_calls = seq_calls(args.warmup, args.steps)
    n_launch = len(timed_calls)
    for c in warm_calls:
        c()
    torch.cuda.synchronize()
    warm_graph = capture(lambda: [c() for c in warm_calls])
    timed_graph = capture(lambda: [c() for c in timed_calls])
    warm_graph.replay()
    ms_guess = time_graph(timed_graph, 3)
    reps = max(MIN_REPLAYS, int(REPLAY_SECONDS * 1e3 / max(ms_guess, 1e-3)))
    sampler = ClockSampler(uuid)
    sampler.start()
    time.sleep(0.25)                      # the sampler's first reading is not part of the region
    evs = [(ev(), ev()) for _ in range(reps)]
    barrier()
    sampler.mark(True)
    for a, b in evs:
        a.record()
        timed_graph.replay()
        b.record()
    barrier()
    sampler.mark(False)
    clocks = sampler.stop()
    replay_ms = sorted(a.elapsed_time(b) for a, b in evs)
    elapsed_ms = statistics.median(replay_ms)
    if q4k.q4k_device_error() != 0:
        raise RuntimeError("a GEMV kernel gave up a bounded wait during the timed region")

    # ---------------- decode in engine order (each group reads the previous
    # group's output): one layer as 4 launches, one layer as one q4k_gemv_seq
    # launch with waits, and the 36-layer token as q4k_gemv_seq launches
    def decode_step_4launch(i):
        layer = copies[i % n_copies]
        for names in launch_groups:
            rows = [shape[n][0] for n in names]
            cols, inp = shape[names[0]][1], shape[names[0]][2]
            if len(names) == 1:
                q4k.q4k_gemv(layer[names[0]], rows[0], cols, xs[inp], y=ys[names[0]])
            else:
                q4k.q4k_gemv_multi([layer[n] for n in names], rows, cols, xs[inp], ys=[ys[n] for n in names])

    for i in range(3):
        decode_step_4launch(i)
    torch.cuda.synchronize()
    ms_4launch = time_graph(capture(lambda: [decode_step_4launch(i) for i in range(args.steps)]), 20)
    chain_calls = seq_calls(0, args.steps, max_per=1, wait_groups=True)
    for c in chain_calls[:3]:
        c()
    ms_chain = time_graph(capture(lambda: [c() for c in chain_calls]), 20)

    def stack_token(batch, wait_groups):
        """One decode token over the 36-layer stack (layer L reads copy L %
        n_copies): 252 jobs, 3 launches."""
        xs_b = {name: torch.from_numpy(synth.activations(batch, cols, synth.layer_seed(synth.WL_STACK_4B, 0, 100 + j)))
                .to(dev) for j, (name, cols) in enumerate(synth.QWEN3_4B_INPUTS)}
        ys_b = {n: torch.empty((batch, shape[n][0]), device=dev) for n in shape}
        jobs = []
        for L in range(36):
            lj = layer_jobs(copies[L % n_copies], wait_groups, xs_b, ys_b)
            lj[0]["wait"] = wait_groups and L > 0      # layer L's QKV reads layer L-1's output
            jobs += lj
        tok = gemv_seq(jobs, batch)
        tok()
        torch.cuda.synchronize()
        n_tok = 10
        ms = time_graph(capture(lambda: [tok() for _ in range(n_tok)]), 10) / n_tok
        return {"tokens_per_s": batch / (ms * 1e-3), "ms_per_token": ms,
                "GB/s": 36 * set_bytes(batch) / (ms * 1e-3) / 1e9}

    token_engine = {f"batch{b}": stack_token(b, True) for b in (1, 4)}
    stack_indep = {f"batch{b}": stack_token(b, False) for b in (1, 4)}

    # Q4_K_M-style stack: v and down in Q6_K (GPU layout) in every other layer,
    # one token in engine order through the job list (mixed formats)
    q6_mats = {}
    for n in ("v", "down"):
        rows, cols, _ = shape[n]
        f6 = synth.q6k_fields(rows, cols, [795, rows])
        q6w = q4k.q6k_pack(torch.from_numpy(f6["d"].view(np.int16)).to(dev), torch.from_numpy(f6["sc"]).to(dev),
                           torch.from_numpy(f6["q"]).to(dev))
        q6_mats[n] = [q6w] + [q6w.clone() for _ in range(n_copies - 1)]
        del f6

    def q4km_token():
        batch = 1
        xs_b = {name: torch.from_numpy(synth.activations(batch, cols, synth.layer_seed(synth.WL_STACK_4B, 0, 200 + j)))
                .to(dev) for j, (name, cols) in enumerate(synth.QWEN3_4B_INPUTS)}
        ys_b = {n: torch.empty((batch, shape[n][0]), device=dev) for n in shape}
        jobs, nbytes = [], 0
        for L in range(36):
            lj = layer_jobs(copies[L % n_copies], True, xs_b, ys_b)
            lj[0]["wait"] = L > 0
            for j in lj:
                name = next(n for n in shape if ys_b[n] is j["y"])
                rows, cols, _ = shape[name]
                if L % 2 == 0 and name in q6_mats:
                    j["w"], j["format"] = q6_mats[name][L % n_copies], 1
                    nbytes += rows * (cols // 256) * 210
                else:
                    nbytes += rows * (cols // 256) * 144
                nbytes += batch * (rows + cols) * 4
            jobs += lj
        tok = gemv_seq(jobs, batch)
        tok()
        torch.cuda.synchronize()
        n_tok = 10
        ms = time_graph(capture(lambda: [tok() for _ in range(n_tok)]), 10) / n_tok
        return {"tokens_per_s": batch / (ms * 1e-3), "ms_per_token": ms, "GB/s": nbytes / (ms * 1e-3) / 1e9,
                "weight_bytes": nbytes,
                "note": "36 layers in engine order, v and down in Q6_K in layers 0, 2, ..., 34 (252 jobs)"}

    token_q4km = q4km_token()
    del q6_mats

    def q8_layers(batch, n_layers=20):
        """Decode layers at `batch` tokens through the q8_1 GEMV (MMQ form): per
        layer q8_1 of the four inputs and one q4k_gemv_q8 launch per matrix."""
        xs_b = {name: torch.from_numpy(synth.activations(batch, cols, [77, j, batch])).to(dev)
                for j, (name, cols) in enumerate(synth.QWEN3_4B_INPUTS)}
        q8b = {k: q4k.q8_quantize(v) for k, v in xs_b.items()}
        ys_b = {n: torch.empty((batch, shape[n][0]), device=dev) for n in shape}

        def run():
            for L in range(n_layers):
                layer = copies[L % n_copies]
                for k, v in xs_b.items():
                    q4k.q8_quantize(v, *q8b[k])
                for n in shape:
                    rows, cols, inp = shape[n]
                    q4k.q4k_gemv_q8(layer[n], rows, cols, *q8b[inp], y=ys_b[n])
        run()
        torch.cuda.synchronize()
        ms = time_graph(capture(run), 10) / n_layers
        return {"us_per_layer": 1e3 * ms, "tokens_per_s_36_layers": batch / (36 * ms * 1e-3),
                "GB/s": layer_bytes / (ms * 1e-3) / 1e9,
                "note": "q8_1 of the 4 inputs + 7 q4k_gemv_q8 launches per layer, layers in sequence (graph)"}

    q8_decode = {f"batch{b}": q8_layers(b) for b in (1, 4, 8)}

    # ---------------- Q6_K decode GEMV (GPU layout): the Q6_K matrices of a
    # Q4_K_M Qwen3-4B -- the output head and a down projection
    def q6k_case(rows, cols, batch, seed, calls=12, reps=10, q8=False):
        f = synth.q6k_fields(rows, cols, seed)
        w = q4k.q6k_pack(torch.from_numpy(f["d"].view(np.int16)).to(dev), torch.from_numpy(f["sc"]).to(dev),
                         torch.from_numpy(f["q"]).to(dev))
        del f
        n_c = max(2, math.ceil(4 * l2 / w.numel()))
        wc = [w] + [w.clone() for _ in range(n_c - 1)]
        x = torch.from_numpy(synth.activations(batch, cols, [seed, 1])).to(dev)
        y = torch.empty((batch, rows), device=dev)
        xq = q4k.q8_quantize(x) if q8 else None

        def run():
            for i in range(calls):
                if q8:
                    q4k.q6k_gemm(wc[i % n_c], rows, cols, *xq, y=y)
                else:
                    q4k.q6k_gemv(wc[i % n_c], rows, cols, x, y=y)
        run()
        torch.cuda.synchronize()
        ms = time_graph(capture(run), reps) / calls
        alg = rows * (cols // 256) * 210 + batch * (rows + cols) * 4
        del wc, w
        return {"rows": rows, "cols": cols, "batch": batch, "us": 1e3 * ms, "GB/s": alg / (ms * 1e-3) / 1e9,
                "frac_of_measured_hbm": alg / (ms * 1e-3) / 1e9 / hbm_peak, "weight_copies": n_c}

    q6k_decode = {"output_head_151936x2560_b1": q6k_case(151936, 2560, 1, 760),
                  "down_2560x9728_b1": q6k_case(2560, 9728, 1, 761, calls=40),
                  "down_2560x9728_b4": q6k_case(2560, 9728, 4, 762, calls=40),
                  "v_1024x2560_b1": q6k_case(1024, 2560, 1, 763, calls=60),
                  "down_2560x9728_q8_1_b1": q6k_case(2560, 9728, 1, 764, calls=40, q8=True),
                  "down_2560x9728_q8_1_b8": q6k_case(2560, 9728, 8, 765, calls=40, q8=True),
                  "down_2560x9728_q8_1_33_tokens": q6k_case(2560, 9728, 33, 766, calls=20, q8=True)}
    torch.cuda.empty_cache()

    # ---------------- single 2048x2048 GEMV, batch 1 (L2-resident: latency)
    f0, x0 = synth.single_gemv_2048(0)
    d0 = {k: torch.from_numpy(v.view(np.int16) if v.dtype == np.uint16 else v).to(dev) for k, v in f0.items()}
    w0 = q4k.q4k_pack(d0["d"], d0["dmin"], d0["sc"], d0["m"], d0["q"])
    x0d = torch.from_numpy(x0).to(dev)
    y0 = torch.empty((1, 2048), device=dev)
    q4k.q4k_gemv(w0, 2048, 2048, x0d, y=y0)
    torch.cuda.synchronize()
    n_small = 100
    us_gemv = 1e3 * time_graph(capture(lambda: [q4k.q4k_gemv(w0, 2048, 2048, x0d, y=y0) for _ in range(n_small)]),
                               10) / n_small
    seq0 = gemv_seq([{"w": w0, "rows": 2048, "cols": 2048, "x": x0d, "y": y0}])
    seq0()
    us_seq0 = 1e3 * time_graph(capture(lambda: [seq0() for _ in range(n_small)]), 10) / n_small
    bytes0 = 2048 * 2048 * BYTES_PER_WEIGHT + 2 * 2048 * 4

    # ---------------- e2e: public API with host buffers, copies in the region.
    # Every step (decode set) has its own 4 input vectors and 7 outputs, rows
    # of one pinned host array each way.  The steps run in the headline's
    # launches (even split, at most MAX_SETS_PER_LAUNCH sets per launch), one
    # q4k_gemv_seq_launch_host call per launch (GemvSeq.step on buffers bound
    # before the timed region): the copy of its sets' inputs, the planned
    # launch, the copy of its sets' outputs.
    in_off, off = {}, 0
    for k, v in xs_np.items():
        in_off[k] = (off, v.shape)
        off += v.size
    set_in = off
    out_off, off = {}, 0
    for name, rows, _, _ in synth.QWEN3_4B_LAYER:
        out_off[name] = off
        off += rows
    set_out = off
    n_sets = args.warmup + args.steps
    x_host = torch.empty((n_sets, set_in), dtype=torch.float32).pin_memory()
    for i in range(n_sets):
        for j, (k, v) in enumerate(xs_np.items()):
            o = in_off[k][0]
            x_host[i, o:o + v.size] = torch.from_numpy(
                synth.activations(v.shape[0], v.shape[1], [synth.WL_DECODE_4B, 900 + i, j]).reshape(-1))
    x_dev = torch.empty((n_sets, set_in), dtype=torch.float32, device=dev)
    y_dev = torch.empty((n_sets, set_out), dtype=torch.float32, device=dev)
    y_host = torch.empty((n_sets, set_out), dtype=torch.float32).pin_memory()

    def set_views(i):
        xv = {k: x_dev[i, o:o + int(np.prod(shp))].view(shp) for k, (o, shp) in in_off.items()}
        yv = {name: y_dev[i, out_off[name]:out_off[name] + rows].view(1, rows)
              for name, rows, _, _ in synth.QWEN3_4B_LAYER}
        return xv, yv

    def e2e_launches(first, count, max_per):
        calls, i = [], first
        for n in even_split(count, max_per):
            jobs = []
            for k in range(i, i + n):
                jobs += layer_jobs(copies[k % n_copies], False, *set_views(k))
            seq = gemv_seq(jobs)
            seq.bind_host(x_host[i:i + n], x_dev[i:i + n], y_host[i:i + n], y_dev[i:i + n])
            calls.append(seq)
            i += n
        return calls

    h2d = set_in * 4
    d2h = set_out * 4

    def e2e_time(max_per):
        warm = e2e_launches(0, args.warmup, max_per)
        timed = e2e_launches(args.warmup, args.steps, max_per)
        for seq in warm:
            seq.step()
        barrier()
        e0, e1 = ev(), ev()
        t0 = time.perf_counter()
        e0.record()
        for seq in timed:
            seq.step()
        e1.record()
        t1 = time.perf_counter()
        barrier()
        return e0.elapsed_time(e1), 1e6 * (t1 - t0) / args.steps, len(timed)

    e2e_ms, e2e_host_us, e2e_launch_n = e2e_time(MAX_SETS_PER_LAUNCH)
    e2e_one_ms, e2e_one_host_us, _ = e2e_time(1)
    if q4k.q4k_device_error() != 0:
        raise RuntimeError("a GEMV kernel gave up a bounded wait in the end-to-end leg")

    # ---------------- prefill GEMMs (q8_1 + MMQ)
    def prefill_case(mats, xs_in, tokens, layers=1, rotate=True, form="h16"):
        """mats: [(name, fields, rows, cols, input)].  Times one step = q8_1 of
        every input + every GEMM, `layers` times over rotating weight copies.
        form "h16": q8_quantize_h16 + q4k_gemm_h16; "int8": q8_quantize + q4k_gemm;
        "f16": x_split_f16 + q4k_gemm_f16 (fp16 activations, no q8_1 step)."""
        quant = {"h16": q4k.q8_quantize_h16, "int8": q4k.q8_quantize, "f16": q4k.x_split_f16}[form]
        gemm = {"h16": q4k.q4k_gemm_h16, "int8": q4k.q4k_gemm, "f16": q4k.q4k_gemm_f16}[form]
        w = {}
        for name, f, rows, cols, inp in mats:
            d = {k: torch.from_numpy(v.view(np.int16) if v.dtype == np.uint16 else v).to(dev) for k, v in f.items()}
            w[name] = q4k.q4k_pack(d["d"], d["dmin"], d["sc"], d["m"], d["q"])
        x = {k: torch.from_numpy(v).to(dev) for k, v in xs_in.items()}
        wbytes = sum(v.numel() for v in w.values())
        n_c = max(2, math.ceil(4 * l2 / wbytes)) if rotate else 1
        wsets = [w] + [{k: v.clone() for k, v in w.items()} for _ in range(n_c - 1)]
        q8 = {k: quant(v) for k, v in x.items()}
        y = {name: torch.empty((tokens, rows), device=dev) for name, _, rows, _, _ in mats}

        def step(gemm_only=False):
            for L in range(layers):
                ws = wsets[L % n_c]
                if not gemm_only:
                    for k, v in x.items():
                        if form == "f16":
                            quant(v, out=q8[k])
                        else:
                            quant(v, *q8[k])
                for name, _, rows, cols, inp in mats:
                    gemm(ws[name], rows, cols, *q8[inp], y=y[name])

        step()
        torch.cuda.synchronize()
        ops = layers * sum(2.0 * tokens * rows * cols for _, _, rows, cols, _ in mats)
        reps = 3 if layers > 1 else 10
        ms = time_graph(capture(step), reps)
        ms_gemm = time_graph(capture(lambda: step(True)), reps)
        launches = layers * (len(x) + len(mats))
        del wsets, w
        return {"tokens": tokens, "form": form, "ms_per_step": ms, "tok_s": tokens / (ms * 1e-3),
                "int_tops": ops / (ms * 1e-3) / 1e12, "gemm_ms": ms_gemm,
                "gemm_tops": ops / (ms_gemm * 1e-3) / 1e12, "gemm_frac_of_bf16": ops / (ms_gemm * 1e-3) / 1e12 / bf16,
                "gpu_launches": launches, "l2": f"{n_c} rotating weight copies"}

    pf, pxs = synth.prefill_4b_512()
    mats512 = [("gate", pf["gate"], 9728, 2560, "mlp_in"), ("down", pf["down"], 2560, 9728, "down_in")]
    prefill512 = prefill_case(mats512, pxs, 512)
    prefill512["workload"] = "512-token prefill: q8_1 X[512x2560] x gate 9728x2560, X_down[512x9728] x down 2560x9728"
    p512_int8 = prefill_case(mats512, pxs, 512, form="int8")
    prefill512["int8_entry_point"] = {k: p512_int8[k] for k in ("ms_per_step", "tok_s", "gemm_tops")}
    p512_f16 = prefill_case(mats512, pxs, 512, form="f16")
    prefill512["f16_activations"] = {k: p512_f16[k] for k in ("ms_per_step", "tok_s", "gemm_tops",
                                                              "gemm_frac_of_bf16")}
    # short prompts (the pages' 18-33-token regime) on the same two matrices
    short = {}
    for T in (8, 16, 33, 64):
        sx = {k: np.ascontiguousarray(v[:T]) for k, v in pxs.items()}
        for form in ("h16", "int8"):
            r = prefill_case(mats512, sx, T, form=form)
            short[f"tokens{T}_{form}"] = {k: r[k] for k in ("ms_per_step", "tok_s", "gemm_tops", "gemm_frac_of_bf16")}
    # 2048-token prefill of the 36-layer Qwen3-4B stack (7 projections a layer)
    x2048 = {name: synth.activations(2048, cols, synth.layer_seed(synth.WL_STACK_4B, 0, 300 + j))
             for j, (name, cols) in enumerate(synth.QWEN3_4B_INPUTS)}
    mats_layer = [(n, fields[n], shape[n][0], shape[n][1], shape[n][2]) for n in shape]
    prefill2048 = prefill_case(mats_layer, x2048, 2048, layers=36)
    prefill2048["workload"] = ("2048-token prefill of the 36-layer Qwen3-4B-shaped stack: per layer q8_1 of 4 inputs "
                               "and 7 GEMMs (q 4096x2560, k/v 1024x2560, o 2560x4096, gate/up 9728x2560, down 2560x9728)")
    del x2048
    # 4096-token prefill of the Qwen3-8B MLP
    f8, x8 = synth.prefill_8b_4096()
    mats8 = [(n, f8[n], rows, cols, inp) for n, rows, cols, inp in synth.QWEN3_8B_MLP]
    prefill8b = prefill_case(mats8, x8, 4096)
    prefill8b["workload"] = "4096-token prefill, Qwen3-8B MLP: gate/up 12288x4096, down 4096x12288"
    p8_f16 = prefill_case(mats8, x8, 4096, form="f16")
    prefill8b["f16_activations"] = {k: p8_f16[k] for k in ("ms_per_step", "tok_s", "gemm_tops", "gemm_frac_of_bf16")}
    del f8, x8

    # Q6_K prefill: the down projection (Q6_K in Q4_K_M) at 512 tokens through
    # the fp16-activation tensor-core GEMM, and through the q8_1 GEMV launches
    def q6k_prefill(rows, cols, tokens, seed, reps=10):
        f = synth.q6k_fields(rows, cols, seed)
        w = q4k.q6k_pack(torch.from_numpy(f["d"].view(np.int16)).to(dev), torch.from_numpy(f["sc"]).to(dev),
                         torch.from_numpy(f["q"]).to(dev))
        del f
        n_c = max(2, math.ceil(4 * l2 / w.numel()))
        wc = [w] + [w.clone() for _ in range(n_c - 1)]
        x = torch.from_numpy(synth.activations(tokens, cols, [seed, 1])).to(dev)
        y = torch.empty((tokens, rows), device=dev)
        sp = q4k.x_split_f16(x)
        xq = q4k.q8_quantize(x)
        out = {}
        for form in ("f16", "q8_1"):
            def run(calls=6):
                for i in range(calls):
                    if form == "f16":
                        q4k.q6k_gemm_f16(wc[i % n_c], rows, cols, *sp, y=y)
                    else:
                        q4k.q6k_gemm(wc[i % n_c], rows, cols, *xq, y=y)
            run()
            torch.cuda.synchronize()
            ms = time_graph(capture(run), reps) / 6
            out[form] = {"ms": ms, "tops": 2.0 * tokens * rows * cols / (ms * 1e-3) / 1e12,
                         "tok_s": tokens / (ms * 1e-3)}
        del wc, w
        return {"tokens": tokens, "rows": rows, "cols": cols, **out,
                "note": "GEMM only (x_split_f16 / q8_quantize outside the timed graph); q8_1 form = one q6k_gemv_q8 "
                        "launch per 8 tokens"}

    prefill_q6k = q6k_prefill(2560, 9728, 512, 780)
    torch.cuda.empty_cache()

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
    e2e_one_ms = max_over_ranks(e2e_one_ms)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    value = job_throughput(step_bytes, args.steps, world, elapsed_ms)
    e2e_value = job_throughput(step_bytes, args.steps, world, e2e_ms)
    e2e_one_value = job_throughput(step_bytes, args.steps, world, e2e_one_ms)
    # the timed replay holds nothing but this kernel's launches: the average
    # launch duration is the replay over its launches, and each launch
    # processes its sets' algorithmic bytes
    achieved = step_bytes * args.steps / (elapsed_ms * 1e-3) / 1e9
    traffic_rec = profile_traffic("gemv_seq", ["gemv_seq_kernel.cuh", "gemv_common.cuh"])
    traffic = None
    if traffic_rec is not None:
        # the record is for a launch of MAX_SETS_PER_LAUNCH sets: scale to this run's average launch
        traffic = traffic_rec * (args.steps / n_launch) / MAX_SETS_PER_LAUNCH

    cpu = None
    cpu_single = None
    cpu_gemm = None
    if world == 1 and not args.no_cpu_baseline:
        gbs, spent, desc = oracle_decode_sample(args.cpu_seconds)
        cpu = {"value": gbs, "unit": "GB/s", "cores": cpu_threads(), "kind": "oracle", "sample": desc,
               "seconds": round(spent, 2)}
        cpu_single = single_core_decode(args.cpu_seconds)
        tops, tok_s, spent, desc = oracle_gemm_sample(args.cpu_seconds)
        cpu_gemm = {"value": tok_s, "unit": "tok/s", "int_tops": tops, "cores": cpu_threads(), "kind": "oracle",
                    "sample": desc, "seconds": round(spent, 2)}

    sm_mhz = (clocks or {}).get("sm_mhz")
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": 1, "parallelism": "replicas" if world > 1 else "single",
                   "timing": (f"median of {reps} back-to-back replays of one CUDA graph of exactly `steps` steps "
                              f"(replay times: min {replay_ms[0]:.4f} ms, median {elapsed_ms:.4f} ms, "
                              f"max {replay_ms[-1]:.4f} ms); each step is the seven GEMVs of the decode linear "
                              f"set (independent N(0,1) inputs); the steps are split evenly over "
                              f"{n_launch} q4k_gemv_seq launches ({even_split(args.steps, MAX_SETS_PER_LAUNCH)} "
                              f"sets)"),
                   "l2": f"inputs larger than L2: {n_copies} rotating layer copies "
                         f"({n_copies * layer_bytes / 1e6:.0f} MB, L2 {l2 / 1e6:.0f} MB)",
                   "launches": n_launch},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "frac_of_nominal_8TBs": achieved / NOMINAL_HBM_GBS,
                     "traffic": traffic, "peak_kind": f"{peak_kind} hbm_gbs",
                     "kernel": "gemv_seq_kernel<1, 0>",
                     "duration": "CUDA events on the launching stream around each replay (one graph of the "
                                 "launches of this kernel, nothing else), divided by its launches; algorithmic "
                                 "bytes per launch = the sets it holds x bytes per set"},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "us_per_step": 1e3 * e2e_ms / args.steps, "host_issue_us_per_step": e2e_host_us,
                "launches": e2e_launch_n,
                "one_set_per_call": {"value": e2e_one_value, "us_per_step": 1e3 * e2e_one_ms / args.steps,
                                     "host_issue_us_per_step": e2e_one_host_us},
                "note": "each step (decode set) has its own inputs and outputs in pinned host memory; the steps run "
                        "in the headline's launches, one q4k_gemv_seq_launch_host call each: the copy of its sets' "
                        "inputs, the prepared plan's launch, the copy of its sets' outputs; no graph.  "
                        "one_set_per_call: one call (one launch) per step"},
        "gpu_launches": n_launch,
        "clocks": clocks,
        "time_x_sm_mhz": (elapsed_ms / args.steps * 1e3 * sm_mhz) if sm_mhz else None,
        "decode_engine_order": {
            "note": "each input group reads the previous group's output (QKV | o | gate,up | down)",
            "layer_4_launches": {"us_per_layer": 1e3 * ms_4launch / args.steps,
                                 "GB/s": step_bytes * args.steps / (ms_4launch * 1e-3) / 1e9},
            "layer_gemv_seq_with_waits": {"us_per_layer": 1e3 * ms_chain / args.steps,
                                          "GB/s": step_bytes * args.steps / (ms_chain * 1e-3) / 1e9},
            "token_36_layers_gemv_seq_with_waits": token_engine,
            "token_36_layers_q4_k_m_mixed_formats_batch1": token_q4km},
        "decode_q8_1_gemv_per_layer": q8_decode,
        "decode_q6k_gemv": {**q6k_decode,
                            "note": "q6k_gemv launches (fp32 activations) or q6k_gemm (q8_1 activations, one "
                                    "launch per 8 tokens) over Q6K_LAYOUT_GPU weights, rotating copies (inputs larger "
                                    "than L2), median of graph replays; algorithmic bytes = 210 per 256 weights "
                                    "+ x + y (weights counted once per call)"},
        "decode_stack_36_layers_independent_jobs": {
            "note": "the 252 GEMVs of the stack with no dependencies between them (not a decode token)",
            **stack_indep},
        "single_gemv_2048x2048_b1": {"us_q4k_gemv": us_gemv, "us_gemv_seq": us_seq0,
                                     "GB/s_q4k_gemv": bytes0 / (us_gemv * 1e-6) / 1e9,
                                     "note": "2.4 MB of weights, L2-resident: a latency case"},
        "cpu_baseline": cpu,
        "cpu_baseline_single_core": cpu_single,
        "cpu_baseline_gemm_prefill512": cpu_gemm,
        "pack": {"ms": pack_ms, "GB/s": pack_bytes / (pack_ms * 1e-3) / 1e9, "note": "one-off, 7 matrices"},
        "prefill": {
            **prefill512,
            "roofline": {"bound": "tensor", "achieved": prefill512["gemm_tops"], "unit": "TOPS", "peak": bf16,
                         "frac": prefill512["gemm_tops"] / bf16, "peak_kind": f"{peak_kind} bf16_tflops (fp16 rate)",
                         "note": "the GEMM's MMAs are tcgen05 kind::f16 on exact small integers, so its own-dtype "
                                 "peak is the dense fp16 = bf16 rate; sm_103a has no integer tcgen05 MMA",
                         "int8_peak_mma_sync_s8": int8_peak, "frac_of_int8_peak": prefill512["gemm_tops"] / int8_peak,
                         "tcgen05_f16_probe_tflops": f16_peak},
            "timing": "median of CUDA-graph replays of exactly one step (q8_quantize_h16 + q4k_gemm_h16 for "
                      "gate and down); gemm_tops from a graph of the GEMM launches alone",
        },
        "prefill_short_prompts": short,
        "prefill_2048_stack": prefill2048,
        "prefill_q6k_down_512": prefill_q6k,
        "prefill_4096_qwen3_8b_mlp": prefill8b,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=52)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
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
