"""Decode-step throughput of the GB300 Q8_0 decode path.

One step = one launch of the captured decode-step graph (a memset and the
persistent step kernel): every Q8_0 matvec (196 layer matvecs + lm_head),
every layer's KV append + split-K attention, all glue, argmax; token and
position stay in device memory.

Workload (default): 7B-shaped model (hidden 3584, 28 layers, 28/4 heads,
head_dim 128, FFN 18944, vocab 152064, Q8_0 weights = 7.51 GB + 0.58 GB
embedding), f16 KV cache, context 2048 at the first timed step.  Inputs are
seeded synthetic tensors drawn on the device; the weights streamed each
step (7.5 GB) are 58x the 129 MB L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl q8d|reference]

Prints one JSON line (rank 0).  Under torchrun (N > 1) every rank runs an
independent replica (the decode step does not shard: replicas only) and
`value` is the sum of the ranks' tokens over the max of their times.
Besides the workload's own step the line carries kernel legs through the
C ABI (q8d_matvec over the step's matrices, q8d_gqa_decode_attn per layer
at the context and at 8192, the batch-8 ragged stress, q8d_matmul_small_m)
and, under "configs", decode steps of the other configurations
(Qwen3-0.6B at 2048, Qwen2.5-0.5B at 512/2048/4096, 7B at 2048/8192).
The reference arm (--impl reference) times the scalar C oracle on all host
cores: W untimed and exactly K timed whole decode steps of the workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "q8_matvec & gqa_decode_attn HBM GB/s (% of GB300 peak); decode-step tokens/s"


def bf16_peak():
    """Measured dense bf16 TFLOP/s (cuBLAS burst), else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 1900.0


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during a region
    (every 20 ms; samples are kept with their host arrival time so that the
    summary covers the timed window only)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 20):
        self.index = index
        self.period_ms = period_ms
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)  # the first sample is in before the region starts
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def __exit__(self, *a):
        if self.proc:
            time.sleep(2 * self.period_ms / 1e3)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self, t0=None, t1=None):
        """Median SM clock and active throttle reasons of the samples taken
        in [t0, t1] (host monotonic time; the whole run if not given).  A
        window shorter than the sampling period keeps the nearest sample
        on each side."""
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = self.lines
        if t0 is not None and rows:
            inside = [r for r in rows if t0 <= r[0] <= t1]
            if not inside:
                before = [r for r in rows if r[0] < t0][-1:]
                after = [r for r in rows if r[0] > t1][:1]
                inside = before + after
            rows = inside
        for _, ln in rows:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "period_ms": self.period_ms}


def gpu_index():
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    import torch
    cur = torch.cuda.current_device()
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if cur < len(ids) and ids[cur].isdigit():
            return int(ids[cur])
    return cur


# ---------------------------------------------------------------------------- sizes
def matvec_bytes(n, p):
    return 34 * p * (n // 32) + 4 * n + 4 * p


def attn_bytes(L, Hk, D, H, esize, append=True):
    return L * Hk * D * 2 * esize + 4 * 2 * H * D + (2 * Hk * D * esize if append else 0)


STEP_KERNEL_SOURCES = ("q8d_megastep.cu", "q8d_megastep.cuh", "q8d_gemv.cuh", "q8d_mma_frag.cuh",
                       "q8d_internal.cuh", "q8d_attn.cuh", "q8d_attn_common.cuh", "q8d_step.cu")


class L2Flush:
    """Evicts L2 before a timed launch: writes one 256 MB buffer (twice the
    129 MB L2), then reads another 256 MB buffer, so the written lines are
    back in HBM before the timed region starts and the launch meets a cold,
    clean L2 (it pays for no other kernel's write-backs)."""

    DESC = "L2 flushed (256 MB written, then another 256 MB read)"

    def __init__(self):
        import torch
        self.w = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
        self.r = torch.zeros(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")

    def __call__(self, v: int):
        import torch
        self.w.fill_(v & 0xFF)
        torch.amax(self.r)


def kernel_source_sha():
    """Hash of the step kernel's sources (ties an ncu summary to a build)."""
    h = hashlib.sha256()
    for nm in STEP_KERNEL_SOURCES:
        with open(os.path.join(ROOT, "q8_block_quantized_matvec_gb300", "csrc", nm), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def step_bytes(shape, context: int, esize: int) -> float:
    """Algorithmic HBM bytes of one decode step at attended length `context`:
    every weight byte once (layers + lm_head + one embedding row), each
    layer's K and V rows read once and the new row written."""
    kv = shape.n_layers * (2 * context * shape.kv_width * esize + 2 * shape.kv_width * esize)
    return float(shape.weight_bytes() + kv)


def ncu_traffic(algorithmic_bytes: float):
    """DRAM bytes per launch of the step kernel: the committed ncu summary's
    measured DRAM bytes per algorithmic byte (a 4-layer capture of the same
    layer shapes) times this launch's algorithmic bytes, if the summary was
    taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "q8_step_kernel_7b_decode.md")
    try:
        txt = open(path).read()
    except OSError:
        return None
    sha = ratio = None
    for ln in txt.splitlines():
        if ln.startswith("kernel_source_sha:"):
            sha = ln.split(":", 1)[1].strip()
        if ln.startswith("dram_bytes_per_algorithmic_byte:"):
            ratio = float(ln.split(":", 1)[1].strip())
    if sha != kernel_source_sha() or ratio is None:
        return None
    return ratio * algorithmic_bytes


# ---------------------------------------------------------------------------- oracle
def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith(("model name", "cpu part")):
                return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def oracle_model(shape_name: str, context: int, n_layers: int = 0):
    """Host weights and caches of the workload for the oracle: the model's
    shapes (optionally truncated to n_layers), KV filled to context - 1
    rows; every timed step appends row context - 1 and attends `context`."""
    import synth
    from oracle import oracle as orc
    full = synth.MODELS[shape_name]
    shape = full
    if n_layers:
        shape = synth.ModelShape(full.name + f"-{n_layers}layer", full.hidden, n_layers,
                                 full.n_heads, full.n_kv_heads, full.head_dim, full.ffn,
                                 full.vocab, full.qk_norm, full.qkv_bias, full.kv_dtype,
                                 full.rms_eps, full.rope_theta)
    w = synth.step_weights(shape, seed=0)
    caches = [synth.kv_prefix(shape, 0, li, context, context - 1) for li in range(shape.n_layers)]
    return w, orc.HostStep(w, context, caches)


def oracle_full_steps(shape_name: str, context: int, steps: int, warmup: int, threads: int):
    """Wall times of `steps` whole decode steps of the oracle (every layer,
    lm_head, argmax) after `warmup` untimed ones, on `threads` host threads."""
    _, host = oracle_model(shape_name, context)
    for _ in range(warmup):
        host.step(17, context - 1, threads)
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        host.step(17, context - 1, threads)
        times.append(time.perf_counter() - t0)
    return times


def oracle_single_thread(shape_name: str, context: int, runs: int = 5):
    """One host thread, a bounded sample: the model truncated to 2 layers
    (lm_head included), median of `runs` steps after one warm-up, with the
    lm_head timed alone so that the full step projects as
    t(lm_head) + n_layers / 2 * (t(2-layer step) - t(lm_head))."""
    import synth
    from oracle import oracle as orc
    full = synth.MODELS[shape_name]
    w, host = oracle_model(shape_name, context, n_layers=2)
    x = synth.normal_f32(0, "bench.x", full.hidden)
    host.step(17, context - 1, 1)
    heads, steps = [], []
    for _ in range(runs):
        t0 = time.perf_counter()
        orc.q8_matvec(w.lm_head, x, full.hidden, full.vocab, 1)
        heads.append(time.perf_counter() - t0)
        t0 = time.perf_counter()
        host.step(17, context - 1, 1)
        steps.append(time.perf_counter() - t0)
    t_head, t_step2 = statistics.median(heads), statistics.median(steps)
    t_full = t_head + full.n_layers * max(t_step2 - t_head, 1e-9) / 2
    return {"value": 1.0 / t_full, "unit": "tokens/s", "cores": 1,
            "sample": (f"2 of {full.n_layers} layers (+lm_head, KV context {context}), median of "
                       f"{runs} steps: {t_step2:.3f} s, lm_head alone {t_head:.3f} s; projected "
                       f"full step {t_full:.2f} s")}


def cpu_baseline_leg(shape_name: str, context: int, runs: int = 5):
    """The oracle as it stands on this host: all cores on whole decode steps
    (median of `runs` after one warm-up), plus the single-thread mode on a
    2-layer sample; the CPU model is recorded."""
    from oracle import oracle as orc
    threads = orc.default_threads()
    t0 = time.perf_counter()
    times = oracle_full_steps(shape_name, context, runs, 1, threads)
    t_all = time.perf_counter() - t0
    single = oracle_single_thread(shape_name, context, runs)
    med = statistics.median(times)
    return {"value": 1.0 / med, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": (f"whole {shape_name}-shaped decode steps (every layer + lm_head, KV context "
                       f"{context}), median of {runs} after one warm-up: {med:.3f} s per step "
                       f"({t_all:.1f} s of wall time incl. the warm-up)"),
            "cpu_model": cpu_model(), "single_thread": single}


# ---------------------------------------------------------------------------- profiling
def run_profile(args):
    """Fixed workloads for ncu.  step: one decode-step graph launch of the
    bench workload after warm-up.  matvec: q8d_matvec on the 7B gate/up
    shape (3584 -> 18944, 72 MB), 3 launches.  attn: q8d_gqa_decode_attn on
    7B heads at --context (default 2048: 4.2 MB of KV), 3 launches.  ncu's default
    cache control flushes L2 before every profiled launch."""
    import torch
    from __graft_entry__ import build
    build()
    import q8_block_quantized_matvec_gb300 as q8d
    import synth
    torch.cuda.set_device(0)
    cudart = torch.cuda.cudart()
    if args.profile == "step":
        import dataclasses
        from q8_block_quantized_matvec_gb300.device import DeviceStep
        shape = synth.MODELS[args.model]
        if args.layers:
            # the same layer shapes with fewer layers: a capture-sized step
            shape = dataclasses.replace(shape, n_layers=args.layers)
        ctx = args.context
        cap = ctx + 16
        wts = synth.TorchStepWeights(shape, seed=0)
        kdt = torch.float16 if shape.kv_dtype == synth.KV_F16 else torch.float32
        caches = []
        for li in range(shape.n_layers):
            kc = synth.normal_torch(0, f"l{li}.kprefix", (cap, shape.kv_width), kdt)
            vc = synth.normal_torch(0, f"l{li}.vprefix", (cap, shape.kv_width), kdt)
            caches.append((kc, vc))
        ds = DeviceStep(wts, cap, caches)
        ds.set_state(17, ctx - 1)
        for _ in range(3):
            ds.launch()
        ds.set_state(17, ctx - 1)
        torch.cuda.synchronize()
        cudart.cudaProfilerStart()
        ds.launch()
        torch.cuda.synchronize()
        cudart.cudaProfilerStop()
        assert ds.step.status() == 0
        ds.close()
    elif args.profile == "matvec_sweep":
        # the bench's q8d_matvec launches for two 7B-shaped layers + lm_head
        # (the per-shape traffic scales to the 28-layer sweep by launch counts)
        shape = synth.MODELS[args.model]
        mats = []
        for li in range(2):
            for nm, n, p in [("wq", shape.hidden, shape.q_width), ("wk", shape.hidden, shape.kv_width),
                             ("wv", shape.hidden, shape.kv_width), ("wo", shape.q_width, shape.hidden),
                             ("wg", shape.hidden, shape.ffn), ("wu", shape.hidden, shape.ffn),
                             ("wd", shape.ffn, shape.hidden)]:
                mats.append((synth.q8_matrix_torch(0, f"l{li}.{nm}", p, n), n, p))
        mats.append((synth.q8_matrix_torch(0, "lm_head", shape.vocab, shape.hidden), shape.hidden,
                     shape.vocab))
        xs = {n: synth.normal_torch(0, f"x{n}", n, torch.float32) for _, n, _ in mats}
        y = torch.empty(max(p for _, _, p in mats), device="cuda")
        for w, n, p in mats:
            q8d.q8d_matvec(xs[n], w, y, n, p)
        torch.cuda.synchronize()
        cudart.cudaProfilerStart()
        for w, n, p in mats:
            q8d.q8d_matvec(xs[n], w, y, n, p)
        torch.cuda.synchronize()
        cudart.cudaProfilerStop()
    elif args.profile in ("matvec", "matvec_down", "matvec_kv"):
        n, p = {"matvec": (3584, 18944), "matvec_down": (18944, 3584),
                "matvec_kv": (3584, 512)}[args.profile]
        w = synth.q8_matrix_torch(0, "prof.w", p, n)
        x = synth.normal_torch(0, "prof.x", n, torch.float32)
        y = torch.empty(p, device="cuda")
        q8d.q8d_matvec(x, w, y, n, p)
        torch.cuda.synchronize()
        cudart.cudaProfilerStart()
        for _ in range(3):
            q8d.q8d_matvec(x, w, y, n, p)
        torch.cuda.synchronize()
        cudart.cudaProfilerStop()
    elif args.profile in ("mma16", "mma64"):
        m = 16 if args.profile == "mma16" else 64
        w, x, y, n, p = small_m_inputs(m)
        need = q8d.q8d_matmul_small_m_workspace_bytes(m, n)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        q8d.q8d_matmul_small_m_ws(x, n, w, y, p, m, n, p, ws, need)
        torch.cuda.synchronize()
        cudart.cudaProfilerStart()
        q8d.q8d_matmul_small_m_ws(x, n, w, y, p, m, n, p, ws, need)
        torch.cuda.synchronize()
        cudart.cudaProfilerStop()
    elif args.profile in ("attn_stress_q8", "attn_window"):
        s = torch.cuda.Stream()
        flush = L2Flush()
        fn = attn_stress_q8 if args.profile == "attn_stress_q8" else attn_window_leg
        fn(q8d, 28, 4, 128, 1, s, flush)  # warm-up launches (not profiled)
        torch.cuda.synchronize()
        cudart.cudaProfilerStart()
        fn(q8d, 28, 4, 128, 0, s, flush)  # four launches
        torch.cuda.synchronize()
        cudart.cudaProfilerStop()
    elif args.profile == "attn_stress":
        lens, args_, err = stress_inputs(q8d, 28, 4, 128)
        q8d.q8d_gqa_decode_attn(*args_)
        torch.cuda.synchronize()
        cudart.cudaProfilerStart()
        q8d.q8d_gqa_decode_attn(*args_)
        torch.cuda.synchronize()
        cudart.cudaProfilerStop()
        assert err.item() == 0
    else:
        H, Hk, D, L = 28, 4, 128, args.context
        kc = synth.normal_torch(0, "prof.k", (L, Hk * D), torch.float16)
        vc = synth.normal_torch(0, "prof.v", (L, Hk * D), torch.float16)
        q = synth.normal_torch(0, "prof.q", H * D, torch.float32)
        out = torch.empty(H * D, device="cuda")
        wsb = q8d.q8d_gqa_workspace_bytes(1, H, Hk, D, L)
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        lens = torch.tensor([L], dtype=torch.int32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        args_ = (q, None, None, kc, vc, q8d.Q8D_KV_F16, out, 1, H, Hk, D, L, 0, lens,
                 1 / math.sqrt(D), ws, wsb, err)
        q8d.q8d_gqa_decode_attn(*args_)
        torch.cuda.synchronize()
        cudart.cudaProfilerStart()
        for _ in range(3):
            q8d.q8d_gqa_decode_attn(*args_)
        torch.cuda.synchronize()
        cudart.cudaProfilerStop()
        assert err.item() == 0


# ---------------------------------------------------------------------------- attention stress
STRESS_CAP = 32768


def graph_seconds_per_call(calls, stream, reps=3):
    """Seconds per call of `calls` (zero-argument callables, each one library
    call on `stream`) captured once in a CUDA graph and replayed back to
    back; the median of `reps` replays, one timed region per replay."""
    import torch
    with torch.cuda.stream(stream):
        for c in calls:
            c()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="relaxed"):
        for c in calls:
            c()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    with torch.cuda.stream(stream):
        for rep in range(reps + 1):
            a.record(stream)
            graph.replay()
            b.record(stream)
            b.synchronize()
            if rep:
                times.append(a.elapsed_time(b) / 1e3 / len(calls))
    del graph
    return statistics.median(times)


def stress_inputs(q8d, H, Hk, D, rank=0):
    """The long-context attention workload: 8 sequences of the model's heads,
    lengths drawn uniformly from [1, 32768] (seeded), an f16 cache of 32768
    rows per sequence, no append."""
    import torch

    import synth
    cap, kvw = STRESS_CAP, Hk * D
    lens = synth.stream(0, "ragged.lens").integers(1, cap + 1, 8).tolist()
    kc = synth.normal_torch(rank, "stress.k", (8, cap, kvw), torch.float16)
    vc = synth.normal_torch(rank, "stress.v", (8, cap, kvw), torch.float16)
    q = synth.normal_torch(rank, "stress.q", (8, H * D), torch.float32)
    out = torch.empty(8, H * D, device="cuda")
    wsb = q8d.q8d_gqa_workspace_bytes(8, H, Hk, D, cap)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    lt = torch.tensor(lens, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    args_ = (q, None, None, kc, vc, q8d.Q8D_KV_F16, out, 8, H, Hk, D, cap, cap * kvw, lt,
             1 / math.sqrt(D), ws, wsb, err)
    return lens, args_, err


def attn_stress(q8d, H, Hk, D, reps, stream, flush, rank=0):
    """q8d_gqa_decode_attn on the stress workload (K/V of all 8 sequences
    ~0.27 GB, L2 flushed before each timed launch); GB/s of algorithmic
    bytes (the K/V rows read once, q and the output)."""
    import torch
    lens, args_, err = stress_inputs(q8d, H, Hk, D, rank)
    ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    with torch.cuda.stream(stream):
        for rep in range(max(reps, 3) + 1):
            flush(rep)
            ev[0].record(stream)
            q8d.q8d_gqa_decode_attn(*args_, stream)
            ev[1].record(stream)
            ev[1].synchronize()
            if rep:
                times.append(ev[0].elapsed_time(ev[1]) / 1e3)
    assert err.item() == 0
    t = statistics.median(times)
    # back to back: 8 calls in one CUDA graph alternating over two copies of
    # the inputs (2 x 0.54 GB, far beyond L2)
    _, args2, err2 = stress_inputs(q8d, H, Hk, D, rank)
    calls = [(lambda a_=a_: q8d.q8d_gqa_decode_attn(*a_, stream)) for a_ in (args_, args2) * 4]
    t_seq = graph_seconds_per_call(calls, stream, reps)
    assert err.item() == 0 and err2.item() == 0
    del args2
    nbytes = sum(attn_bytes(L, Hk, D, H, 2, append=False) for L in lens)
    return {"kernel": "gqa_mma_kernel + gqa_combine_kernel (q8d_gqa_decode_attn)",
            "GB_s": nbytes / t / 1e9, "us_per_launch": t * 1e6, "kv_bytes": nbytes,
            "batch": 8, "lengths": "seeded uniform in [1, 32768]", "sum_lengths": int(sum(lens)),
            "l2": L2Flush.DESC + " before each launch",
            "back_to_back": {"us_per_call": t_seq * 1e6, "GB_s": nbytes / t_seq / 1e9,
                             "timing": "8 calls in one CUDA graph over two copies of the inputs, "
                                       "replay timed with CUDA events"}}


def attn_stress_q8(q8d, H, Hk, D, reps, stream, flush, rank=0):
    """The same batch-8 ragged workload over a packed Q8_0 cache (34 bytes
    per 32 elements: 0.53x the f16 bytes), L2 flushed before each launch."""
    import torch

    import synth
    cap, kvw = STRESS_CAP, Hk * D
    lens = synth.stream(0, "ragged.lens").integers(1, cap + 1, 8).tolist()
    kc = synth.q8_matrix_torch(rank, "stress.kq8", 8 * cap, kvw, scale_lo=4e-3, scale_hi=3e-2)
    vc = synth.q8_matrix_torch(rank, "stress.vq8", 8 * cap, kvw, scale_lo=4e-3, scale_hi=3e-2)
    q = synth.normal_torch(rank, "stress.q", (8, H * D), torch.float32)
    out = torch.empty(8, H * D, device="cuda")
    wsb = q8d.q8d_gqa_workspace_bytes(8, H, Hk, D, cap)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    lt = torch.tensor(lens, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    with torch.cuda.stream(stream):
        for rep in range(max(reps, 3) + 1):
            flush(rep)
            ev[0].record(stream)
            q8d.q8d_gqa_decode_attn(q, None, None, kc, vc, q8d.Q8D_KV_Q8_0, out, 8, H, Hk, D, cap,
                                    cap * kvw, lt, 1 / math.sqrt(D), ws, wsb, err, stream)
            ev[1].record(stream)
            ev[1].synchronize()
            if rep:
                times.append(ev[0].elapsed_time(ev[1]) / 1e3)
    assert err.item() == 0
    t = statistics.median(times)
    # back to back: 8 calls in one CUDA graph alternating over two copies of
    # the caches (2 x 0.57 GB, far beyond L2)
    kc2 = synth.q8_matrix_torch(rank, "stress.kq8", 8 * cap, kvw, scale_lo=4e-3, scale_hi=3e-2)
    vc2 = synth.q8_matrix_torch(rank, "stress.vq8", 8 * cap, kvw, scale_lo=4e-3, scale_hi=3e-2)

    def call(k_, v_):
        return lambda: q8d.q8d_gqa_decode_attn(q, None, None, k_, v_, q8d.Q8D_KV_Q8_0, out, 8, H,
                                               Hk, D, cap, cap * kvw, lt, 1 / math.sqrt(D), ws,
                                               wsb, err, stream)
    t_seq = graph_seconds_per_call([call(kc, vc), call(kc2, vc2)] * 4, stream, reps)
    assert err.item() == 0
    del kc2, vc2
    row_bytes = kvw // 32 * 34
    nbytes = sum(2 * L * row_bytes + 4 * 2 * H * D for L in lens)
    return {"kernel": "gqa_q8kv_kernel + gqa_combine_kernel (q8d_gqa_decode_attn, packed Q8_0 KV)",
            "GB_s": nbytes / t / 1e9, "us_per_launch": t * 1e6, "kv_bytes": nbytes,
            "batch": 8, "lengths": "seeded uniform in [1, 32768]", "sum_lengths": int(sum(lens)),
            "l2": L2Flush.DESC + " before each launch",
            "back_to_back": {"us_per_call": t_seq * 1e6, "GB_s": nbytes / t_seq / 1e9,
                             "timing": "8 calls in one CUDA graph over two copies of the caches, "
                                       "replay timed with CUDA events"}}


def attn_window_leg(q8d, H, Hk, D, reps, stream, flush, rank=0):
    """q8d_gqa_decode_attn_window on a shared-prefix batch: 8 sequences read
    one f16 cache (stride 0), each a 8192-row shared prefix run plus its own
    1024-row run; L2 flushed before each launch.  GB/s over the rows the
    sequences attend (the prefix counted once per sequence) and over the
    distinct rows."""
    import torch

    import synth
    pre, own, B = 8192, 1024, 8
    cap, kvw = pre + B * own, Hk * D
    kc = synth.normal_torch(rank, "win.k", (cap, kvw), torch.float16)
    vc = synth.normal_torch(rank, "win.v", (cap, kvw), torch.float16)
    q = synth.normal_torch(rank, "win.q", (B, H * D), torch.float32)
    runs = torch.zeros((B, 4, 2), dtype=torch.int32)
    for s in range(B):
        runs[s, 0] = torch.tensor([0, pre])
        runs[s, 1] = torch.tensor([pre + s * own, own])
    runs = runs.cuda()
    out = torch.empty(B, H * D, device="cuda")
    wsb = q8d.q8d_gqa_workspace_bytes(B, H, Hk, D, cap)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    with torch.cuda.stream(stream):
        for rep in range(max(reps, 3) + 1):
            flush(rep)
            ev[0].record(stream)
            q8d.q8d_gqa_decode_attn_window(q, None, None, kc, vc, q8d.Q8D_KV_F16, out, B, H, Hk, D,
                                           cap, 0, runs, 1 / math.sqrt(D), ws, wsb, err, stream)
            ev[1].record(stream)
            ev[1].synchronize()
            if rep:
                times.append(ev[0].elapsed_time(ev[1]) / 1e3)
    assert err.item() == 0
    t = statistics.median(times)
    attended = B * attn_bytes(pre + own, Hk, D, H, 2, append=False)
    distinct = 2 * cap * kvw * 2 + B * 8 * H * D
    return {"kernel": "gqa_mma_kernel + gqa_combine_kernel (q8d_gqa_decode_attn_window)",
            "us_per_launch": t * 1e6, "attended_GB_s": attended / t / 1e9,
            "distinct_GB_s": distinct / t / 1e9, "attended_bytes": attended,
            "distinct_bytes": distinct,
            "workload": "8 sequences, one f16 cache: shared 8192-row prefix + own 1024-row run each",
            "l2": L2Flush.DESC + " before each launch"}


# ---------------------------------------------------------------------------- small M
SMALL_M = (1, 4, 16, 64, 128, 256)


def small_m_inputs(m, rank=0):
    """The 7B gate/up shape (3584 -> 18944, 72 MB of Q8_0) against m
    activation rows."""
    import torch

    import synth
    n, p = 3584, 18944
    w = synth.q8_matrix_torch(rank, "smallm.w", p, n)
    x = synth.normal_torch(rank, f"smallm.x{m}", (m, n), torch.float32)
    y = torch.empty(m, p, device="cuda")
    return w, x, y, n, p


def small_m_leg(q8d, reps, stream, flush, hbm, rank=0):
    """q8d_matmul_small_m on the 7B gate/up shape at m = 1, 4, 16, 64 (m >= 16
    on tcgen05), L2 flushed before each timed launch; GB/s of algorithmic
    bytes (weights once, X and Y)."""
    import torch

    import synth
    out = {}
    ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for m in SMALL_M:
        w, x, y, n, p = small_m_inputs(m, rank)
        need = q8d.q8d_matmul_small_m_workspace_bytes(m, n)
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
        times = []
        with torch.cuda.stream(stream):
            for rep in range(max(reps, 3) + 1):
                flush(rep)
                ev[0].record(stream)
                q8d.q8d_matmul_small_m_ws(x, n, w, y, p, m, n, p, ws, need, stream)
                ev[1].record(stream)
                ev[1].synchronize()
                if rep:
                    times.append(ev[0].elapsed_time(ev[1]) / 1e3)
        t = statistics.median(times)
        # back to back: 6 calls in one CUDA graph rotating over three copies
        # of the weights (216 MB, beyond L2)
        ws_ = [w] + [synth.q8_matrix_torch(rank, "smallm.w", p, n) for _ in range(2)]

        def call(w_):
            return lambda: q8d.q8d_matmul_small_m_ws(x, n, w_, y, p, m, n, p, ws, need, stream)
        t_seq = graph_seconds_per_call([call(w_) for w_ in ws_] * 2, stream, reps)
        del ws_
        nbytes = p * n // 32 * 34 + 4 * m * n + 4 * m * p
        out[f"m{m}"] = {"us": t * 1e6, "GB_s": nbytes / t / 1e9, "frac_of_peak": nbytes / t / 1e9 / hbm,
                        "back_to_back": {"us_per_call": t_seq * 1e6, "frac_of_peak": nbytes / t_seq / 1e9 / hbm,
                                         "TFLOP_s": 2.0 * m * n * p / t_seq / 1e12},
                        "TFLOP_s": 2.0 * m * n * p / t / 1e12,
                        "kernel": ("q8_ximage_kernel + q8_mma_kernel (tcgen05)" if m >= 16
                                   else "q8_gemv_kernel / q8_rows_kernel"),
                        "bf16_tensor_frac_of_measured": 2.0 * m * n * p / t / 1e12 / bf16_peak()}
        del w, x, y, ws
    out["shape"] = ("3584 -> 18944 (7B gate/up), " + L2Flush.DESC + " before each call; m >= 9 through "
                    "q8d_matmul_small_m_ws with a preallocated workspace; back_to_back: 6 calls "
                    "in one CUDA graph over three copies of the weights")
    return out


# ---------------------------------------------------------------------------- replicas
def replica_throughput(local_seconds: float, steps: int, dist=None, device="cuda") -> float:
    """Whole-job steps per second of independent replicas: every rank ran
    `steps` steps in `local_seconds`; the job takes the slowest rank's time
    (max over ranks), and the ranks' steps add up."""
    world = 1
    t = local_seconds
    if dist is not None and dist.is_initialized():
        import torch
        world = dist.get_world_size()
        tt = torch.tensor([t], dtype=torch.float64, device=device)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        t = float(tt.item())
    return world * steps / t


# ---------------------------------------------------------------------------- main
def run_reference(args, rank, world):
    """The reference arm: the oracle as it stands, whole decode steps of the
    workload (every layer, lm_head, argmax) on all host cores, W untimed and
    exactly K timed; rank 0 only."""
    if rank != 0:
        return
    from oracle import oracle as orc
    threads = orc.default_threads()
    times = oracle_full_steps(args.model, args.context, args.steps, args.warmup, threads)
    total = sum(times)
    tps = args.steps / total
    desc = (f"whole {args.model}-shaped decode steps (every layer + lm_head + argmax, KV context "
            f"{args.context}): {args.warmup} untimed, {args.steps} timed, {total:.1f} s; median "
            f"{statistics.median(times):.3f} s per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": tps, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": workload_name(args)},
        "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": desc, "cpu_model": cpu_model()},
        "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_name(args):
    return (f"{args.model}-shaped decode step, Q8_0 weights, "
            f"{'f16' if args.model != 'qwen2.5-0.5b' else 'f32'} KV cache, context {args.context}")


def device_caches(shape, ctx, cap, rank):
    """Per-layer KV caches of `cap` rows with ctx - 1 seeded rows."""
    import torch

    import synth
    kdt = torch.float16 if shape.kv_dtype == synth.KV_F16 else torch.float32
    caches = []
    for li in range(shape.n_layers):
        kc = torch.zeros((cap, shape.kv_width), dtype=kdt, device="cuda")
        vc = torch.zeros((cap, shape.kv_width), dtype=kdt, device="cuda")
        kc[:ctx - 1] = synth.normal_torch(rank, f"l{li}.kprefix", (ctx - 1, shape.kv_width), kdt)
        vc[:ctx - 1] = synth.normal_torch(rank, f"l{li}.vprefix", (ctx - 1, shape.kv_width), kdt)
        caches.append((kc, vc))
    return caches


def config_leg(shape, wts, ctx, steps, warmup, stream, hbm, rank):
    """Decode steps of another configuration (graph launches, everything
    resident), CUDA-event timed on the launching stream."""
    import torch

    import synth
    from q8_block_quantized_matvec_gb300.device import DeviceStep
    cap = ctx + warmup + steps + 64
    caches = device_caches(shape, ctx, cap, rank)
    ds = DeviceStep(wts, cap, caches, stream=stream)
    with torch.cuda.stream(stream):
        ds.set_state(17, ctx - 1)
        for _ in range(warmup):
            ds.launch(stream)
        ds.set_state(17, ctx - 1)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        ds.launch(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) / 1e3
    assert ds.step.status(stream) == 0, "device error word set"
    ds.close()
    del caches
    esize = 2 if shape.kv_dtype == synth.KV_F16 else 4
    b = statistics.mean(step_bytes(shape, ctx + s, esize) for s in range(steps))
    return {"tokens_s": steps / t, "ms_per_step": 1e3 * t / steps, "steps": steps,
            "context_first_step": ctx, "kv": "f16" if esize == 2 else "f32",
            "weight_bytes_per_step": shape.weight_bytes(),
            "roofline": {"bound": "hbm", "achieved_GB_s": b / (t / steps) / 1e9,
                         "frac": b / (t / steps) / 1e9 / hbm,
                         "algorithmic_bytes_per_launch": b}}


def attn_layer_leg(q8d, shape, caches, ctx, cap, reps, stream, flush, rank):
    """q8d_gqa_decode_attn over every layer's cache at attended length ctx,
    one launch per layer with an L2 flush (L2Flush) between layers; returns
    the median over reps of the per-step sum."""
    import torch

    import synth
    esize = 2 if shape.kv_dtype == synth.KV_F16 else 4
    H, Hk, D = shape.n_heads, shape.n_kv_heads, shape.head_dim
    qv = synth.normal_torch(rank, "bench.q", H * D, torch.float32)
    aout = torch.empty(H * D, device="cuda")
    wsb = q8d.q8d_gqa_workspace_bytes(1, H, Hk, D, cap)
    aws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    lens = torch.tensor([ctx], dtype=torch.int32, device="cuda")
    aerr = torch.zeros(1, dtype=torch.int32, device="cuda")
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    at_times = []
    with torch.cuda.stream(stream):
        for rep in range(reps + 1):
            tot = 0.0
            for li in range(shape.n_layers):
                flush(li)  # evict the previous layer's KV from L2 (same stream)
                a.record(stream)
                q8d.q8d_gqa_decode_attn(qv, None, None, caches[li][0], caches[li][1],
                                        shape.kv_dtype, aout, 1, H, Hk, D, cap, 0, lens,
                                        1 / math.sqrt(D), aws, wsb, aerr, stream)
                b.record(stream)
                b.synchronize()
                tot += a.elapsed_time(b) / 1e3
            if rep:
                at_times.append(tot)
    # the layers back to back: the 28 calls captured in one CUDA graph and
    # replayed after an L2 flush (every layer reads its own rows from
    # HBM), one timed region per replay
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="relaxed"):
        for li in range(shape.n_layers):
            q8d.q8d_gqa_decode_attn(qv, None, None, caches[li][0], caches[li][1],
                                    shape.kv_dtype, aout, 1, H, Hk, D, cap, 0, lens,
                                    1 / math.sqrt(D), aws, wsb, aerr, stream)
    seq_times = []
    with torch.cuda.stream(stream):
        for rep in range(reps + 1):
            flush(rep)
            a.record(stream)
            graph.replay()
            b.record(stream)
            b.synchronize()
            if rep:
                seq_times.append(a.elapsed_time(b) / 1e3)
    del graph
    assert aerr.item() == 0
    t = statistics.median(at_times)
    t_seq = statistics.median(seq_times)
    nbytes = attn_bytes(ctx, Hk, D, H, esize, append=False)
    return {"kernel": "gqa_mma_kernel + gqa_combine_kernel (q8d_gqa_decode_attn)"
            if esize == 2 else "gqa_split_kernel + gqa_combine_kernel (q8d_gqa_decode_attn)",
            "GB_s": nbytes * shape.n_layers / t / 1e9, "us_per_layer": t / shape.n_layers * 1e6,
            "bytes_per_layer": nbytes, "context": ctx, "l2": L2Flush.DESC + " between layers",
            "back_to_back": {"us_per_layer": t_seq / shape.n_layers * 1e6,
                             "GB_s": nbytes * shape.n_layers / t_seq / 1e9,
                             "timing": "the 28 layers' calls captured in one CUDA graph, "
                                       "replayed after an L2 flush"}}


# The other configurations of the workload set, measured as extra keys:
# (model, context) pairs; the line's own workload is skipped.
CONFIG_LEGS = [("qwen3-0.6b", 2048), ("qwen2.5-0.5b", 512), ("qwen2.5-0.5b", 2048),
               ("qwen2.5-0.5b", 4096), ("qwen2.5-7b", 2048), ("qwen2.5-7b", 8192)]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="q8d", choices=["q8d", "reference"])
    ap.add_argument("--model", default="qwen2.5-7b", choices=["qwen2.5-7b", "qwen3-0.6b", "qwen2.5-0.5b"])
    ap.add_argument("--context", type=int, default=2048)
    ap.add_argument("--layers", type=int, default=0,
                    help="--profile step only: use this many layers of the model's shape")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the other configurations")
    ap.add_argument("--kernel-reps", type=int, default=3)
    ap.add_argument("--profile",
                    choices=["step", "matvec", "matvec_down", "matvec_kv", "attn", "attn_stress", "mma16", "mma64",
                             "matvec_sweep", "attn_stress_q8", "attn_window"],
                    default=None,
                    help="run a short fixed workload between cudaProfilerStart/Stop for ncu "
                         "(--profile-from-start off) and print no JSON")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.profile:
        run_profile(args)
        return

    import torch
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    from __graft_entry__ import build
    build()
    import q8_block_quantized_matvec_gb300 as q8d
    import synth
    from q8_block_quantized_matvec_gb300.device import DeviceStep

    shape = synth.MODELS[args.model]
    ctx = args.context
    cap = ctx + args.warmup + 2 * args.steps + 64
    wts = synth.TorchStepWeights(shape, seed=rank)
    caches = device_caches(shape, ctx, cap, rank)
    stream = torch.cuda.Stream()
    ds = DeviceStep(wts, cap, caches, stream=stream)
    torch.cuda.synchronize()
    kernels_per_step = ds.kernel_count()

    def barrier():
        if dist:
            dist.barrier()
        torch.cuda.synchronize()

    # ---- device-timed steps (inputs resident) ----
    with torch.cuda.stream(stream):
        ds.set_state(17, ctx - 1)
        for _ in range(args.warmup):
            ds.launch(stream)
        ds.set_state(17, ctx - 1)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_index()) as clk:
        h0 = time.monotonic()
        e0.record(stream)
        for _ in range(args.steps):
            ds.launch(stream)
        e1.record(stream)
        barrier()
        h1 = time.monotonic()
    t_dev = e0.elapsed_time(e1) / 1e3
    assert ds.step.status(stream) == 0, "device error word set during the timed steps"
    value = replica_throughput(t_dev, args.steps, dist)
    t_dev = world * args.steps / value  # the slowest rank's time

    # ---- end to end through the public API: every step copies its token id
    # and position from pinned host memory, runs the graph and copies the
    # next token id back (q8d_step_launch_host: one call), and the host
    # waits for it and feeds it to the next step ----
    h_in = torch.tensor([17, ctx - 1], dtype=torch.int32).pin_memory()
    h_out = torch.empty(1, dtype=torch.int32).pin_memory()
    barrier()
    t0 = time.perf_counter()
    for s in range(args.steps):
        h_in[1] = ctx - 1 + s
        ds.launch_host(h_in, h_out, stream)   # H2D token + position, step, D2H next token
        stream.synchronize()
        h_in[0] = int(h_out[0])
    t_e2e = time.perf_counter() - t0
    e2e = {"value": replica_throughput(t_e2e, args.steps, dist), "unit": "tokens/s",
           "h2d_bytes_per_step": 8, "d2h_bytes_per_step": 4}
    ds.close()

    # ---- kernel legs: q8_matvec over the step's matrices, attention per layer ----
    mats = []
    for li, L in enumerate(ds.layers):
        for nm in ("wq", "wk", "wv", "wo", "wg", "wu", "wd"):
            n = shape.hidden if nm not in ("wo", "wd") else (shape.q_width if nm == "wo" else shape.ffn)
            p = {"wq": shape.q_width, "wk": shape.kv_width, "wv": shape.kv_width, "wo": shape.hidden,
                 "wg": shape.ffn, "wu": shape.ffn, "wd": shape.hidden}[nm]
            mats.append((L[nm], n, p))
    mats.append((ds.lm_head, shape.hidden, shape.vocab))
    xin = {n: synth.normal_torch(rank, f"bench.x{n}", n, torch.float32) for _, n, _ in mats}
    yout = torch.empty(max(p for _, _, p in mats), device="cuda")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in mats]
    mv_times, mv_big = [], []
    for rep in range(args.kernel_reps + 1):
        torch.cuda.synchronize()
        for (w, n, p), (a, b) in zip(mats, ev):
            a.record(stream)
            q8d.q8d_matvec(xin[n], w, yout, n, p, stream)
            b.record(stream)
        torch.cuda.synchronize()
        if rep:
            mv_times.append(sum(a.elapsed_time(b) for a, b in ev) / 1e3)
            mv_big.append(sum(a.elapsed_time(b) for (w, n, p), (a, b) in zip(mats, ev)
                              if p == shape.ffn or n == shape.ffn) / 1e3)
    mv_time = statistics.median(mv_times)
    # the same 197 calls back to back, captured once in a CUDA graph (as a
    # serving loop runs them) and replayed, one timed region per replay: no
    # host work or event between launches (7.5 GB per step, far beyond L2)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="relaxed"):
        for (w, n, p) in mats:
            q8d.q8d_matvec(xin[n], w, yout, n, p, stream)
    mv_seq = []
    for rep in range(args.kernel_reps + 1):
        torch.cuda.synchronize()
        a, b = ev[0]
        with torch.cuda.stream(stream):
            a.record(stream)
            graph.replay()
            b.record(stream)
        torch.cuda.synchronize()
        if rep:
            mv_seq.append(a.elapsed_time(b) / 1e3)
    mv_seq_time = statistics.median(mv_seq)
    del graph
    mv_bytes = sum(matvec_bytes(n, p) for _, n, p in mats)
    big_bytes = sum(matvec_bytes(n, p) for _, n, p in mats if p == shape.ffn or n == shape.ffn)
    hbm, peak_kind = peaks()
    mv_gbs = mv_bytes / mv_time / 1e9
    big_gbs = big_bytes / statistics.median(mv_big) / 1e9

    flush = L2Flush()
    attn = attn_layer_leg(q8d, shape, caches, ctx, cap, args.kernel_reps, stream, flush, rank)
    attn["frac_of_peak"] = attn["GB_s"] / hbm
    attn["back_to_back"]["frac_of_peak"] = attn["back_to_back"]["GB_s"] / hbm
    attn_long = None
    H, Hk, D = shape.n_heads, shape.n_kv_heads, shape.head_dim
    if shape.name == "qwen2.5-7b" and ctx != 8192:
        del caches
        caches = device_caches(shape, 8192, 8192, rank)
        attn_long = attn_layer_leg(q8d, shape, caches, 8192, 8192, args.kernel_reps, stream, flush,
                                   rank)
        attn_long["frac_of_peak"] = attn_long["GB_s"] / hbm
        attn_long["back_to_back"]["frac_of_peak"] = attn_long["back_to_back"]["GB_s"] / hbm
    del caches
    stress = attn_stress(q8d, H, Hk, D, args.kernel_reps, stream, flush, rank) \
        if shape.kv_dtype == synth.KV_F16 else None
    if stress is not None:
        stress["frac_of_peak"] = stress["GB_s"] / hbm
    window = attn_window_leg(q8d, H, Hk, D, args.kernel_reps, stream, flush, rank) \
        if shape.kv_dtype == synth.KV_F16 else None
    if window is not None:
        window["distinct_frac_of_peak"] = window["distinct_GB_s"] / hbm
    stress_q8 = attn_stress_q8(q8d, H, Hk, D, args.kernel_reps, stream, flush, rank) \
        if shape.kv_dtype == synth.KV_F16 else None
    if stress_q8 is not None:
        stress_q8["frac_of_peak"] = stress_q8["GB_s"] / hbm
    small_m = small_m_leg(q8d, args.kernel_reps, stream, flush, hbm, rank) \
        if shape.name == "qwen2.5-7b" else None

    # ---- the other configurations (decode steps, extra keys) ----
    configs = {}
    if not args.no_configs:
        csteps = max(args.steps, 20)
        for mname, cctx in CONFIG_LEGS:
            if (mname, cctx) == (args.model, ctx):
                continue
            cshape = synth.MODELS[mname]
            cw = wts if mname == args.model else synth.TorchStepWeights(cshape, seed=rank)
            configs[f"{mname}@{cctx}"] = config_leg(cshape, cw, cctx, csteps, args.warmup, stream,
                                                    hbm, rank)
            if cw is not wts:
                del cw
            torch.cuda.empty_cache()

    # dominant kernel: the persistent step kernel, one launch per step
    esize = 2 if shape.kv_dtype == synth.KV_F16 else 4
    step_b = statistics.mean(step_bytes(shape, ctx + s, esize) for s in range(args.steps))
    step_s = t_dev / args.steps
    traffic = ncu_traffic(step_b)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_leg(args.model, ctx)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_dev / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": workload_name(args), "model_shape": shape.name,
                       "context_first_step": ctx, "context_last_step": ctx + args.steps - 1,
                       "weight_bytes_per_step": shape.weight_bytes(),
                       "l2": "inputs larger than L2 (7.5 GB of weights streamed per step)"
                       if shape.name == "qwen2.5-7b" else "weights streamed per step exceed L2",
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "kernel": "q8_step_kernel (q8d_step_launch)",
                         "achieved": step_b / step_s / 1e9, "peak": hbm,
                         "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": step_b / step_s / 1e9 / hbm, "traffic": traffic,
                         "algorithmic_bytes_per_launch": step_b,
                         "avg_launch_us": step_s * 1e6, "launches": args.steps},
            "kernels": {
                "q8_matvec": {"kernel": "q8_gemv_kernel (q8d_matvec, one launch per matrix)",
                              "GB_s": mv_gbs, "frac_of_peak": mv_gbs / hbm,
                              "us_per_step_sum": mv_time * 1e6,
                              "avg_launch_us": mv_time / len(mats) * 1e6,
                              "algorithmic_bytes_per_launch": mv_bytes / len(mats),
                              "ffn_matrices_GB_s": big_gbs, "ffn_matrices_frac_of_peak": big_gbs / hbm,
                              "back_to_back": {
                                  "us_per_step": mv_seq_time * 1e6,
                                  "GB_s": mv_bytes / mv_seq_time / 1e9,
                                  "frac_of_peak": mv_bytes / mv_seq_time / 1e9 / hbm,
                                  "timing": "the step's 197 calls captured in one CUDA graph, "
                                            "replay timed with CUDA events"}},
                "gqa_decode_attn": attn,
                "gqa_decode_attn_ctx8192": attn_long,
                "gqa_decode_attn_batch8_ragged": stress,
                "gqa_decode_attn_batch8_ragged_q8_0_kv": stress_q8,
                "gqa_decode_attn_window_shared_prefix": window,
                "q8_matmul_small_m": small_m,
            },
            "configs": configs,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "gpu_launches": kernels_per_step * args.steps,
            "clocks": clk.summary(h0, h1),
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
