"""Benchmark of the block-quantised GEMV library on one GB300 (or N replicas).

Default workload: the GEMVs of a Llama-3.1-8B decode step at batch 1, Q4_K_M
mix (Q4_K q/k/v/o/gate/up, Q6_K down), W4A8, 32 layers: per layer q/k/v (one
job of three matrices), o, gate/up (one job of two), down, each GEMV after the
previous one completes.  The step runs as one chain launch (qx_gemv_chain);
the same step as 128 separate launches with programmatic dependent launch is
reported beside it.  `value` is the faster of the two forms (named in
config.launch); both are in the JSON line.  Weights (4.41 GB per step) are resident in HBM and far
larger than L2, so every step streams them from DRAM.

Prints one JSON line:
  value       weight-GB/s over the timed region (device-resident inputs)
  e2e         the same metric through the public API with pinned host
              activations copied in and all outputs copied back every step
  roofline    the dominant kernel of the faster form (the chain kernel, or the
              gate/up GEMV launch of the per-launch form): algorithmic bytes per
              launch / its CUDA-event duration vs measured HBM bandwidth
  cpu_baseline  the CPU oracle on a bounded sample of the same workload

`--impl reference` times the CPU oracle itself on the same metric.  Other
workloads (`--workload`): q4k_1024 (Q4_K 1024x1024), lmhead_q6k (Q6_K
128256x4096), qwen05b (Qwen2-0.5B decode step, 24 layers + Q8_0 lm_head),
prefill (Q4_K 14336x4096, X[512, 4096]).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "quantized GEMV weight-GB/s & % of HBM peak (Llama-8B decode shapes, batch 1)"


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1916.5)), "measured"
    return 6800.0, 1900.0, "fallback"


CHAIN_SOURCES = ["qx_chain.cu", "qx_lanes.cuh", "qx_device.cuh", "qx_api.cu", "qx_internal.h"]
CHAIN_PROFILE_NAME = "profiles/gemv_chain_llama8b.md"
GEMV_SOURCES = ["qx_gemv.cu", "qx_stage.cuh", "qx_lanes.cuh", "qx_device.cuh", "qx_api.cu", "qx_internal.h"]
GATEUP_PROFILE_NAME = "profiles/gemv_q4k_w4a8_gateup_llama8b.md"


def kernel_sources_hash(files) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "block_quantized_gemv_q8_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profile_fields(path):
    fields = {}
    if os.path.exists(path):
        for line in open(path):
            if ":" in line:
                k, v = line.split(":", 1)
                fields[k.strip()] = v.strip()
    return fields


def chain_traffic(layers: int):
    """DRAM bytes of one chain launch of `layers` layers from the committed ncu
    summary of a smaller chain (traffic grows with the layers streamed), or
    None once the kernel sources differ from the captured ones."""
    f = profile_fields(os.path.join(ROOT, CHAIN_PROFILE_NAME))
    if "traffic_bytes_per_layer" not in f or f.get("source_sha256_16") != kernel_sources_hash(CHAIN_SOURCES):
        return None
    return int(f["traffic_bytes_per_layer"]) * layers


def gateup_traffic():
    """DRAM bytes of one gate/up GEMV launch from its committed ncu summary, or
    None once the kernel sources differ from the captured ones."""
    f = profile_fields(os.path.join(ROOT, GATEUP_PROFILE_NAME))
    if "traffic_bytes_per_launch" not in f or f.get("source_sha256_16") != kernel_sources_hash(GEMV_SOURCES):
        return None
    return int(f["traffic_bytes_per_launch"])


# ---------------------------------------------------------------- clocks ----

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.device_index = device_index

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------- workloads ----

class LlamaDecode:
    """Llama-3.1-8B decode GEMVs at batch 1, W4A8, 32 layers (Q4_K_M mix)."""
    name = "llama-3.1-8b decode GEMVs (q,k,v,o,gate,up Q4_K; down Q6_K), W4A8, batch 1, 32 layers"
    unit = "GB/s"
    higher_is_better = True

    def __init__(self, layers: int = synth.LLAMA8B_LAYERS, down_layout: str = "soa"):
        self.layers = layers
        # the Q6_K down projection as stored (GGUF blocks) or repacked at load time
        # into QX_Q6_K_SOA (the same values and, for 14336 columns, the same bytes per row)
        self.down_layout = down_layout
        self.shapes = {n: (f, r, c) for n, f, r, c in synth.LLAMA8B_LAYER}
        self.bytes_per_step = layers * sum(r * synth.row_bytes(f, c) for f, r, c in self.shapes.values())
        self.launches_per_step = layers * 4
        self.dominant = "gemv_chain_kernel (the whole step: 128 dependent W4A8 GEMV jobs)"
        self.dominant_bytes = self.bytes_per_step
        # dominant launch of the per-launch form: the Q4_K gate/up pair (2 x 14336 x 4096)
        self.dominant_pdl = "gemv_kernel<Q4_K, W4A8> (gate/up: 2 x 14336 rows x 4096 cols, one launch)"
        self.dominant_pdl_bytes = 2 * 14336 * synth.row_bytes(synth.Q4_K, 4096)

    def setup(self, qx, torch, seed_base: int = 0):
        self.W, self.y = [], []
        self.host_layer0 = None
        for L in range(self.layers):
            Wl, yl = {}, {}
            for j, (n, (f, r, c)) in enumerate(self.shapes.items()):
                Wh = synth.weights(f, r, c, seed=synth.seed_for(1, L + seed_base, j))
                if L == 0:
                    self.host_layer0 = self.host_layer0 or {}
                    self.host_layer0[n] = Wh
                Wl[n] = torch.from_numpy(Wh).cuda()
                if n == "down" and self.down_layout == "soa":
                    Wl["down_soa"] = qx.qx_repack(qx.QX_Q6_K, qx.QX_Q6_K_SOA, Wl[n], r, c)
                yl[n] = torch.empty(r, dtype=torch.float32, device="cuda")
            self.W.append(Wl)
            self.y.append(yl)
        # activations: per layer x_qkv, x_o, x_ffn [4096] and x_down [14336], in one buffer
        self.xcols = [4096, 4096, 4096, 14336]
        per_layer = sum(self.xcols)
        xs = np.concatenate([synth.activation(1, per_layer, seed=synth.seed_for(1, L + seed_base, 100))[0]
                             for L in range(self.layers)])
        self.x_host = xs
        self.x_dev = torch.from_numpy(xs).cuda()
        self.x_views = []
        off = 0
        for L in range(self.layers):
            views = []
            for c in self.xcols:
                views.append(self.x_dev[off:off + c])
                off += c
            self.x_views.append(views)
        # one output buffer so that the e2e path copies it back in one piece
        outs = [(L, n) for L in range(self.layers) for n in self.shapes]
        total = sum(self.shapes[n][1] for _, n in outs)
        self.y_all = torch.empty(total, dtype=torch.float32, device="cuda")
        self.bufs = [(self.x_views, self.y, self.x_dev, self.y_all)]
        off = 0
        for L, n in outs:
            r = self.shapes[n][1]
            self.y[L][n] = self.y_all[off:off + r]
            off += r

    def add_buffer_set(self, torch):
        """A second set of device activations and outputs (same shapes), so that
        one step's copies can overlap another step's GEMVs."""
        x_dev = torch.empty_like(self.x_dev)
        y_all = torch.empty_like(self.y_all)
        x_views, off = [], 0
        for L in range(self.layers):
            views = []
            for c in self.xcols:
                views.append(x_dev[off:off + c])
                off += c
            x_views.append(views)
        y, off = [{} for _ in range(self.layers)], 0
        for L in range(self.layers):
            for n in self.shapes:
                r = self.shapes[n][1]
                y[L][n] = y_all[off:off + r]
                off += r
        self.bufs.append((x_views, y, x_dev, y_all))

    def make_chain(self, qx):
        F = qx.QX_Q4_K
        jobs = []
        for L in range(self.layers):
            W, y, xv = self.W[L], self.y[L], self.x_views[L]
            jobs.append(qx.GemvJob(F, [W["q"], W["k"], W["v"]], [4096, 1024, 1024], 4096, xv[0],
                                   [y["q"], y["k"], y["v"]]))
            jobs.append(qx.GemvJob(F, [W["o"]], [4096], 4096, xv[1], [y["o"]]))
            jobs.append(qx.GemvJob(F, [W["gate"], W["up"]], [14336, 14336], 4096, xv[2], [y["gate"], y["up"]]))
            jobs.append(qx.GemvJob(qx.QX_Q6_K, [W["down"]], [4096], 14336, xv[3], [y["down"]]))
        self.jobs = jobs
        self.chain = qx.make_chain(jobs)
        self.scratch = qx.chain_scratch(len(jobs))

    def step_chain(self, qx, stream, events=None):
        """One decode step as one chain launch."""
        if events is not None:
            events[0].record(stream)
        qx.qx_gemv_chain(self.jobs, self.scratch, stream=stream, marshalled=self.chain)
        if events is not None:
            events[1].record(stream)

    def step(self, qx, stream, dom_events=None, buf: int = 0):
        """One decode step as 128 launches: per layer q/k/v (one launch), o, gate/up (one launch), down.

        Each launch quantises its f32 activation in-kernel (W4A8) and is
        launched with programmatic dependent launch, so it streams its weights
        while the previous launch finishes."""
        F = qx.QX_Q4_K
        mode = qx.QX_MODE_W4A8_FUSED | qx.QX_FLAG_PDL
        x_views, ys = self.bufs[buf][0], self.bufs[buf][1]
        for L in range(self.layers):
            W, y, xv = self.W[L], ys[L], x_views[L]
            qx.qx_gemv_multi([F, F, F], [W["q"], W["k"], W["v"]], [4096, 1024, 1024], 4096, xv[0],
                             ys=[y["q"], y["k"], y["v"]], mode=mode, stream=stream)
            qx.qx_gemv(F, W["o"], 4096, 4096, xv[1], y=y["o"], mode=mode, stream=stream)
            if dom_events is not None:
                dom_events[L][0].record(stream)
            qx.qx_gemv_multi([F, F], [W["gate"], W["up"]], [14336, 14336], 4096, xv[2],
                             ys=[y["gate"], y["up"]], mode=mode, stream=stream)
            if dom_events is not None:
                dom_events[L][1].record(stream)
            if self.down_layout == "soa":
                qx.qx_gemv(qx.QX_Q6_K_SOA, W["down_soa"], 4096, 14336, xv[3], y=y["down"], mode=mode, stream=stream)
            else:
                qx.qx_gemv(qx.QX_Q6_K, W["down"], 4096, 14336, xv[3], y=y["down"], mode=mode, stream=stream)

    def cpu_sample(self, oracle, budget_s: float = 10.0, threads: int | None = None):
        """Oracle on layer 0 (quantise + 7 W4A8 GEMVs), repeated for ~budget_s
        (at least once), on `threads` host threads (default: every core)."""
        threads = threads or oracle.default_threads()
        x = self.x_host
        acts = {}
        nbytes, reps = 0, 0
        t0 = time.perf_counter()
        while True:
            off = 0
            for k, c in enumerate(self.xcols):
                q, d, _ = oracle.quantize_act_q8(x[off:off + c][None])
                acts[k] = (q[0], d[0])
                off += c
            which = {"q": 0, "k": 0, "v": 0, "o": 1, "gate": 2, "up": 2, "down": 3}
            for n, (f, r, c) in self.shapes.items():
                q, d = acts[which[n]]
                oracle.gemv_w4a8(f, self.host_layer0[n], r, c, q, d, threads=threads, with_absdot=False)
                nbytes += r * synth.row_bytes(f, c)
            reps += 1
            el = time.perf_counter() - t0
            if el >= budget_s:
                break
        return {"value": nbytes / el / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
                "sample": f"layer 0 of the same workload (7 W4A8 GEMVs + 4 activation quantisations, "
                          f"{nbytes // reps} weight bytes) x {reps} repetitions, {el:.1f} s, "
                          + ("OpenMP over rows" if threads > 1 else "one thread")}


# ------------------------------------------------------------------ main ----

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(torch, value: float) -> float:
    """The largest `value` over all ranks of the initialised process group (the
    job's time is its slowest rank's); the value itself without one.  The
    tensor lives where the backend needs it: CUDA for NCCL, host for gloo."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    device = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world_size: int, bytes_per_step: int, steps: int, max_ms: float) -> float:
    """Whole-job weight GB/s: every rank streams bytes_per_step per step (weak
    scaling), over the slowest rank's time."""
    return world_size * bytes_per_step * steps / (max_ms * 1e-3) / 1e9


def reference_step_budget(steps: int) -> float:
    """Seconds of oracle work per timed step of the reference arm: about 2 s,
    less when there are many steps, so that the whole --steps K --warmup W run
    stays near a minute and a half (each step still runs at least one
    repetition of layer 0, about 40 ms on 16 host cores)."""
    return min(float(os.environ.get("QX_REF_STEP_S", "2.0")),
               float(os.environ.get("QX_REF_TOTAL_S", "90")) / max(1, steps))


def run_reference(args):
    """Time the CPU oracle itself on bounded samples of the workload (rank 0 only)."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    wl = LlamaDecode(layers=1)
    # host-only set-up: layer 0 weights and activations
    wl.shapes = {n: (f, r, c) for n, f, r, c in synth.LLAMA8B_LAYER}
    wl.host_layer0 = {n: synth.weights(f, r, c, seed=synth.seed_for(1, 0, j))
                      for j, (n, (f, r, c)) in enumerate(wl.shapes.items())}
    wl.xcols = [4096, 4096, 4096, 14336]
    wl.x_host = synth.activation(1, sum(wl.xcols), seed=synth.seed_for(1, 0, 100))[0]
    per_step_budget = reference_step_budget(args.steps)
    for _ in range(args.warmup):
        wl.cpu_sample(oracle, budget_s=0.0)
    vals, t0 = [], time.perf_counter()
    cb = None
    for _ in range(args.steps):
        cb = wl.cpu_sample(oracle, budget_s=per_step_budget)
        vals.append(cb["value"])
    el = time.perf_counter() - t0
    value = statistics.mean(vals)
    cb["value"] = value
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / max(1, args.steps) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int64+f64",
            "data": "synthetic",
            "config": {"workload": wl.name, "sample": "layer 0 per step (bounded, CPU oracle)"},
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------- secondary workloads ----

def graph_time_ms(torch, fn, reps: int, stream):
    """Mean device time of fn() captured once in a CUDA graph, replayed `reps` times."""
    with torch.cuda.stream(stream):
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def gemv_roofline(nbytes: int, us: float, hbm: float, peak_kind: str, kernel: str) -> dict:
    achieved = nbytes / (us * 1e-6) / 1e9
    return {"bound": "hbm", "kernel": kernel, "achieved": achieved, "peak": hbm, "unit": "GB/s",
            "frac": achieved / hbm, "peak_kind": peak_kind, "bytes_per_launch": nbytes, "mean_launch_us": us}


def measure_config(name: str, qx, torch, stream, hbm: float, bf16: float, peak_kind: str,
                   prefill_m: int = 0, prefill_path: int = 3) -> dict:
    """One of the other workloads (Q4_K 1024 x 1024, the Q6_K lm_head, the
    Qwen2-0.5B step, the prefill sweep), timed with CUDA events on `stream`
    around CUDA-graph replays; one dict with its own roofline figures."""
    out = {"workload": name}
    FUSED, F32, PDL = qx.QX_MODE_W4A8_FUSED, qx.QX_MODE_F32, qx.QX_FLAG_PDL
    if name == "q4k_1024":
        fmt, rows, cols = synth.Q4_K, 1024, 1024
        nbytes = rows * synth.row_bytes(fmt, cols)
        copies = 512  # 302 MB rotating pool, larger than L2
        pool = torch.from_numpy(np.concatenate([synth.weights(fmt, rows, cols, seed=i) for i in range(8)])).cuda()
        pool = pool.repeat(copies // 8, 1).reshape(copies, rows, -1)
        x = torch.from_numpy(synth.activation(1, cols, seed=9)[0]).cuda()
        y = torch.empty(rows, dtype=torch.float32, device="cuda")
        out["config"] = ("Q4_K GEMV 1024 x 1024, batch 1; a rotating pool of 512 weight copies (302 MB, larger "
                         "than L2) streamed by back-to-back PDL launches in a CUDA graph; single serial launches "
                         "on one L2-resident copy reported beside")
        for mname, mode in (("w4a8", FUSED | PDL), ("f32", F32 | PDL)):
            def rot():
                for c in range(copies):
                    qx.qx_gemv(fmt, pool[c], rows, cols, x, y=y, mode=mode, stream=stream)
            us = graph_time_ms(torch, rot, 5, stream) / copies * 1e3
            def hot():
                for _ in range(64):
                    qx.qx_gemv(fmt, pool[0], rows, cols, x, y=y, mode=mode & 0xFF, stream=stream)
            us_hot = graph_time_ms(torch, hot, 5, stream) / 64 * 1e3
            out[mname] = {"GB_per_s_rotating_pool": nbytes / (us * 1e-6) / 1e9, "us_per_gemv_rotating": us,
                          "us_per_gemv_l2_hot_serial": us_hot,
                          "roofline": gemv_roofline(nbytes, us, hbm, peak_kind,
                                                    f"gemv_kernel<Q4_K, {mname}> (rotating pool)")}
        del pool
    elif name == "lmhead_q6k":
        fmt, rows, cols = synth.LLAMA8B_LM_HEAD_Q6K[1:]
        nbytes = rows * synth.row_bytes(fmt, cols)
        W = torch.from_numpy(synth.weights(fmt, rows, cols, seed=20)).cuda()
        x = torch.from_numpy(synth.activation(1, cols, seed=21)[0]).cuda()
        y = torch.empty(rows, dtype=torch.float32, device="cuda")
        # the GGUF layout, and the same weights repacked at load time into QX_Q6_K_SOA (same bytes per row)
        Ws = qx.qx_repack(qx.QX_Q6_K, qx.QX_Q6_K_SOA, W, rows, cols)
        out["config"] = "Q6_K lm_head 128256 x 4096 (430.9 MB, larger than L2), batch 1, f32 and W4A8 modes"
        for mname, f, Wm, mode in (("w4a8", fmt, W, FUSED | PDL), ("f32", fmt, W, F32 | PDL),
                                   ("w4a8_soa", qx.QX_Q6_K_SOA, Ws, FUSED | PDL),
                                   ("f32_soa", qx.QX_Q6_K_SOA, Ws, F32 | PDL)):
            us = graph_time_ms(torch, lambda: qx.qx_gemv(f, Wm, rows, cols, x, y=y, mode=mode, stream=stream),
                               50, stream) * 1e3
            out[mname] = {"GB_per_s": nbytes / (us * 1e-6) / 1e9, "us": us, "frac_of_hbm": nbytes / (us * 1e-6) / 1e9 / hbm,
                          "roofline": gemv_roofline(nbytes, us, hbm, peak_kind,
                                                    ("gemv_f32_mma_kernel" if mname.startswith("f32") else "gemv_kernel")
                                                    + f" lm_head {mname}")}
        out["weight_bytes"] = nbytes
        del W, Ws
    elif name == "qwen05b":
        shapes = {n: (f, r, c) for n, f, r, c in synth.QWEN05B_LAYER}
        L = synth.QWEN05B_LAYERS
        Ws = [{n: torch.from_numpy(synth.weights(f, r, c, seed=synth.seed_for(3, l, j))).cuda()
               for j, (n, (f, r, c)) in enumerate(shapes.items())} for l in range(L)]
        lf, lr, lc = synth.QWEN05B_LM_HEAD[1:]
        Wlm = torch.from_numpy(synth.weights(lf, lr, lc, seed=31)).cuda()
        xs = [torch.from_numpy(synth.activation(1, 1024, seed=40 + k, valid_cols=896 if k == 2 else None)[0]).cuda()
              for k in range(3)]
        xd = torch.from_numpy(synth.activation(1, 4864, seed=44)[0]).cuda()
        ys = {n: torch.empty(r, dtype=torch.float32, device="cuda") for n, (f, r, c) in shapes.items()}
        ylm = torch.empty(lr, dtype=torch.float32, device="cuda")
        nbytes = L * sum(r * synth.row_bytes(f, c) for f, r, c in shapes.values()) + lr * synth.row_bytes(lf, lc)
        mode = FUSED | PDL
        Q8, Q4 = synth.Q8_0, synth.Q4_K

        def step():
            for l in range(L):
                W = Ws[l]
                qx.qx_gemv_multi([Q8] * 3, [W["q"], W["k"], W["v"]], [896, 128, 128], 896, xs[0][:896],
                                 ys=[ys["q"], ys["k"], ys["v"]], mode=mode, stream=stream)
                qx.qx_gemv(Q8, W["o"], 896, 896, xs[1][:896], y=ys["o"], mode=mode, stream=stream)
                qx.qx_gemv_multi([Q4, Q4], [W["gate"], W["up"]], [4864, 4864], 1024, xs[2],
                                 ys=[ys["gate"], ys["up"]], mode=mode, stream=stream)
                qx.qx_gemv(Q4, W["down"], 896, 4864, xd, y=ys["down"], mode=mode, stream=stream)
            qx.qx_gemv(Q8, Wlm, lr, lc, xs[0][:896], y=ylm, mode=mode, stream=stream)
        us = graph_time_ms(torch, step, 50, stream) * 1e3
        jobs = []
        for l in range(L):
            W = Ws[l]
            jobs += [qx.GemvJob(Q8, [W["q"], W["k"], W["v"]], [896, 128, 128], 896, xs[0][:896],
                                [ys["q"], ys["k"], ys["v"]]),
                     qx.GemvJob(Q8, [W["o"]], [896], 896, xs[1][:896], [ys["o"]]),
                     qx.GemvJob(Q4, [W["gate"], W["up"]], [4864, 4864], 1024, xs[2], [ys["gate"], ys["up"]]),
                     qx.GemvJob(Q4, [W["down"]], [896], 4864, xd, [ys["down"]])]
        jobs.append(qx.GemvJob(Q8, [Wlm], [lr], lc, xs[0][:896], [ylm]))
        arr, scratch = qx.make_chain(jobs), qx.chain_scratch(len(jobs))
        us_chain = graph_time_ms(torch, lambda: qx.qx_gemv_chain(jobs, scratch, stream=stream, marshalled=arr),
                                 50, stream) * 1e3
        best = min(us, us_chain)
        out.update({"config": "Qwen2-0.5B decode step, 24 layers + Q8_0 lm_head 896 -> 151936, W4A8, batch 1 "
                              "(Q4_K gate/up stored with 896 columns padded to 1024)",
                    "weight_bytes_per_token": nbytes, "us_per_token_pdl_launches": us,
                    "us_per_token_chain": us_chain, "us_per_token": best,
                    "GB_per_s_pdl": nbytes / (us * 1e-6) / 1e9, "GB_per_s_chain": nbytes / (us_chain * 1e-6) / 1e9,
                    "launches_per_token_pdl": 4 * L + 1, "hbm_bound_us": nbytes / (hbm * 1e9) * 1e6,
                    "roofline": gemv_roofline(nbytes, best, hbm, peak_kind,
                                              "the whole step (" + ("PDL launches" if us <= us_chain else "chain") + ")")})
        del Ws, Wlm
    elif name == "prefill":
        fmt, rows, cols = synth.PREFILL[1:]
        W = torch.from_numpy(synth.weights(fmt, rows, cols, seed=70)).cuda()
        X = torch.from_numpy(synth.activation(synth.PREFILL_M, cols, seed=71)).cuda()
        act = qx.qx_quantize_act_q8(X)
        torch.cuda.synchronize()
        nbytes = rows * synth.row_bytes(fmt, cols)
        sweep = []
        for m in ([prefill_m] if prefill_m else synth.PREFILL_SWEEP_M):
            a = qx.ActQ8(act.q[:m], act.d[:m], act.sum[:m])
            Y = torch.empty((m, rows), dtype=torch.float32, device="cuda")
            rec = {"m": m}
            for path in ((prefill_path,) if prefill_m else (1, 2, 3, 4)):
                if path in (1, 4) and m > 64:
                    continue
                ms = graph_time_ms(torch, lambda: qx.qx_gemm_prefill_ex(fmt, W, rows, cols, a, Y=Y, path=path,
                                                                        stream=stream), 10, stream)
                rec[f"path{path}_us"] = ms * 1e3
                rec[f"path{path}_tflops"] = 2.0 * m * rows * cols / (ms * 1e-3) / 1e12
                rec[f"path{path}_weight_GB_per_s"] = nbytes / (ms * 1e-3) / 1e9
                if path == 3:  # three bf16 passes over K on tcgen05
                    rec["path3_bf16_tflops"] = 3 * 2.0 * m * rows * cols / (ms * 1e-3) / 1e12
                    rec["path3_frac_of_bf16_peak"] = rec["path3_bf16_tflops"] / bf16
            paths = {k[:-3]: v for k, v in rec.items() if k.endswith("_us")}
            rec["fastest"] = min(paths, key=paths.get)
            sweep.append(rec)
        # measured on this device, for context: the int8 tensor rate a prefill can use on sm_103a
        # (legacy mma.sync; no int8 tcgen05) and the f16 mma.sync rate path 2 runs on
        out["mma_sync_int8_tops_measured"] = qx.qx_debug_mma_rate(0, stream=stream) / 1e12
        out["mma_sync_f16_tflops_measured"] = qx.qx_debug_mma_rate(1, stream=stream) / 1e12
        for rec in sweep:
            for path in (2, 3, 4):
                if f"path{path}_tflops" in rec:  # int8-equivalent multiply-adds x 2 per second
                    rec[f"path{path}_frac_of_int8_mma_sync"] = (rec[f"path{path}_tflops"]
                                                                / out["mma_sync_int8_tops_measured"])
        tensor_from = [r["m"] for r in sweep if r["fastest"] in ("path2", "path3")]
        out["crossover_m"] = min(tensor_from) if tensor_from else None
        top = max(sweep, key=lambda r: r["m"])
        if "path3_us" in top:
            fl = 3 * 2.0 * top["m"] * rows * cols
            out["roofline"] = {"bound": "tensor", "kernel": f"tcgen05 prefill (path 3) at M = {top['m']}",
                               "achieved": fl / (top["path3_us"] * 1e-6) / 1e12, "peak": bf16, "unit": "TFLOP/s",
                               "frac": fl / (top["path3_us"] * 1e-6) / 1e12 / bf16, "peak_kind": peak_kind,
                               "flops_per_launch": fl, "mean_launch_us": top["path3_us"],
                               "note": "bf16 FLOP of the three split products (Xh Wh + Xh Wl + Xl Wh)"}
        out.update({"config": "prefill X[M, 4096] x Q4_K [14336, 4096], M in " + str(list(synth.PREFILL_SWEEP_M)),
                    "sweep": sweep, "flops_per_row": 2 * rows * cols, "bf16_dense_peak_tflops": bf16,
                    "note": "path 1 = one W4A8 GEMV launch per row; path 2 = tensor cores (mma.sync f16 with "
                            "integer-valued operands); path 3 = tcgen05 bf16 GEMM over the split dequantised "
                            "operands (3 passes of K); path 4 = small-batch GEMV, one weight stream per 8 rows of "
                            "X while five or more remain (int8 mma.sync for rows of up to 4096 columns, else "
                            "dp4a lanes), else per up to 4 (dp4a lanes); tflops count the int8-equivalent "
                            "multiply-adds x2; crossover_m = the smallest swept M whose fastest path is a "
                            "tensor-core one"})
        del W, X
    torch.cuda.synchronize()
    return out


def run_extra(args):
    """One of the other configurations, as its own JSON line."""
    import torch
    import block_quantized_gemv_q8_gb300 as qx
    qx.build_library()
    torch.cuda.set_device(0)
    stream = torch.cuda.Stream()
    hbm, bf16, peak_kind = measured_peaks()
    with ClockSampler(0) as clk:
        out = measure_config(args.workload, qx, torch, stream, hbm, bf16, peak_kind, args.prefill_m, args.prefill_path)
    out.update({"peak_hbm_gbs": hbm, "peak_kind": peak_kind, "clocks": clk.summary()})
    print(json.dumps(out), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="qx", choices=["qx", "reference"])
    ap.add_argument("--prefill-m", type=int, default=0,
                    help="prefill workload: time only one path (--prefill-path) at this many rows of X")
    ap.add_argument("--prefill-path", type=int, default=3, choices=[1, 2, 3, 4],
                    help="prefill workload with --prefill-m: the path timed")
    ap.add_argument("--workload", default="llama8b", choices=["llama8b", "q4k_1024", "lmhead_q6k", "qwen05b",
                                                               "prefill"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="default workload: skip the sub-records of the other configurations")
    ap.add_argument("--layers", type=int, default=synth.LLAMA8B_LAYERS)
    ap.add_argument("--down-layout", default="soa", choices=["soa", "gguf"],
                    help="Llama step: the Q6_K down projection repacked at load time (QX_Q6_K_SOA) or as stored")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import block_quantized_gemv_q8_gb300 as qx

    if args.workload != "llama8b":
        return run_extra(args)

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    qx.build_library()
    qx.lib()

    wl = LlamaDecode(layers=args.layers, down_layout=args.down_layout)
    wl.setup(qx, torch, seed_base=0)
    wl.make_chain(qx)
    stream = torch.cuda.Stream()
    # Timing events recorded inside a captured graph need external record nodes.
    ev = (torch.cuda.Event(enable_timing=True, external=True), torch.cuda.Event(enable_timing=True, external=True))

    # eager warm-up (first-call device set-up) of both step forms, then graphs
    with torch.cuda.stream(stream):
        wl.step_chain(qx, stream)
        wl.step(qx, stream)
    torch.cuda.synchronize()
    assert qx.qx_device_check(stream) == qx.QX_OK
    g = torch.cuda.CUDAGraph()                 # the step: one chain launch
    with torch.cuda.graph(g, stream=stream):
        wl.step_chain(qx, stream)
    g_ev = torch.cuda.CUDAGraph()              # the same with events around the launch
    with torch.cuda.graph(g_ev, stream=stream):
        wl.step_chain(qx, stream, events=ev)
    g_pdl = torch.cuda.CUDAGraph()             # the step as 128 PDL launches
    with torch.cuda.graph(g_pdl, stream=stream):
        wl.step(qx, stream)
    # the same with events around every gate/up launch (the dominant launch)
    dom_ev = [(torch.cuda.Event(enable_timing=True, external=True),
               torch.cuda.Event(enable_timing=True, external=True)) for _ in range(wl.layers)]
    g_pdl_ev = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_pdl_ev, stream=stream):
        wl.step(qx, stream, dom_events=dom_ev)
    # e2e graph: pinned host activations in, step, all outputs back
    x_pin = torch.from_numpy(wl.x_host).pin_memory()
    y_pin = torch.empty(wl.y_all.numel(), dtype=torch.float32).pin_memory()
    ge = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ge, stream=stream):
        wl.x_dev.copy_(x_pin, non_blocking=True)
        wl.step_chain(qx, stream)
        y_pin.copy_(wl.y_all, non_blocking=True)
    # per-launch form: S steps per graph over two buffer sets, each step's
    # input copied in on an upload stream while the previous step computes and
    # its outputs copied back on a download stream while the next one does
    # (every step still moves its own inputs and outputs through pinned host
    # memory); S divides the timed steps
    e2e_steps = max(d for d in range(1, 11) if args.steps % d == 0)
    wl.add_buffer_set(torch)
    y_pins = [y_pin, torch.empty_like(y_pin).pin_memory()]
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ge_pdl = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ge_pdl, stream=stream):
        fork = torch.cuda.Event()
        fork.record(stream)
        up.wait_event(fork)
        down.wait_event(fork)
        h, c, d = {}, {}, {}

        def upload(k):
            with torch.cuda.stream(up):
                if k >= 2:
                    up.wait_event(c[k - 2])  # step k - 2 has read this buffer set's inputs
                wl.bufs[k % 2][2].copy_(x_pin, non_blocking=True)
                h[k] = torch.cuda.Event()
                h[k].record(up)

        upload(0)
        if e2e_steps > 1:
            upload(1)
        for k in range(e2e_steps):
            stream.wait_event(h[k])
            if k >= 2:
                stream.wait_event(d[k - 2])  # step k - 2's outputs are back on the host
            wl.step(qx, stream, buf=k % 2)
            c[k] = torch.cuda.Event()
            c[k].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(c[k])
                y_pins[k % 2].copy_(wl.bufs[k % 2][3], non_blocking=True)
                d[k] = torch.cuda.Event()
                d[k].record(down)
            if k + 2 < e2e_steps:
                upload(k + 2)
        for k in range(max(0, e2e_steps - 2), e2e_steps):
            stream.wait_event(d[k])

    def timed(graph, steps):
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(torch, e0.elapsed_time(e1))

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g.replay()
        with ClockSampler(local) as clk:
            ms = timed(g, args.steps)
            # the chain kernel's own duration: events around its launch, each
            # of K instrumented steps read back one by one
            dom_ms = []
            for _ in range(args.steps):
                g_ev.replay()
                ev[1].synchronize()
                dom_ms.append(ev[0].elapsed_time(ev[1]))
            for _ in range(args.warmup):
                g_pdl.replay()
            ms_pdl = timed(g_pdl, args.steps)
            # the gate/up launches' own durations, K instrumented steps read back one by one
            dom_pdl_ms = []
            for _ in range(args.steps):
                g_pdl_ev.replay()
                dom_ev[-1][1].synchronize()
                dom_pdl_ms.extend(a.elapsed_time(b) for a, b in dom_ev)
        for _ in range(args.warmup):
            ge.replay()
        ms_e2e_chain = timed(ge, args.steps)
        for _ in range(args.warmup):
            ge_pdl.replay()
        ms_e2e_pdl = timed(ge_pdl, args.steps // e2e_steps)
    st = qx.qx_device_check(stream)
    if st != qx.QX_OK:
        raise RuntimeError(f"device error after the timed region: {qx.qx_status_string(st)}")
    assert int(wl.scratch.sum()) == 0

    hbm, bf16, peak_kind = measured_peaks()
    per_s = lambda m: job_throughput(ws, wl.bytes_per_step, args.steps, m)  # noqa: E731
    value_chain, value_pdl = per_s(ms), per_s(ms_pdl)
    chain_is_faster = ms <= ms_pdl
    ms_e2e = ms_e2e_chain if chain_is_faster else ms_e2e_pdl
    value_e2e = per_s(ms_e2e)
    ms_best = ms if chain_is_faster else ms_pdl
    value, ms_step = per_s(ms_best), ms_best / args.steps
    def roofline(kernel, nbytes, launch_ms, traffic, source, note):
        achieved = nbytes / (launch_ms * 1e-3) / 1e9
        return {"bound": "hbm", "kernel": kernel, "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "peak_kind": peak_kind, "bytes_per_launch": nbytes,
                "mean_launch_ms": launch_ms, "traffic": traffic, "traffic_source": source if traffic else None,
                "note": note}
    t_chain = chain_traffic(wl.layers)
    roof_chain = roofline(wl.dominant, wl.dominant_bytes, statistics.mean(dom_ms), t_chain, CHAIN_PROFILE_NAME,
                          "the chain kernel carries the whole step; timed with CUDA events around its launch")
    t_gu = gateup_traffic()
    roof_pdl = roofline(wl.dominant_pdl, wl.dominant_pdl_bytes, statistics.mean(dom_pdl_ms), t_gu,
                        GATEUP_PROFILE_NAME,
                        "the largest launch of the Q4_K kernel, which takes 66% of the per-launch form's "
                        "device time (ncu launch list; gate/up is 48% of the step's weight bytes); timed with "
                        "CUDA events around each of its 32 launches in an instrumented copy of the step graph; "
                        "algorithmic bytes = the two Q4_K matrices (scales included)")
    configs = None
    if rank == 0 and not args.no_configs:
        # the other configurations, each with its own roofline and clock record
        configs = {}
        for name in ("q4k_1024", "lmhead_q6k", "qwen05b", "prefill"):
            with ClockSampler(local) as cclk:
                rec = measure_config(name, qx, torch, stream, hbm, bf16, peak_kind)
            rec["clocks"] = cclk.summary()
            configs[name] = rec
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        cpu = wl.cpu_sample(oracle, budget_s=10.0)
        one = wl.cpu_sample(oracle, budget_s=5.0, threads=1)
        cpu["single_thread"] = {"value": one["value"], "unit": one["unit"], "cores": 1, "sample": one["sample"]}
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "s8xu4/u6->s32 (dp4a) + f32 scales", "data": "synthetic",
            "config": {"workload": wl.name, "weight_bytes_per_step": wl.bytes_per_step,
                       "layers": wl.layers, "batch": 1, "jobs_per_step": len(wl.jobs),
                       "launch": ("one qx_gemv_chain launch per step" if chain_is_faster else
                                  "128 qx_gemv / qx_gemv_multi launches per step with programmatic dependent "
                                  "launch") + ", captured in a CUDA graph",
                       "activation_quantisation": "in-kernel (same codes as qx_quantize_act_q8)",
                       "down_projection_layout": ("Q6_K repacked at load time into QX_Q6_K_SOA (qx_repack; same "
                                                  "values, same 11760 bytes per row; the chain form reads the "
                                                  "GGUF blocks)") if wl.down_layout == "soa" else "GGUF Q6_K blocks",
                       "l2": "inputs larger than L2 (4.41 GB of weights streamed per step)",
                       "parallelism": "replicas" if ws > 1 else "single"},
            "pct_of_hbm_peak": value / ws / hbm,
            "us_per_token": ms_step * 1e3,
            "roofline": roof_chain if chain_is_faster else roof_pdl,
            "roofline_other_form": roof_pdl if chain_is_faster else roof_chain,
            "e2e": {"value": value_e2e, "unit": "GB/s", "h2d_bytes_per_step": int(wl.x_host.nbytes),
                    "d2h_bytes_per_step": int(wl.y_all.numel() * 4), "ms_per_step": ms_e2e / args.steps,
                    "copies": ("one pinned host->device copy of the step's activations and one device->host copy "
                               "of all its outputs per step" +
                               ("" if chain_is_faster else
                                f"; {e2e_steps} steps per graph over two device buffer sets, each step's upload "
                                "and download overlapping a neighbouring step's GEMVs"))},
            "per_launch_pdl": {"value": value_pdl, "unit": "GB/s", "ms_per_step": ms_pdl / args.steps,
                               "launches_per_step": wl.launches_per_step},
            "chain": {"value": value_chain, "unit": "GB/s", "ms_per_step": ms / args.steps, "launches_per_step": 1},
            "gpu_launches": args.steps * (1 if chain_is_faster else wl.launches_per_step),
            "clocks": clk.summary(),
            "cpu_baseline": cpu,
            "configs": configs,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
