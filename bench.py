"""Throughput of the routed-expert MoE layer on GB300, in tokens/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config C | --workload NAME]
                    [--impl ours|reference] [--no-sweep]

A step is one forward of the whole layer (router GEMV, top-k, permutation,
expert FFNs, combine) over one batch of T tokens, through the C ABI.  The
default workload is the T = 1 decode layer (hidden 2048, 256 experts, top-8 +
shared, intermediate 512, int4 g64 experts, 8-bit router); --config picks
another of the named workloads in quantised_moe_expert_gb300.synth.WORKLOADS,
--workload any workload by name (the 8-bit and NVFP4 expert layers of WORKLOADS_B8 and
WORKLOADS_NVFP4 too).

Timing: W warm-up steps, then exactly K steps replayed from one CUDA graph,
bracketed by a barrier and a device synchronize, timed with CUDA events on
the capturing stream; the max over ranks is reported.  Inputs are resident in
HBM.  Each step uses its own copy of the layer weights and its own x (copies
rotate), so a step never finds its weights in L2.  Under torchrun every rank
runs its own replica (weak scaling, no collective on the data path).

The JSON line also carries: the roofline of the expert-FFN stage (CUDA events
around it in a second graph of the same steps), the FP64 oracle's own
throughput on the host cores (cpu_baseline), an end-to-end number through the
public API with host buffers (e2e), the number of kernel launches, and SM
clocks sampled with nvidia-smi while the GPU is under load.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from quantised_moe_expert_gb300 import synth  # noqa: E402

METRIC = "MoE-layer tokens/s at T=1/16/512/4096; % HBM roofline / % bf16 TC peak"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--config", type=int, default=1)
    ap.add_argument("--workload", default=None,
                    help="a workload by name (any of synth.WORKLOADS, WORKLOADS_B8 or WORKLOADS_NVFP4); overrides --config")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--copies", type=int, default=0, help="weight copies to rotate (0: enough to defeat L2)")
    ap.add_argument("--profile", action="store_true",
                    help="warm-up and timed steps only (for a profiler's launch list): no clocks, stage, e2e, "
                         "CPU baseline or sweep")
    ap.add_argument("--timeline", action="store_true",
                    help="decode workloads: print the per-phase timeline of single launches (fused decode kernel "
                         "stamps) as one JSON line and exit")
    return ap.parse_args()


def default_steps(wl):
    return {1: 2000, 16: 400, 512: 40, 4096: 10}.get(wl.tokens, 50)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


# ----------------------------------------------------------------- distributed

def dist_setup(gpus):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local, pg


def barrier(pg):
    import torch
    if pg is not None:
        pg.barrier()
    if torch.cuda.is_available():
        torch.cuda.synchronize()


def max_over_ranks(pg, v):
    """Largest value over all ranks (the slowest rank's time); identity without a process group."""
    import torch
    if pg is None:
        return v
    dev = "cuda" if pg.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def whole_job_tokens_per_s(world, steps, tokens, max_ms):
    """Weak scaling: every rank processes `steps` batches of `tokens`; the job takes the slowest rank's time."""
    return world * steps * tokens / (max_ms / 1e3)


# ----------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=timestamp," + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, on):
        self.marks.append((time.time(), on))

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(2)
        except Exception:
            self.proc.kill()
        # samples taken while the GPU was under load (between mark(True) and mark(False))
        spans, start = [], None
        for t, on in self.marks:
            if on:
                start = t
            elif start is not None:
                spans.append((start, t))
                start = None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, line in self.lines:
            if not any(a <= t <= b for a, b in spans):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- workload

class Workload:
    """Rotating weight copies and inputs of one named workload on the current device."""

    def __init__(self, wl, copies):
        import torch
        import quantised_moe_expert_gb300 as qm
        self.wl = wl
        self.qm = qm
        host = synth.make_weights(wl.shape, wl.seed)
        base = qm.DeviceLayer(host)
        self.layers = [base]
        for _ in range(copies - 1):
            t = {k: v.clone() for k, v in base.tensors.items()}
            self.layers.append(qm.DeviceLayer.from_tensors(wl.shape, t))
        self.weight_bytes = host.nbytes()
        T = wl.tokens
        self.x_host = [synth.make_x(wl.shape, T, wl.seed, stream=i) for i in range(copies)]
        self.x = [torch.from_numpy(x.view(np.int16)).cuda() for x in self.x_host]
        self.bias = None
        if wl.zipf_s > 0:
            self.bias = torch.from_numpy(synth.zipf_bias(wl.shape, wl.zipf_s, wl.seed)).cuda()
        self.ws = [qm.workspace(base.cfg, T) for _ in range(copies)]
        self.y = [torch.empty((T, wl.shape.hidden), dtype=torch.int16, device="cuda") for _ in range(copies)]
        self.ids = [torch.full((T, wl.shape.top_k), -1, dtype=torch.int32, device="cuda") for _ in range(copies)]
        self.copies = copies
        self.executed = set()        # copies whose step has run (their ids are real)

    def step(self, i, stream):
        c = i % self.copies
        self.executed.add(c)
        L = self.layers[c]
        self.qm.moe_forward(L.cfg, L.w, self.x[c], self.wl.tokens, self.bias, None, self.y[c], self.ids[c],
                            None, None, self.qm.MOE_PATH_AUTO, self.ws[c], stream)

    def path(self):
        # NVFP4 experts take the grouped GEMMs at every T (the library resolves the decode path to them)
        return self.qm.MOE_PATH_DECODE if self.wl.tokens <= 16 else self.qm.MOE_PATH_PREFILL

    def kernels_per_step(self):
        # decode: the one fused kernel (8-bit experts: router GEMV, top-k, permute, gate/up, down,
        # slot sum); prefill: router GEMV (gamma), router MMA, top-k, permute, x conversion, two
        # small-tile (4-bit experts only) and two tensor-memory GEMMs, slot sum
        # NVFP4 experts (grouped GEMMs at every T): router GEMV (logits at T <= 16, and gamma), router MMA
        # (T > 16), top-k, permute, x conversion, two tensor-memory GEMMs, slot sum
        b8 = self.wl.shape.bits == 8
        if self.wl.shape.fmt == "nvfp4":
            return 7 if self.wl.tokens <= 16 else 8
        if self.wl.tokens <= 16:
            return 6 if b8 else 1
        return 8 if b8 else 10

    def distinct_experts(self):
        """Distinct routed experts (plus the shared expert) of each copy whose step was executed."""
        out = []
        for c in sorted(self.executed):
            ids = self.ids[c].cpu().numpy()
            assert ids.min() >= 0, "a copy marked executed has no routing"
            out.append(len(np.unique(ids)) + self.wl.shape.has_shared)
        return out


def capture(fn, nsteps, stream):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for i in range(nsteps):
                fn(i)
    return g


def algorithmic(wl, W, distinct):
    """Bytes and expert FLOPs of one step (weights of every touched expert once)."""
    sh = wl.shape
    ex = synth.active_expert_bytes(sh)
    io = 2 * 2 * wl.tokens * sh.hidden
    d = float(np.mean(distinct))
    bytes_step = synth.router_bytes(sh) + io + d * ex
    flops = wl.tokens * synth.expert_flops_per_token(sh)
    return bytes_step, d * ex, flops


def run_ours(args, wl, rank, world, pg, steps, warmup, want_extras):
    import torch
    import quantised_moe_expert_gb300 as qm
    qm.load()
    sh = wl.shape
    act = synth.active_expert_bytes(sh) * (min(sh.n_experts, wl.tokens * sh.top_k) + 1)
    l2 = 129 * 2 ** 20
    copies = int(max(2, min(64, np.ceil(3 * l2 / max(act, 1)) + 1)))
    if getattr(args, "copies", 0):
        copies = args.copies
    W = Workload(wl, copies)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    g_warm = capture(lambda i: W.step(i, stream), max(warmup, 1), stream)
    g_timed = capture(lambda i: W.step(i, stream), steps, stream)

    def replay(g):
        # CUDAGraph.replay() launches on the current stream: make it the timed stream
        with torch.cuda.stream(stream):
            g.replay()

    for _ in range(2):
        replay(g_warm)
    torch.cuda.synchronize()
    st = qm.moe_get_device_status(W.ws[0], stream)
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")

    clocks = ClockSampler(torch.cuda.current_device()) if want_extras and not args.profile else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
        clocks.mark(True)
        t_end = time.time() + 1.0          # keep the GPU busy so clocks settle under load
        while time.time() < t_end:
            replay(g_warm)
            torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(pg)
    ev0.record(stream)
    replay(g_timed)
    ev1.record(stream)
    barrier(pg)
    if clocks:
        t_end = time.time() + 0.5
        while time.time() < t_end:
            replay(g_warm)
            torch.cuda.synchronize()
        clocks.mark(False)
    ms = ev0.elapsed_time(ev1)
    ms = max_over_ranks(pg, ms)
    for c in range(copies):
        if qm.moe_get_device_status(W.ws[c], stream) != 0:
            raise RuntimeError("device status set during the timed steps")
    distinct = W.distinct_experts()
    value = whole_job_tokens_per_s(world, steps, wl.tokens, ms)
    res = dict(value=value, ms_per_step=ms / steps, copies=copies, distinct=distinct)
    bytes_step, expert_bytes, flops = algorithmic(wl, W, distinct)
    res["bytes_step"] = bytes_step
    res["flops_step"] = flops
    res["kernels"] = steps * W.kernels_per_step()
    res["clocks"] = clocks.stop() if clocks else None
    if want_extras and not args.profile:
        res["e2e"] = e2e_timing(W, stream, steps, warmup)
        if wl.tokens <= 16:
            res["cold"] = cold_call_latency(W, stream)
    if not args.profile:
        res["stage"] = stage_timing(W, stream, steps, expert_bytes, flops)
    del g_warm, g_timed
    return res


def stage_timing(W, stream, steps, expert_bytes, flops):
    """Mean duration of the expert-FFN stage, from CUDA events recorded inside a graph of the same steps."""
    import torch
    qm = W.qm
    wl = W.wl
    sh = wl.shape
    T = wl.tokens
    n = min(steps, 4 * W.copies)
    bufs = []
    for c in range(W.copies):
        d = dict(ids=torch.empty((T, sh.top_k), dtype=torch.int32, device="cuda"),
                 p=torch.empty((T, sh.top_k), dtype=torch.int16, device="cuda"),
                 w_s=torch.empty((T,), dtype=torch.int16, device="cuda"),
                 counts=torch.empty(sh.n_experts, dtype=torch.int32, device="cuda"),
                 offsets=torch.empty(sh.n_experts + 1, dtype=torch.int32, device="cuda"),
                 perm=torch.empty(T * sh.top_k, dtype=torch.int32, device="cuda"),
                 inv=torch.empty(T * sh.top_k, dtype=torch.int32, device="cuda"),
                 acc=torch.zeros((T, sh.hidden), dtype=torch.float32, device="cuda"))
        bufs.append(d)
    evs = [(torch.cuda.Event(enable_timing=True, external=True), torch.cuda.Event(enable_timing=True, external=True))
           for _ in range(n)]
    path = W.path()

    def step(i):
        c = i % W.copies
        L, b = W.layers[c], bufs[c]
        qm.moe_route(L.cfg, L.w, W.x[c], T, W.bias, None, None, b["ids"], b["p"], b["w_s"], W.ws[c], stream)
        qm.moe_permute(L.cfg, b["ids"], T, b["counts"], b["offsets"], b["perm"], b["inv"], W.ws[c], stream)
        evs[i][0].record(stream)
        qm.moe_expert_ffn(L.cfg, L.w, W.x[c], T, b["ids"], b["p"], b["w_s"], b["counts"], b["offsets"], b["perm"],
                          b["acc"], path, W.ws[c], stream)
        evs[i][1].record(stream)
        qm.moe_combine(L.cfg, T, b["acc"], W.y[c], stream)

    g = capture(step, n, stream)
    with torch.cuda.stream(stream):
        g.replay()
        g.replay()
    torch.cuda.synchronize()
    times = [a.elapsed_time(b) for a, b in evs]
    ms = float(np.mean(times))
    del g
    return dict(ms=ms, expert_bytes=expert_bytes, flops=flops, launches=n)


def cold_call_latency(W, stream, reps=20):
    """One moe_forward after an L2-flushing write (a buffer larger than L2), device time per call."""
    import torch
    qm = W.qm
    wl = W.wl
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device="cuda")
    times = []
    for i in range(reps):
        c = i % W.copies
        L = W.layers[c]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            flush.fill_(i & 0xFF)
            e0.record(stream)
            qm.moe_forward(L.cfg, L.w, W.x[c], wl.tokens, W.bias, None, W.y[c], None, None, None,
                           qm.MOE_PATH_AUTO, W.ws[c], stream)
            e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    del flush
    return dict(ms_median=float(np.median(times)), ms_min=float(np.min(times)), calls=reps,
                flush="512 MiB write before each call")


TIMELINE = ["start", "router_published", "logits_seen", "x_staged", "topk_done", "list_done", "routing_done",
            "first_gate_chunk", "first_down_chunk", "first_down_done", "units_done", "units_counter",
            "combine_loads_done", "combine_done"]


def timeline(W, stream, graph_steps=200):
    """Per-phase times of the fused decode kernel in steady state: a graph of back-to-back steps is
    replayed, then each weight copy's workspace holds the stamps of its last launch (us from the
    launch's earliest CTA start; median CTA and last CTA), and consecutive launches give the gap
    from one launch's last CTA to the next launch's first."""
    import torch
    qm = W.qm
    wl = W.wl
    g = capture(lambda i: W.step(i, stream), graph_steps, stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
    torch.cuda.synchronize()
    traces = []
    for c in range(W.copies):
        L = W.layers[c]
        traces.append(qm.moe_decode_timeline(L.cfg, wl.tokens, W.ws[c], stream).astype(np.int64))
    med, last = [], []
    for st in traces:
        rel = (st - st[:, 0].min()) / 1e3
        med.append(np.median(rel, axis=0))
        last.append(rel.max(axis=0))
    # launches of the last replay in order: copies (graph_steps - copies .. graph_steps - 1) % copies
    order = [(graph_steps - W.copies + j) % W.copies for j in range(W.copies)]
    gaps = [(traces[b][:, 0].min() - traces[a][:, -1].max()) / 1e3 for a, b in zip(order[:-1], order[1:])]
    del g
    return {"workload": wl.name, "launches_read": W.copies, "ctas": int(traces[0].shape[0]),
            "median_cta_us": dict(zip(TIMELINE, [round(float(v), 3) for v in np.median(np.stack(med), axis=0)])),
            "last_cta_us": dict(zip(TIMELINE, [round(float(v), 3) for v in np.median(np.stack(last), axis=0)])),
            "gap_between_launches_us": round(float(np.median(gaps)), 3) if gaps else None}


def e2e_timing(W, stream, steps, warmup):
    """Same metric through the public API per step: pinned-host x -> device, forward, y -> pinned host."""
    import torch
    qm = W.qm
    wl = W.wl
    T = wl.tokens
    n = min(steps, 200 if T <= 16 else steps)
    xh = [torch.from_numpy(x.view(np.int16)).pin_memory() for x in W.x_host]
    yh = [torch.empty((T, wl.shape.hidden), dtype=torch.int16).pin_memory() for _ in range(W.copies)]
    xd = torch.empty_like(W.x[0])
    yd = torch.empty_like(W.y[0])

    def one(i):
        c = i % W.copies
        L = W.layers[c]
        xd.copy_(xh[c], non_blocking=True)
        qm.moe_forward(L.cfg, L.w, xd, T, W.bias, None, yd, None, None, None, qm.MOE_PATH_AUTO, W.ws[c], stream)
        yh[c].copy_(yd, non_blocking=True)

    with torch.cuda.stream(stream):
        for i in range(max(3, warmup)):
            one(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n):
            one(i)
        e1.record(stream)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    return dict(value=n * T / (ms / 1e3), unit="tokens/s", h2d_bytes_per_step=int(xh[0].numel() * 2),
                d2h_bytes_per_step=int(yh[0].numel() * 2), steps=n)


# ----------------------------------------------------------------- oracle (CPU) legs

def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def oracle_single_core(wl, seconds=5.0):
    """The same oracle sample on one core: a fresh process with OMP_NUM_THREADS=1."""
    code = ("import sys, json; sys.path.insert(0, %r); import bench; "
            "r, n, dt = bench.oracle_sample(bench.workload_named(%r), seconds=%r); print(json.dumps(r))"
            % (ROOT, wl.name, seconds))
    env = dict(os.environ, OMP_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    try:
        out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120, env=env)
        return json.loads(out.stdout.strip().splitlines()[-1])
    except Exception as e:
        return {"error": str(e)[:200]}


def oracle_sample(wl, seconds=12.0, max_tokens=None):
    """FP64 oracle throughput on this host's cores over a bounded sample of the workload's tokens."""
    import oracle
    oracle.build()
    w = synth.make_weights(wl.shape, wl.seed)
    x = synth.make_x(wl.shape, max(wl.tokens, 1), wl.seed)
    bias = synth.zipf_bias(wl.shape, wl.zipf_s, wl.seed) if wl.zipf_s > 0 else None
    t0 = time.time()
    oracle.forward(wl.shape, w, x[:1], bias=bias)
    per = max(time.time() - t0, 1e-3)
    n = int(max(1, min(seconds / per, max_tokens or 1e9)))
    reps = int(np.ceil(n / x.shape[0]))
    xs = np.concatenate([synth.make_x(wl.shape, x.shape[0], wl.seed, stream=r) for r in range(reps)])[:n]
    t0 = time.time()
    oracle.forward(wl.shape, w, xs, bias=bias)
    dt = time.time() - t0
    return dict(value=n / dt, unit="tokens/s", cores=oracle.num_threads(), kind="oracle",
                sample=f"{n} tokens of the {wl.name} workload through the FP64 oracle (router, top-k, "
                       f"{wl.shape.top_k}+{wl.shape.has_shared} expert FFNs, combine)"), n, dt


def run_reference(args, wl, rank, world, steps, warmup):
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = synth.make_weights(wl.shape, wl.seed)
    bias = synth.zipf_bias(wl.shape, wl.zipf_s, wl.seed) if wl.zipf_s > 0 else None
    per_step_tokens = max(1, min(wl.tokens, 8))
    xs = [synth.make_x(wl.shape, max(wl.tokens, 1), wl.seed, stream=i)[:per_step_tokens] for i in range(4)]
    for i in range(warmup):
        oracle.forward(wl.shape, w, xs[i % 4], bias=bias)
    t0 = time.time()
    for i in range(steps):
        oracle.forward(wl.shape, w, xs[i % 4], bias=bias)
    dt = time.time() - t0
    v = steps * per_step_tokens / dt
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world, "steps": steps,
            "warmup": warmup, "ms_per_step": 1e3 * dt / steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "tokens_per_step_sampled": per_step_tokens, "tokens": wl.tokens},
            "cpu_baseline": {"kind": "oracle", "cores": oracle.num_threads(), "value": v, "unit": "tokens/s",
                             "sample": f"each step: {per_step_tokens} tokens of the {wl.name} workload through "
                                       f"the FP64 oracle"},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def stage_roofline(wl, st, hbm, tc, peak_src):
    """Roofline of the expert-FFN stage from its CUDA-event time: HBM below the ridge point, else tensor."""
    decode = wl.tokens <= 16
    if decode:
        ach = st["expert_bytes"] / (st["ms"] / 1e3) / 1e9
        return {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                "traffic": traffic_for("decode_expert_ffn", wl.name),
                "kernel": ("expert-FFN stage (tensor-memory GEMMs and slot sum)" if wl.shape.fmt == "nvfp4"
                           else "expert-FFN stage (decode gate/up, down and reduce kernels)" if wl.shape.bits == 8
                           else "expert-FFN stage (fused decode kernel: units + combine)"),
                "kernel_us": st["ms"] * 1e3, "algorithmic_bytes_per_launch": st["expert_bytes"],
                "peak_source": peak_src}
    if st["flops"] / max(st["expert_bytes"], 1.0) < tc * 1e12 / (hbm * 1e9):
        # below the ridge point (e.g. T = 512: ~16 tokens per expert) the weights bound the stage
        ach = st["expert_bytes"] / (st["ms"] / 1e3) / 1e9
        return {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                "traffic": traffic_for("prefill_expert_ffn", wl.name),
                "kernel": "expert-FFN stage (grouped GEMMs)", "kernel_us": st["ms"] * 1e3,
                "algorithmic_bytes_per_launch": st["expert_bytes"],
                "tensor_frac": st["flops"] / (st["ms"] / 1e3) / 1e12 / tc, "peak_source": peak_src}
    ach = st["flops"] / (st["ms"] / 1e3) / 1e12
    return {"bound": "tensor", "achieved": ach, "peak": tc, "unit": "TFLOP/s", "frac": ach / tc,
            "traffic": traffic_for("prefill_expert_ffn", wl.name),
            "kernel": "expert-FFN stage (grouped GEMMs)", "kernel_us": st["ms"] * 1e3,
            "algorithmic_flops_per_launch": st["flops"], "peak_source": peak_src}


def traffic_for(kernel_key, workload):
    """DRAM bytes per launch from a committed ncu summary, if no source of the stage has changed since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        ent = d[kernel_key][workload]
        for src, sha in zip(ent["sources"], ent["source_shas"]):
            h = hashlib.sha256(open(os.path.join(ROOT, src), "rb").read()).hexdigest()[:16]
            if h != sha:
                return None
        return float(ent["bytes_per_launch"])
    except Exception:
        return None


def workload_named(name):
    for wl in synth.WORKLOADS + synth.WORKLOADS_B8 + synth.WORKLOADS_NVFP4:
        if wl.name == name:
            return wl
    raise SystemExit(f"unknown workload {name!r}")


def main():
    args = parse()
    wl = workload_named(args.workload) if args.workload else synth.WORKLOADS[args.config]
    steps = args.steps or default_steps(wl)
    warmup = max(3, args.warmup if args.warmup is not None else 20)
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", "1"))
        run_reference(args, wl, rank, world, steps, warmup)
        return
    import torch
    rank, world, local, pg = dist_setup(args.gpus)
    hbm, tc, tc_sus, peak_src = peaks()
    if args.timeline:
        import quantised_moe_expert_gb300 as qm
        qm.load()
        W = Workload(wl, args.copies or 8)
        stream = torch.cuda.Stream()
        if rank == 0:
            print(json.dumps(timeline(W, stream)), flush=True)
        return
    r = run_ours(args, wl, rank, world, pg, steps, warmup, want_extras=True)
    if args.profile:
        if rank == 0:
            print(json.dumps({"profile_run": wl.name, "ms_per_step": r["ms_per_step"], "steps": steps}), flush=True)
        return
    roof = stage_roofline(wl, r["stage"], hbm, tc, peak_src)
    line = {"metric": METRIC, "value": r["value"], "unit": "tokens/s", "n_gpus": world, "steps": steps,
            "warmup": warmup, "ms_per_step": r["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "data": "synthetic",
            "dtype": ("nvfp4 (e2m1 codes, e4m3 block scales)/bf16 in, fp32 accumulate" if wl.shape.fmt == "nvfp4"
                      else f"int{wl.shape.bits}-affine/bf16 in, fp32 accumulate"),
            "config": {"workload": wl.name, "tokens": wl.tokens, "hidden": wl.shape.hidden,
                       "inter": wl.shape.inter, "experts": wl.shape.n_experts, "top_k": wl.shape.top_k,
                       "shared": wl.shape.has_shared, "expert_bits": wl.shape.bits, "expert_format": wl.shape.fmt,
                       "parallelism": f"replicas x{world}",
                       "l2": f"{r['copies']} rotating weight copies and inputs: no step finds its weights in L2"},
            "roofline": roof,
            "layer_hbm": {"bytes_per_step": r["bytes_step"], "achieved_gbs": r["bytes_step"] / (r["ms_per_step"] / 1e3) / 1e9,
                          "frac_of_peak": r["bytes_step"] / (r["ms_per_step"] / 1e3) / 1e9 / hbm,
                          "frac_of_8tbs": r["bytes_step"] / (r["ms_per_step"] / 1e3) / 8e12,
                          "distinct_experts_mean": float(np.mean(r["distinct"]))},
            "layer_tensor": {"flops_per_step": r["flops_step"],
                             "frac_of_peak": r["flops_step"] / (r["ms_per_step"] / 1e3) / 1e12 / tc},
            "e2e": r["e2e"], "gpu_launches": r["kernels"], "clocks": r["clocks"]}
    if "cold" in r:
        line["cold_single_call"] = r["cold"]
    if rank == 0 and not args.no_cpu_baseline:
        cb, _, _ = oracle_sample(wl)
        one = oracle_single_core(wl)
        cb["cpu_model"] = cpu_model()
        cb["host_cores"] = os.cpu_count()
        cb["single_core"] = {"value": one.get("value"), "unit": "tokens/s", "cores": 1,
                             "sample": one.get("sample", one.get("error"))}
        line["cpu_baseline"] = cb
    if not args.no_sweep and rank == 0:
        sweep = {}
        others = [o for o in synth.WORKLOADS[1:] + synth.WORKLOADS_B8 + synth.WORKLOADS_NVFP4
                  if o.name != wl.name]                                              # not the tiny layer
        for other in others:
            try:
                rr = run_ours(args, other, 0, 1, None, default_steps(other) // 2, 3, want_extras=False)
                sweep[other.name] = {"value": rr["value"], "ms_per_step": rr["ms_per_step"],
                                     "hbm_frac": rr["bytes_step"] / (rr["ms_per_step"] / 1e3) / 1e9 / hbm,
                                     "tc_frac": rr["flops_step"] / (rr["ms_per_step"] / 1e3) / 1e12 / tc,
                                     "distinct_experts_mean": float(np.mean(rr["distinct"])),
                                     "stage_roofline": stage_roofline(other, rr["stage"], hbm, tc, peak_src)}
            except Exception as e:  # a path not built yet reports why
                sweep[other.name] = {"error": str(e)[:200]}
        line["sweep"] = sweep
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
