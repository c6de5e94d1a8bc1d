"""Benchmark of the sparse MoE layer forward on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one full layer forward (router, capacity + dispatch, expert FFNs,
combine) over one batch of the workload, inputs resident in HBM, replayed as a
CUDA graph of those launches. The default
workload is the largest single-GPU one: the bf16 prefill shape T=16384,
d=4096, N=8, k=2, d_ff=14336 with no capacity limit. The step is
issued as the four stage calls of the C ABI (moe_route, moe_dispatch,
moe_expert_ffn, moe_combine: exactly the launches moe_forward makes). The
value's timed region records CUDA events at the step boundaries only, on the
launching stream; a second timed region of the same K steps puts events around
the expert FFN launch for its roofline, and a third pass with an event after
every stage gives the stage breakdown. Between timed steps L2 is flushed (a
512 MiB write, then a 1 GiB read, outside the events) unless a step streams at
least twice the L2 size, in which case its inputs are larger than L2. The
roofline and stage-breakdown regions launch the stage calls directly. ``e2e`` times
moe_forward with each step's batch copied in from pinned host memory and its
output copied back inside the timed region, the copies of neighbouring steps
overlapping the forward on a second stream (double-buffered x and y).

Multi-GPU: replicas only (capacity couples every token of a batch, so a batch
is not split); every rank runs its own batch and value = all tokens / the
slowest rank's time. ``--gpus N`` without a launcher re-runs this script under
torch.distributed.run with N ranks. Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_mixture_experts_66_b300 import moe  # noqa: E402
from sparse_mixture_experts_66_b300.workload import PREFILL, WORKLOADS, as_f32_numpy, draw  # noqa: E402

METRIC = "MoE-layer fwd tokens/s on 1 B300; % of bf16 tensor / HBM roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
L2_BYTES = 126 * 1024 * 1024


def kernels_per_step(w) -> int:
    """Launches of one forward: router, capacity, permute, the expert FFN (one
    fused launch for bf16, two SIMT GEMMs for fp32) and the combine."""
    return 5 if w.dtype == "bf16" else 6


def measured_traffic(workload: str):
    """DRAM bytes of one expert-FFN launch from the committed ncu summary
    (profiles/traffic.txt), or None when there is none for this workload or
    the kernel sources changed since the capture."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        f = line.split("#", 1)[0].split()
        if len(f) != 4 or f[0] != workload:
            continue
        m = hashlib.sha1()
        for src in f[1].split(","):
            m.update(open(os.path.join(ROOT, "sparse_mixture_experts_66_b300", "csrc", src), "rb").read())
        if m.hexdigest()[:12] == f[2]:
            return float(f[3])
    return None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# distributed plumbing (barrier + max over ranks only; no data-path collective)
# ---------------------------------------------------------------------------
def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(value: float, world: int, device) -> float:
    if world == 1:
        return value
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(units_per_rank: float, seconds_per_rank: float, world: int, device) -> tuple:
    """Whole-job throughput of replicas: the units every rank processed in one
    step (tokens), summed over ranks, over the slowest rank's step time."""
    slowest = max_over_ranks(seconds_per_rank, world, device)
    return units_per_rank * world / slowest, slowest


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.file,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        self.t0 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
class Stages:
    """The four stage calls of one forward, on workspace buffers."""

    def __init__(self, cfg, dev, ws):
        self.cfg, self.dev, self.ws = cfg, dev, ws
        self.v = ws.views()
        self.y = torch.empty_like(dev["x"])

    def route(self, s):
        d, v = self.dev, self.v
        moe.moe_route(self.cfg, d["x"], d["w_g"], d["router_bias"], v["topk_idx"], v["gate"], v["score"], self.ws.buf,
                      s)

    def dispatch(self, s):
        d, v = self.dev, self.v
        moe.moe_dispatch(self.cfg, d["x"], v["topk_idx"], v["gate"], v["score"], v["counts_raw"], v["counts_kept"],
                         v["offsets"], v["row_of"], v["row_token"], v["row_gate"], v["x_perm"], self.ws.buf, s)

    def ffn(self, s):
        d, v = self.dev, self.v
        moe.moe_expert_ffn(self.cfg, v["x_perm"], v["offsets"], d["w1"], d["b1"], d["w2"], d["b2"], v["row_gate"],
                           v["h"], v["y_perm"], self.ws.buf, s)

    def combine(self, s):
        v = self.v
        moe.moe_combine(self.cfg, v["y_perm"], v["row_of"], v["gate"], self.dev["x"], self.y, self.ws.buf, s)

    def all(self, s):
        self.route(s)
        self.dispatch(s)
        self.ffn(s)
        self.combine(s)


def l2_policy(w, streamed_bytes):
    """Whether timed steps flush L2, and the sentence that says so: a step that
    streams at least twice the L2 size has inputs larger than L2; otherwise a
    512 MiB write and a 1 GiB read evict L2 between timed steps."""
    use_flush = streamed_bytes < 2 * L2_BYTES
    note = ("flushed between timed steps outside the events (512 MiB write, then 1 GiB read)" if use_flush else
            f"inputs larger than L2: {streamed_bytes / 1e9:.2f} GB streamed per step, "
            f"{streamed_bytes / L2_BYTES:.0f}x the 126 MB L2; no flush")
    return use_flush, note


def config_dict(w, capacity, counts_kept, world):
    """The workload as both arms report it (the same dict in both lines)."""
    alg = algorithmic(w, counts_kept)
    return {"workload": w.name, "T": w.T, "d": w.d, "N": w.N, "k": w.k, "d_ff": w.d_ff,
            "capacity_factor": None if math.isinf(w.capacity_factor) else w.capacity_factor,
            "router_bias": w.router_bias, "capacity": int(capacity), "kept_rows": alg["R"],
            "active_experts": alg["A"], "parallelism": f"replicas{world}", "l2": l2_policy(w, alg["bytes"])[1]}


def algorithmic(w, counts_kept):
    """Algorithmic FLOPs and bytes of one forward (kept rows only; padding and
    intermediates excluded)."""
    s = 2 if w.dtype == "bf16" else 4
    R = int(np.sum(counts_kept))
    A = int(np.sum(np.asarray(counts_kept) > 0))
    flops_router = 2.0 * w.T * w.d * w.N
    flops_ffn = 4.0 * R * w.d * w.d_ff
    bytes_total = 2.0 * w.T * w.d * s + w.N * w.d * s + A * (2.0 * w.d * w.d_ff + w.d_ff + w.d) * s
    bytes_ffn_weights = A * (2.0 * w.d * w.d_ff + w.d_ff + w.d) * s
    return dict(R=R, A=A, flops=flops_router + flops_ffn, flops_ffn=flops_ffn, bytes=bytes_total,
                bytes_ffn_weights=bytes_ffn_weights)


def timing_events(n, per, stream):
    """n lists of `per` timing events, each recorded once and synchronised
    here: torch creates a CUDA event at its first record, and hundreds of
    creations inside a timed loop can make it host-bound."""
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(per)] for _ in range(n)]
    for row in evs:
        for e in row:
            e.record(stream)
    stream.synchronize()
    return evs


def run_ours(args, world, rank, local):
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    w = WORKLOADS[args.workload]
    inp = draw(w)
    dev = {k: (None if v is None else v.to(device)) for k, v in inp.items()}
    cfg = moe.config_of(w)
    ws = moe.Workspace(cfg, device=device)
    st = Stages(cfg, dev, ws)
    stream = torch.cuda.current_stream(device)
    flush_bufs = []

    def flush():
        """Evict L2: write 512 MiB, then read 1 GiB, so that L2 holds none of
        the step's data and no dirty lines whose write-back would land in the
        next step. (The buffers are allocated on first use: workloads whose
        steps stream more than twice the L2 size never flush.)"""
        if not flush_bufs:
            flush_bufs.append(torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=device))
            flush_bufs.append(torch.zeros(256 * 1024 * 1024, dtype=torch.float32, device=device))
        flush_bufs[0].zero_()
        flush_bufs[1].sum()

    for _ in range(max(args.warmup, 3)):
        st.all(stream)
    torch.cuda.synchronize(device)
    ws.status(stream)
    counts_kept = st.v["counts_kept"].cpu().numpy()
    alg = algorithmic(w, counts_kept)
    # L2 between timed steps: when a step streams at least twice the L2 size
    # (the weights of the active experts), its inputs are larger than L2 and
    # no flush is needed; otherwise a 512 MiB write evicts L2 before each step.
    use_flush, _ = l2_policy(w, alg["bytes"])

    K = args.steps
    # The step as a CUDA graph: the four stage calls (the launches moe_forward
    # makes) captured once and replayed once per step, as a serving loop
    # would; the programmatic-dependent-launch edges between the kernels are
    # kept in the graph.
    graph = torch.cuda.CUDAGraph()
    cap_stream = torch.cuda.Stream(device)
    cap_stream.wait_stream(stream)
    with torch.cuda.graph(graph, stream=cap_stream):
        st.all(cap_stream)
    stream.wait_stream(cap_stream)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize(device)
    ws.status(stream)
    # Timed region 1 (the value): events at the step boundaries only, around
    # each replay, so the launches inside a step overlap through programmatic
    # dependent launch as they do for a user.
    ev = timing_events(K, 2, stream)
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize(device)
    t_wall0 = time.perf_counter()
    for i in range(K):
        if use_flush:
            flush()  # evict L2 between steps, outside the step's events
        e = ev[i]
        e[0].record(stream)
        graph.replay()
        e[1].record(stream)
    torch.cuda.synchronize(device)
    barrier(world)
    t_wall = time.perf_counter() - t_wall0
    ws.status(stream)
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    ms = statistics.mean(step_ms)

    # Timed region 2 (the roofline): the same K steps with events around the
    # expert FFN launch, the dominant kernel (events there stop its launch
    # from overlapping its neighbours, so this region does not give the value).
    ev_f = timing_events(K, 2, stream)
    for i in range(K):
        if use_flush:
            flush()
        st.route(stream)
        st.dispatch(stream)
        ev_f[i][0].record(stream)
        st.ffn(stream)
        ev_f[i][1].record(stream)
        st.combine(stream)
    torch.cuda.synchronize(device)
    ws.status(stream)
    ffn_ms = statistics.mean(a.elapsed_time(b) for a, b in ev_f)

    # Stage breakdown (reported, not timed for the value): an event after every
    # stage call, which serialises the stages.
    K2 = min(K, 20)
    ev2 = timing_events(K2, 5, stream)
    for i in range(K2):
        if use_flush:
            flush()
        e = ev2[i]
        e[0].record(stream)
        for j, fn in enumerate((st.route, st.dispatch, st.ffn, st.combine)):
            fn(stream)
            e[j + 1].record(stream)
    torch.cuda.synchronize(device)
    ws.status(stream)
    stage_ms = {n: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in ev2)
                for j, n in enumerate(["route", "dispatch", "expert_ffn", "combine"])}
    stage_ms["serialised_step"] = statistics.mean(e[0].elapsed_time(e[4]) for e in ev2)
    clk = clocks.stop()
    value, slowest_s = aggregate_throughput(w.T, ms * 1e-3, world, device)
    ms_max = slowest_s * 1e3

    # End to end through moe_forward with host buffers: every step copies its
    # batch in from pinned host memory and its output back, inside the timed
    # region. When the workload needs no L2 flush the steps are pipelined: x of
    # step i+1 is copied in (copy stream) and y of step i-1 copied out (a second
    # copy stream) while step i computes, with x and y double-buffered on the
    # device. Workloads timed with L2 flushes run the copies and the forward
    # serially, each step between its own events with the flush outside them.
    x_host = inp["x"].pin_memory()
    y_host = [torch.empty_like(x_host).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(dev["x"]) for _ in range(2)]
    y_dev = [torch.empty_like(dev["x"]) for _ in range(2)]

    def fwd(xd, yd):
        moe.moe_forward(cfg, xd, dev["w_g"], dev["router_bias"], dev["w1"], dev["b1"], dev["w2"], dev["b2"], yd,
                        ws.buf, stream)

    for i in range(3):
        x_dev[0].copy_(x_host, non_blocking=True)
        fwd(x_dev[0], y_dev[0])
        y_host[0].copy_(y_dev[0], non_blocking=True)
    torch.cuda.synchronize(device)
    barrier(world)
    if use_flush:
        e2e_mode = "serial: copy in, forward, copy out per step; L2 flushed between steps outside the events"
        e2e_ev = timing_events(K, 2, stream)
        for i in range(K):
            flush()
            e2e_ev[i][0].record(stream)
            x_dev[0].copy_(x_host, non_blocking=True)
            fwd(x_dev[0], y_dev[0])
            y_host[0].copy_(y_dev[0], non_blocking=True)
            e2e_ev[i][1].record(stream)
        torch.cuda.synchronize(device)
        e2e_ms = statistics.mean(a.elapsed_time(b) for a, b in e2e_ev)
    else:
        e2e_mode = ("pipelined: step i+1's x copied in and step i-1's y copied out on two copy streams while step "
                    "i computes (x, y double-buffered); one event pair around all K steps")
        s_in = torch.cuda.Stream(device)
        s_out = torch.cuda.Stream(device)

        def pipelined(n):
            ev = lambda: torch.cuda.Event()  # noqa: E731
            in_done = [ev() for _ in range(n)]
            fwd_done = [ev() for _ in range(n)]
            out_done = [ev() for _ in range(n)]
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            # torch creates a CUDA event at its first record: do that here, not
            # inside the timed steps (hundreds of creations made the first timed
            # run host-bound)
            for e in in_done + fwd_done + out_done + [t0, t1]:
                e.record(stream)
            torch.cuda.synchronize(device)
            t0.record(stream)
            s_in.wait_event(t0)
            s_out.wait_event(t0)
            for i in range(n):
                b = i % 2
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(fwd_done[i - 2])  # the forward of step i-2 has read x_dev[b]
                    x_dev[b].copy_(x_host, non_blocking=True)
                    in_done[i].record(s_in)
                stream.wait_event(in_done[i])
                if i >= 2:
                    stream.wait_event(out_done[i - 2])  # y_dev[b] of step i-2 is back on the host
                fwd(x_dev[b], y_dev[b])
                fwd_done[i].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(fwd_done[i])
                    y_host[b].copy_(y_dev[b], non_blocking=True)
                    out_done[i].record(s_out)
            t1.record(s_out)
            torch.cuda.synchronize(device)
            return t0.elapsed_time(t1) / n

        # untimed warm-up: the same pattern, as many steps as the timed run, on
        # the same streams and buffers (torch's pinned-memory allocator records
        # an event per asynchronous copy and grows its event pool during the
        # first long run)
        pipelined(K)
        barrier(world)
        e2e_ms = pipelined(K)
    barrier(world)
    ws.status(stream)
    e2e_value, _ = aggregate_throughput(w.T, e2e_ms * 1e-3, world, device)
    es = 2 if w.dtype == "bf16" else 4

    peaks, peak_src = load_peaks()
    t_ffn = ffn_ms * 1e-3
    t_tensor = alg["flops"] / (peaks["bf16_tflops"] * 1e12)
    t_hbm = alg["bytes"] / (peaks["hbm_gbs"] * 1e9)
    if t_tensor >= t_hbm:
        achieved = alg["flops_ffn"] / t_ffn / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"],
                "frac_of_sustained": achieved / peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]),
                "peak_source": f"{peak_src} bf16 dense (burst)"}
    else:
        achieved = alg["bytes_ffn_weights"] / t_ffn / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "frac_of_8TBs": achieved / 8000.0,
                "peak_source": f"{peak_src} HBM copy"}
    roof["traffic"] = measured_traffic(w.name)
    roof["traffic_scope"] = "DRAM read+write bytes of one expert-FFN launch (ncu, profiles/traffic.txt)"
    roof["kernel"] = ("expert FFN: grouped GEMM1 (+b1, GELU) and GEMM2 (+b2, gate scale), one fused launch per step"
                      if w.dtype == "bf16" else "expert FFN: two SIMT grouped GEMMs per step")
    roof["ms_per_launch"] = ffn_ms
    roof["timing"] = "CUDA events around the FFN launch over a second timed region of the same K steps"
    roof["algorithmic_per_step"] = alg["flops_ffn"] if roof["bound"] == "tensor" else alg["bytes_ffn_weights"]

    step_flops = alg["flops"] / (ms * 1e-3) / 1e12
    step_gbs = alg["bytes"] / (ms * 1e-3) / 1e9
    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic: seeded normal draws (torch CPU generator, seed 0), fan-in scaled weights",
        "config": config_dict(w, ws.layout.capacity, counts_kept, world),
        "roofline": roof,
        "step": {"tflops": step_flops, "gbs": step_gbs,
                 "frac_tensor_roofline": (alg["flops"] / (peaks["bf16_tflops"] * 1e12)) / (ms * 1e-3),
                 "frac_hbm_roofline": (alg["bytes"] / (peaks["hbm_gbs"] * 1e9)) / (ms * 1e-3),
                 "stages_ms": stage_ms, "ms_min": min(step_ms), "ms_median": statistics.median(step_ms),
                 "wall_s": t_wall,
                 "timing": "CUDA events around each replay of a CUDA graph of one forward's launches"},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": w.T * w.d * es,
                "d2h_bytes_per_step": w.T * w.d * es, "ms_per_step": e2e_ms, "mode": e2e_mode},
        "gpu_launches": kernels_per_step(w) * K,
        "clocks": clk,
    }
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(w, inp, budget_s=args.cpu_budget)
    return out


# ---------------------------------------------------------------------------
# the CPU oracle as a baseline
# ---------------------------------------------------------------------------
def _oracle_inputs(inp):
    return tuple(as_f32_numpy(inp[n]) for n in ("x", "w_g", "w1", "b1", "w2", "b2")), as_f32_numpy(inp["router_bias"])


def _oracle_step(orc, w, arrays, rb, n_tok):
    """Route and apply capacity to the whole batch, run the FFNs and combine for
    the first n_tok tokens; returns seconds."""
    t0 = time.perf_counter()
    orc.forward(*arrays, k=w.k, cf=w.capacity_factor, router_bias=rb, sel=np.arange(n_tok, dtype=np.int64))
    return time.perf_counter() - t0


def _oracle_costs(orc, w, arrays, rb, budget_s):
    """Fixed cost (routing + capacity of the batch) and per-token cost (expert
    FFNs + combine) of the oracle, and the sample size that fits the budget."""
    fixed = _oracle_step(orc, w, arrays, rb, 0)
    probe = min(w.T, 16)
    t = _oracle_step(orc, w, arrays, rb, probe)
    per_tok = max(t - fixed, 1e-9) / probe
    n = int(max(probe, min(w.T, (budget_s - fixed) / per_tok)))
    return fixed, per_tok, n


def cpu_baseline(w, inp, budget_s=15.0):
    import oracle

    orc = oracle.load()
    arrays, rb = _oracle_inputs(inp)
    fixed, per_tok, n = _oracle_costs(orc, w, arrays, rb, budget_s)
    t = _oracle_step(orc, w, arrays, rb, n)
    per_tok = max(t - fixed, 1e-9) / n
    est = fixed + per_tok * w.T
    cores = len(os.sched_getaffinity(0))
    return {"value": w.T / est, "unit": "tokens/s", "cores": int(os.environ.get("OMP_NUM_THREADS", cores)),
            "kind": "oracle",
            "sample": f"routing+capacity over all {w.T} tokens ({fixed:.2f} s) and expert FFNs+combine for "
                      f"{n} of {w.T} tokens ({t - fixed:.2f} s); tokens/s extrapolated to the whole batch",
            "seconds": t}


def run_reference(args, world, rank):
    """The oracle timed on the host cores as the reference arm, on the same
    workload and config as the GPU arm. A step runs the whole batch when that
    fits the per-step budget (--ref-budget over warm-up plus timed steps);
    otherwise routing and capacity of the whole batch plus the expert FFNs and
    combine of the first n tokens (a bounded sample), and the tokens/s value is
    extrapolated to the whole batch. ms_per_step is the measured time of the
    steps actually run, so ms_per_step x steps is the time spent timing."""
    w = WORKLOADS[args.workload]
    inp = draw(w)
    import oracle

    orc = oracle.load()
    arrays, rb = _oracle_inputs(inp)
    steps = args.steps + args.warmup
    fixed, per_tok, _ = _oracle_costs(orc, w, arrays, rb, 1e9)
    per_step_budget = args.ref_budget / max(steps, 1)
    full = fixed + per_tok * w.T <= per_step_budget
    n = w.T if full else int(max(1, min(w.T, (per_step_budget - fixed) / per_tok)))
    for _ in range(args.warmup):
        _oracle_step(orc, w, arrays, rb, n)
    ts = [_oracle_step(orc, w, arrays, rb, n) for _ in range(args.steps)]
    t = statistics.mean(ts)
    est = t if full else fixed + max(t - fixed, 1e-9) / n * w.T
    value = w.T / est
    ref0 = orc.forward(*arrays, k=w.k, cf=w.capacity_factor, router_bias=rb, sel=np.arange(0, dtype=np.int64))
    cores = int(os.environ.get("OMP_NUM_THREADS", len(os.sched_getaffinity(0))))
    if full:
        sample = f"each step: the whole batch of {w.T} tokens (fp64 CPU oracle)"
    else:
        sample = (f"each step: routing+capacity over all {w.T} tokens and expert FFNs+combine for {n} of {w.T} "
                  f"tokens (fp64 CPU oracle, {t:.2f} s measured per step); tokens/s extrapolated to the whole "
                  f"batch ({est:.1f} s per full step)")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic: seeded normal draws (torch CPU generator, seed 0), fan-in scaled weights",
            "config": config_dict(w, ref0["C"], ref0["counts_kept"], world),
            "timed_region_s": t * args.steps, "tokens_per_timed_step": n, "extrapolated": not full,
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "note": "host-core arm: no L2 flush applies; the config's l2 entry describes the GPU arm"}


def relaunch(n):
    """Re-run this script under torch.distributed.run with n ranks on this
    node (one per GPU), passing the same arguments; returns its exit code."""
    import socket

    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", f"--master-port={port}", os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=PREFILL, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-budget", type=float, default=90.0)
    args = ap.parse_args()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(relaunch(args.gpus))
    world, rank, local = dist_info()
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, world, rank)), flush=True)
        return
    init_dist(world, "nccl")
    out = run_ours(args, world, rank, local)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
