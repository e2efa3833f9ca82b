"""Benchmark of the block-coreset MoE FFN on GB300.

One step = one pass of the whole layer over one batch: route -> coreset ->
forward, through the C ABI of libmoeblock (moe_block_pass), replayed as a CUDA
graph with the inputs resident in HBM.  L2 is flushed between steps, outside the timed
events: a 256 MiB write, then a 256 MiB read of another buffer, so the step
starts with no dirty lines to write back.  Prints ONE JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on the host cores

Under torchrun (N > 1) every rank runs the same workload shape on its own
GPU with its own rows (weak scaling); rank 0 prints the line with the
maximum time over ranks.  On one GPU the line also carries, under
"workloads", the other full-size workloads (512 Zipf rows, 2048 rows with the
coreset on and off, 8192 rows) timed the same way in the same run.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from sparse_moe_layer_row_gb300 import workloads as W  # noqa: E402

METRIC = "MoE block-layer rows/s and expert-weight HBM GB/s (% of roofline) on 1 GB300"
DEFAULT_WORKLOAD = W.BLOCK32.name
FLUSH_BYTES = 256 << 20


def kernels_per_step(w: W.Workload) -> int:
    """This library's kernels in one step (one moe_block_pass) of the workload."""
    if w.R <= 32:  # small path: router, coreset, one-CTA scatter, gate/up, down, combine
        return 6
    tc_route = w.R >= 256 and w.E <= 256 and w.E % 16 == 0 and w.k <= 16 and w.H <= 8192
    route = 3 if tc_route else 1  # norms + tensor-core screen + exact; or the SIMT router
    return route + 1 + 3 + 3      # coreset; hist, scan, place; gate/up, down, combine


# --------------------------------------------------------------------------- helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return ws, rank, local


def rank_workload(w: W.Workload, rank: int) -> int:
    """x seed of a rank: same shape, distinct rows (weak scaling; no data exchange)."""
    return w.x_seed + 7919 * rank


def reduce_max(value: float, ws: int, device=None) -> float:
    if ws == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm_gbs=float(p["hbm_gbs"]), bf16_tflops=float(p["bf16_tflops"]),
                    bf16_tflops_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


def gemm_source_hash() -> str:
    """Hash of the GEMM kernels' code: their sources without comments and blank
    lines (a comment edit leaves recorded counters valid)."""
    h = hashlib.sha256()
    for f in ("gemm.cu", "gemm_pair.cu", "common.cuh", "kernels.cuh"):
        with open(os.path.join(ROOT, "sparse_moe_layer_row_gb300", "csrc", f)) as fh:
            for line in fh:
                code = line.split("//", 1)[0].rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per gate/up launch from a committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "gateup_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    entry = rec.get(workload)
    if not entry or entry.get("source_hash") != gemm_source_hash():
        return None
    return float(entry["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi samples (200 ms) during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
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
        if not getattr(self, "out", ""):
            return None
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def weight_bytes_per_element(qbits: int = 0) -> float:
    """Bytes per expert weight as stored: bf16, or a b-bit code plus a bf16
    scale per 32 weights."""
    return 2.0 if not qbits else qbits / 8.0 + 2.0 / W.QBLOCK


def accounting(w: W.Workload, R: int, n_core_experts: int, n_pairs: int, qbits: int = 0):
    """Algorithmic bytes and flops of one step and of one gate/up launch."""
    H, E, I, Is = w.H, w.E, w.I, w.Is
    wb = weight_bytes_per_element(qbits)
    expert_bytes = 3 * H * I * wb
    shared_bytes = 3 * H * Is * wb
    router_bytes = E * H * 2
    step_bytes = n_core_experts * expert_bytes + shared_bytes + router_bytes + 2 * R * H * 2
    step_flops = 2.0 * R * H * E + n_pairs * 6.0 * H * I + R * 6.0 * H * Is
    # gate/up launch: the touched experts' and the shared expert's gate and up
    # weights plus the rows of x, each read once (intermediates are not counted)
    gu_bytes = n_core_experts * 2 * H * I * wb + 2 * H * Is * wb + R * H * 2
    # gate/up FLOPs: two H x I products per surviving pair, two H x Is per row
    gu_flops = 4.0 * H * (n_pairs * I + R * Is)
    weight_bytes = n_core_experts * expert_bytes + shared_bytes + router_bytes
    return dict(step_bytes=step_bytes, step_flops=step_flops, gu_bytes=gu_bytes,
                gu_flops=gu_flops, weight_bytes=weight_bytes)


# --------------------------------------------------------------------------- oracle arm

def oracle_step(w: W.Workload, x_u16, wr_u16, off, bias, experts_fn, shared, nthreads):
    import oracle
    idx, wt, _, _ = oracle.route(x_u16, wr_u16, off, w.k, bias=bias, nthreads=nthreads)
    keep, core, wr, empty, _ = oracle.coreset(off, idx, wt, w.E, w.tau)
    used = oracle.surviving_experts(idx, keep, off, w.E)
    y = oracle.forward(x_u16, off, idx, wr, keep, experts_fn(used), shared, w.E,
                       nthreads=nthreads)
    return y, len(used)


def oracle_inputs(w: W.Workload, x_seed: int):
    """Inputs of the workload as numpy bf16 bit patterns (generated on a GPU when
    one is present, for speed; the generator is device-independent)."""
    import oracle  # noqa: F401
    dev = "cuda" if torch.cuda.is_available() else "cpu"

    def u16(t):
        return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)

    x = u16(W.make_x(w, dev, seed=x_seed))
    wr = u16(W.make_router(w, dev))
    sg, su, sd = (u16(t) for t in W.make_shared(w, dev))
    bias = W.zipf_bias(w, seed=x_seed)
    bias = None if bias is None else bias.numpy()
    cache = {}

    def experts_fn(used):
        need = [e for e in used if e not in cache]
        for e in need:
            cache[e] = tuple(u16(W.make_expert_slice(w, which, e, e + 1, dev)[0])
                             for which in ("gate", "up", "down"))
        return {e: cache[e] for e in used}

    return x, wr, np.asarray(w.block_offsets(), np.int32), bias, experts_fn, (sg, su, sd)


def cpu_baseline(w: W.Workload, x_seed: int, budget_s: float = 10.0, max_steps: int = 50):
    import oracle
    nthreads = oracle.default_threads()
    x, wr, off, bias, experts_fn, shared = oracle_inputs(w, x_seed)
    oracle_step(w, x, wr, off, bias, experts_fn, shared, nthreads)  # warm: experts generated
    t0 = time.perf_counter()
    n = 0
    while n < max_steps:
        oracle_step(w, x, wr, off, bias, experts_fn, shared, nthreads)
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": w.R * n / dt, "unit": "rows/s", "cores": nthreads, "kind": "oracle",
            "sample": f"{n} full steps of {w.name} ({w.R} rows; route+coreset+fp64 FFN), "
                      f"{dt:.2f} s"}


def run_reference(args, w: W.Workload):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    nthreads = oracle.default_threads()
    x, wr, off, bias, experts_fn, shared = oracle_inputs(w, rank_workload(w, 0))
    for _ in range(args.warmup):
        oracle_step(w, x, wr, off, bias, experts_fn, shared, nthreads)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(w, x, wr, off, bias, experts_fn, shared, nthreads)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = w.R * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, "CPU oracle; no GPU"),
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": nthreads, "kind": "oracle",
                         "sample": f"{args.steps} full steps of {w.name} ({w.R} rows each)"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_of(w: W.Workload, l2: str):
    return {"workload": w.name, "rows": w.R, "blocks": w.nb, "block_rows": w.block_rows[0],
            "hidden": w.H, "experts": w.E, "top_k": w.k, "intermediate": w.I,
            "shared_intermediate": w.Is, "coreset_mass": w.tau, "l2": l2,
            "parallelism": "replicas (weak scaling by rows)"}


# --------------------------------------------------------------------------- GPU arm

class StepTimer:
    """The launch stream and the L2 flush run between timed steps (a 256 MiB
    write, then a 256 MiB read of another buffer, so no dirty lines are left)."""

    def __init__(self, dev):
        self.dev = dev
        self.stream = torch.cuda.Stream(device=dev)
        self._wr = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self._rd = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self._out = torch.empty((), dtype=torch.float32, device=dev)

    def flush_l2(self, i):
        self._wr.fill_(float(i))
        torch.sum(self._rd, dim=0, out=self._out)

    def median_us(self, replay, n):
        """Median of n replays (after 3 untimed ones), each behind the flush."""
        ts = []
        with torch.cuda.stream(self.stream):
            for i in range(n + 3):
                self.flush_l2(i)
                a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a_.record(self.stream)
                replay()
                b_.record(self.stream)
                b_.synchronize()
                if i >= 3:
                    ts.append(a_.elapsed_time(b_))
        return 1e3 * statistics.median(ts)


def routing_facts(w: W.Workload, layer, live=None):
    """Experts kept and (row, expert) pairs evaluated, from the routing on the device."""
    idx = layer._topk_idx[:w.R].cpu().numpy()
    keep = layer._keep[:w.nb].cpu().numpy().view(np.uint32)
    off = np.asarray(w.block_offsets())
    used, pairs = set(), 0
    for b in range(w.nb):
        for r in range(off[b], off[b + 1]):
            if live is not None and not live[r]:
                continue
            for e in idx[r]:
                if (keep[b, e // 32] >> (e % 32)) & 1:
                    used.add(int(e))
                    pairs += 1
    return used, pairs


def measure(w: W.Workload, T, layer, steps: int, tm: StepTimer, clock_index: int, warmup: int,
            ws: int = 1):
    """One step (route -> coreset -> forward through the C ABI) as a CUDA graph,
    replayed `steps` times behind the L2 flush, CUDA events on the launch stream;
    then the forward's kernels timed by its own event records, and the three
    calls as separate graphs.  Returns the raw times and the routing facts."""
    stream, dev = tm.stream, tm.dev
    y = torch.empty(w.R, w.H, dtype=torch.bfloat16, device=dev)
    # the layer's weights and buffers (zeroed workspace, quantised codes) were
    # made on the default stream: finish that work before `stream` uses them
    torch.cuda.synchronize()

    def step():
        layer(T.x, T.block_offsets, w.tau, bias=T.bias, y=y)

    with torch.cuda.stream(stream):
        for _ in range(max(warmup, 3)):
            step()
    torch.cuda.synchronize()
    st = layer.status()
    if st["wait_timeout"] or st["bad_expert_id"]:
        raise RuntimeError(f"device status after warm-up of {w.name}: {st}")
    used, pairs = routing_facts(w, layer)

    # the step as a graph (timed); and the same step with the forward's 5 event
    # records around its kernels (the records sit between the kernels, so that
    # graph is replayed separately)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    fwd_ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    layer.plan.set_forward_events(fwd_ev)
    graph_ev = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_ev, stream=stream):
        step()
    layer.plan.set_forward_events(None)
    torch.cuda.synchronize()

    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(clock_index) as clk:
        with torch.cuda.stream(stream):
            for i in range(steps):
                tm.flush_l2(i)
                step_ev[i][0].record(stream)
                graph.replay()
                step_ev[i][1].record(stream)
            torch.cuda.synchronize()
        torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    barrier(ws)
    total_ms = reduce_max(sum(step_ms), ws, dev)
    # front: router + coreset + scatter (the kernels before the gate/up GEMM)
    kern = {"front": [], "gate_up": [], "down": [], "combine": []}
    with torch.cuda.stream(stream):
        for i in range(min(steps, 100)):
            tm.flush_l2(i)
            graph_ev.replay()
            fwd_ev[4].synchronize()   # the next replay overwrites the events
            for j, name in enumerate(kern):
                kern[name].append(fwd_ev[j].elapsed_time(fwd_ev[j + 1]))
    torch.cuda.synchronize()

    # per-phase breakdown (not the headline): the three calls as separate graphs,
    # replayed back to back behind the L2 flush so no host gap falls inside
    phase_ms = {"route": [], "coreset": [], "forward": []}
    idx_t, w_t = layer._topk_idx[:w.R], layer._topk_w[:w.R]
    keep_t, wr_t = layer._keep[:w.nb], layer._w_renorm[:w.R]
    calls = {
        "route": lambda: layer.route(T.x, T.block_offsets, T.bias),
        "coreset": lambda: layer.coreset(T.block_offsets, idx_t, w_t, w.tau),
        "forward": lambda: layer.forward(T.x, T.block_offsets, idx_t, wr_t, keep_t, y=y),
    }
    graphs = {}
    for name, fn in calls.items():
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        graphs[name] = g
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(min(steps, 50)):
            tm.flush_l2(i)
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            evs[0].record(stream)
            for j, name in enumerate(phase_ms):
                graphs[name].replay()
                evs[j + 1].record(stream)
            evs[3].synchronize()
            for j, name in enumerate(phase_ms):
                phase_ms[name].append(evs[j].elapsed_time(evs[j + 1]))
    torch.cuda.synchronize()
    return dict(total_ms=total_ms, steps=steps, kern=kern, phase_ms=phase_ms, used=used,
                pairs=pairs, clocks=clk.summary(), y=y)


def summarize(w: W.Workload, m: dict, peaks: dict, ws: int = 1, qbits: int = 0) -> dict:
    """Throughput, the gate/up kernel's roofline and the whole step's fraction."""
    from sparse_moe_layer_row_gb300 import moe_block
    acc = accounting(w, w.R, len(m["used"]), m["pairs"], qbits)
    t_step = m["total_ms"] / 1e3 / m["steps"]
    t_gu = statistics.mean(m["kern"]["gate_up"]) / 1e3
    traffic = recorded_traffic(w.name)
    # the gate/up GEMM's binding roof: the larger of its HBM time (algorithmic
    # bytes at the measured copy bandwidth) and its tensor time (bf16 FLOPs at
    # the measured burst peak); the other is reported alongside
    t_hbm = acc["gu_bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_tc = acc["gu_flops"] / (peaks["bf16_tflops"] * 1e12)
    if t_tc > t_hbm:
        achieved = acc["gu_flops"] / t_gu / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                "algorithmic_flops_per_launch": acc["gu_flops"],
                "hbm_gbs_alongside": acc["gu_bytes"] / t_gu / 1e9}
    else:
        achieved = acc["gu_bytes"] / t_gu / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"],
                "algorithmic_bytes_per_launch": acc["gu_bytes"],
                "tflops_alongside": acc["gu_flops"] / t_gu / 1e12,
                "tensor_frac_alongside": acc["gu_flops"] / t_gu / 1e12 / peaks["bf16_tflops"]}
    gu_kernel = (f"k_gemm<kGateUp, 32, 5, {qbits}> (tcgen05, {qbits}-bit experts)" if qbits
                 else "k_gemm<kGateUp, 32, 5> (tcgen05)" if w.R <= moe_block.SMALL_ROWS
                 else "k_gateup_pair (tcgen05 cta_group::2)")
    roof = {"bound": roof.pop("bound"), "kernel": gu_kernel, **roof,
            "traffic": traffic, "launch_us": t_gu * 1e6, "peak_source": peaks["source"]}
    step_frac = max(acc["step_bytes"] / (peaks["hbm_gbs"] * 1e9),
                    acc["step_flops"] / (peaks["bf16_tflops_sustained"] * 1e12)) / t_step
    return {
        "value": w.R * ws * m["steps"] / (m["total_ms"] / 1e3), "unit": "rows/s",
        "ms_per_step": m["total_ms"] / m["steps"],
        "expert_weight_gbs": acc["weight_bytes"] / t_step / 1e9,
        "step_roofline_frac": step_frac,
        "step_roofline_bound": ("hbm" if acc["step_bytes"] / (peaks["hbm_gbs"] * 1e9) >=
                                acc["step_flops"] / (peaks["bf16_tflops_sustained"] * 1e12)
                                else "tensor"),
        "roofline": roof,
        "kernel_us": {k: 1e3 * statistics.mean(v) for k, v in m["kern"].items()},
        "phase_us": {k: 1e3 * statistics.median(v) for k, v in m["phase_ms"].items()},
        "coreset": {"experts": len(m["used"]), "pairs": m["pairs"]},
        "clocks": m["clocks"],
    }


# Workloads timed in the same run next to the main one (their own JSON object,
# not the headline): the 512-row Zipf batch, 2048 rows in 32-row blocks with
# the coreset on and off, and the 8192-row prefill shape; on request, the main
# workload's layer with 8-bit and 4-bit experts (same router and inputs).
EXTRA_WORKLOADS = ("blocks16x32-zipf1.1", "rows2048-b32-tau0.9", "rows2048-b32-tau1",
                   "prefill8192-b32")
QUANT_BITS = (8, 4)


def tensors_like(we: W.Workload, base: W.Workload, T, dev, x_seed: int):
    """Inputs of workload `we`, sharing the weights of `base` when they are the same
    synthetic layer (same shapes and weight seed)."""
    same = (we.H, we.E, we.k, we.I, we.Is, we.w_seed, we.sigma_w, we.sigma_r) == \
        (base.H, base.E, base.k, base.I, base.Is, base.w_seed, base.sigma_w, base.sigma_r)
    if not same:
        return W.make_tensors(we, device=dev, x_seed=x_seed)
    bias = W.zipf_bias(we, seed=x_seed)
    return W.Tensors(W.make_x(we, dev, seed=x_seed), T.w_router, T.w_gate, T.w_up, T.w_down,
                     T.ws_gate, T.ws_up, T.ws_down, None if bias is None else bias.to(dev),
                     torch.tensor(we.block_offsets(), dtype=torch.int32, device=dev))


def run_gpu(args, w: W.Workload):
    from sparse_moe_layer_row_gb300 import moe_block

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    moe_block.load()
    x_seed = rank_workload(w, rank)
    T = W.make_tensors(w, device=dev, x_seed=x_seed)
    layer = moe_block.MoeBlockLayer(T.w_router, T.w_gate, T.w_up, T.w_down, T.ws_gate, T.ws_up,
                                    T.ws_down, k=w.k, max_rows=w.R, max_blocks=w.nb)
    tm = StepTimer(dev)
    stream = tm.stream
    m = measure(w, T, layer, args.steps, tm, local, args.warmup, ws)
    y = m["y"]
    idx_t, keep_t, wr_t = layer._topk_idx[:w.R], layer._keep[:w.nb], layer._w_renorm[:w.R]

    # live-row passes (informational): the forward on a seeded subset of the
    # rows, the others keeping their cached output
    live_us = {}
    for frac in args.live_fracs:
        live = W.live_rows(w.R, frac, seed=x_seed + 7, device=dev)
        lv = live.cpu().numpy().astype(bool)
        lused, lpairs = routing_facts(w, layer, live=lv)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            layer.forward(T.x, T.block_offsets, idx_t, wr_t, keep_t, y=y, live=live)
        torch.cuda.synchronize()
        live_us[f"{frac:g}"] = {"live_rows": int(lv.sum()), "experts": len(lused),
                                "pairs": lpairs,
                                "forward_us": tm.median_us(g.replay, min(args.steps, 50))}
    torch.cuda.synchronize()

    # several layers as one pass (informational): each layer its own weights, the
    # pass captured as one CUDA graph and replayed behind the same L2 flush
    stack_info = None
    if args.layers > 1:
        import dataclasses
        stack_layers, biases = [layer], [T.bias]
        for i in range(1, args.layers):
            wi = dataclasses.replace(w, w_seed=w.w_seed + 1000 * i)
            Ti = W.make_tensors(wi, device=dev, x_seed=x_seed)
            stack_layers.append(moe_block.MoeBlockLayer(
                Ti.w_router, Ti.w_gate, Ti.w_up, Ti.w_down, Ti.ws_gate, Ti.ws_up, Ti.ws_down,
                k=w.k, max_rows=w.R, max_blocks=w.nb))
            biases.append(Ti.bias)
        stack = moe_block.MoeStack(stack_layers)   # every layer reads the block's x
        g_stack, _ = stack.capture(T.x, T.block_offsets, w.tau, biases)
        t_pass = tm.median_us(g_stack.replay, min(args.steps, 50))
        stack_info = {"layers": args.layers, "pass_us": t_pass, "per_layer_us": t_pass / args.layers,
                      "launches_per_pass": 1}
    torch.cuda.synchronize()

    # end to end through the public API with host buffers (pinned), no graph
    x_host = T.x.cpu().pin_memory()
    off_host = T.block_offsets.cpu().pin_memory()
    y_host = torch.empty(w.R, w.H, dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty_like(T.x)
    off_dev = torch.empty_like(T.block_offsets)
    e2e_steps = max(3, min(args.steps, 200))
    with torch.cuda.stream(stream):
        for _ in range(3):
            x_dev.copy_(x_host, non_blocking=True)
            off_dev.copy_(off_host, non_blocking=True)
            y_host.copy_(layer(x_dev, off_dev, w.tau, bias=T.bias), non_blocking=True)
        torch.cuda.synchronize()
        barrier(ws)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2e_ms = 0.0
        for i in range(e2e_steps):
            tm.flush_l2(i)
            e0.record(stream)
            x_dev.copy_(x_host, non_blocking=True)
            off_dev.copy_(off_host, non_blocking=True)
            y_host.copy_(layer(x_dev, off_dev, w.tau, bias=T.bias), non_blocking=True)
            e1.record(stream)
            e1.synchronize()
            e2e_ms += e0.elapsed_time(e1)
    e2e_ms = reduce_max(e2e_ms, ws, dev)
    h2d = x_host.numel() * 2 + off_host.numel() * 4
    d2h = y_host.numel() * 2

    if rank != 0:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0

    peaks = load_peaks()
    summ = summarize(w, m, peaks, ws)
    line = {
        "metric": METRIC, "value": summ["value"], "unit": "rows/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": summ["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,s) bf16 inputs and weights; no trained weights)",
        "config": config_of(w, f"flushed between steps ({FLUSH_BYTES >> 20} MiB write, then "
                               f"{FLUSH_BYTES >> 20} MiB read of another buffer)"),
        **{k: summ[k] for k in ("expert_weight_gbs", "step_roofline_frac", "roofline",
                                "kernel_us", "phase_us", "coreset")},
        "gpu_launches": kernels_per_step(w) * args.steps,
        "clocks": summ["clocks"],
        "e2e": {"value": w.R * ws * e2e_steps / (e2e_ms / 1e3), "unit": "rows/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
    }
    if live_us:
        line["live_pass"] = live_us
    if stack_info:
        line["stack"] = stack_info
    # the other full-size workloads, timed in the same run (1 GPU only)
    if ws == 1 and not args.no_extra_workloads:
        extra = {}
        for name in (EXTRA_WORKLOADS if args.extras is None else args.extras):
            we = W.BY_NAME[name]
            if we.name == w.name:
                continue
            Te = tensors_like(we, w, T, dev, rank_workload(we, rank))
            le = moe_block.MoeBlockLayer(Te.w_router, Te.w_gate, Te.w_up, Te.w_down, Te.ws_gate,
                                         Te.ws_up, Te.ws_down, k=we.k, max_rows=we.R,
                                         max_blocks=we.nb)
            me = measure(we, Te, le, args.extra_steps, tm, local, args.warmup)
            se = summarize(we, me, peaks)
            se["gpu_launches_per_step"] = kernels_per_step(we)
            se["config"] = {"rows": we.R, "blocks": we.nb, "block_rows": we.block_rows[0],
                            "coreset_mass": we.tau, "zipf_bias": we.zipf_s or None,
                            "steps": args.extra_steps}
            extra[name] = se
            del le, Te, me
            torch.cuda.empty_cache()
        for bits in (QUANT_BITS if args.quant_workloads else ()):
            qe = W.quantize_experts(T, bits)
            lq = moe_block.MoeBlockLayer.quantized(T.w_router, qe, k=w.k, max_rows=w.R,
                                                   max_blocks=w.nb)
            mq = measure(w, T, lq, args.extra_steps, tm, local, args.warmup)
            sq = summarize(w, mq, peaks, qbits=bits)
            sq["gpu_launches_per_step"] = kernels_per_step(w)
            sq["config"] = {"rows": w.R, "blocks": w.nb, "block_rows": w.block_rows[0],
                            "coreset_mass": w.tau, "expert_bits": bits,
                            "expert_bytes_per_weight": weight_bytes_per_element(bits),
                            "steps": args.extra_steps}
            extra[f"{w.name}-q{bits}"] = sq
            del lq, qe, mq
            torch.cuda.empty_cache()
        line["workloads"] = extra
    if ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, x_seed, budget_s=args.cpu_budget)
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.BY_NAME))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quant-workloads", action="store_true",
                    help="also time the main workload's layer with 8-bit and 4-bit experts")
    ap.add_argument("--no-extra-workloads", action="store_true",
                    help="skip the other full-size workloads (reported under workloads)")
    ap.add_argument("--extras", type=lambda v: [t for t in v.split(",") if t and t != "none"],
                    default=None,
                    help="comma-separated names of the other full-size workloads to time "
                         "(default: all of them; 'none': none, e.g. with --quant-workloads only)")
    ap.add_argument("--extra-steps", type=int, default=30,
                    help="timed steps of each extra workload")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--layers", type=int, default=1,
                    help="also time a pass over this many layers (own weights each) captured "
                         "as one CUDA graph, reported under stack")
    ap.add_argument("--live-fracs", type=lambda v: [float(t) for t in v.split(",") if t],
                    default=[], help="also time live-row passes with these live fractions "
                                     "(comma separated), reported under live_pass")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    for name in args.extras or ():
        if name not in W.BY_NAME:
            ap.error(f"--extras: unknown workload {name!r}")
    w = W.BY_NAME[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_gpu(args, w)


if __name__ == "__main__":
    sys.exit(main())
