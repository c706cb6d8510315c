"""Benchmark of the MoE-layer forward pass on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--only]
                    [--impl ours|reference] [--no-cpu-baseline]

A step is one pass of the whole layer (moe_forward: route -> permute ->
grouped FFN -> combine) over one batch of seeded synthetic tokens, through
the C ABI, replayed from one CUDA graph.  The headline workload is the largest
one a single GPU holds among the problem statement's: the Mixtral-shaped layer
(T=8192, 4096 -> 14336 -> 4096, E=8, top-2 on logits, bf16).  Every other
workload is measured in the same run and printed as a sub-record under
"workloads" (--only skips them).  Prints one JSON line (rank 0).

Timing: W untimed warm-up steps; then K steps bracketed by a barrier and a
device synchronise.  L2 is flushed (a 256 MB write) before every step, outside
the per-step CUDA events whose sum gives the device time.  The grouped FFN
(the dominant kernel pair, the roofline figure), routing, permute and the
combine are then timed the same way from graphs of their own entry points on
the same stream.  The
end-to-end figure repeats the step through moe_forward with the tokens copied
in from pinned host memory and the output (and aux) copied back every step.

N > 1 (torchrun): every rank runs an independent replica of the layer on its
own GPU (the path has no exchange step); value = all ranks' tokens / the
slowest rank's time.

--impl reference times the CPU oracle (the plain float64 restatement of the
pages) on the host cores, on a bounded token sample of the same workload,
drawn from the same seeded generator.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "mixtral_top2"
# the other workloads, measured in the same run as sub-records of the line
SUB_WORKLOADS = ["switch_top1_cap", "deepseek_v3_top8", "decode_zipf_top2", "tiny_fp32_top2",
                 "switch_expert_choice", "mixtral_swiglu_top2", "switch_top1_cap_mxfp8",
                 "decode_zipf_top2_mxfp8", "mixtral_top2_mxfp8"]
HEADLINE_TIMED_MS = 1500.0     # device time of the headline's timed region (auto steps)
SUB_TIMED_MS = 600.0           # the same for each sub-record
METRIC = "MoE-layer fwd tokens/s"
L2_FLUSH_BYTES = 256 << 20
PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
PROFILE_DIR = os.path.join(ROOT, "profiles")
GEMM_SOURCES = ["gemm_tc.cuh", "gemm_tc2.cuh", "gemm_mx2.cuh", "ptx_sm100.cuh", "groups.cuh",
                "mxfp8.cuh"]
# oracle rows (tokens whose FFN output the CPU baseline computes) per workload
CPU_SAMPLE_ROWS = {"tiny_fp32_top2": 256, "switch_top1_cap": 4096, "mixtral_top2": 128,
                   "deepseek_v3_top8": 16, "decode_zipf_top2": 64, "mixtral_swiglu_top2": 128,
                   "switch_expert_choice": 4096}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0,
                    help="timed steps; 0 = enough for >= 1.5 s of timed device work")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--dispatch-only", action="store_true",
                    help="run moe_route, moe_permute and moe_combine three times on the "
                         "workload's token batch (no expert weights) and exit: the command "
                         "for per-kernel ncu captures of those steps at full size")
    ap.add_argument("--forward-only", action="store_true",
                    help="run moe_forward W + K times on the workload (eager, no graphs) and "
                         "exit: the command behind the per-kernel launch lists and captures")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", action="store_true",
                    help="measure the named workload alone (no sub-records)")
    ap.add_argument("--cpu-rows", type=int, default=None)
    return ap.parse_args()


def load_peaks():
    if os.path.exists(PEAKS_PATH):
        with open(PEAKS_PATH) as fh:
            p = json.load(fh)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def gemm_source_hash() -> str:
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        with open(os.path.join(ROOT, "sparse_mixture_experts_52_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per grouped-FFN call from the committed ncu summary, if it was
    taken on the current kernel source (else None)."""
    path = os.path.join(PROFILE_DIR, f"gffn_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_hash = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_gffn_call:\s*([0-9.eE+]+)", text)
    if not m_hash or not m_bytes or m_hash.group(1) != gemm_source_hash():
        return None
    return float(m_bytes.group(1))


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi every 100 ms in the background; keeps the samples whose
    arrival falls inside [begin(), end()]."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        import threading
        self.lines, self.t0, self.t1, self.proc = [], None, None, None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line))

    def begin(self):
        self.t0 = time.perf_counter()

    def end(self):
        self.t1 = time.perf_counter()

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
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, line in self.lines:
            if self.t0 is None or not (self.t0 <= t <= self.t1 + 0.1):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ our arm
def mx_experts(cfg) -> bool:
    return cfg.get("experts", "dense") == "mxfp8"


def algorithmic_ffn(cfg, kept, elem):
    """Bytes and FLOPs the grouped FFN must move / do at least, for this batch:
    the active experts' weights once, the rows in, the hidden activation out
    and back, the expert outputs out.  MX FP8 operands take 1 + 1/32 bytes an
    element (codes and block scales); the expert outputs stay in the layer
    dtype."""
    d, F, S, T = cfg["d_model"], cfg["d_ff"], cfg.get("n_shared", 0), cfg["T"]
    F1 = 2 * F if cfg.get("act", "gelu") == "swiglu" else F   # SwiGLU: gate and up rows
    n_a = int(sum(kept))
    active = int(sum(1 for v in kept if v > 0))
    op = 33 / 32 if mx_experts(cfg) else elem
    weights = (active + S) * (F1 + F) * d * op
    acts = (n_a + S * T) * ((d + F + F) * op + d * elem)
    flops = 2 * (n_a + S * T) * d * (F1 + F)
    return int(weights + acts), flops, n_a, active


def rpc_bytes(cfg, n_a, elem) -> int:
    """Algorithmic bytes of routing + permute + combine: x read by the router,
    W_g, the indices and weights; x read and N_a rows written by the permute;
    N_a rows read and T rows written by the combine (shared-expert rows, when
    present, read once more)."""
    T, d, E, k, S = cfg["T"], cfg["d_model"], cfg["E"], cfg["k"], cfg.get("n_shared", 0)
    route = T * d * elem + d * E * elem + T * k * 8
    permute = T * d * elem + n_a * d * elem
    combine = n_a * d * elem + T * d * elem + S * T * d * elem
    return route + permute + combine


def kernel_launches_per_step(cfg) -> int:
    """Kernels one moe_forward enqueues (see moe_api.cu).
    Top-k routing: the routing grid, with the W_g transpose ahead of it for
    bf16 layers with E > 64 or T > 512 - then either the tensor-core router
    with the gating in its epilogue (E <= 16) or the router GEMM plus a gating
    grid - the permute, the up- and down-projections, and the combine unless a
    bf16 top-1 layer without shared experts folds it into the down-projection.
    Expert Choice: (W_g transpose and router GEMM for bf16), the per-token
    scores, the per-expert selection, the row gather, the two projections and
    the combine."""
    bf16 = cfg["dtype"] == "bf16"
    if cfg.get("route") == "expert_choice":
        return (2 if bf16 else 0) + 2 + 1 + 2 + 1
    tc_router = bf16 and (cfg["E"] > 64 or cfg["T"] > 512)
    fused_router = (tc_router and cfg["E"] <= 16
                    and ((cfg["T"] + 127) // 128) * (cfg["E"] + 1) <= 257 * 512)
    route = 2 if fused_router else (3 if tc_router else 1)
    fused = bf16 and cfg["k"] == 1 and cfg.get("n_shared", 0) == 0
    return route + 1 + 2 + (0 if fused else 1)


def _timed_graph_loop(graph, flush, stream, steps, before=None):
    """Replays `graph` `steps` times, flushing L2 before each replay outside the
    replay's event pair; returns the per-replay device times in ms."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        if before is not None:
            before()
        ev[i][0].record(stream)
        graph.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def run_dispatch_only(args):
    """Routing, dispatch and combine of one workload's token batch, three
    times, through the step entry points; no expert weights are allocated
    (the combine sums seeded rows standing in for the expert outputs)."""
    import torch
    from sparse_mixture_experts_52_b300 import moe, synth

    cfg = synth.workload(args.workload)
    if moe.expert_choice(cfg):
        raise SystemExit("--dispatch-only covers the top-k routing forms")
    T, d, E, k, S = cfg["T"], cfg["d_model"], cfg["E"], cfg["k"], cfg.get("n_shared", 0)
    dt = moe.TORCH_DTYPES[cfg["dtype"]]
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    rnd = lambda shape, std=1.0: (torch.randn(shape, generator=g, device="cuda") * std).to(dt)
    x, w_g = rnd((T, d)), rnd((d, E), d ** -0.5)
    sb = (torch.randn((E,), generator=g, device="cuda") * cfg.get("select_bias_std", 0.0)
          if cfg["route"] == "biased_softmax" else None)
    ws = moe.new_workspace(cfg, "cuda")
    z = lambda s, t: torch.empty(s, dtype=t, device="cuda")
    idx, w = z((T, k), torch.int32), z((T, k), torch.float32)
    f, P, aux = z((E,), torch.float32), z((E,), torch.float32), z((1,), torch.float32)
    counts, kept, offs = z((E,), torch.int32), z((E,), torch.int32), z((E + 1,), torch.int32)
    pt, so, xp = z((T * k,), torch.int32), z((T * k,), torch.int32), z((T * k, d), dt)
    y, ys, out = rnd((T * k, d)), (rnd((S, T, d)) if S else None), z((T, d), dt)
    for _ in range(3):
        moe.route(cfg, x, w_g, idx, w, f, P, aux, ws, select_bias=sb)
        moe.permute(cfg, x, idx, counts, kept, offs, pt, so, xp, ws)
        moe.combine(cfg, y, so, w, out, y_shared=ys)
    torch.cuda.synchronize()
    moe.check_status(ws)


def run_forward_only(args):
    """moe_forward on one workload, W + K times in eager mode, then exit."""
    import torch
    from sparse_mixture_experts_52_b300 import moe, synth

    cfg = synth.workload(args.workload)
    inp = draw_inputs(cfg, cfg.get("seed", 0), torch.device("cuda", 0))
    layer = moe.MoELayer(cfg, inp, device="cuda")
    for _ in range(max(1, args.warmup + args.steps)):
        layer(inp["x"])
    torch.cuda.synchronize()
    moe.check_status(layer.ws)


def max_over_ranks(values, world, device):
    """Element-wise maximum of per-rank timings over the process group (the
    slowest replica sets the whole-job time); the values themselves at N = 1."""
    import torch
    if world <= 1:
        return [float(v) for v in values]
    t = torch.tensor(values, dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def whole_job_tokens_per_s(T, world, steps, slowest_ms):
    """Weak scaling: every replica processes T tokens a step, so the job
    processes world * T * steps tokens in the slowest replica's time."""
    return world * T * steps / (slowest_ms / 1e3)


def line_config(cfg, world) -> dict:
    """The `config` object of a JSON line: the workload as the layer's problem
    statement names it.  Both arms print the same dict for the same workload."""
    return {"workload": cfg["name"], "T": cfg["T"], "d_model": cfg["d_model"],
            "d_ff": cfg["d_ff"], "E": cfg["E"], "k": cfg["k"], "act": cfg.get("act", "gelu"),
            "n_shared": cfg.get("n_shared", 0), "capacity_factor": cfg["capacity_factor"],
            "route": cfg["route"], "dtype": cfg["dtype"],
            "experts": cfg.get("experts", "dense"), "parallelism": f"replicas x{world}",
            "l2": "flushed (256 MB write) before every step, outside the step events"}


def draw_inputs(cfg, seed, device):
    """The seeded inputs of one workload.  Both arms draw them with the same
    generator on the GPU when there is one (the reference arm then copies them
    to the host), so they route the same numbers."""
    import torch
    from sparse_mixture_experts_52_b300 import synth
    if device is None:
        device = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    return synth.make_inputs(cfg, device=device, seed=seed)


def measure(args, cfg, rank, world, local_rank, steps, timed_ms, cpu_leg):
    """Times one workload on this rank's GPU: the whole-layer step (a CUDA
    graph of moe_forward), the grouped FFN, routing, permute and combine each
    in a graph of their own, and the end-to-end step through the public API
    with host buffers.  Returns the raw figures (max over ranks)."""
    import torch
    from sparse_mixture_experts_52_b300 import moe

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    inp = draw_inputs(cfg, cfg.get("seed", 0) + rank, dev)
    T, d, E, k, S = cfg["T"], cfg["d_model"], cfg["E"], cfg["k"], cfg.get("n_shared", 0)
    dt = moe.TORCH_DTYPES[cfg["dtype"]]
    elem = 2 if cfg["dtype"] == "bf16" else 4
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    # ---- the step: moe_forward on device-resident tokens, one CUDA graph
    layer = moe.MoELayer(cfg, inp, device=dev)
    layer(inp["x"])                        # eager warm-up: kernel attributes, tensor maps
    torch.cuda.synchronize(dev)
    moe.check_status(layer.ws)
    g_fwd = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_fwd):
        layer(inp["x"])

    # ---- the dominant kernel pair (grouped FFN), routing, permute and the
    # combine through their own entry points, each in its own graph
    z = lambda shape, t: torch.empty(shape, dtype=t, device=dev)
    f32 = torch.float32
    ec = moe.expert_choice(cfg)
    R = moe.routed_rows(cfg)
    o = dict(counts=z((E,), torch.int32), kept=z((E,), torch.int32),
             offsets=z((E + 1,), torch.int32), perm_token=z((T * k,), torch.int32),
             slot_of=z((T * k,), torch.int32), x_perm=z((R, d), dt),
             y_perm=z((R, d), dt), out=z((T, d), dt))
    y_sh = z((S, T, d), dt) if S else None
    ws2 = moe.new_workspace(cfg, dev)
    r_stats = dict(f=z((E,), f32), P=z((E,), f32), aux=z((1,), f32))
    if ec:
        C = moe.expert_capacity(cfg)
        o["ec_slot"] = z((E, T), torch.int32)
        r_sel = (z((E, C), torch.int32), z((E, C), f32), o["ec_slot"])

        def part_route():
            moe.route_expert_choice(cfg, inp["x"], inp["w_g"], *r_sel, r_stats["f"],
                                    r_stats["P"], r_stats["aux"], ws2,
                                    logit_bias=inp.get("logit_bias"))

        def part_permute():
            moe.permute_expert_choice(cfg, inp["x"], r_sel[0], o["offsets"], o["x_perm"])
        o["kept"].fill_(C)
    else:
        r_sel = (z((T, k), torch.int32), z((T, k), f32))

        def part_route():
            moe.route(cfg, inp["x"], inp["w_g"], *r_sel, r_stats["f"], r_stats["P"],
                      r_stats["aux"], ws2, logit_bias=inp.get("logit_bias"),
                      select_bias=inp.get("select_bias"))

        def part_permute():
            moe.permute(cfg, inp["x"], r_sel[0], o["counts"], o["kept"], o["offsets"],
                        o["perm_token"], o["slot_of"], o["x_perm"], ws2)

    def part_ffn():   # the layer's weights: packed MX FP8 buffers for MX experts
        moe.grouped_ffn(cfg, o["x_perm"], o["offsets"], layer.w["w1"], layer.w["w2"],
                        o["y_perm"], ws2, b1=inp.get("b1"), b2=inp.get("b2"), x=inp["x"],
                        ws1=inp.get("ws1"),
                        wsb1=inp.get("wsb1"), ws2=inp.get("ws2"), wsb2=inp.get("wsb2"),
                        y_shared=y_sh)

    def part_combine():
        if ec:
            moe.combine_expert_choice(cfg, o["y_perm"], o["ec_slot"], r_sel[1], o["out"],
                                      y_shared=y_sh)
        else:
            moe.combine(cfg, o["y_perm"], o["slot_of"], r_sel[1], o["out"], y_shared=y_sh)

    part_route()
    part_permute()
    part_ffn()
    part_combine()
    torch.cuda.synchronize(dev)
    moe.check_status(ws2)
    kept = o["kept"].cpu().tolist()
    byt, flops, n_a, active = algorithmic_ffn(cfg, kept, elem)
    g_route, g_perm = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    g_ffn, g_comb = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    g_chain = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_route):
        part_route()
    with torch.cuda.graph(g_perm):
        part_permute()
    with torch.cuda.graph(g_ffn):
        part_ffn()
    with torch.cuda.graph(g_comb):
        part_combine()
    with torch.cuda.graph(g_chain):   # the three dispatch-side calls back to back
        part_route()
        part_permute()
        part_combine()

    warm = max(3, args.warmup)
    w_ms = _timed_graph_loop(g_fwd, flush, stream, warm)
    moe.check_status(layer.ws)
    if steps <= 0:
        t_step = max(min(w_ms), 1e-3)
        steps = int(min(20000, max(20, math.ceil(timed_ms / t_step))))

    sampler = ClockSampler(local_rank)
    time.sleep(0.5)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.perf_counter()
    sampler.begin()
    step_ms = _timed_graph_loop(g_fwd, flush, stream, steps)
    sampler.end()
    t_wall = time.perf_counter() - t_wall0
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    moe.check_status(layer.ws)
    dev_ms = sum(step_ms)

    n_part = max(20, steps // 4)
    _timed_graph_loop(g_ffn, flush, stream, 3)
    ffn_ms = statistics.fmean(_timed_graph_loop(g_ffn, flush, stream, n_part))
    cb_ms = statistics.fmean(_timed_graph_loop(g_comb, flush, stream, n_part))
    ro_ms = statistics.fmean(_timed_graph_loop(g_route, flush, stream, n_part))
    pe_ms = statistics.fmean(_timed_graph_loop(g_perm, flush, stream, n_part))
    ch_ms = statistics.fmean(_timed_graph_loop(g_chain, flush, stream, n_part))
    moe.check_status(ws2)
    del g_route, g_perm, g_ffn, g_comb, g_chain, o, ws2, y_sh, r_sel, r_stats

    # ---- end to end through the public API, host buffers: StreamedMoELayer
    # (graphed moe_forward, the copy-in of step i+1 and the copy-out of step
    # i-1 overlapping step i on their own streams); every step copies x in from
    # pinned host memory and out and aux back
    x_host = inp["x"].cpu().pin_memory()
    out_host = torch.empty((T, d), dtype=dt).pin_memory()
    aux_host = torch.empty((1,), dtype=torch.float32).pin_memory()
    slayer = moe.StreamedMoELayer(cfg, inp, device=dev)
    for _ in range(warm):
        slayer.submit(x_host, out_host, aux_host)
    slayer.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    e0.record(slayer.s_in)       # before the first copy-in (the other streams follow it)
    for _ in range(steps):
        slayer.submit(x_host, out_host, aux_host)
    e1.record(slayer.s_out)      # after the last copy-out
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1)
    slayer.synchronize()
    del slayer

    # ---- max over ranks
    dev_ms, e2e_ms, ffn_ms, ro_ms, pe_ms, cb_ms, ch_ms = max_over_ranks(
        [dev_ms, e2e_ms, ffn_ms, ro_ms, pe_ms, cb_ms, ch_ms], world, dev)

    res = dict(cfg=cfg, steps=steps, warmup=warm, dev_ms=dev_ms, e2e_ms=e2e_ms,
               ffn_ms=ffn_ms, ro_ms=ro_ms, pe_ms=pe_ms, cb_ms=cb_ms, ch_ms=ch_ms,
               rpc_bytes=rpc_bytes(cfg, n_a, elem), bytes=byt, flops=flops,
               n_a=n_a, active=active, clocks=clocks, wall_s=t_wall,
               counts=layer.counts.cpu().tolist(), aux=float(layer.aux.cpu()[0]),
               h2d=x_host.numel() * x_host.element_size(),
               d2h=out_host.numel() * out_host.element_size() + 4)
    del layer, g_fwd, x_host, out_host, aux_host, flush
    if cpu_leg and rank == 0 and world == 1:
        res["cpu"] = cpu_baseline(cfg, inp, args)
    del inp
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return res


def _oracle_seconds(cfg, host, rows):
    from oracle import compare
    t0 = time.perf_counter()
    compare.run_oracle(cfg, host, rows=rows)
    return time.perf_counter() - t0


def host_cores() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


def cpu_sample(cfg, args):
    """Rows (tokens) whose expert FFNs the timed oracle computes, and the
    description of that sample."""
    import numpy as np
    rows_n = min(args.cpu_rows or CPU_SAMPLE_ROWS.get(cfg["name"], 256), cfg["T"])
    text = (f"float64 numpy oracle: routing, statistics and dispatch of all {cfg['T']} "
            f"tokens, expert FFNs of the first {rows_n} tokens; value = {rows_n} tokens / "
            f"wall time")
    return np.arange(rows_n), text


class BlasThreads:
    """Sets the thread count of the BLAS library numpy loaded, through its own
    set/get entry points (OpenBLAS builds export them under a few names), for
    the duration of a `with` block.  `available` is False when no such library
    or entry point is found."""
    NAMES = [("scipy_openblas_set_num_threads64_", "scipy_openblas_get_num_threads64_"),
             ("openblas_set_num_threads64_", "openblas_get_num_threads64_"),
             ("openblas_set_num_threads", "openblas_get_num_threads")]

    def __init__(self, n: int):
        import ctypes
        import numpy  # noqa: F401  (loads its BLAS)
        self.n, self.set, self.get, self.old = n, None, None, None
        paths = []
        try:
            with open("/proc/self/maps") as fh:
                for line in fh:
                    p = line.split()[-1]
                    name = os.path.basename(p)
                    if "openblas" in name and ".so" in name and p not in paths:
                        paths.append(p)
        except OSError:
            pass
        for p in paths:
            try:
                lib = ctypes.CDLL(p)
            except OSError:
                continue
            for s_name, g_name in self.NAMES:
                if hasattr(lib, s_name) and hasattr(lib, g_name):
                    self.set, self.get = getattr(lib, s_name), getattr(lib, g_name)
                    self.set.argtypes, self.get.restype = [ctypes.c_int], ctypes.c_int
                    return

    @property
    def available(self) -> bool:
        return self.set is not None

    def __enter__(self):
        if self.available:
            self.old = int(self.get())
            self.set(int(self.n))
        return self

    def __exit__(self, *exc):
        if self.available and self.old is not None:
            self.set(self.old)
        return False


def cpu_baseline(cfg, inp, args):
    """The oracle as it stands, on the host cores, on a bounded token sample:
    once with every core this process may run on (BLAS threads = the affinity
    mask) and once single-threaded.  `value` is the all-cores figure."""
    import torch
    rows, text = cpu_sample(cfg, args)
    host = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    cores = host_cores()
    why = None
    runs = {}
    for n in (cores, 1):
        ctl = BlasThreads(n)
        if not ctl.available:      # no thread control: one run at the library's default
            runs[n] = _oracle_seconds(cfg, host, rows)
            why = "no BLAS thread-count entry point found"
            break
        with ctl:
            runs[n] = _oracle_seconds(cfg, host, rows)
    out = {"value": len(rows) / runs[cores], "unit": "tokens/s", "cores": cores,
           "kind": "oracle", "seconds": runs[cores], "sample": text}
    if 1 in runs and cores != 1:
        out["single_thread"] = {"value": len(rows) / runs[1], "unit": "tokens/s", "cores": 1,
                                "seconds": runs[1]}
    elif why:
        out["single_thread"] = {"unavailable": why}
    return out


def record(res, world, peaks, peak_src) -> dict:
    """The measured figures of one workload as JSON fields."""
    cfg = res["cfg"]
    T, steps = cfg["T"], res["steps"]
    ms = res["dev_ms"] / steps
    tokens_s = whole_job_tokens_per_s(T, world, steps, res["dev_ms"])
    ffn_s = res["ffn_ms"] / 1e3
    gbs = res["bytes"] / ffn_s / 1e9
    tfl = res["flops"] / ffn_s / 1e12
    t_hbm = res["bytes"] / (peaks["hbm_gbs"] * 1e9)
    # back-to-back steps for more than 200 ms run under the power cap: their tensor fraction is
    # taken against the sustained peak; the burst (dense) peak is reported beside it
    long_region = res["dev_ms"] > 200.0
    # MX FP8 contractions: the measured bf16 peak times the nominal fp8 / bf16
    # ratio of the tensor cores (4.5 / 2.25 PFLOP/s dense)
    ratio = 2.0 if mx_experts(cfg) else 1.0
    tc_dense = peaks["bf16_tflops"] * ratio
    tc_peak = (peaks["bf16_tflops_sustained"] if long_region else peaks["bf16_tflops"]) * ratio
    t_tc = res["flops"] / (tc_peak * 1e12)
    if cfg["dtype"] == "bf16" and t_tc > t_hbm:
        roof = {"bound": "tensor", "achieved": round(tfl, 2), "peak": tc_peak,
                "unit": "TFLOP/s", "frac": round(tfl / tc_peak, 4),
                "frac_dense": round(tfl / tc_dense, 4)}
    else:
        roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4)}
    roof["traffic"] = profiled_traffic(cfg["name"])
    roof["kernel"] = "grouped FFN (tcgen05 up-projection + activation and down-projection)"
    sustained = long_region and roof["unit"] == "TFLOP/s"
    roof["peak_source"] = (f"{peak_src} ({'sustained' if sustained else 'burst'})" +
                           (", bf16 x 2 for fp8" if ratio != 1.0 and roof["unit"] == "TFLOP/s" else ""))
    roof["algorithmic_bytes"] = res["bytes"]
    roof["algorithmic_flops"] = res["flops"]
    roof["ms_per_launch"] = round(res["ffn_ms"], 4)
    e2e_val = whole_job_tokens_per_s(T, world, steps, res["e2e_ms"])
    rpc_ms = res["ch_ms"]
    rpc_gbs = res["rpc_bytes"] / (rpc_ms / 1e3) / 1e9
    rpc_sep_ms = res["ro_ms"] + res["pe_ms"] + res["cb_ms"]
    counts = res["counts"]
    mean_count = max(sum(counts) / len(counts), 1e-30)
    return {
        "value": round(tokens_s, 1), "unit": "tokens/s", "steps": steps,
        "warmup": res["warmup"], "ms_per_step": round(ms, 4),
        "dtype": "mxfp8" if mx_experts(cfg) else cfg["dtype"],
        "config": line_config(cfg, world),
        "roofline": roof,
        "grouped_ffn": {"tflops": round(tfl, 2), "gbs": round(gbs, 1),
                        "tensor_frac": round(tfl / tc_peak, 4),
                        "tensor_frac_dense": round(tfl / tc_dense, 4),
                        "hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
                        "rows": res["n_a"], "active_experts": res["active"]},
        "routing_stats": {"aux": res["aux"], "max_count": max(counts),
                          "min_count": min(counts),
                          "imbalance_ratio": round(max(counts) / mean_count, 3)},
        "e2e": {"value": round(e2e_val, 1), "unit": "tokens/s", "h2d_bytes_per_step": res["h2d"],
                "d2h_bytes_per_step": res["d2h"],
                "api": "StreamedMoELayer (graphed moe_forward; copy-in of step i+1 and copy-out of step i-1 overlap step i), pinned host x in, out+aux back every step"},
        "parts_ms": {"route": round(res["ro_ms"], 4), "permute": round(res["pe_ms"], 4),
                     "grouped_ffn": round(res["ffn_ms"], 4), "combine": round(res["cb_ms"], 4)},
        "route_permute_combine": {
            "ms": round(rpc_ms, 4), "algorithmic_bytes": res["rpc_bytes"],
            "achieved": round(rpc_gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(rpc_gbs / peaks["hbm_gbs"], 4),
            "ms_separate_graphs": round(rpc_sep_ms, 4),
            "api": "moe_route, moe_permute, moe_combine back to back in one CUDA graph, L2 "
                   "flushed before it (the combine reads expert outputs of an earlier grouped "
                   "FFN call); ms_separate_graphs: the three calls each in a graph of its own, "
                   "each after a flush (parts_ms)"},
        "gpu_launches": kernel_launches_per_step(cfg) * steps,
        "clocks": res["clocks"],
        "wall_s_timed": round(res["wall_s"], 3),
    }


def run_ours(args, rank, world, local_rank) -> dict:
    """The headline workload, then (unless --only) every other workload as a
    sub-record of the same line."""
    from sparse_mixture_experts_52_b300 import synth

    peaks, peak_src = load_peaks()
    cfg = synth.workload(args.workload)
    res = measure(args, cfg, rank, world, local_rank, args.steps, HEADLINE_TIMED_MS,
                  cpu_leg=not args.no_cpu_baseline)
    rec = record(res, world, peaks, peak_src)
    line = {"metric": METRIC, "value": rec["value"], "unit": "tokens/s", "n_gpus": world,
            "steps": rec["steps"], "warmup": rec["warmup"], "ms_per_step": rec["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": rec["dtype"], "data": "synthetic (seeded: x~N(0,1), weights~N(0,1/fan_in))"}
    line.update({k: v for k, v in rec.items() if k not in line})
    if "cpu" in res:
        line["cpu_baseline"] = res["cpu"]
    if not args.only:
        subs = {}
        for name in SUB_WORKLOADS:
            if name == cfg["name"]:
                continue
            r = measure(args, synth.workload(name), rank, world, local_rank, 0, SUB_TIMED_MS,
                        cpu_leg=False)
            subs[name] = record(r, world, peaks, peak_src)
        line["workloads"] = subs
    return line


# ------------------------------------------------------------------ reference arm
def run_reference(args, rank, world):
    """The oracle timed as it stands on the host cores (rank 0 only), on the
    same config and the same seeded inputs as our arm."""
    if rank != 0:
        return
    import torch
    from sparse_mixture_experts_52_b300 import synth

    cfg = synth.workload(args.workload)
    inp = draw_inputs(cfg, cfg.get("seed", 0), None)
    host = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    del inp
    rows, text = cpu_sample(cfg, args)
    samples = []
    for i in range(args.warmup + args.steps):
        t = _oracle_seconds(cfg, host, rows)
        if i >= args.warmup:
            samples.append(t)
    t = sum(samples)
    value = len(rows) * max(args.steps, 1) / max(t, 1e-12)
    line = {"metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * t / max(args.steps, 1), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded: x~N(0,1), weights~N(0,1/fan_in))",
            "config": line_config(cfg, world),
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": host_cores(),
                             "kind": "oracle", "sample": text},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.dispatch_only:
        run_dispatch_only(args)
        return
    if args.forward_only:
        run_forward_only(args)
        return
    import torch
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        line = run_ours(args, rank, world, local_rank)
        if rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
