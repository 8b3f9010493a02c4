"""Benchmark of the INT4-weight / rotated-INT4-KV decode block on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

One step = one ft_decode_block call (prep, QKV, attention with the new token's
cache write, O, gate/up + SwiGLU, down) over one batch of seeded synthetic
inputs of the workload's shape (default: Llama-3-8B layer shape, batch 1,
context 1024).  The timed region replays a CUDA graph of R consecutive steps
over R distinct replicas of weights + KV cache + workspace, R chosen so the
replicas together are >= 4x the L2 size (each step's inputs are cold in L2).
Rank 0 prints one JSON line.  Under torchrun (N > 1) every rank runs its own
replica on its own GPU (the path has no cross-GPU exchange: replicas only) and
the reported time is the maximum over ranks.

--impl reference times the CPU oracle (the reference implementation of this
build) on the same workload, on the host cores, one bounded sample per step.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np

METRIC = "decode-block µs/step and achieved HBM GB/s (% of GB300 roofline), batch 1–32"
DEFAULT_WORKLOAD = "8b_b1_ctx1024"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------- helpers
def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f)
    return {}


def hbm_peak() -> tuple[float, str]:
    pk = measured_peaks()
    if "hbm_gbs" in pk:
        return float(pk["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def algorithmic_bytes(shape, B: int, ctx: int, weight_format: int = 0) -> dict:
    """Minimum bytes one step must move: the codes (INT4, or E4M3 with
    weight_format 1) + BF16 group scales of every weight, the KV history read
    (codes + scales) and the new entry written, and the BF16 activations in and
    out."""
    import int4_weight_kv_gb300 as ft
    cfg = ft.cfg_from_shape(shape)
    cfg.weight_format = weight_format
    w = {r: ft.ft_packed_weight_bytes(cfg, r) for r in ft.ROLES}
    kv_tok = shape.n_kv * 2 * (shape.head_dim // 2 + 2 * (shape.head_dim // shape.kvg))
    kv = B * ctx * kv_tok + B * kv_tok
    act = B * shape.hidden * 2 * 2
    return {"weights": sum(w.values()), "per_role": w, "kv": kv, "act": act,
            "total": sum(w.values()) + kv + act}


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the GPU works."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------- multi-rank helpers
def dist_env() -> tuple[int, int, int]:
    """(world size, rank, local rank) from the torchrun environment (1, 0, 0 when run directly)."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value: float, device, world: int) -> float:
    """The largest of every rank's value (the job's time is set by its slowest rank); identity at N=1."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------- our arm
def setup_replicas(wl, R: int, device, weight_format: int = 0):
    import torch
    import synth
    import int4_weight_kv_gb300 as ft
    from int4_weight_kv_gb300 import runtime as rt
    s = wl.shape
    cfg = ft.cfg_from_shape(s)
    cfg.weight_format = weight_format
    w = synth.layer_weights(s, wl.config_id, 0)
    packed = rt.pack_layer(cfg, w, device=device)
    del w
    B, ctx = wl.batch, wl.ctx
    max_ctx = ctx + 1
    kb, _ = synth.kv_history(s, wl.config_id, B, ctx, which="k")
    vb, _ = synth.kv_history(s, wl.config_id, B, ctx, which="v")
    cache = rt.alloc_cache(cfg, B, max_ctx, device=device)
    rt.fill_history(cfg, cache, B, max_ctx, kb, vb)
    del kb, vb
    xb, _ = synth.activations(s, wl.config_id, B)
    reps = []
    for r in range(R):
        reps.append({
            "w": packed if r == 0 else {k: v.clone() for k, v in packed.items()},
            "cache": cache if r == 0 else cache.clone(),
            "x": rt.bits_tensor(xb, device=device),
            "y": torch.empty((B, s.hidden), dtype=torch.int16, device=device),
            "ws": rt.alloc_workspace(cfg, B, max_ctx, device=device),
        })
    pos = torch.full((B,), ctx, dtype=torch.int32, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    return cfg, reps, pos, status, max_ctx, xb


def run_ours(args):
    import torch
    import torch.distributed as dist
    import synth
    import int4_weight_kv_gb300 as ft

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    from int4_weight_kv_gb300 import build
    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        dist.barrier(device_ids=[local])
    ft.lib()

    wl = synth.workload(args.workload)
    s, B, ctx = wl.shape, wl.batch, wl.ctx
    wfmt = 1 if args.weights == "e4m3" else 0
    ab = algorithmic_bytes(s, B, ctx, wfmt)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    footprint = ab["weights"] + ab["kv"]
    R = max(2, int(np.ceil(4 * l2 / footprint)))
    cfg, reps, pos, status, max_ctx, xb = setup_replicas(wl, R, device, wfmt)
    stream = torch.cuda.current_stream(device)

    def step(r):
        p = reps[r]
        ft.check(ft.ft_decode_block(cfg, p["w"], p["cache"], B, max_ctx, p["x"], p["y"], ft.FT_BF16, pos, B, p["ws"],
                                    status), "ft_decode_block")

    for r in range(R):     # eager warm-up: sets kernel attributes before capture
        step(r)
    torch.cuda.synchronize()
    side = torch.cuda.Stream(device)
    side.wait_stream(stream)
    graphs = {}

    def graph_of(n):
        if n not in graphs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for i in range(n):
                    step(i % R)
            graphs[n] = g
        return graphs[n]

    def run_steps(k):
        full, rem = divmod(k, R)
        for _ in range(full):
            graph_of(R).replay()
        if rem:
            graph_of(rem).replay()

    run_steps(max(args.warmup, 3))
    torch.cuda.synchronize()

    # timed region: exactly K steps, barrier + synchronize on both sides
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier(device_ids=[local])
    torch.cuda.synchronize()
    e0.record(stream)
    run_steps(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier(device_ids=[local])
    ms = e0.elapsed_time(e1)
    # keep the GPU under the same load long enough for the clock sampler
    t_end = time.time() + (0.0 if args.profile else max(0.0, 1.0 - ms / 1000.0))
    while time.time() < t_end:
        run_steps(R * 50)
        torch.cuda.synchronize()
    clk = clocks.stop()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {status.item()}")
    ms = max_over_ranks(ms, device, world)
    us_step = ms * 1000.0 / args.steps

    # dominant kernel (gate/up projection) timed alone with CUDA events on its stream
    dom_role = max(ab["per_role"], key=lambda r: ab["per_role"][r])
    stage = {ft.FT_W_QKV: ft.FT_STAGE_QKV, ft.FT_W_O: ft.FT_STAGE_O, ft.FT_W_GATEUP: ft.FT_STAGE_GU,
             ft.FT_W_DOWN: ft.FT_STAGE_DOWN}[dom_role]
    n_dom = R if args.profile else max(R * 20, min(args.steps, 2000))
    for i in range(R):
        p = reps[i]
        ft.check(ft.ft_decode_block_stages(cfg, p["w"], p["cache"], B, max_ctx, p["x"], p["y"], ft.FT_BF16, pos, B,
                                           p["ws"], stage, status))
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(n_dom):
        p = reps[i % R]
        ft.ft_decode_block_stages(cfg, p["w"], p["cache"], B, max_ctx, p["x"], p["y"], ft.FT_BF16, pos, B, p["ws"],
                                  stage, status)
    e1.record(stream)
    torch.cuda.synchronize()
    dom_us = e0.elapsed_time(e1) * 1000.0 / n_dom
    dom_bytes = ab["per_role"][dom_role] + B * (s.hidden * 2 + s.inter * 2)
    peak, peak_kind = hbm_peak()
    achieved = dom_bytes / dom_us / 1e3
    traffic = None
    tr_path = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tr_path):
        with open(tr_path) as f:
            traffic = json.load(f).get(args.workload + ("_e4m3" if wfmt else ""))

    # end to end through the C ABI with host buffers (pinned), copies inside the timed region
    n_e2e = R if args.profile else min(args.steps, 500)
    x_host = torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).pin_memory()
    pos_host = torch.full((B,), ctx, dtype=torch.int32).pin_memory()
    y_host = torch.empty((B, s.hidden), dtype=torch.int16).pin_memory()
    for i in range(R):
        step(i)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(n_e2e):
        p = reps[i % R]
        p["x"].copy_(x_host, non_blocking=True)
        pos.copy_(pos_host, non_blocking=True)
        step(i % R)
        y_host.copy_(p["y"], non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_us = e0.elapsed_time(e1) * 1000.0 / n_e2e

    # per-replay spread of the headline (outside the timed region)
    g_all = graph_of(R)
    spread = _time_graph(g_all, max(10, min(args.steps, 200)), R)
    sweep = None if (args.profile or args.no_sweep) else run_sweep(args, device, hbm_peak()[0])
    sweep_e4m3 = None if (args.profile or args.no_sweep) else run_sweep(args, device, hbm_peak()[0], SWEEP_E4M3,
                                                                         weight_format=1, full_step=False)

    line = {
        "metric": METRIC, "value": round(us_step, 3), "unit": "us/step", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": us_step / 1000.0, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic (seeded N(0,0.02) weights, outlier-laden BF16 "
                                                  "activations and K/V history)",
        "config": {"workload": args.workload, "hidden": s.hidden, "n_q": s.n_q, "n_kv": s.n_kv,
                   "head_dim": s.head_dim, "inter": s.inter, "batch": B, "ctx": ctx, "replicas": R,
                   "l2": f"inputs larger than L2: {R} replicas of weights+KV ({R * footprint / 1e6:.0f} MB) cycled",
                   "graph": True, "pdl": True, "weights": args.weights,
                   "precision": ("E4M3" if wfmt else "INT4") + " weights and INT4 KV (BF16 scales), FP16 MMA "
                                "operands, FP32 accumulate, BF16 block I/O"},
        "block_gbs": round(ab["total"] / us_step / 1e3, 1),
        "pct_of_8tbs": round(100.0 * ab["total"] / us_step / 1e3 / NOMINAL_HBM_GBS, 1),
        "pct_of_measured_hbm": round(100.0 * ab["total"] / us_step / 1e3 / peak, 1),
        "algorithmic_bytes_per_step": ab["total"],
        "roofline": {"bound": "hbm", "kernel": "gemv_kernel (gate/up + SwiGLU)", "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 3), "traffic": traffic,
                     "peak_kind": f"{peak_kind} copy bandwidth (burst; kernel timed alone)",
                     "launch_us": round(dom_us, 3), "algorithmic_bytes": dom_bytes},
        "e2e": {"value": round(e2e_us, 3), "unit": "us/step", "h2d_bytes_per_step": B * s.hidden * 2 + B * 4,
                "d2h_bytes_per_step": B * s.hidden * 2},
        "gpu_launches": ft.ft_decode_block_launches(cfg, B) * args.steps,
        "clocks": clk,
        "us_p10": round(float(np.percentile(spread, 10)), 3), "us_median": round(float(np.median(spread)), 3),
        "us_p90": round(float(np.percentile(spread, 90)), 3),
        "sweep": sweep,
        "sweep_e4m3": sweep_e4m3,
    }
    if rank == 0:
        line["cpu_baseline"] = None if args.profile else cpu_baseline(wl)
        if args.profile:
            line["note"] = "profiler run: timings are not bench values"
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier(device_ids=[local])
        dist.destroy_process_group()


# ---------------------------------------------------------------------------- the metric's sweep
# (shape, [(batch, context)]) of the metric's batch range on the 8B and 70B layer shapes; the 8B rows at
# context 1024 (batch 1 is the headline workload), 8B batch 32 at context 4096 (the attention-dominated
# configuration), the 70B rows at context 2048 and 70B batch 1 at context 32768 (the split-KV reduction).
SWEEP = (("8B", 2, ((1, 1024), (2, 1024), (4, 1024), (8, 1024), (16, 1024), (32, 1024), (32, 4096))),
         ("70B", 4, ((1, 2048), (2, 2048), (4, 2048), (8, 2048), (16, 2048), (32, 2048), (1, 32768))))
# the same points with E4M3 decode weights (the pages' FP8 decode variant), beside the INT4 ones
SWEEP_E4M3 = (("8B", 2, ((1, 1024), (32, 1024))), ("70B", 4, ((1, 2048), (32, 2048))))


def stage_bytes(shape, B: int, ctx: int, per_role: dict) -> dict:
    """Algorithmic bytes of each stage that streams a large operand (one launch)."""
    import int4_weight_kv_gb300 as ft
    s = shape
    kv_tok = s.n_kv * 2 * (s.head_dim // 2 + 2 * (s.head_dim // s.kvg))
    return {ft.FT_STAGE_ATTN: B * (ctx + 1) * kv_tok,
            ft.FT_STAGE_GU: per_role[ft.FT_W_GATEUP] + B * (s.hidden + s.inter) * 2,
            ft.FT_STAGE_DOWN: per_role[ft.FT_W_DOWN] + B * (s.inter + 2 * s.hidden) * 2,
            ft.FT_STAGE_QKV: per_role[ft.FT_W_QKV] + B * (s.hidden * 2 + s.n_qkv * 4)}


STAGE_NAMES = {1: "prep", 2: "qkv projection", 4: "attention", 8: "o projection", 16: "mid", 32: "gate/up + SwiGLU",
               64: "down projection"}


def _pct(a: float, b: float) -> float:
    return round(100.0 * a / b, 1)


def _time_graph(g, n: int, per: int) -> list:
    """Per-step times (us) of n replays of a graph holding `per` steps."""
    import torch
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    evs[0].record()
    for i in range(n):
        g.replay()
        evs[i + 1].record()
    torch.cuda.synchronize()
    return [evs[i].elapsed_time(evs[i + 1]) * 1000.0 / per for i in range(n)]


def run_sweep(args, device, peak: float, sweep=SWEEP, weight_format: int = 0, full_step: bool = True) -> list:
    """Every (layer shape, batch, context) of the metric: one graph of R steps over R replicas
    (R * footprint >= 4x L2), per-replay CUDA events; the stage with the most algorithmic bytes timed
    alone for its roofline.  weight_format 1 runs the points with E4M3 decode weights."""
    import torch
    import synth
    import int4_weight_kv_gb300 as ft
    from int4_weight_kv_gb300 import runtime as rt
    shapes = {"8B": synth.L8B, "70B": synth.L70B}
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    tr_path = os.path.join(ROOT, "profiles", "traffic.json")
    traffic = json.load(open(tr_path)) if os.path.exists(tr_path) else {}  # DRAM bytes per dominant launch (ncu)
    out = []
    n_rep = max(10, min(args.steps, 200))
    tag = "_e4m3" if weight_format else ""
    for sname, cid, points in sweep:
        s = shapes[sname]
        cfg = ft.cfg_from_shape(s)
        cfg.weight_format = weight_format
        w = synth.device_layer_weights(s, cid, 0, device)
        packed = [rt.pack_layer(cfg, {k: v for k, v in w.items()}, device=device)]
        del w
        per_role = {r: ft.ft_packed_weight_bytes(cfg, r) for r in ft.ROLES}
        wbytes = sum(per_role.values())
        for B, ctx in points:
            ab = algorithmic_bytes(s, B, ctx, weight_format)
            R = max(2, int(np.ceil(4 * l2 / (ab["weights"] + ab["kv"]))))
            while len(packed) < R:
                packed.append({k: v.clone() for k, v in packed[0].items()})
            max_ctx = ctx + 1
            cache0 = rt.alloc_cache(cfg, B, max_ctx, device=device)
            chunk = max(1, (1 << 26) // (B * s.n_kv * s.head_dim))
            for t0 in range(0, ctx, chunk):
                t1 = min(ctx, t0 + chunk)
                kb = synth.device_kv_history(s, cid, B, t0, t1, "k", device)
                vb = synth.device_kv_history(s, cid, B, t0, t1, "v", device)
                pos0 = torch.full((B,), t0, dtype=torch.int32, device=device)
                ft.check(ft.ft_kv_append_int4(cfg, cache0, B, max_ctx, kb, vb, pos0, B, t1 - t0), "ft_kv_append_int4")
                del kb, vb
            reps = [{"w": packed[r], "cache": cache0 if r == 0 else cache0.clone(),
                     "x": synth.device_activations(s, cid, B, device),
                     "y": torch.empty((B, s.hidden), dtype=torch.int16, device=device),
                     "ws": rt.alloc_workspace(cfg, B, max_ctx, device=device)} for r in range(R)]
            pos = torch.full((B,), ctx, dtype=torch.int32, device=device)
            st = torch.zeros(1, dtype=torch.int32, device=device)

            def step(r, mask=ft.FT_STAGE_ALL):
                p = reps[r]
                ft.check(ft.ft_decode_block_stages(cfg, p["w"], p["cache"], B, max_ctx, p["x"], p["y"], ft.FT_BF16,
                                                   pos, B, p["ws"], mask, st), "ft_decode_block")
            for r in range(R):
                step(r)
            torch.cuda.synchronize()
            side = torch.cuda.Stream(device)
            side.wait_stream(torch.cuda.current_stream(device))
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for r in range(R):
                    step(r)
            for _ in range(max(args.warmup, 3)):
                g.replay()
            torch.cuda.synchronize()
            ts = _time_graph(g, n_rep, R)
            if int(st.item()) != 0:
                raise RuntimeError(f"device status {st.item()} at {sname} B={B} ctx={ctx}")
            med = float(np.median(ts))
            # dominant stage: the most algorithmic bytes; timed alone, replicas cycled
            sb = stage_bytes(s, B, ctx, per_role)
            dom = max(sb, key=lambda k: sb[k])
            n_dom = R * 20
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for i in range(n_dom):
                step(i % R, dom)
            e1.record()
            torch.cuda.synchronize()
            st.zero_()  # stages re-run alone may re-accumulate offsets: timing only
            dom_us = e0.elapsed_time(e1) * 1000.0 / n_dom
            ach = sb[dom] / dom_us / 1e3
            out.append({
                "workload": f"{sname.lower()}_b{B}_ctx{ctx}{tag}", "batch": B, "ctx": ctx, "replicas": R,
                "us_step": round(med, 2), "us_p10": round(float(np.percentile(ts, 10)), 2),
                "us_p90": round(float(np.percentile(ts, 90)), 2), "replays": n_rep,
                "algorithmic_bytes": ab["total"], "gbs": round(ab["total"] / med / 1e3, 1),
                "pct_of_measured_hbm": _pct(ab["total"] / med / 1e3, peak),
                "pct_of_8tbs": _pct(ab["total"] / med / 1e3, NOMINAL_HBM_GBS),
                "dominant": {"stage": STAGE_NAMES[dom], "launch_us": round(dom_us, 2), "algorithmic_bytes": sb[dom],
                             "achieved_gbs": round(ach, 1), "frac": round(ach / peak, 3),
                             "traffic": traffic.get(f"{sname.lower()}_b{B}_ctx{ctx}{tag}")},
            })
            print(json.dumps(out[-1]), file=sys.stderr, flush=True)
            del reps, cache0, g
            torch.cuda.empty_cache()
        del packed
        torch.cuda.empty_cache()
    if full_step:
        out.append(run_full_step(args, device, peak))
    return out


def run_full_step(args, device, peak: float) -> dict:
    """The full 32-layer Llama-3.1-8B decode step at batch 1, context 4096: embedding, 32 decode blocks
    (FP32 residual between layers), final RMSNorm + BF16 LM head (vocab 128256), one CUDA graph."""
    import torch
    import synth
    import int4_weight_kv_gb300 as ft
    from int4_weight_kv_gb300 import runtime as rt
    wl = synth.workload("8b_full_b1_ctx4096")
    s, B, ctx, nl, V = wl.shape, wl.batch, wl.ctx, wl.layers, wl.vocab
    cfg = ft.cfg_from_shape(s)
    max_ctx = ctx + 1
    layers, caches = [], []
    for li in range(nl):
        w = synth.device_layer_weights(s, wl.config_id, li, device)
        layers.append(rt.pack_layer(cfg, w, device=device))
        del w
        c = rt.alloc_cache(cfg, B, max_ctx, device=device)
        kb = synth.device_kv_history(s, wl.config_id, B, 0, ctx, "k", device, layer=li)
        vb = synth.device_kv_history(s, wl.config_id, B, 0, ctx, "v", device, layer=li)
        ft.check(ft.ft_kv_append_int4(cfg, c, B, max_ctx, kb, vb, torch.zeros(B, dtype=torch.int32, device=device),
                                      B, ctx), "ft_kv_append_int4")
        caches.append(c)
        del kb, vb
    mt = synth.device_model_tensors(s, wl.config_id, V, B, device)
    pos = torch.full((B,), ctx, dtype=torch.int32, device=device)
    bufs = {"x": torch.empty((B, s.hidden), dtype=torch.float32, device=device),
            "y": torch.empty((B, s.hidden), dtype=torch.float32, device=device),
            "logits": torch.empty((B, V), dtype=torch.float32, device=device)}
    ws = [rt.alloc_workspace(cfg, B, max_ctx, device=device)]
    st = torch.zeros(1, dtype=torch.int32, device=device)

    def step():
        rt.model_step(cfg, layers, caches, B, max_ctx, mt["emb_bits"], mt["lm_bits"], mt["gamma_final"],
                      mt["tokens"], pos, bufs, ws, st)
    step()
    torch.cuda.synchronize()
    side = torch.cuda.Stream(device)
    side.wait_stream(torch.cuda.current_stream(device))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        step()
    for _ in range(max(args.warmup, 3)):
        g.replay()
    torch.cuda.synchronize()
    n = max(10, min(args.steps, 100))
    ts = _time_graph(g, n, 1)
    if int(st.item()) != 0:
        raise RuntimeError(f"device status {st.item()} in the full step")
    med = float(np.median(ts))
    per_role = {r: ft.ft_packed_weight_bytes(cfg, r) for r in ft.ROLES}
    kv_tok = s.n_kv * 2 * (s.head_dim // 2 + 2 * (s.head_dim // s.kvg))
    lm_bytes = V * s.hidden * 2
    floor = nl * (sum(per_role.values()) + B * (ctx + 1) * kv_tok) + lm_bytes
    # the LM head (the largest single launch) timed alone
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    k = 20
    e0.record()
    for _ in range(k):
        ft.check(ft.ft_lm_head_bf16(bufs["x"], mt["gamma_final"], mt["lm_bits"], bufs["logits"], B, V, s.hidden,
                                    cfg.rms_eps), "ft_lm_head_bf16")
    e1.record()
    torch.cuda.synchronize()
    lm_us = e0.elapsed_time(e1) * 1000.0 / k
    res = {"workload": "8b_full_b1_ctx4096", "layers": nl, "batch": B, "ctx": ctx, "vocab": V,
           "us_step": round(med, 1), "us_p10": round(float(np.percentile(ts, 10)), 1),
           "us_p90": round(float(np.percentile(ts, 90)), 1), "replays": n,
           "algorithmic_bytes": floor, "gbs": round(floor / med / 1e3, 1),
           "pct_of_measured_hbm": _pct(floor / med / 1e3, peak), "pct_of_8tbs": _pct(floor / med / 1e3, NOMINAL_HBM_GBS),
           "dominant": {"stage": "lm head (BF16, final RMSNorm fused)", "launch_us": round(lm_us, 2),
                        "algorithmic_bytes": lm_bytes, "achieved_gbs": round(lm_bytes / lm_us / 1e3, 1),
                        "frac": round(lm_bytes / lm_us / 1e3 / peak, 3)},
           "context": "the pages quote 2.8 ms per full Llama-3.1-8B decode step at batch 1 on one H100 (not comparable)"}
    print(json.dumps(res), file=sys.stderr, flush=True)
    del layers, caches, mt, g
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------------- oracle timing
def _oracle_inputs(wl):
    import synth
    from oracle.block import BlockWeightsOracle
    from oracle.kv import KVCacheOracle
    s = wl.shape
    w = synth.layer_weights(s, wl.config_id, 0)
    wts = BlockWeightsOracle(s, w)
    B, ctx = wl.batch, wl.ctx
    kb, kf = synth.kv_history(s, wl.config_id, B, ctx, which="k")
    vb, vf = synth.kv_history(s, wl.config_id, B, ctx, which="v")
    cache = KVCacheOracle(B, s.n_kv, ctx + 1, s.head_dim, s.hb, s.kvg)
    cache.append(kf, vf, np.zeros(B, int))
    _, x = synth.activations(s, wl.config_id, B)
    return wts, cache, x.astype(np.float64), np.full(B, ctx, np.int32)


def oracle_sample_us(wl, inputs, rows=1) -> tuple[float, str]:
    """One bounded sample of the oracle: the full block for `rows` request(s),
    scaled to the whole batch (requests are independent)."""
    from oracle.block import decode_block
    wts, cache, x, pos = inputs
    t0 = time.perf_counter()
    decode_block(wl.shape, wts, cache, x, pos, batch_idx=list(range(min(rows, wl.batch))), write_cache=False)
    dt = time.perf_counter() - t0
    n = min(rows, wl.batch)
    return dt * 1e6 * wl.batch / n, f"full FP64 oracle block for {n} of {wl.batch} request(s), scaled to the batch"


def _cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(wl) -> dict:
    inputs = _oracle_inputs(wl)
    us, sample = oracle_sample_us(wl, inputs)
    return {"value": round(us, 1), "unit": "us/step", "cores": _cores(), "kind": "oracle", "sample": sample}


def run_reference(args):
    import synth
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    wl = synth.workload(args.workload)
    inputs = _oracle_inputs(wl)
    for _ in range(max(0, min(args.warmup, 1))):
        oracle_sample_us(wl, inputs)
    # each step is one bounded sample; cap the run at a few minutes of CPU time
    budget_s, times, sample = 150.0, [], ""
    t_start = time.perf_counter()
    for i in range(args.steps):
        us, sample = oracle_sample_us(wl, inputs)
        times.append(us)
        if time.perf_counter() - t_start > budget_s:
            break
    val = float(np.mean(times))
    line = {
        "impl": "reference", "metric": METRIC, "value": round(val, 1), "unit": "us/step", "n_gpus": 1,
        "steps": len(times), "warmup": args.warmup, "ms_per_step": val / 1000.0, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "hidden": wl.shape.hidden, "batch": wl.batch, "ctx": wl.ctx},
        "cpu_baseline": {"value": round(val, 1), "unit": "us/step", "cores": _cores(), "kind": "oracle",
                         "sample": sample + (f"; {len(times)} of {args.steps} steps within {budget_s:.0f} s"
                                             if len(times) < args.steps else "")},
        "e2e": {"value": round(val, 1), "unit": "us/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--weights", choices=["int4", "e4m3"], default="int4",
                    help="decode-weight format of the headline workload (the sweep reports both)")
    ap.add_argument("--no-sweep", action="store_true",
                    help="only the headline workload (skip the batch 1-32 sweep and the full 32-layer step)")
    ap.add_argument("--profile", action="store_true",
                    help="short run for a profiler: no clock hold, no oracle baseline; numbers are not bench values")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
