#!/usr/bin/env python
"""Benchmark of the routed-expert (MoE) layer on GB300.

One step = one pass of the whole layer over one batch: router (+ optional RMSNorm) + bias +
top-k + weights, route list, expert gated FFN (phase 1, phase 2), shared expert, slot-ordered
combine.  Default workload: the gpt-oss-shaped decode layer, T=8 tokens, H=I=2880, E=32, k=4,
MXFP4 experts (the configuration the headline metric is quoted on).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--T T] [--impl ours|reference]

Prints ONE JSON line on rank 0.  Under torchrun (N > 1) every rank runs an independent replica
on its own GPU (the layer has no exchange step): weak scaling, value = all ranks' tokens / the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s; decode HBM GB/s and prefill TFLOPS as % of GB300 peak"
DEFAULT_T = {1: 4, 2: 8, 3: 512, 4: 8, 5: 2048}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--config", type=int, default=2)
    p.add_argument("--T", type=int, default=None)
    p.add_argument("--layers", type=int, default=None, help="rotating weight sets")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--path", default="auto", choices=["auto", "gemv", "gemm", "gemm_dequant"],
                   help="expert path passed to ts_moe_forward_path")
    p.add_argument("--gemma-tail", action="store_true",
                   help="append the Gemma sandwich tail (ts_moe_gemma_tail) to every step")
    p.add_argument("--no-per-config", action="store_true",
                   help="measure only the selected configuration (no per_config entries)")
    p.add_argument("--profile", action="store_true",
                   help="short run for profiler captures: one timed repetition, few samples")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while active."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = str(gpu_index)
        try:
            import torch
            u = str(torch.cuda.get_device_properties(gpu_index).uuid)
            self.gpu = u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            pass
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-i", self.gpu, "-lms", "200"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def slowest_rank_ms(ms, ws, device):
    """Every rank passes its own time per step; returns the largest over the ranks (the job's
    time per step).  With one rank, the rank's own time."""
    if ws == 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.item()


def job_tokens_per_s(ws, T, ms_max):
    """Whole-job throughput: each of the ws ranks runs T tokens per step, and a step of the job
    takes the slowest rank's time."""
    return ws * T / (ms_max * 1e-3)


def captured_traffic(kernel, workload):
    """DRAM bytes (read + write) per launch of `kernel` on `workload` from a committed ncu summary
    under profiles/, or None.  A summary records its number on a line
    `traffic-record: kernel=K workload=W bytes=N files=a,b,c src_sha256=H`; the number is used only
    while the listed kernel sources still hash to H (a changed kernel makes it stale)."""
    import glob
    import hashlib
    here = os.path.dirname(os.path.abspath(__file__))
    csrc = os.path.join(here, "mixture_experts_routed_logits_gb300", "csrc")
    for path in sorted(glob.glob(os.path.join(here, "profiles", "*.md"))):
        for line in open(path):
            if not line.strip().startswith("traffic-record:"):
                continue
            kv = dict(tok.split("=", 1) for tok in line.split()[1:] if "=" in tok)
            if kv.get("kernel") != kernel or kv.get("workload") != workload:
                continue
            h = hashlib.sha256()
            try:
                for f in kv["files"].split(","):
                    with open(os.path.join(csrc, f), "rb") as fh:
                        h.update(fh.read())
            except OSError:
                return None
            return int(kv["bytes"]) if h.hexdigest() == kv.get("src_sha256") else None
    return None


def touched_bytes(cfg, idx_np, ex_mat_bytes, shared_bytes):
    """Algorithmic HBM bytes of one step: each touched expert's packed weights once, plus the
    activations in/out, router weights and the shared expert."""
    import numpy as np
    c = cfg
    n_touched = len(np.unique(idx_np))
    w_bytes = n_touched * ex_mat_bytes["total"]
    H, T = c["H"], idx_np.shape[0]
    act_bytes = T * H * 2 * 2 + c["E"] * H * 2          # x in, y out, router weights
    return n_touched, w_bytes + act_bytes + shared_bytes


def run_reference(args, cfg_id, T, rank, ws):
    """Reference arm: the CPU oracle, as it stands, on the machine's host cores."""
    if rank != 0:
        return
    import numpy as np
    from mixture_experts_routed_logits_gb300 import synth
    import oracle
    from tests._helpers import bits16, oracle_layer, oracle_route
    oracle.build()
    L = synth.make_layer(cfg_id, T=T, device="cpu")
    c = L["cfg"]
    cores = os.cpu_count() or 1
    ntok = max(1, min(T, cores))
    toks = np.arange(ntok, dtype=np.int32)
    xb = bits16(L["x"])
    oex, osh = oracle_layer(L)

    def step():
        xn, lg, idx, w = oracle_route(L, xb[:ntok] if not c["rmsnorm"] else xb[:ntok])
        xin = xn if xn is not None else xb[:ntok]
        oracle.moe_forward(xin, c["adt"], oex, idx, w, shared=osh, nthreads=min(cores, ntok))

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    val = ntok * args.steps / dt
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_name(c, T), "T": T, "sample_tokens_per_step": ntok},
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": min(cores, ntok),
                             "kind": "oracle",
                             "sample": f"first {ntok} of the {T} tokens of the batch per step, "
                                       f"{args.steps} steps"},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_baseline(cfg_id, T):
    """The oracle timed on the host cores on a bounded sample of the same workload."""
    import numpy as np
    from mixture_experts_routed_logits_gb300 import synth
    import oracle
    from tests._helpers import bits16, oracle_layer, oracle_route
    oracle.build()
    L = synth.make_layer(cfg_id, T=T, device="cpu")
    c = L["cfg"]
    cores = os.cpu_count() or 1
    ntok = max(1, min(T, cores))
    xb = bits16(L["x"])[:ntok]
    oex, osh = oracle_layer(L)
    n, t0 = 0, time.perf_counter()
    while True:
        xn, lg, idx, w = oracle_route(L, xb)
        oracle.moe_forward(xn if xn is not None else xb, c["adt"], oex, idx, w, shared=osh,
                           nthreads=min(cores, ntok))
        n += ntok
        if time.perf_counter() - t0 > 8.0:
            break
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": "tokens/s", "cores": min(cores, ntok), "kind": "oracle",
            "sample": f"{n} tokens ({ntok} per pass) of the same layer, routing + experts, "
                      f"{dt:.1f} s"}


def workload_name(cfg, T):
    """Workload label of a configuration at T tokens (the same string on both bench arms)."""
    import re
    base = re.sub(r"_T\d+", "", cfg["name"])
    prefix, rest = base.split("_H", 1)
    return f"{prefix}_T{T}_H{rest}"


def dtype_label(cfg, gemm_path, mx_path=False):
    """The arithmetic the path computes in (inputs -> multiply -> accumulate)."""
    fmt, adt = cfg["fmt"], cfg["adt"]
    if mx_path:
        return f"{adt}-in/exact 2-term e4m3 split·e2m1, e8m0 block scales, tcgen05 mma/f32-acc"
    if gemm_path:
        if fmt == "mxfp4":
            return f"{adt}-in/f16(exact prescale)·e2m1→f16 tcgen05 mma/f32-acc"
        return f"{adt}·{fmt} tcgen05 mma/f32-acc"
    if fmt in ("mxfp4", "int4"):
        w = "e2m1" if fmt == "mxfp4" else "int4-affine"
        return f"{adt}-in/f16(exact prescale)·{w} mma.sync/f32-acc"
    if fmt == "bf16":
        return "bf16·bf16 mma.sync/f32-acc"
    return f"{adt}-in/f16·f16 mma.sync/f32-acc"


def measure(cfg_id, T, args, ws, rank, local, hbm_peak, bf16_sust, peak_src, min_wall, want_e2e):
    """Builds the layers of one configuration, captures a CUDA graph per layer and times K-step
    loops of graph replays (L2 flushed between steps) under clock sampling; returns the
    configuration's measurement (rank-local time and the slowest rank's)."""
    import numpy as np
    import torch
    import mixture_experts_routed_logits_gb300 as moe
    from mixture_experts_routed_logits_gb300 import synth

    cfg = dict(synth.CONFIGS[cfg_id])
    cfg["T"] = T
    H, I, E, k = cfg["H"], cfg["I"], cfg["E"], cfg["k"]

    # ---- rotating weight sets (layers), inputs resident in HBM -----------------------------------
    # one layer's touched experts can fit in the 129 MB L2 at T=1, so steps rotate over several
    # independent layers AND the L2 is flushed (512 MB write) between timed steps
    per_layer = 3 * E * H * I * (0.53 if cfg["fmt"] == "mxfp4" else 0.625 if cfg["fmt"] == "int4" else 2.0)
    n_layers = args.layers or int(max(2, min(8, (2 << 30) // max(1, int(per_layer)))))
    layers = []
    for li in range(n_layers):
        L = synth.make_layer(cfg_id, T=T, seed=synth.default_seed(cfg_id) + 1000 * li + 7919 * rank,
                             device="cuda")
        ex = moe.Experts.from_canonical(cfg["fmt"], cfg["act"], L["experts"])
        sh = moe.Experts.from_canonical("f16", cfg["act"], L["shared"]) if L["shared"] is not None else None
        del L["experts"], L["shared"]
        wsb = moe.alloc_workspace(T, k, ex, sh)
        outs = dict(idx=torch.empty((T, k), dtype=torch.int32, device="cuda"),
                    w=torch.empty((T, k), dtype=torch.float32, device="cuda"),
                    xn=torch.empty_like(L["x"]) if cfg["rmsnorm"] else None,
                    y=torch.empty_like(L["x"]))
        if args.gemma_tail:
            # the tail's other inputs: the dense branch h1, the residual stream, the two
            # post-FFN norm weights (around 1) and the layer scalar
            g = torch.Generator(device="cuda").manual_seed(li)
            outs.update(h1=torch.randn(L["x"].shape, generator=g, device="cuda").to(L["x"].dtype),
                        xres=torch.randn(L["x"].shape, generator=g, device="cuda").to(L["x"].dtype),
                        w_post2=(1 + 0.1 * torch.randn(H, generator=g, device="cuda")).to(torch.bfloat16),
                        w_post=(1 + 0.1 * torch.randn(H, generator=g, device="cuda")).to(torch.bfloat16))
        layers.append(dict(L=L, ex=ex, sh=sh, ws=wsb, **outs))
    torch.cuda.synchronize()

    def step(ly, stream=None):
        # the whole layer through ts_moe_route_forward: the router, then the experts (the router
        # launch also does the decode kernels' prep when they take the call); with the Gemma
        # sandwich tail, the router then ts_moe_forward_tail (the tail inside the GEMV phase 2
        # at decode sizes)
        L = ly["L"]
        if not args.gemma_tail:
            moe.route_forward(L["x"], L["Wr"], k, ly["ex"], mode=cfg["mode"], router_bias=L["router_bias"],
                              per_expert_scale=L["scale"], rmsnorm=cfg["rmsnorm"], shared=ly["sh"],
                              ws=ly["ws"], path=args.path,
                              out=(ly["y"], None, ly["idx"], ly["w"], ly["xn"]), stream=stream)
            return
        moe.router_route(L["x"], L["Wr"], k, mode=cfg["mode"], router_bias=L["router_bias"],
                         per_expert_scale=L["scale"], rmsnorm=cfg["rmsnorm"],
                         out=(ly["idx"], ly["w"], ly["xn"], None), stream=stream)
        moe.forward_tail(ly["xn"] if cfg["rmsnorm"] else L["x"], ly["ex"], ly["idx"], ly["w"], ly["h1"],
                         ly["xres"], ly["w_post2"], ly["w_post"], 0.5, shared=ly["sh"], ws=ly["ws"],
                         path=args.path, out=(ly["y"], None), stream=stream)

    # ---- CUDA graphs: one per layer, plus a copy with per-phase events -------------------------------
    nph = 8
    phase_ev = [torch.cuda.Event(enable_timing=True) for _ in range(nph)]
    for ev in phase_ev:      # the library records them inside the graphs; torch only lets
        ev.record()          # elapsed_time() read events it has seen recorded once
    cs = torch.cuda.Stream()
    graphs, graphs_ev = [], []
    with torch.cuda.stream(cs):
        for ly in layers:          # warm (not captured) so lazy init happens outside capture
            step(ly, cs)
    torch.cuda.synchronize()
    for ly in layers:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cs):
            step(ly, cs)
        graphs.append(g)
        ge = torch.cuda.CUDAGraph()
        moe.set_phase_events(phase_ev)
        with torch.cuda.graph(ge, stream=cs):
            step(ly, cs)
        moe.set_phase_events(None)
        graphs_ev.append(ge)
    torch.cuda.synchronize()

    flush = synth.make_l2_flush("cuda")
    # the library's automatic choice: tensor-core grouped GEMM above 8 tokens for MXFP4 and for
    # 16-bit weights of the activation type (H, I multiples of 64), else the streaming GEMV
    gemm_ok = H % 64 == 0 and I % 64 == 0 and (cfg["fmt"] == "mxfp4" or cfg["fmt"] == cfg["adt"])
    mx_ok = cfg["fmt"] == "mxfp4" and cfg["adt"] == "bf16"
    # decode batches with MXFP4 + bf16 take the block-scaled decode kernels (prep, then one
    # launch for both phases and the combine) on "gemm", and on "auto" from 3 tokens
    mxd_path = (mx_ok and T <= 8 and T * k <= 64 and k <= 8 and H <= 4096
                and (args.path == "gemm" or (args.path == "auto" and T >= 3)))
    gemm_path = mxd_path or ((gemm_ok or mx_ok) and (args.path in ("gemm", "gemm_dequant") or (args.path == "auto" and T > 8)))
    # GEMV decode (T*k <= 512): router, phase 1, phase 2 (+ fused route list and combine);
    # otherwise router, route list, [gather], phase 1, phase 2, combine; + 2 shared-expert GEMVs
    fused_decode = (not gemm_path) and T * k <= 512
    # MXFP4 with bf16 activations takes the block-scaled MMA (activation split + two GEMMs);
    # "gemm_dequant" the f16 MMA over dequantised weights (gather, h conversion)
    mx_path = (gemm_path and not mxd_path and cfg["fmt"] == "mxfp4" and cfg["adt"] == "bf16"
               and args.path != "gemm_dequant")
    # the block-scaled grouped GEMM runs both phases in one launch unless K is split (<= 64 routes)
    mx_one = mx_path and T * k > 64
    # the decode kernels' prep (x split, counters) done by the router launch
    route_fold = mxd_path
    # the Gemma tail runs inside the GEMV phase 2 (fused combine), else as a launch of its own
    tail_fused = bool(args.gemma_tail) and fused_decode and not mxd_path
    if args.gemma_tail and mxd_path:
        route_fold = False          # the step is router_route + forward_tail: the prep launches
    n_launch_step = ((2 if route_fold else 3 if mxd_path else 3 if fused_decode else 5 if mx_one
                      else 5 + (1 if gemm_path else 0)
                      + (1 if gemm_path and cfg["fmt"] == "mxfp4" and not mx_path else 0))
                     + (2 if cfg.get("shared_I") else 0) + (1 if args.gemma_tail and not tail_fused else 0))

    def timed(K):
        b = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        e = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        for i in range(K):
            flush.zero_()
            b[i].record()
            graphs[i % n_layers].replay()
            e[i].record()
        torch.cuda.synchronize()
        return [b[i].elapsed_time(e[i]) for i in range(K)]

    # ---- warm-up + timed region ---------------------------------------------------------------------
    timed(max(3, args.warmup))
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # the K-step timed loop is repeated (each repetition exactly K steps, bracketed by
    # synchronisation) for >= min_wall seconds so that the 200 ms clock sampler sees the work;
    # the median repetition is reported
    reps = []
    with ClockSampler(local) as clk:
        t_wall0 = time.perf_counter()
        while True:
            torch.cuda.synchronize()
            times = timed(args.steps)
            reps.append(statistics.mean(times))
            if args.profile or (time.perf_counter() - t_wall0 > min_wall and len(reps) >= 3):
                break
        torch.cuda.synchronize()
        wall = time.perf_counter() - t_wall0
    if ws > 1:
        torch.distributed.barrier()
    ms = statistics.median(reps)
    ms_max = slowest_rank_ms(ms, ws, "cuda")

    # ---- per-phase breakdown: graphs carrying event-record nodes after every launch ----------------
    # event order in a step: 6 router, 0 route list, 1 phase 1, [2 shared phase 1], 3 phase 2,
    # [4 shared phase 2], 5 combine, [7 Gemma sandwich tail]
    if mxd_path:   # router (+ prep), [shared phase 1, shared phase 2], both phases + combine
        order = [6] + ([] if route_fold else [0]) + ([2, 4] if cfg.get("shared_I") else []) + [1]
    elif mx_one:   # router, route list + split, both phases, combine
        order = [6, 0, 1, 5]
    elif gemm_path:
        order = [6, 0, 1, 3, 5]
    else:   # GEMV: routed phase 1, shared phase 1, shared phase 2, routed phase 2 (+ combine)
        order = [6, 0, 1] + ([2, 4] if cfg.get("shared_I") else []) + [3, 5]
    if args.gemma_tail and not tail_fused:
        order = order + [7]
    samples = {moe.PHASES[j]: [] for j in order}
    for i in range(3 if args.profile else min(args.steps, 50)):
        flush.zero_()
        b = torch.cuda.Event(enable_timing=True)
        b.record()
        graphs_ev[i % n_layers].replay()
        torch.cuda.synchronize()
        prev = b
        for j in order:
            samples[moe.PHASES[j]].append(prev.elapsed_time(phase_ev[j]))
            prev = phase_ev[j]
    phases = {n: statistics.mean(v) for n, v in samples.items()}
    if mxd_path:   # the router launch splits x as well; one launch runs both phases
        phases = {("router_and_prep" if n == "router" and route_fold else "prep_x_split" if n == "route_list"
                   else "experts_fused" if n == "experts_phase1" else n): v for n, v in phases.items()}
    if mx_one:     # one launch runs both phases
        phases = {("experts_fused" if n == "experts_phase1" else n): v for n, v in phases.items()}

    # ---- algorithmic bytes / FLOPs of the dominant kernel (expert phase 1) ---------------------------
    idx_np = layers[0]["idx"].cpu().numpy()
    n_touched = len(np.unique(idx_np))
    fmt = cfg["fmt"]
    if fmt in ("mxfp4", "int4"):
        mat_gu = moe.packed_bytes(fmt, 1, I, H)
        mat_d = moe.packed_bytes(fmt, 1, H, I)
    else:
        mat_gu, mat_d = I * H * 2, H * I * 2
    bias_gu = 2 * I * 2 if cfg.get("expert_bias_std") else 0
    bias_d = H * 2 if cfg.get("expert_bias_std") else 0
    p1_bytes = n_touched * (2 * mat_gu + bias_gu) + T * H * 2 + T * k * I * 2
    p2_bytes = n_touched * (mat_d + bias_d) + T * k * I * 2 + T * k * H * 4
    shared_bytes = 0
    if cfg.get("shared_I"):
        shared_bytes = 3 * H * cfg["shared_I"] * 2
    step_bytes = p1_bytes + p2_bytes + shared_bytes + E * H * 2 + T * H * 2 * 2 + T * k * H * 4
    p1_ms = phases["experts_fused" if (mxd_path or mx_one) else "experts_phase1"]
    routes = T * k
    p1_flop = 2.0 * routes * 2 * I * H
    p2_flop = 2.0 * routes * H * I
    wl = workload_name(cfg, T)
    if gemm_path and fmt != "mxfp4":
        # tensor-bound: FLOPs of the phase-1 grouped GEMM over its launch time, against the
        # sustained bf16 peak (the kernel runs inside a seconds-long loop)
        achieved = p1_flop / (p1_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "kernel": "experts_phase1 (tcgen05 grouped GEMM, gate/up)",
                "achieved": achieved, "peak": bf16_sust, "unit": "TFLOP/s",
                "frac": achieved / bf16_sust, "peak_source": peak_src + " (bf16 sustained)",
                "traffic": None, "algorithmic_flop": p1_flop, "launch_ms": p1_ms}
        step_tf = (p1_flop + p2_flop) / (ms_max * 1e-3) / 1e12
    else:
        # the decode kernels, and the block-scaled grouped GEMM above 64 routes, run both phases in
        # one launch: its bytes are both phases'
        k_bytes = p1_bytes + p2_bytes if (mxd_path or mx_one) else p1_bytes
        achieved = k_bytes / (p1_ms * 1e-3) / 1e9
        traffic = (captured_traffic("mxd_fused", wl) if mxd_path
                   else captured_traffic("mx_fused", wl) if mx_one
                   else None if gemm_path else captured_traffic(f"gemv_{fmt}_phase1", wl))
        roof = {"bound": "hbm",
                "kernel": ("experts_fused (tcgen05 block-scaled decode kernel: gate/up, down, combine; "
                           "stream-K, cooperative)" if mxd_path else
                           "experts_fused (tcgen05 block-scaled grouped GEMM: gate/up and down in one "
                           "cooperative launch, items from one counter)" if mx_one else
                           "experts_phase1 (tcgen05 block-scaled grouped GEMM, MXFP4 gate/up)"
                           if mx_path else
                           "experts_phase1 (tcgen05 grouped GEMM over packed MXFP4, gate/up)"
                           if gemm_path else "experts_phase1 (gate/up GEMV)"),
                "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak, "peak_source": peak_src,
                "traffic": traffic, "algorithmic_bytes": k_bytes, "launch_ms": p1_ms}
        step_tf = None

    # ---- end to end through the public API with host buffers ---------------------------------------
    e2e = None
    if want_e2e:
        ly = layers[0]
        x_host = ly["L"]["x"].cpu().pin_memory()
        y_host = torch.empty_like(x_host).pin_memory()
        e2e_t = []
        for i in range(max(3, args.warmup) + (3 if args.profile else args.steps)):
            lyr = layers[i % n_layers]
            flush.zero_()
            b = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            b.record()
            lyr["L"]["x"].copy_(x_host, non_blocking=True)
            step(lyr)
            y_host.copy_(lyr["y"], non_blocking=True)
            e.record()
            e.synchronize()
            if i >= max(3, args.warmup):
                e2e_t.append(b.elapsed_time(e))
        e2e_ms = statistics.mean(e2e_t)
        e2e = {"value": T * ws / (e2e_ms * 1e-3), "unit": "tokens/s",
               "h2d_bytes_per_step": T * H * 2, "d2h_bytes_per_step": T * H * 2,
               "ms_per_step": e2e_ms}

    out = {
        "ms": ms, "ms_max": ms_max, "value": job_tokens_per_s(ws, T, ms_max), "wall": wall,
        "n_layers": n_layers, "reps": len(reps), "gemm_path": gemm_path,
        "n_launch_step": n_launch_step, "n_touched": int(n_touched), "phases": phases,
        "roofline": roof, "clocks": clk.summary(), "e2e": e2e,
        "step_tflops": None if step_tf is None else {"TFLOPs": step_tf, "frac": step_tf / bf16_sust},
        "step_hbm": {"bytes": step_bytes, "GBps": step_bytes / (ms_max * 1e-3) / 1e9,
                     "frac": step_bytes / (ms_max * 1e-3) / 1e9 / hbm_peak},
        "dtype": dtype_label(cfg, gemm_path, mx_path or mxd_path), "workload": wl, "cfg": cfg,
        "path": ("tcgen05 block-scaled decode kernels (kind::mxf8f6f4, stream-K over every SM, TMA + TMEM; "
                 + ("router launch with the prep folded in, " if route_fold else "prep, ")
                 + "gate/up, down + fused combine)" if mxd_path
                 else "tcgen05 block-scaled grouped GEMM (kind::mxf8f6f4, TMA + TMEM; gate/up and down in one "
                      "launch)" if mx_one
                 else "tcgen05 block-scaled grouped GEMM (kind::mxf8f6f4, TMA + TMEM)" if mx_path
                 else "tcgen05 grouped GEMM (TMA + TMEM)" if gemm_path
                 else "gemv (mma.sync m16n8k16 over streamed tiles)"),
    }
    del layers, graphs, graphs_ev, flush
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


# the other configurations reported beside the headline one (config id, tokens)
PER_CONFIG = [(1, 4), (2, 1), (3, 512), (4, 8), (5, 2048)]


def main():
    args = parse()
    ws, rank, local = dist_setup(args)
    cfg_id = args.config
    T = args.T or DEFAULT_T[cfg_id]
    if args.impl == "reference":
        run_reference(args, cfg_id, T, rank, ws)
        return

    import torch
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    if ws > 1:
        torch.distributed.barrier()

    hbm_peak, bf16_peak, bf16_sust, peak_src = peaks()
    m = measure(cfg_id, T, args, ws, rank, local, hbm_peak, bf16_sust, peak_src, 1.5, True)
    cfg = m["cfg"]

    per_config = None
    if not args.profile and not args.no_per_config and args.config == 2 and args.T is None:
        per_config = {}
        for cid, tt in PER_CONFIG:
            r = measure(cid, tt, args, ws, rank, local, hbm_peak, bf16_sust, peak_src, 0.4, False)
            per_config[r["workload"]] = {
                "config": cid, "T": tt, "tokens_per_s": r["value"], "ms_per_step": r["ms_max"],
                "dtype": r["dtype"], "path": r["path"], "touched_experts": r["n_touched"],
                "roofline": r["roofline"], "step_hbm": r["step_hbm"], "step_tflops": r["step_tflops"],
                "phase_ms": r["phases"], "clocks": r["clocks"], "launches_per_step": r["n_launch_step"],
                "timing": f"{r['reps']} repetitions of {args.steps} steps, median; L2 flushed "
                          f"between steps; {r['n_layers']} rotating weight sets"}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline and not args.profile:
        try:
            cpu = cpu_baseline(cfg_id, T)
        except Exception as ex:     # reported, not fatal
            cpu = {"error": str(ex)}

    H, I, E, k = cfg["H"], cfg["I"], cfg["E"], cfg["k"]
    line = {
        "metric": METRIC, "value": m["value"], "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": m["ms_max"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": m["dtype"],
        "data": "synthetic",
        "config": {"workload": m["workload"], "T": T, "H": H,
                   "I": I, "E": E, "k": k, "weights": cfg["fmt"], "activations": cfg["adt"],
                   "accumulate": "f32", "path": m["path"],
                   "l2": "flushed between timed steps (512 MB write, outside the step events); "
                         f"{m['n_layers']} rotating weight sets",
                   "timing": "CUDA graph per step, CUDA events per step; the K-step loop repeated "
                             f"{m['reps']}x under clock sampling, median repetition",
                   "touched_experts": m["n_touched"], "parallelism": f"replicas x{ws}",
                   "gemma_tail": bool(args.gemma_tail)},
        "roofline": m["roofline"],
        "step_tflops": m["step_tflops"],
        "step_hbm": m["step_hbm"],
        "phase_ms": m["phases"],
        "cpu_baseline": cpu,
        "e2e": m["e2e"],
        "gpu_launches": m["n_launch_step"] * args.steps,
        "clocks": m["clocks"],
        "wall_s_timed": m["wall"],
        "per_config": per_config,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
