"""Benchmark of the NVFP4 fused-MoE forward on GB300 (one JSON line on stdout).

Headline workload (one step = one fused forward pass over one batch): the
large-batch w4a16 case -- M=131072 tokens, H=6144, I=2048, E=256, top_k=8,
BF16 activations, NVFP4 weights, uniform distinct top-8 routing with
Dirichlet(1) weights, seed 0 (the route-window workload of the FlashInfer
PR #4440 page, results table).  Weights are generated once and stay
resident; each step re-runs routing, x into slot order, GEMM1 + SwiGLU,
GEMM2 and finalize.  The line also carries the other single-GPU workloads
under "workloads" (decode w4a16, skewed w4a16, prefill w4a4), each with its
own roofline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload large_w4a16|...] [--also decode_w4a16,...|none]

`--impl reference` times the CPU oracle (test infrastructure, never tuned)
on the host cores over bounded samples of the same workload.  Under torchrun
every rank runs its own replica (independent batches, no collective on the
data path: weak scaling); times are the max over ranks.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused-MoE tokens/s"
UNIT = "tokens/s"
SECONDARY = "decode_w4a16,skewed_w4a16,prefill_w4a4"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="large_w4a16")
    ap.add_argument("--also", default=SECONDARY,
                    help="comma-separated workloads measured after the headline and reported "
                         "under 'workloads' ('none' for the headline alone)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=20.0,
                    help="seconds of oracle work for the cpu_baseline leg (bounded sample)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override M (a smaller case of the workload, e.g. for a profiler)")
    ap.add_argument("--experts", type=int, default=0, help="override E")
    ap.add_argument("--route-tile", type=int, default=0, help="override the route tile T")
    ap.add_argument("--no-localized", action="store_true",
                    help="skip the two-domain timing (ncu cannot profile kernels launched into "
                         "green contexts)")
    ap.add_argument("--parallel", default="replicas", choices=["replicas", "ep"],
                    help="N > 1: independent replicas per rank (weak scaling), or one batch with "
                         "the experts split over the ranks and one all-reduce (strong scaling)")
    ap.add_argument("--locality", action="store_true",
                    help="print the GEMM1 gather-locality measurement instead of the bench line")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(v, world, device=None):
    """Max of a per-rank float over all ranks (the job's time is its slowest rank)."""
    if world == 1:
        return float(v)
    import torch
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replica_cfg(cfg, rank):
    """Rank r's replica draws its own batch and weights (seed + r): weak scaling."""
    return cfg.with_(seed=cfg.seed + rank) if rank else cfg


def tokens_per_s(world, tokens_per_rank, ms):
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank / (ms * 1e-3)


def workload_config(cfg, T):
    return {"workload": cfg.name, "M": cfg.M, "H": cfg.H, "I": cfg.I, "E": cfg.E,
            "top_k": cfg.top_k, "mode": cfg.mode, "routing": cfg.routing, "route_tile": T,
            "seed": cfg.seed}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def oracle_tokens(cfg, inp):
    """Tokens the oracle is timed on: every token of the small workloads, the
    seeded sample (1024 tokens) of the large ones."""
    import numpy as np
    return np.asarray(inp.sample_tokens) if cfg.sample else np.arange(cfg.M)


def time_oracle_bounded(orc, toks, budget_s, max_runs=3):
    """Time the oracle on a prefix of `toks` sized to about `budget_s` seconds
    of host work: a 1-thread-per-token calibration pass on a few tokens picks
    the prefix, then up to `max_runs` timed passes.  Returns (tokens/s,
    seconds per pass, threads, tokens per pass, runs)."""
    ncpu = os.cpu_count() or 1
    probe = toks[:min(len(toks), ncpu)]
    t0 = time.perf_counter()
    orc.forward(probe, nthreads=min(ncpu, len(probe)))
    per_round = time.perf_counter() - t0          # one token per thread
    rounds = max(1, int(budget_s / max(per_round, 1e-9)))
    n = min(len(toks), rounds * ncpu)
    sub = toks[:n]
    cores = min(ncpu, n)
    runs = max(1, min(max_runs, int(budget_s / max(per_round * -(-n // cores), 1e-9))))
    t0 = time.perf_counter()
    for _ in range(runs):
        orc.forward(sub, nthreads=cores)
    dt = (time.perf_counter() - t0) / runs
    return n / dt, dt, cores, n, runs


def cpu_baseline(cfg, inp, T, budget_s):
    import oracle
    oracle.build()
    orc = oracle.OracleMoE.from_inputs(inp, T=T)
    toks = oracle_tokens(cfg, inp)
    v, dt, cores, n, runs = time_oracle_bounded(orc, toks, budget_s)
    if cfg.sample:
        what = ("the first %d of the %d seeded sampled tokens of %s, %d timed pass(es); the full "
                "M=%d batch would take ~%.0f s on these cores (extrapolated from the sample)"
                % (n, len(toks), cfg.name, runs, cfg.M, cfg.M / v))
    else:
        what = "%d of the %d tokens of one %s batch, %d timed pass(es)" % (n, cfg.M, cfg.name, runs)
    return {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": what,
            "host_cpus": os.cpu_count()}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def src_digest(*names):
    """Digest of kernel sources: a stored ncu traffic figure is used only while
    the sources it was taken on are unchanged."""
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "block_scaled_fp4_sort_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# the sources of each GEMM kernel family (its own file and the shared headers)
_SHARED = ("gemm_common.cuh", "common.cuh", "decode.cuh", "nvfp4.cuh", "internal.h")
GEMM_SOURCES = {"tcgen05": ("moe_gemm.cu",) + _SHARED,
                "nvfp4": ("moe_gemm_nvfp4.cu",) + _SHARED,
                "gemv": ("moe_gemv.cu",) + _SHARED}


def gemm_family(cfg, T, native):
    if native:
        return "nvfp4"
    return "gemv" if cfg.mode == "w4a16" and T <= 16 else "tcgen05"


def stored_traffic(workload, family, T=None, cfg=None):
    """DRAM bytes per GEMM1 launch from a committed ncu summary of this
    workload's GEMM1 (scaled to the full launch where the capture ran a
    smaller case), or None if none was taken on the current sources of the
    kernel family that runs it, or the run changed the workload's sizes or
    route tile."""
    path = os.path.join(ROOT, "profiles", "gemm1_traffic.json")
    if not os.path.exists(path):
        return None, None
    with open(path) as f:
        tj = json.load(f)
    ent = tj.get(workload)
    if not ent or ent.get("src_digest") != src_digest(*GEMM_SOURCES[family]):
        return None, None
    if T is not None and ent.get("route_tile") != T:
        return None, None
    if cfg is not None:
        import synth
        if workload in synth.CONFIGS and cfg != synth.CONFIGS[workload]:
            return None, None
    return ent.get("dram_bytes_per_launch"), ent.get("source")


def native_mma(cfg, T):
    """GEMM1's block-scaled tensor-core MMA, if any: 'nvfp4' (w4a4, K a
    multiple of 256), 'mxfp8' (w4a8, K a multiple of 128; the packed E2M1
    weights unpacked on the way into shared memory), route tiles of 32 or
    more; else None."""
    if T >= 32 and cfg.mode == "w4a4" and cfg.H % 256 == 0:
        return "nvfp4"
    if T >= 32 and cfg.mode == "w4a8" and cfg.H % 128 == 0:
        return "mxfp8"
    return None


def mma_dtype(cfg, T, native):
    """Operand type of GEMM1's MMAs: the native block-scaled MMAs (NVFP4, or
    E4M3 x E4M3 with E8M0 block scales), the decode-size w4a16 kernel's FP16
    (hardware E2M1 -> FP16 decode, activations as FP16 rows with a
    power-of-two scale each), the other w4a16 / expanded kernels BF16."""
    if native:
        return native
    return "f16" if cfg.mode == "w4a16" and T <= 16 else "bf16"


def gemm1_kernel_name(cfg, T, native):
    if cfg.mode == "w4a16" and T <= 16:
        return "moe_gemv_kernel (GEMM1 + SwiGLU, warp MMA, f16)"
    if native:
        return "moe_gemm_nvfp4_kernel<%d> (GEMM1 + SwiGLU, tcgen05 %s)" % (
            T, "kind::mxf4nvf4" if native == "nvfp4" else "kind::mxf8f6f4")
    return "moe_gemm_kernel<%d> (GEMM1 + SwiGLU, tcgen05 kind::f16)" % T


def measure(cfg, args, rank, world, local, dev, headline):
    """Time one workload: the fused step (device-resident inputs), the atomic
    finalize variant, the two-domain variant (headline only), the per-kernel
    breakdown through the staged entry points, and the end-to-end step
    through pinned host buffers.  Returns (line dict, inputs, route tile)."""
    import numpy as np
    import torch

    import block_scaled_fp4_sort_gb300 as fm
    import synth
    from block_scaled_fp4_sort_gb300.buffers import MoEBuffers, problem_for

    cfg = replica_cfg(cfg, rank)
    T = args.route_tile or synth.route_tile_for(cfg)
    inp = synth.generate(cfg, device=dev)
    p = problem_for(cfg, T)
    B = MoEBuffers(p, dev).prepare(inp.w1, inp.w1_sf, inp.w2, inp.w2_sf)
    ids = inp.token_selected_experts.to(dev)
    wts = inp.token_final_scales.to(dev)
    x = inp.x if inp.x is not None else inp.x_q
    out = torch.zeros(cfg.M, cfg.H, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    warm = max(args.warmup, 3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(fn, clocks=False):
        for _ in range(warm):
            fn()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        clk = ClockSampler(local) if clocks else None
        if clk:
            clk.__enter__()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        if clk:
            clk.__exit__(None, None, None)
        ms_ = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
        if world > 1:
            torch.distributed.barrier()
        return ms_, (clk.summary() if clk else None)

    # ---------------- device-resident timed region
    def step():
        B.forward(x, inp.x_sf, ids, wts, inp.w1_alpha, inp.w2_alpha, out, inp.fc2_input_scale,
                  stream=stream)
    ms, clocks = timed(step, clocks=True)
    err = fm.read_error(B.fused_ws)
    if err:
        raise RuntimeError("device error word %d" % err)

    # ---------------- the same step with the atomic finalize (y never stored)
    def step_atomic():
        B.forward(x, inp.x_sf, ids, wts, inp.w1_alpha, inp.w2_alpha, out, inp.fc2_input_scale,
                  finalize_mode=fm.FINALIZE_ATOMIC, stream=stream)
    ms_atomic, _ = timed(step_atomic)

    # ---------------- the same step over two locality domains: FC1 split on I,
    # FC2 on H, each half on a green context holding half of the SMs
    localized = None
    if headline and cfg.I % 256 == 0 and cfg.H % 256 == 0 and not args.no_localized:
        try:
            doms = fm.Domains(local)
        except fm.Fp4MoeError as exc:
            localized = {"unavailable": str(exc)}
        else:
            B.prepare_domains(inp.w1, inp.w1_sf, inp.w2, inp.w2_sf)

            def step_local():
                B.forward_localized(x, inp.x_sf, ids, wts, inp.w1_alpha, inp.w2_alpha, out,
                                    doms.streams, doms.sm_count, None, inp.fc2_input_scale,
                                    stream=stream)
            ms_local, _ = timed(step_local)
            if fm.read_error(B.local_ws):
                raise RuntimeError("device error word in the localized forward")
            localized = {"ms_per_step": ms_local, "value": tokens_per_s(world, cfg.M, ms_local),
                         "unit": UNIT, "sm_per_domain": doms.sm_count,
                         "streams": "green contexts"}
            B.w1d = B.w2d = None
            B.local_ws = None
            torch.cuda.synchronize()
            doms.close()

    # ---------------- per-kernel breakdown through the staged entry points
    # (the fused call's kernels in its order: x into slot order, then GEMM1 on
    # plain row tiles; events on the launching stream around each launch)
    kernels = {}
    names = ["route_sort", "permute", "gemm1_swiglu", "gemm2", "finalize"]
    ev = {n: [] for n in names}
    px, pxsf = B.alloc_permuted()
    h, hsf = B.alloc_h()
    y = torch.zeros(B.S, cfg.H, dtype=torch.float32, device=dev)

    def launch(name):
        if name == "route_sort":
            fm.moe_route_sort(p, ids, B.e2p, B.p2e, B.tile_expert, B.tile_mn, B.num_tiles, None,
                              B.route_ws, stream)
        elif name == "permute":
            fm.moe_permute(p, x, inp.x_sf, B.p2e, B.num_tiles, px, pxsf, stream)
        elif name == "gemm1_swiglu":
            fm.moe_gemm1_swiglu(p, px, pxsf, None, B.w1p, inp.w1_alpha, inp.fc2_input_scale,
                                B.tile_expert, B.tile_mn, B.num_tiles, h, hsf, B.gemm1_ws, stream)
        elif name == "gemm2":
            fm.moe_gemm2(p, h, hsf, B.w2p, inp.w2_alpha, B.tile_expert, B.tile_mn, B.num_tiles, y,
                         B.gemm2_ws, stream)
        elif name == "finalize":
            fm.moe_finalize(p, y, B.e2p, wts, 1.0, False, out, stream)

    for it in range(warm + args.steps):
        for n in names:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            launch(n)
            b.record(stream)
            if it >= warm:
                ev[n].append((a, b))
    torch.cuda.synchronize()
    for n in names:
        kernels[n] = statistics.mean(a.elapsed_time(b) for a, b in ev[n])
    del px, pxsf, h, hsf, y

    # ---------------- end to end through host buffers.  Every step copies its
    # inputs from pinned host memory and its output back; the copies run on
    # their own streams, double-buffered, so that step i's inputs travel while
    # step i-1 computes (the way a serving loop feeds the library)
    pin = lambda t: t.detach().cpu().pin_memory()
    hx = pin(x)
    hxsf = pin(inp.x_sf) if inp.x_sf is not None else None
    hids = pin(inp.token_selected_experts)
    hw = pin(inp.token_final_scales)
    houts = [torch.empty(cfg.M, cfg.H, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dev_in = [dict(x=torch.empty_like(x), ids=torch.empty_like(ids), w=torch.empty_like(wts),
                   xsf=torch.empty_like(inp.x_sf) if inp.x_sf is not None else None)
              for _ in range(2)]
    outs = [torch.empty_like(out) for _ in range(2)]
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    in_ready, done, out_back = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    h2d = sum(t.numel() * t.element_size() for t in (hx, hids, hw) + ((hxsf,) if hxsf is not None else ()))
    d2h = houts[0].numel() * houts[0].element_size()

    def e2e_run(n):
        # step i uses buffer set b = i % 2; its copy-in waits for step i-2's
        # compute (same inputs buffer), its compute for its copy-in and for
        # step i-2's copy-out (same output buffer)
        for i in range(n):
            b = i % 2
            d = dev_in[b]
            with torch.cuda.stream(h2d_s):
                if i >= 2:
                    h2d_s.wait_event(done[b])
                d["x"].copy_(hx, non_blocking=True)
                if d["xsf"] is not None:
                    d["xsf"].copy_(hxsf, non_blocking=True)
                d["ids"].copy_(hids, non_blocking=True)
                d["w"].copy_(hw, non_blocking=True)
                in_ready[b].record(h2d_s)
            stream.wait_event(in_ready[b])
            if i >= 2:
                stream.wait_event(out_back[b])
            B.forward(d["x"], d["xsf"], d["ids"], d["w"], inp.w1_alpha, inp.w2_alpha, outs[b],
                      inp.fc2_input_scale, stream=stream)
            done[b].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(done[b])
                houts[b].copy_(outs[b], non_blocking=True)
                out_back[b].record(d2h_s)
        stream.wait_event(out_back[(n - 1) % 2])
        if n >= 2:
            stream.wait_event(out_back[(n - 2) % 2])

    e2e_run(max(args.warmup, 3))
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0.record(stream)
    h2d_s.wait_stream(stream)
    e2e_run(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
    if world > 1:
        torch.distributed.barrier()
    # the pipelined outputs are the forward's outputs
    if not torch.equal(outs[(args.steps - 1) % 2].view(torch.int16).cpu(),
                       houts[(args.steps - 1) % 2].view(torch.int16)):
        raise RuntimeError("end-to-end output copy mismatch")
    del dev_in, outs, hx, hxsf, houts

    # ---------------- roofline of the dominant kernel (GEMM1)
    peaks, peak_src = load_peaks()
    ids_np = inp.token_selected_experts.numpy()
    touched = len(np.unique(ids_np))
    H, I, M, R = cfg.H, cfg.I, cfg.M, cfg.routes
    sb = 32 if cfg.mode == "w4a8" else 16       # weight scale block: MXFP4 / NVFP4
    w1_bytes_per_expert = 2 * I * H // 2 + 2 * I * H // sb
    w2_bytes_per_expert = H * I // 2 + H * I // sb
    act1 = {"w4a16": M * H * 2, "w4a4": M * H // 2 + M * H // 16,
            "w4a8": M * H + M * H // 32}[cfg.mode]
    h_bytes = {"w4a16": R * I * 2, "w4a4": R * I // 2 + R * I // 16, "w4a8": R * I + R * I // 32}[cfg.mode]
    g1_bytes = touched * w1_bytes_per_expert + act1 + h_bytes
    g1_ms = kernels["gemm1_swiglu"]
    g1_flops = 4.0 * R * H * I
    # w4a4 (K % 256 == 0) and w4a8 (K % 128 == 0) with route tiles >= 32
    # multiply on the native block-scaled tensor-core MMAs (NVFP4; MXFP8 x
    # E4M3-stored MXFP4); everything else on BF16 / FP16 MMAs of decoded
    # weights.  Their peaks: the measured BF16 peak times the nominal dense
    # ratios 13.5 / 2.25 (FP4) and 4.5 / 2.25 (FP8) PFLOP/s.
    native = native_mma(cfg, T)
    ratio = {"nvfp4": 13.5 / 2.25, "mxfp8": 4.5 / 2.25}.get(native, 1.0)
    # a kernel timed inside a loop that lasts about a second or more runs
    # under the power cap: its denominator is the sustained cuBLAS rate
    sustained = args.steps * ms > 500.0
    bf16_peak = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
    mma_peak = bf16_peak * ratio
    # the roofline of GEMM1 is the HBM rate below the ridge (peak flops / peak
    # bytes) and the tensor rate of its MMA dtype above it
    tensor_bound = g1_flops / g1_bytes > mma_peak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    achieved_bw = g1_bytes / (g1_ms * 1e-3) / 1e9
    achieved_tf = g1_flops / (g1_ms * 1e-3) / 1e12
    step_bytes = touched * (w1_bytes_per_expert + w2_bytes_per_expert) + act1 + M * H * 2
    traffic, traffic_src = stored_traffic(cfg.name, gemm_family(cfg, T, native), T, cfg)
    g2_ms = kernels["gemm2"]
    roof = {"kernel": gemm1_kernel_name(cfg, T, native), "mma_dtype": mma_dtype(cfg, T, native)}
    if tensor_bound:
        roof.update({"bound": "tensor", "achieved": achieved_tf, "peak": mma_peak,
                     "unit": "TFLOP/s", "frac": achieved_tf / mma_peak,
                     "algorithmic_flops": g1_flops})
    else:
        roof.update({"bound": "hbm", "achieved": achieved_bw, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved_bw / peaks["hbm_gbs"],
                     "algorithmic_bytes": g1_bytes})
    roof.update({
        "traffic": traffic, "traffic_source": traffic_src,
        "peak_source": "%s (%s)" % (
            peak_src, ("bf16_tflops_sustained: GEMM1 timed inside a %.1f s loop" % (args.steps * ms / 1e3)
                       if sustained else "bf16_tflops burst") + (
                {"nvfp4": " x 13.5/2.25 nominal fp4 ratio", "mxfp8": " x 4.5/2.25 nominal fp8 ratio"}
                .get(native, ""))
            if tensor_bound else "hbm_gbs"),
        "touched_experts": touched,
        "tensor_frac": achieved_tf / mma_peak,
        "tensor_frac_of_burst": achieved_tf / (peaks["bf16_tflops"] * ratio),
        "hbm_frac": achieved_bw / peaks["hbm_gbs"],
        "gemm2": {"ms": g2_ms, "tflops": 2.0 * R * H * I / (g2_ms * 1e-3) / 1e12,
                  "tensor_frac": 2.0 * R * H * I / (g2_ms * 1e-3) / 1e12 / mma_peak},
    })
    routes_kernels = 1 if R <= 4096 else 3
    line = {
        "metric": METRIC, "value": tokens_per_s(world, cfg.M, ms), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": warm, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": (native or ("f16" if mma_dtype(cfg, T, native) == "f16" else
                             {"w4a16": "bf16", "w4a4": "nvfp4->bf16", "w4a8": "mxfp8->bf16"}[cfg.mode])),
        "data": "synthetic (seeded generator; random NVFP4 weights)",
        "config": dict(workload_config(cfg, T), l2="inputs larger than L2: %.2f GB of weights "
                       "and activations per step vs 126 MB L2" % (step_bytes / 1e9),
                       parallelism="replicas" if world > 1 else "1 GPU"),
        "tflops": world * cfg.flops() / (ms * 1e-3) / 1e12,
        "step_hbm_gbs": step_bytes / (ms * 1e-3) / 1e9,
        "roofline": roof,
        "kernels_ms": kernels,
        "atomic_finalize": {"ms_per_step": ms_atomic, "value": tokens_per_s(world, cfg.M, ms_atomic),
                            "unit": UNIT},
        "localized": localized,
        "e2e": {"value": tokens_per_s(world, cfg.M, e2e_ms), "unit": UNIT, "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "copies": "pinned host buffers; every step copies its inputs in and its output "
                          "back on two copy streams, double-buffered so that step i's copies "
                          "overlap step i-1's compute"},
        "clocks": clocks,
        # per fused step: routing (1 kernel up to 4096 routes, else 3), x in slot
        # order, GEMM1, one pass over h before GEMM2 (BF16 expansion for w4a4 on
        # BF16 MMAs and w4a8 on them, the MXFP8 scales' chunk-major copy for w4a8
        # on the MX MMA, FP16 rows for decode-size w4a16), GEMM2, finalize
        "gpu_launches": args.steps * (routes_kernels + 1 + 3 + (
            1 if (cfg.mode == "w4a16" and T <= 16) or (cfg.mode != "w4a16" and native != "nvfp4")
            else 0)),
    }
    del B, out
    torch.cuda.synchronize()
    return line, inp, T


def run_ours(args, rank, world, local):
    import torch

    import synth
    from block_scaled_fp4_sort_gb300 import build as fbuild

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        fbuild.build()
    if world > 1:
        torch.distributed.barrier()
    fbuild.build()

    def cfg_of(name):
        cfg = synth.CONFIGS[name]
        if args.tokens or args.experts:
            cfg = cfg.with_(M=args.tokens or cfg.M, E=args.experts or cfg.E, sample=0)
        return cfg

    cfg = cfg_of(args.workload)
    line, inp, T = measure(cfg, args, rank, world, local, dev, headline=True)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp.cfg, inp, T, args.cpu_budget)
    del inp
    torch.cuda.empty_cache()
    others = [] if args.also in ("", "none") else [w for w in args.also.split(",")
                                                    if w != args.workload]
    if others:
        line["workloads"] = {}
    for name in others:
        sub, sinp, sT = measure(cfg_of(name), args, rank, world, local, dev, headline=False)
        if rank == 0 and not args.no_cpu_baseline:
            sub["cpu_baseline"] = cpu_baseline(sinp.cfg, sinp, sT, args.cpu_budget / 4)
        line["gpu_launches"] += sub["gpu_launches"]
        line["workloads"][name] = {k: sub[k] for k in (
            "value", "unit", "ms_per_step", "tflops", "step_hbm_gbs", "dtype", "config", "roofline",
            "kernels_ms", "atomic_finalize", "e2e", "clocks", "gpu_launches") + (
            ("cpu_baseline",) if "cpu_baseline" in sub else ())}
        del sinp
        torch.cuda.empty_cache()
    return line


def pages_per_tile(groups, top_k, row_bytes, page=2 << 20):
    """Distinct `page`-byte pages of the activation matrix that each group of
    route slots (one GEMM1 tile) gathers from; a row may straddle two pages."""
    import numpy as np
    out = []
    for g in groups:
        rows = g[g >= 0].astype(np.int64) // top_k
        if rows.size == 0:
            continue
        lo = rows * row_bytes // page
        hi = (rows * row_bytes + row_bytes - 1) // page
        out.append(np.unique(np.concatenate([lo, hi])).size)
    return np.array(out)


def expert_groups(p2e, tile_expert, tile_mn, num_tiles, T, group):
    """Each local expert's valid slots in slot order, cut into groups of `group` routes."""
    import numpy as np
    by_e = {}
    for tau in range(num_tiles):
        e = int(tile_expert[tau])
        sl = p2e[tau * T:min(tau * T + T, int(tile_mn[tau]))]
        by_e.setdefault(e, []).append(sl)
    groups = []
    for e, parts in by_e.items():
        v = np.concatenate(parts)
        groups += [v[i:i + group] for i in range(0, v.size, group)]
    return groups


def shuffled_within_experts(p2e, tile_expert, tile_mn, num_tiles, T, seed=0):
    """Arrival-order model: each expert's routes in a seeded random order."""
    import numpy as np
    rng = np.random.default_rng(seed)
    out = p2e.copy()
    start = {}
    for tau in range(num_tiles):
        start.setdefault(int(tile_expert[tau]), []).append(tau)
    for e, taus in start.items():
        idx = np.concatenate([np.arange(t * T, min(t * T + T, int(tile_mn[t]))) for t in taus])
        out[idx] = rng.permutation(p2e[idx])
    return out


def run_locality(args):
    """Gather locality of GEMM1 (the pages' M1/M2 table): 2 MiB pages of x per
    tile under this build's stable routing order and under an arrival-order
    model, plus GEMM1 time with either order at the large batch."""
    import numpy as np
    import torch

    import block_scaled_fp4_sort_gb300 as fm
    import synth
    from block_scaled_fp4_sort_gb300 import build as fbuild
    from block_scaled_fp4_sort_gb300.buffers import MoEBuffers, problem_for

    fbuild.build()
    base = synth.CONFIGS["large_w4a16"]
    res = {"metric": "2 MiB pages of x per GEMM1 tile", "unit": "pages", "rows": []}
    for M in (65536, 131072, 262144):
        cfg = base.with_(M=M)
        ids, _ = synth.generate_routing(cfg)
        for EL, group in ((32, 256), (256, 128)):   # the pages' setting; this build's large config
            p = problem_for(cfg, 128, EL, 0)
            B = MoEBuffers(p)
            B.route(torch.from_numpy(ids).cuda())
            torch.cuda.synchronize()
            nt = int(B.num_tiles[0])
            p2e, te, tm = B.p2e.cpu().numpy(), B.tile_expert.cpu().numpy(), B.tile_mn.cpu().numpy()
            row = {"M": M, "local_experts": EL, "tile_routes": group}
            for name, order in (("stable", p2e),
                                ("arrival_model", shuffled_within_experts(p2e, te, tm, nt, 128))):
                pg = pages_per_tile(expert_groups(order, te, tm, nt, 128, group), cfg.top_k,
                                    cfg.H * 2)
                row[name] = {"mean": float(pg.mean()), "max": int(pg.max()), "tiles": int(pg.size)}
            res["rows"].append(row)
            del B
    # GEMM1 with the stable against the shuffled permutation, M = 131072
    cfg = base
    inp = synth.generate(cfg, device="cuda")
    p = problem_for(cfg, 128)
    B = MoEBuffers(p).prepare(inp.w1, inp.w1_sf, inp.w2, inp.w2_sf)
    B.route(inp.token_selected_experts.cuda())
    torch.cuda.synchronize()
    nt = int(B.num_tiles[0])
    shuf = torch.from_numpy(shuffled_within_experts(B.p2e.cpu().numpy(), B.tile_expert.cpu().numpy(),
                                                    B.tile_mn.cpu().numpy(), nt, 128)).cuda()
    h = torch.zeros(B.S, cfg.I, dtype=torch.bfloat16, device="cuda")
    times = {}
    for name, rows in (("stable", B.p2e), ("arrival_model", shuf)):
        def g1():
            fm.moe_gemm1_swiglu(p, inp.x, None, rows, B.w1p, inp.w1_alpha, None, B.tile_expert,
                                B.tile_mn, B.num_tiles, h, None, B.gemm1_ws)
        for _ in range(3):
            g1()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            g1()
        e1.record()
        torch.cuda.synchronize()
        times[name] = e0.elapsed_time(e1) / args.steps
    res["gemm1_ms_at_131072"] = times
    print(json.dumps(res))


def run_ep(args, rank, world, local):
    """Expert parallelism: every rank holds the same batch, owns a contiguous
    range of the experts, computes its fp32 partial output and joins one
    all-reduce (NCCL); moe_combine rounds the sum.  The whole job processes
    one batch: strong scaling."""
    import torch

    import synth
    from block_scaled_fp4_sort_gb300 import build as fbuild
    from block_scaled_fp4_sort_gb300.buffers import problem_for
    from block_scaled_fp4_sort_gb300.ep import ExpertParallelMoE, expert_range

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        fbuild.build()
    torch.distributed.barrier()
    fbuild.build()
    cfg = synth.CONFIGS[args.workload]
    T = args.route_tile or synth.route_tile_for(cfg)
    inp = synth.generate(cfg, device=dev)          # the same seed on every rank
    epm = ExpertParallelMoE(problem_for(cfg, T), world, rank, dev).prepare(
        inp.w1, inp.w1_sf, inp.w2, inp.w2_sf)
    ids = inp.token_selected_experts.to(dev)
    wts = inp.token_final_scales.to(dev)
    x = inp.x if inp.x is not None else inp.x_q
    out = torch.zeros(cfg.M, cfg.H, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(xx=x, ii=ids, ww=wts):
        epm.forward(xx, inp.x_sf, ii, ww, inp.w1_alpha, inp.w2_alpha, out, inp.fc2_input_scale,
                    stream=stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(fn, clocks=False):
        for _ in range(max(args.warmup, 3)):
            fn()
        torch.cuda.synchronize()
        torch.distributed.barrier()
        clk = ClockSampler(local) if clocks else None
        if clk:
            clk.__enter__()
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        if clk:
            clk.__exit__(None, None, None)
        ms_ = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
        torch.distributed.barrier()
        return ms_, (clk.summary() if clk else None)
    ms, clocks = timed(step, clocks=True)
    hx = x.detach().cpu().pin_memory()
    hids = inp.token_selected_experts.pin_memory()
    hw = inp.token_final_scales.pin_memory()
    hout = torch.empty(cfg.M, cfg.H, dtype=torch.bfloat16).pin_memory()
    dx, dids, dw = torch.empty_like(x), torch.empty_like(ids), torch.empty_like(wts)

    def e2e_step():
        dx.copy_(hx, non_blocking=True)
        dids.copy_(hids, non_blocking=True)
        dw.copy_(hw, non_blocking=True)
        step(dx, dids, dw)
        hout.copy_(out, non_blocking=True)
    e2e_ms, _ = timed(e2e_step)
    h2d = sum(t.numel() * t.element_size() for t in (hx, hids, hw))
    line = {
        "metric": METRIC, "value": cfg.M / (ms * 1e-3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms,
        "higher_is_better": True, "scaling": "strong", "vs_baseline": None,
        "dtype": mma_dtype(cfg, T, False) if cfg.mode == "w4a16" else cfg.mode,
        "data": "synthetic (seeded generator; random NVFP4 weights)",
        "config": dict(workload_config(cfg, T), parallelism="ep%d" % world,
                       experts_per_rank=[expert_range(cfg.E, world, r)[1] for r in range(world)],
                       l2="inputs larger than L2"),
        "tflops": cfg.flops() / (ms * 1e-3) / 1e12,
        "e2e": {"value": cfg.M / (e2e_ms * 1e-3), "unit": UNIT, "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": hout.numel() * 2},
        "clocks": clocks,
        "collective": "one NCCL all-reduce (sum) of the fp32 [M, H] partial per step",
        "gpu_launches": args.steps * (3 + 1 + 3 + 1),
    }
    return line


def run_reference(args, world):
    """The reference arm: the CPU oracle, as it stands, on the host cores, over
    bounded samples of the headline workload (each step a different slice of
    the seeded token sample, sized so that the whole run stays within a few
    minutes)."""
    import numpy as np
    import torch

    import oracle
    import synth
    cfg = synth.CONFIGS[args.workload]
    T = args.route_tile or synth.route_tile_for(cfg)
    # inputs are drawn on the GPU when there is one (input preparation, not
    # timed), then copied to the host for the oracle
    inp = synth.generate(cfg, device="cuda" if torch.cuda.is_available() else "cpu").to("cpu")
    oracle.build()
    orc = oracle.OracleMoE.from_inputs(inp, T=T)
    toks = oracle_tokens(cfg, inp)
    ncpu = os.cpu_count() or 1
    # calibration: one token per thread
    t0 = time.perf_counter()
    orc.forward(toks[:min(ncpu, len(toks))], nthreads=min(ncpu, len(toks)))
    per_round = time.perf_counter() - t0
    budget = 90.0 / max(1, args.steps + args.warmup)       # seconds per step
    per_step = int(min(len(toks), max(1, int(budget / max(per_round, 1e-9))) * ncpu))
    cores = min(ncpu, per_step)

    def slice_of(i):
        a = (i * per_step) % len(toks)
        return np.take(toks, np.arange(a, a + per_step), mode="wrap")
    for i in range(args.warmup):
        orc.forward(slice_of(i), nthreads=cores)
    t0 = time.perf_counter()
    for i in range(args.steps):
        orc.forward(slice_of(args.warmup + i), nthreads=cores)
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    v = per_step / dt
    sample = ("%d tokens per step from the %d-token %s of %s (each step the next slice)"
              % (per_step, len(toks), "seeded sample" if cfg.sample else "batch", cfg.name))
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(cfg, T),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample, "host_cpus": ncpu},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.locality:
        return run_locality(args)
    if args.impl == "reference":
        # rank 0 alone times the oracle; the other ranks have no work
        if rank == 0:
            run_reference(args, world)
        return
    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    if args.parallel == "ep" and world > 1:
        line = run_ep(args, rank, world, local)
    else:
        line = run_ours(args, rank, world, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
