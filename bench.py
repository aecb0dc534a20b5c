#!/usr/bin/env python
"""Benchmark of the GB300 routed-expert MoE forward.

One step = one whole forward (route -> gather -> grouped GEMM w13 -> SiLU*mul
-> grouped GEMM w2 -> scatter-add) over one batch of the workload, with the
inputs resident in HBM.  Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

Default workload: the largest one, the fine-grained-experts layer (T=4096,
D=7168, H=2048, E=128, top_k=8, bf16, Zipf-skewed routing: 2.89 TFLOP and
11.3 GB of expert weights per step).  --config decode | prefill_fp8 |
padded_fp8 | tiny | decode_zero measures the other workloads.  Under torchrun (N > 1) every rank
runs an independent replica on its own GPU (no data-path collective); the
timing is the max over ranks and the value counts the tokens of all ranks.

--impl reference times the CPU oracle (the plain reference implementation of
the method, on the host cores) on bounded token samples of the same workload.
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
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "routed-MoE tokens/s; gather/scatter HBM GB/s; grouped-GEMM TFLOP/s (1 GB300)"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 4.5 / 2.25   # nominal dense FP8 : BF16 tensor-core ratio


def load_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def workload_desc(cfg):
    tv = f" Tv={cfg.Tv}" if cfg.Tv is not None else ""
    prec = "fp8-rowwise e4m3" if cfg.fp8 else "bf16"
    ub = f" scale_ub={cfg.scale_ub:g}" if cfg.scale_ub else ""
    skew = {"uniform": "uniform routing", "zipf": "Zipf(1.1)-skewed routing",
            "zero_experts": f"experts {list(cfg.zero_experts)} get no token"}[cfg.skew]
    return f"{cfg.name}: T={cfg.T}{tv} D={cfg.D} H={cfg.H} E={cfg.E} top_k={cfg.top_k} {prec}{ub}, {skew}"


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (every 100 ms) of the SM clock and throttle reasons."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.rows, self.proc, self.thread = [], None, None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if gpu_id is not None:
            cmd += ["-i", gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 9:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


def gpu_id_for(dev) -> str | None:
    import torch

    try:
        props = torch.cuda.get_device_properties(dev)
        return f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0"
    except Exception:
        return None


# ------------------------------------------------------------ CPU oracle

def _host_bits(t):
    import numpy as np
    import torch

    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def _layer_weights_host(cfg, router, shared):
    """Router bits and shared-expert arrays (bf16 bits, or fp32 for FP8 layers) for the oracle."""
    if router is None:
        return None
    sh = None
    if shared is not None:
        conv = (lambda t: t.float().cpu().numpy()) if cfg.fp8 else _host_bits
        sh = (conv(shared[0]), conv(shared[1]))
    return _host_bits(router), sh


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), best effort."""
    import subprocess

    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def oracle_forward_tokens(cfg, toks, xb, sb, weights, layer, weighting: str):
    """The oracle forward of the sampled tokens: the routed experts on the given scores, or
    (layer = router bits and shared arrays) the whole layer; input- or output-side weighting."""
    import numpy as np

    import oracle

    if layer is not None:
        return oracle.moe_layer_forward_tokens(toks, xb, layer[0], cfg.top_k, weights, fp8=cfg.fp8, z_bf16=cfg.fp8,
                                               shared=layer[1],
                                               scale_ub=cfg.scale_ub, weighting=weighting)[0]
    if weighting == "output":
        return oracle.moe_forward_output_weighted(np.ascontiguousarray(xb[toks]), np.ascontiguousarray(sb[toks]),
                                                  cfg.top_k, weights, fp8=cfg.fp8, z_bf16=cfg.fp8,
                                                  scale_ub=cfg.scale_ub)["out"]
    return oracle.moe_forward_tokens(toks, xb, sb, cfg.top_k, weights, fp8=cfg.fp8, z_bf16=cfg.fp8,
                                     scale_ub=cfg.scale_ub)[0]


def oracle_tokens_per_s(cfg, x, s, w13, w2, seconds: float, max_tokens: int | None = None, layer=None,
                        weighting: str = "input"):
    """Time the oracle's forward (as it stands) on a bounded sample of tokens.

    Returns (tokens/s, tokens in the sample, threads, wall seconds).  The
    sample is the first n valid tokens, n grown until about `seconds` of work.
    layer: (router bits, shared-expert arrays) to time the whole layer
    (router, shared expert and routed experts) instead of the routed forward.
    """
    import numpy as np

    import oracle

    xb, sb = _host_bits(x), _host_bits(s)
    Tv = cfg.valid_tokens
    cache = {}

    def forward(toks):
        oracle_forward_tokens(cfg, toks, xb, sb, weights, layer, weighting)

    def weights(ids):
        missing = [e for e in ids if e not in cache]
        if missing:
            if cfg.fp8:
                a13, a2 = w13[missing].float().cpu().numpy(), w2[missing].float().cpu().numpy()
            else:
                a13, a2 = _host_bits(w13[missing]), _host_bits(w2[missing])
            for i, e in enumerate(missing):
                cache[e] = (a13[i], a2[i])
        return np.stack([cache[e][0] for e in ids]), np.stack([cache[e][1] for e in ids])

    n = 1
    limit = Tv if max_tokens is None else min(Tv, max_tokens)
    while True:
        toks = np.arange(n)
        weights(sorted(set(oracle.route(sb[toks], cfg.top_k)["expert_indices"].tolist())))  # warm the copy
        t0 = time.perf_counter()
        forward(toks)
        dt = time.perf_counter() - t0
        if dt >= 0.3 * seconds or n >= limit:
            break
        n = int(min(limit, max(n + 1, seconds / max(dt / n, 1e-6))))
    done, total = n, dt
    while total < 0.8 * seconds:          # a small workload is repeated until the sample is long enough
        t0 = time.perf_counter()
        forward(toks)
        total += time.perf_counter() - t0
        done += n
    return done / total, n, oracle.num_threads(), total


# ------------------------------------------------------------ multi-rank

def max_over_ranks(value: float, device) -> float:
    """The largest value over all ranks (the step time that bounds the job)."""
    import torch
    import torch.distributed as dist

    if not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank: int, world: int, max_ms_per_step: float) -> float:
    """Whole-job throughput: every rank's tokens over the slowest rank's step time."""
    return tokens_per_rank * world / (max_ms_per_step * 1e-3)


# ------------------------------------------------------------- our arm

def run_ours(args, cfg):
    import torch
    import torch.distributed as dist

    from moe_token_routing_index_gb300 import binding as mb
    from moe_token_routing_index_gb300 import workloads
    from moe_token_routing_index_gb300.forward import MoELayer

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())

    # inputs: seeded per rank (replicas process different batches of the same shape)
    x = workloads.make_tokens(cfg, seed=rank).to(dev)
    s = workloads.make_scores(cfg, seed=rank).to(dev)
    w13, w2 = workloads.make_weights(cfg, seed=0, device=dev)
    pairs = {"auto": None, "on": True, "off": False}[args.cta_pairs]
    full = args.layer == "full"
    router = shared = None
    if full:
        router = workloads.make_router(cfg, device=dev)
        shared = workloads.make_shared_weights(cfg, device=dev)
    layer = MoELayer.from_weights(cfg, w13, w2, cta_pairs=pairs, router=router, shared=shared,
                                  overlap_shared=not args.no_overlap, weighting=args.weighting)
    if args.no_cpu_baseline or world > 1 or rank != 0:
        # only the oracle baseline needs the source weights (fp32 for FP8 layers)
        del w13, w2
        w13 = w2 = None
        torch.cuda.empty_cache()
    nv = None if cfg.Tv is None else torch.tensor([cfg.Tv], dtype=torch.int32, device=dev)
    out = torch.zeros(cfg.T, cfg.D, dtype=torch.bfloat16, device=dev)
    # one forward through the public call first: it records the per-expert counts that the
    # layer's GEMM tile choice reads, then the stage list is built once for the timed steps
    layer(x, None if full else s, nv, out=out)
    torch.cuda.synchronize()
    stages = layer.stages(x, None if full else s, nv, out, accumulate=False)
    names = [n for n, _, _ in stages]

    def step(ev=None):
        layer.run(stages, events=ev)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if mb.device_error() != 0:
        raise RuntimeError("device-side error during warm-up")
    counts = layer.buffers(cfg.T, dev).route["counts"].cpu().tolist()

    def stage_pass(n_steps, only=None):
        """n_steps more steps with CUDA events around every stage (or the stage `only`)."""
        ev = [{n: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for n in names if only in (None, n)} for _ in range(n_steps)]
        return ev

    def stage_means(ev):  # the median over the steps of each stage's event time
        return {n: statistics.median(e[n][0].elapsed_time(e[n][1]) for e in ev) for n in ev[0]}

    # the dominant stage, from a short pass with events around every stage
    pre = stage_pass(min(args.warmup, 5))
    for e in pre:
        step(e)
    torch.cuda.synchronize()
    pre_ms = stage_means(pre)
    dominant = max(pre_ms, key=pre_ms.get)

    # the timed region: K steps, with events around the dominant stage only
    K = args.steps
    dom_ev = stage_pass(K, only=dominant)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu_id_for(dev))
    time.sleep(0.25)
    t_start.record()
    for k in range(K):
        step(dom_ev[k])
    t_end.record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if world > 1:
        dist.barrier()
    ms = t_start.elapsed_time(t_end) / K
    ms = max_over_ranks(ms, dev)
    # every other stage: a second pass of the same steps with events around every stage
    ev = stage_pass(min(K, 50))
    for e in ev:
        step(e)
    torch.cuda.synchronize()
    stage_ms = stage_means(ev)
    stage_ms[dominant] = stage_means(dom_ev)[dominant]      # the timed region's own measurement
    if mb.device_error() != 0:
        raise RuntimeError("device-side error during the timed steps")

    # the same forward captured into a CUDA graph and replayed K times (no host launch work)
    graph, gout = layer.capture(x, None if full else s, nv)
    for _ in range(3):
        graph.replay()
    g_start, g_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    g_start.record()
    for _ in range(K):
        graph.replay()
    g_end.record()
    torch.cuda.synchronize()
    graph_ms = max_over_ranks(g_start.elapsed_time(g_end) / K, dev)
    if mb.device_error() != 0:
        raise RuntimeError("device-side error during the graph replays")
    del graph

    e2e_ms, h2d, d2h = (None, 0, 0) if args.no_e2e else run_e2e(args, cfg, layer, x, None if full else s, nv,
                                                                 out, world)

    result = None
    if rank == 0:
        result = report(args, cfg, world, ms, stage_ms, counts, clocks, e2e_ms, h2d, d2h, layer, names)
        result["cuda_graph"] = {"value": round(job_tokens_per_s(cfg.valid_tokens, world, graph_ms), 1), "unit": UNIT,
                                "ms_per_step": round(graph_ms, 4),
                                "note": "the same step captured once and replayed K times"}
        if not args.no_cpu_baseline and world == 1:
            tps, n, cores, dt = oracle_tokens_per_s(cfg, x, s, w13, w2, args.cpu_seconds,
                                                    layer=_layer_weights_host(cfg, router, shared),
                                                    weighting=args.weighting)
            result["cpu_baseline"] = {"value": round(tps, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
                                      "cpu": cpu_model(),
                                      "sample": f"first {n} valid tokens of the workload (repeated to {dt:.1f} s of wall time)"}
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return result


def run_e2e(args, cfg, layer, x, s, nv, out, world):
    """The same forward through the public API with pinned host buffers: every
    step copies its inputs host -> device and its result device -> host.  Steps
    are pipelined over two buffer slots, as a serving loop would run them: the
    inputs of step i+1 and the result of step i-1 move on two copy streams
    while step i computes.  The timed region spans all K steps, copies included.
    Only the valid tokens move (the first Tv rows of x, of the scores and of the
    result): the padding rows of a fixed-size token buffer are neither inputs nor
    results (the layer leaves them untouched)."""
    import torch
    import torch.distributed as dist

    K = args.steps
    slots = 2
    Tv = cfg.valid_tokens
    comp = torch.cuda.current_stream()
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    xh = [x[:Tv].cpu().pin_memory() for _ in range(slots)]
    sh = [None if s is None else s[:Tv].cpu().pin_memory() for _ in range(slots)]   # the whole layer routes itself
    nvh = [None if nv is None else nv.cpu().pin_memory() for _ in range(slots)]
    outh = [torch.empty(Tv, cfg.D, dtype=torch.bfloat16).pin_memory() for _ in range(slots)]
    xd = [torch.empty_like(x) for _ in range(slots)]
    sd = [None if s is None else torch.empty_like(s) for _ in range(slots)]
    nvd = [None if nv is None else torch.empty_like(nv) for _ in range(slots)]
    outd = [torch.zeros_like(out) for _ in range(slots)]
    ev_in = [torch.cuda.Event() for _ in range(slots)]
    ev_comp = [torch.cuda.Event() for _ in range(slots)]
    ev_out = [torch.cuda.Event() for _ in range(slots)]
    for i in range(slots):           # every slot starts free
        ev_comp[i].record(comp)
        ev_out[i].record(comp)

    def e2e_step(i):
        j = i % slots
        with torch.cuda.stream(h2d_s):
            h2d_s.wait_event(ev_comp[j])           # the compute that read this slot is done
            xd[j][:Tv].copy_(xh[j], non_blocking=True)
            if sd[j] is not None:
                sd[j][:Tv].copy_(sh[j], non_blocking=True)
            if nvd[j] is not None:
                nvd[j].copy_(nvh[j], non_blocking=True)
            ev_in[j].record(h2d_s)
        comp.wait_event(ev_in[j])
        comp.wait_event(ev_out[j])                 # this slot's previous result has left the device
        layer(xd[j], sd[j], nvd[j], out=outd[j])
        ev_comp[j].record(comp)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(ev_comp[j])
            outh[j].copy_(outd[j][:Tv], non_blocking=True)
            ev_out[j].record(d2h_s)

    for i in range(max(2, min(args.warmup, 10))):
        e2e_step(i)
    torch.cuda.synchronize()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    e_start.record(comp)
    h2d_s.wait_event(e_start)
    d2h_s.wait_event(e_start)
    for i in range(K):
        e2e_step(i)
    for j in range(slots):
        comp.wait_event(ev_out[j])
    e_end.record(comp)
    torch.cuda.synchronize()
    e2e_ms = e_start.elapsed_time(e_end) / K
    e2e_ms = max_over_ranks(e2e_ms, x.device)
    h2d = xh[0].numel() * xh[0].element_size() + (0 if sh[0] is None else sh[0].numel() * sh[0].element_size()) + \
        (0 if nvh[0] is None else 4)
    d2h = outh[0].numel() * outh[0].element_size()
    return e2e_ms, h2d, d2h


def report(args, cfg, world, ms, stage_ms, counts, clocks, e2e_ms, h2d, d2h, layer, names):
    peaks, peak_kind = load_peaks()
    E, D, H, k = cfg.E, cfg.D, cfg.H, cfg.top_k
    a = cfg.routed_rows
    active = sum(1 for c in counts[:E] if c > 0)
    wb = 1 if cfg.fp8 else 2        # weight / activation element bytes into the GEMMs
    tokens = cfg.valid_tokens * world
    value = job_tokens_per_s(cfg.valid_tokens, world, ms)

    # algorithmic work per stage (one launch each per step)
    gemm1 = "gemm_w13_silu_quant" if cfg.fp8 else "gemm_w13_silu"
    mlp_bytes = (active * 3 * H * D * wb + a * D * wb + a * H * 2 * 2 + a * D * 2)
    work = {
        "route": ("hbm", cfg.valid_tokens * E * 2 + a * 12 + 8 * (E + 1)),
        "expert_mlp": ("gemm", mlp_bytes, 2.0 * a * 3 * H * D),
        ("gather_quant" if cfg.fp8 else "gather"): ("hbm", cfg.valid_tokens * D * 2 + a * D * wb + a * (14 if cfg.fp8 else 10)),
        # FP8: the SILU_MUL_QUANT epilogue writes bf16 z, and its row pass reads it and writes e4m3 z + scales
        gemm1: ("gemm", active * 2 * H * D * wb + a * D * wb + a * (H * 2 * 2 + H + 8 if cfg.fp8 else H * 2),
                2.0 * a * 2 * H * D),
        "gemm_w2": ("gemm", active * D * H * wb + a * H * wb + a * D * 2, 2.0 * a * D * H),
        "scatter": ("hbm", a * D * 2 + cfg.valid_tokens * D * 2 + (a * 4 if k > 1 else 0)),
    }
    # top-k finalize: the weighted rows, weights and indices in, the tokens out (+ the shared output read)
    work["finalize"] = ("hbm", a * D * 2 + a * 8 + cfg.valid_tokens * D * 2 * (2 if layer.shared else 1))
    full = args.layer == "full"
    if full:
        Tv = cfg.valid_tokens
        Hs = layer.Hs
        # the router GEMM with the top-k selection in its epilogue, and the routing's emit kernel
        work["router_route"] = ("hbm", Tv * D * 2 + E * D * 2 + Tv * E * 2 + a * 12 + 8 * (E + 1))
        work["shared_mlp"] = ("gemm", 3 * Hs * D * 2 + Tv * D * 2 + Tv * Hs * 2 * 2 + Tv * D * 2,
                              2.0 * Tv * 3 * Hs * D)
        work["shared_w13_silu"] = ("gemm", 2 * Hs * D * 2 + Tv * D * 2 + Tv * Hs * 2, 2.0 * Tv * 2 * Hs * D)
        work["shared_quant"] = ("hbm", Tv * D * 2 + Tv * D + Tv * 16)
        work["shared_w13_silu_quant"] = ("gemm", 2 * Hs * D + Tv * D + Tv * 4 + Tv * (Hs * 2 * 2 + Hs + 4),
                                         2.0 * Tv * 2 * Hs * D)
        work["shared_w2"] = ("gemm", D * Hs * wb + Tv * Hs * wb + Tv * D * 2, 2.0 * Tv * D * Hs)
        # the routed combine adds into the shared expert's output: one more read of it
        comb = layer.combine_stage(names)
        if comb != "finalize":
            kind, *w = work[comb]
            work[comb] = (kind, w[0] + Tv * D * 2, *w[1:])
    peak_t = peaks["bf16_tflops_sustained"] * (FP8_OVER_BF16 if cfg.fp8 else 1.0)
    gemm_stages = [n for n in stage_ms if work[n][0] == "gemm"]
    stages = {}
    for name, t in stage_ms.items():
        kind, *w = work[name]
        d = {"us": round(t * 1e3, 2)}
        if kind == "hbm":
            d["GB/s"] = round(w[0] / (t * 1e-3) / 1e9, 1)
            d["hbm_frac"] = round(d["GB/s"] / peaks["hbm_gbs"], 3)
        else:
            d["GB/s"] = round(w[0] / (t * 1e-3) / 1e9, 1)
            d["TFLOP/s"] = round(w[1] / (t * 1e-3) / 1e12, 1)
            d["hbm_frac"] = round(d["GB/s"] / peaks["hbm_gbs"], 3)
            d["tensor_frac"] = round(d["TFLOP/s"] / peak_t, 3)
        stages[name] = d
    dom = max(stage_ms, key=stage_ms.get)
    kind, *w = work[dom]
    t_dom = stage_ms[dom] * 1e-3
    if kind == "gemm" and w[1] / (peak_t * 1e12) > w[0] / (peaks["hbm_gbs"] * 1e9):
        roof = {"bound": "tensor", "achieved": round(w[1] / t_dom / 1e12, 1), "peak": round(peak_t, 1),
                "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": round(w[0] / t_dom / 1e9, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    roof["kernel"] = dom
    roof["peak_source"] = f"{peak_kind} ({'sustained bf16 x nominal fp8/bf16 ratio' if cfg.fp8 and roof['bound'] == 'tensor' else 'MEASURED_PEAKS.json'})"
    roof["traffic"] = traffic_for(cfg.name, dom)
    roof["algorithmic_bytes"] = int(w[0])
    if kind == "gemm":
        roof["algorithmic_flops"] = w[1]

    res = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3" if cfg.fp8 else "bf16",
        "data": ("synthetic, seeded: x~N(0,1), router N(0,1/D) (logits ~N(0,1)), routed and shared expert "
                 "weights N(0,0.02) random init") if full else
                "synthetic, seeded: x~N(0,1), scores=bf16(sigmoid(N(0,1) logits)), expert weights N(0,0.02) random init",
        "config": {"workload": workload_desc(cfg) + (" + router + shared expert" if full else ""),
                   "layer": "router + shared expert + routed experts" if full else "routed experts",
                   "weighting": args.weighting,
                   "T": cfg.T, "valid_tokens": cfg.valid_tokens, "D": D, "H": H,
                   "E": E, "top_k": k, "routed_rows": a, "active_experts": active,
                   "l2": "inputs larger than L2: each step streams the active experts' weights "
                         f"({(active * 3 * H * D * wb) / 1e9:.2f} GB) from HBM",
                   "parallelism": "replicas" if world == 1 else f"{world} independent replicas (weak scaling)"},
        "roofline": roof,
        "stages": stages,
        "gemm_tflops": round(sum(work[n][2] for n in gemm_stages) / (sum(stage_ms[n] for n in gemm_stages) * 1e-3)
                             / 1e12, 1),
        "e2e": None if e2e_ms is None else {
            "value": round(job_tokens_per_s(cfg.valid_tokens, world, e2e_ms), 1), "unit": UNIT,
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
            "method": "pinned host buffers, 2 slots: step i+1's H2D and step i-1's D2H on copy streams overlap "
                      "step i's compute"},
        "gpu_launches": layer.kernel_launches(cfg.T, with_router=full) * args.steps,
        "clocks": clocks,
    }
    return res


# ncu dram__bytes_read.sum + dram__bytes_write.sum per launch of the stage's kernels, from
# the captures summarised under profiles/, with the hash of the kernel sources they were
# taken on (one file, or a tuple of files for a stage of two kernels): when those sources
# change the figure no longer applies and is reported as null.
TRAFFIC: dict = {
    # the w13 GEMM alone, active experts only (moe_token_routing_index_gb300.cases w13 fine_grained)
    ("fine_grained", "gemm_w13_silu"): (2_077_630_720 + 134_013_184, "grouped_gemm.cu", "e0257906703a"),
    ("decode", "expert_mlp"): (4_037_685_504 + 5_910_016, "grouped_gemm.cu", "e0257906703a"),
    # the GEMM and its quantising row pass (cases w13 prefill_fp8 / padded_fp8)
    ("prefill_fp8", "gemm_w13_silu_quant"): (1_385_728_768 + 126_059_520 + 134_234_624 + 29_979_392,
                                             ("grouped_gemm.cu", "rowwise.cu"), "cd11016e2830"),
    ("padded_fp8", "gemm_w13_silu_quant"): (1_792_874_496 + 128_456_448 + 135_185_152 + 32_439_296,
                                            ("grouped_gemm.cu", "rowwise.cu"), "cd11016e2830"),
}


def _code_only(text: str) -> str:
    """C/C++ source without comments and with whitespace runs collapsed, so that an edit
    of comments or layout does not retire a figure taken on the same code."""
    import re

    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(name) -> str:
    """sha1 (12 hex digits) of the code of a kernel source (or of several, in order) and of
    every local header it reaches through `#include "..."`, in first-reach order (comments
    and whitespace dropped): counters captured on one build are reported only while that
    code is unchanged."""
    import hashlib
    import re

    csrc = ROOT / "moe_token_routing_index_gb300" / "csrc"
    seen, order = set(), []

    def visit(path: Path) -> None:
        path = path.resolve()
        if path in seen:
            return
        seen.add(path)
        order.append(path)
        for inc in re.findall(r'^\s*#\s*include\s+"([^"]+)"', path.read_text(), re.M):
            visit(path.parent / inc)

    for n in ((name,) if isinstance(name, str) else name):
        visit(csrc / n)
    h = hashlib.sha1()
    for f in order:
        h.update(_code_only(f.read_text()).encode())
    return h.hexdigest()[:12]


def traffic_for(workload: str, stage: str):
    t = TRAFFIC.get((workload, stage))
    if t is None or kernel_source_hash(t[1]) != t[2]:
        return None
    return t[0]


# ------------------------------------------------------- reference arm

def run_reference(args, cfg):
    """The CPU oracle, as it stands, on the host cores: each step is a bounded
    token sample of the workload; rank 0 only."""
    import torch

    from moe_token_routing_index_gb300 import workloads

    if int(os.environ.get("RANK", "0")) != 0:
        return None
    import oracle

    x = workloads.make_tokens(cfg)
    s = workloads.make_scores(cfg)
    wdev = "cuda" if torch.cuda.is_available() else "cpu"   # the device the GPU arm draws its weights on
    w13, w2 = workloads.make_weights(cfg, device=wdev)
    layer = None
    if args.layer == "full":
        layer = _layer_weights_host(cfg, workloads.make_router(cfg), workloads.make_shared_weights(cfg, device=wdev))
    budget = 150.0                                  # seconds for the whole --steps/--warmup run
    # calibrate the per-token cost, then size each step's sample to the budget
    tps, n, cores, dt = oracle_tokens_per_s(cfg, x, s, w13, w2, min(3.0, budget / (args.steps + args.warmup)),
                                            layer=layer, weighting=args.weighting)
    per_tok = dt / n
    n_step = int(max(1, min(cfg.valid_tokens, budget / (args.steps + args.warmup) / per_tok)))
    xb, sb = _host_bits(x), _host_bits(s)
    import numpy as np

    cache = {}

    def weights(ids):
        missing = [e for e in ids if e not in cache]
        if missing:
            a13 = w13[missing].float().cpu().numpy() if cfg.fp8 else _host_bits(w13[missing])
            a2 = w2[missing].float().cpu().numpy() if cfg.fp8 else _host_bits(w2[missing])
            for i, e in enumerate(missing):
                cache[e] = (a13[i], a2[i])
        return np.stack([cache[e][0] for e in ids]), np.stack([cache[e][1] for e in ids])

    Tv = cfg.valid_tokens

    def step(i):
        toks = np.unique((np.arange(n_step) + i * n_step) % Tv)
        oracle_forward_tokens(cfg, toks, xb, sb, weights, layer, args.weighting)
        return len(toks)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    done = sum(step(args.warmup + i) for i in range(args.steps))
    dt = time.perf_counter() - t0
    value = done / dt
    res = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 accumulate",
        "data": "synthetic, seeded (same workload generator as the GPU arm)",
        "config": {"workload": workload_desc(cfg) + (" + router + shared expert" if layer else ""),
                   "weighting": args.weighting, "sample_tokens_per_step": n_step},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                         "cpu": cpu_model(),
                         "sample": f"{n_step} valid tokens per step (of {Tv}), tokens cycling through the workload"},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(res), flush=True)
    return res


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=500)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--config", default="fine_grained")
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle CPU-baseline leg")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU work of the oracle baseline sample")
    p.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffer) measurement")
    p.add_argument("--layer", choices=["routed", "full"], default="routed",
                   help="routed: the routed-expert path from router scores; full: router scores, shared "
                        "expert and routed experts (the whole MoE layer)")
    p.add_argument("--weighting", choices=["input", "output"], default="input",
                   help="input: scores scale the expert inputs (gather*score); output: the top-k finalize weights "
                        "the expert outputs")
    p.add_argument("--no-overlap", action="store_true",
                   help="full layer: run the shared expert on the main stream instead of a second one")
    p.add_argument("--cta-pairs", choices=["auto", "on", "off"], default="auto",
                   help="256-row GEMM tiles on CTA pairs (default: when the batch has >= 256 rows per expert)")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be at least 3")
    from moe_token_routing_index_gb300 import workloads

    cfg = workloads.CONFIGS[args.config]
    if args.impl == "reference":
        return run_reference(args, cfg)
    return run_ours(args, cfg)


if __name__ == "__main__":
    main()
