"""Single-GEMM cases at the workloads' shapes, for timing and ncu captures.

    python -m moe_token_routing_index_gb300.cases w13 fine_grained [--tiles pairs|single] [--launches N]
    python -m moe_token_routing_index_gb300.cases fp8_w13 grouped|one [--tiles single|pairs] [--launches N]
    python -m moe_token_routing_index_gb300.cases rowwise <workload> [--launches N]

w13: the workload's w13 grouped GEMM as the layer runs it (SiLU*mul epilogue for bf16
layers, SiLU*mul + row quantisation for FP8 layers, tile-packed weights), with the
per-expert counts of routing the workload's scores (moe_route on the device).  Only
the active experts' weights are allocated: the GEMM never reads the others, so the
launch moves the same bytes as inside the whole forward while holding a few GB
instead of the workload's full weight set.  Inputs are random with the workload's
shapes (the values do not change the traffic or the time).

fp8_w13: the prefill-shaped FP8 w13 GEMM (8192 rows, K = 5120, N = 16384, plain
epilogue), its rows split 16 x 512 over the experts ("grouped", as the prefill
workload routes them) or all in one expert ("one").

rowwise: every bandwidth- or latency-bound kernel of the library at the workload's
shapes, on the routing of its scores: moe_router_scores and moe_router_route (router
weight of the whole-layer workload), moe_route, moe_gather_scale,
moe_gather_scale_quant, moe_silu_mul, moe_silu_mul_quant, moe_scatter_add,
moe_scatter_add_padded (the routed rows as the padded layout with one rank) and
moe_topk_finalize.  Each launch is timed alone with
CUDA events after a 256 MB write that evicts L2; the line gives the mean time, the
algorithmic bytes and GB/s (and the fraction of the measured HBM copy peak when
MEASURED_PEAKS.json sits beside the package).

Each GEMM case runs 2 warm-up launches and then N timed ones (CUDA events), and prints
one JSON line.  Every launch is the library's own kernel.
"""
from __future__ import annotations

import argparse
import json
from pathlib import Path

import torch

from . import binding as mb
from . import workloads


def _time(fn, launches: int) -> float:
    for _ in range(2):
        fn()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(launches):
        fn()
    e.record()
    torch.cuda.synchronize()
    return s.elapsed_time(e) / launches * 1e3


def case_w13(name: str, tiles: str, launches: int) -> dict:
    cfg = workloads.CONFIGS[name]
    dev = torch.device("cuda")
    scores = workloads.make_scores(cfg).to(dev)
    nv = None if cfg.Tv is None else torch.tensor([cfg.Tv], dtype=torch.int32, device=dev)
    counts = mb.moe_route(scores, cfg.top_k, nv)["counts"][: cfg.E].cpu()
    active = counts[counts > 0].to(torch.int32)
    E, D, H = int(active.numel()), cfg.D, cfg.H
    a = int(active.sum())
    g = torch.Generator(device=dev).manual_seed(0)
    w = torch.randn(E, 2 * H, D, device=dev, generator=g) * cfg.weight_std
    x = torch.randn(a, D, device=dev, generator=g)
    cd = active.to(dev)
    flags = mb.MOE_GEMM_CTA_PAIRS if tiles == "pairs" else 0
    if cfg.fp8:
        wq, ws = mb.moe_quantize_rows(w)
        del w
        w = mb.moe_pack_weights(wq)
        xq, xs = mb.moe_quantize_rows(x)
        zb = torch.empty(a, H, dtype=torch.bfloat16, device=dev)
        zq = torch.empty(a, H, dtype=torch.float8_e4m3fn, device=dev)
        zs = torch.empty(a, dtype=torch.float32, device=dev)
        ub = torch.tensor([cfg.scale_ub or 1200.0], dtype=torch.float32, device=dev)
        fn = lambda: mb.moe_grouped_gemm_fp8_rowwise(xq, w, cd, xs, ws, epilogue=mb.MOE_EPILOGUE_SILU_MUL_QUANT | flags,
                                                     out=zb, scale_ub=ub, z_out=zq, z_scale=zs)
        wb = 1
    else:
        w = mb.moe_pack_weights(w.to(torch.bfloat16))
        xb = x.to(torch.bfloat16)
        z = torch.empty(a, H, dtype=torch.bfloat16, device=dev)
        fn = lambda: mb.moe_grouped_gemm(xb, w, cd, epilogue=mb.MOE_EPILOGUE_SILU_MUL | flags, out=z)
        wb = 2
    us = _time(fn, launches)
    flops = 2.0 * a * 2 * H * D
    alg = E * 2 * H * D * wb + a * D * wb + a * H * 2
    if mb.device_error() != 0:
        raise RuntimeError("device-side error")
    return {"case": f"w13 {name}", "tiles": tiles, "experts": E, "rows": a, "max_rows": int(active.max()),
            "us": round(us, 1), "TFLOP/s": round(flops / us / 1e6, 1), "algorithmic_bytes": alg}


def case_fp8_w13(shape: str, tiles: str, launches: int) -> dict:
    cfg = workloads.CONFIGS["prefill_fp8"]
    dev = torch.device("cuda")
    E, D, H, a = cfg.E, cfg.D, cfg.H, 8192
    g = torch.Generator(device=dev).manual_seed(0)
    wq, ws = mb.moe_quantize_rows(torch.randn(E, 2 * H, D, device=dev, generator=g) * cfg.weight_std)
    w = mb.moe_pack_weights(wq)
    del wq
    xq, xs = mb.moe_quantize_rows(torch.randn(a, D, device=dev, generator=g))
    if shape == "grouped":
        counts = torch.full((E,), a // E, dtype=torch.int32, device=dev)
    else:
        counts = torch.zeros(E, dtype=torch.int32, device=dev)
        counts[0] = a
    y = torch.empty(a, 2 * H, dtype=torch.bfloat16, device=dev)
    flags = mb.MOE_GEMM_CTA_PAIRS if tiles == "pairs" else 0
    us = _time(lambda: mb.moe_grouped_gemm_fp8_rowwise(xq, w, counts, xs, ws, epilogue=flags, out=y), launches)
    if mb.device_error() != 0:
        raise RuntimeError("device-side error")
    return {"case": f"fp8_w13 {shape}", "tiles": tiles, "us": round(us, 1),
            "TFLOP/s": round(2.0 * a * 2 * H * D / us / 1e6, 1)}


def _time_cold(fn, launches: int, flush: torch.Tensor) -> float:
    """Mean us of `launches` launches of fn, each timed alone after a write of `flush`."""
    fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(launches)]
    for s, e in ev:
        flush.zero_()
        s.record()
        fn()
        e.record()
    torch.cuda.synchronize()
    return sum(s.elapsed_time(e) for s, e in ev) / launches * 1e3


def case_rowwise(name: str, launches: int) -> dict:
    cfg = workloads.CONFIGS[name]
    dev = torch.device("cuda")
    T, D, H, E, k = cfg.T, cfg.D, cfg.H, cfg.E, cfg.top_k
    Tv = cfg.valid_tokens
    a = Tv * k
    x = workloads.make_tokens(cfg).to(dev)
    scores = workloads.make_scores(cfg).to(dev)
    nv = None if cfg.Tv is None else torch.tensor([cfg.Tv], dtype=torch.int32, device=dev)
    ws = torch.empty(max(mb.moe_route_workspace_size(T, E, k), 1), dtype=torch.uint8, device=dev)
    r = mb.moe_route(scores, k, nv, with_weights=True, workspace=ws)
    ti, ei, inv, tw = r["token_indices"], r["expert_indices"], r["inv_rows"], r["topk_weights"]
    counts = r["counts"][:E].contiguous()
    g = torch.Generator(device=dev).manual_seed(1)
    y = torch.randn(a, 2 * H, device=dev, generator=g).to(torch.bfloat16)
    # GEMM2 rows: T * top_k of them, the layout moe_scatter_add_padded takes (the first a are routed)
    rows = torch.randn(T * k, D, device=dev, generator=g).to(torch.bfloat16)
    xr = torch.empty(a, D, dtype=torch.bfloat16, device=dev)
    xq = torch.empty(a, D, dtype=torch.float8_e4m3fn, device=dev)
    xs = torch.empty(a, dtype=torch.float32, device=dev)
    z = torch.empty(a, H, dtype=torch.bfloat16, device=dev)
    zq = torch.empty(a, H, dtype=torch.float8_e4m3fn, device=dev)
    zs = torch.empty(a, dtype=torch.float32, device=dev)
    out = torch.zeros(T, D, dtype=torch.bfloat16, device=dev)
    fin = torch.empty(Tv, D, dtype=torch.bfloat16, device=dev)
    ub = torch.tensor([cfg.scale_ub], dtype=torch.float32, device=dev) if cfg.scale_ub else None
    valid = r["counts"][E:]   # the routed-row count on the device, as the layer passes it
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    wr = workloads.make_router(cfg, device=dev)
    rs = torch.empty(T, E, dtype=torch.bfloat16, device=dev)
    rws = torch.empty(max(mb.moe_router_workspace_size(T, D, E), 1), dtype=torch.uint8, device=dev)
    rr_ws = torch.empty(max(mb.moe_router_route_workspace_size(T, D, E, k), 1), dtype=torch.uint8, device=dev)
    _, rr_out = mb.moe_router_route(x, wr, k, nv, scores=rs, workspace=rr_ws)   # its outputs, allocated once
    router_bytes = Tv * D * 2 + E * D * 2 + Tv * E * 2
    # (callable, algorithmic bytes per launch; the per-kernel figures of the roofline table)
    kernels = {
        "moe_router_scores": (lambda: mb.moe_router_scores(x, wr, nv, out=rs, workspace=rws), router_bytes),
        "moe_router_route": (lambda: mb.moe_router_route(x, wr, k, nv, scores=rs, out=rr_out, workspace=rr_ws),
                             router_bytes + a * 12 + 8 * (E + 1)),
        "moe_route": (lambda: mb.moe_route(scores, k, nv, with_weights=True, out=r, workspace=ws),
                      Tv * E * 2 + a * 12 + 8 * (E + 1)),
        "moe_gather_scale": (lambda: mb.moe_gather_scale(x, ti, ei, scores, valid, inv_rows=inv, top_k=k, out=xr),
                             Tv * D * 2 + a * D * 2 + 10 * a),
        "moe_gather_scale_quant": (lambda: mb.moe_gather_scale_quant(x, ti, ei, scores, ub, valid, inv_rows=inv,
                                                                     top_k=k, out=xq, out_scale=xs),
                                   Tv * D * 2 + a * D + 14 * a),
        "moe_silu_mul": (lambda: mb.moe_silu_mul(y, H, valid, out=z), a * 2 * H * 2 + a * H * 2),
        "moe_silu_mul_quant": (lambda: mb.moe_silu_mul_quant(y, H, ub, valid, out=zq, out_scale=zs),
                               a * 2 * H * 2 + a * H + 4 * a),
        "moe_scatter_add": (lambda: mb.moe_scatter_add(out, rows, ti, inv, k, valid, accumulate=False),
                            a * D * 2 + Tv * D * 2 + (4 * a if k > 1 else 0)),
        "moe_scatter_add_padded": (lambda: mb.moe_scatter_add_padded(out, rows, counts, ti, inv, k, accumulate=False),
                                   a * D * 2 + Tv * D * 2 + (4 * a if k > 1 else 0)),
        "moe_topk_finalize": (lambda: mb.moe_topk_finalize(rows, tw[: Tv * k].view(Tv, k), inv[: Tv * k].view(Tv, k),
                                                           out=fin),
                              a * D * 2 + Tv * D * 2 + Tv * k * 8),
    }
    peak = None
    peaks_file = Path(__file__).resolve().parent.parent / "MEASURED_PEAKS.json"
    if peaks_file.exists():
        peak = json.loads(peaks_file.read_text()).get("hbm_gbs")
    res = {}
    for kname, (fn, byts) in kernels.items():
        us = _time_cold(fn, launches, flush)
        d = {"us": round(us, 2), "bytes": int(byts), "GB/s": round(byts / us / 1e3, 1)}
        if peak:
            d["hbm_frac"] = round(byts / us / 1e3 / peak, 3)
        res[kname] = d
    if mb.device_error() != 0:
        raise RuntimeError("device-side error")
    return {"case": f"rowwise {name}", "T": T, "valid_tokens": Tv, "routed_rows": a, "D": D, "H": H, "E": E,
            "top_k": k, "hbm_peak_gbs": peak, "kernels": res}


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("case", choices=["w13", "fp8_w13", "rowwise"])
    p.add_argument("which", help="w13, rowwise: a workload name; fp8_w13: grouped or one")
    p.add_argument("--tiles", choices=["single", "pairs"], default=None,
                   help="128-row tiles or 256-row tiles on CTA pairs (default: pairs for bf16, single for FP8)")
    p.add_argument("--launches", type=int, default=20)
    args = p.parse_args(argv)
    if args.case == "rowwise":
        res = case_rowwise(args.which, args.launches)
    elif args.case == "w13":
        cfg = workloads.CONFIGS[args.which]
        tiles = args.tiles or ("single" if cfg.fp8 else "pairs")
        res = case_w13(args.which, tiles, args.launches)
    else:
        if args.which not in ("grouped", "one"):
            p.error("fp8_w13 takes grouped or one")
        res = case_fp8_w13(args.which, args.tiles or "single", args.launches)
    print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
