"""CPU oracle for the routed-expert MoE forward (test infrastructure).

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The CUDA library and its Python binding never import
it; the product path fails loudly when the CUDA library is missing instead of
falling back to anything here.

The arithmetic lives in ``moe_oracle.c`` (plain loops, built with gcc on
first use).  This module marshals numpy arrays and composes the stages in the
order of mslk/moe/layers.py, MetaShufflingMoE._route -> _routed_expert ->
_combine_outputs:

    route -> gather*score (bf16, or e4m3 + per-row scale)
          -> grouped GEMM with w13 -> silu_mul (or silu_mul_quant)
          -> grouped GEMM with w2  -> scatter-add into the output.

The whole layer of _no_comm_forward adds the router scores
sigmoid(tokens @ router_DE) in front and the shared expert, whose output the
routed rows are added into.

bf16 values travel as ``numpy.uint16`` bit patterns, e4m3 as ``numpy.uint8``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "moe_oracle.c"
_LIB = _HERE / "liboracle.so"
_lock = threading.Lock()
_lib = None

BF16, F32 = 0, 1


def build(force: bool = False) -> Path:
    """Compile moe_oracle.c into liboracle.so (OpenMP when the compiler has it)."""
    if not force and _LIB.exists() and _LIB.stat().st_mtime >= _SRC.stat().st_mtime:
        return _LIB
    tmp = _LIB.with_suffix(f".{os.getpid()}.tmp")
    base = ["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-std=c11", str(_SRC), "-o", str(tmp)]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:] + ["-lm"], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-lm"], check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        try:
            lib = ctypes.CDLL(str(build()))
        except OSError:
            lib = ctypes.CDLL(str(build(force=True)))
        P, I, L = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        sig = {
            "oracle_num_threads": ([], I),
            "oracle_bf16_round": ([P, P, L], None),
            "oracle_bf16_to_f32": ([P, P, L], None),
            "oracle_e4m3_encode": ([P, P, L], None),
            "oracle_e4m3_decode": ([P, P, L], None),
            "oracle_quantize_rows": ([P, L, L, P, P, P], None),
            "oracle_route": ([P, I, L, L, I, I, I, I, P, P, P, P, P], I),
            "oracle_gather_scale": ([P, I, P, P, I, P, I, L, L, P], None),
            "oracle_gather_scale_quant": ([P, I, P, P, I, P, I, L, L, P, P, P], None),
            "oracle_grouped_gemm_bf16": ([P, P, P, I, I, I, P], None),
            "oracle_grouped_gemm_fp8": ([P, P, P, P, P, I, I, I, P], None),
            "oracle_silu_mul": ([P, P, L, I, I, P], None),
            "oracle_silu_mul_quant": ([P, P, L, I, I, P, P, P], None),
            "oracle_scatter_add": ([P, I, I, P, P, I], None),
            "oracle_router_scores": ([P, P, I, I, I, I, P, P], None),
            "oracle_topk_finalize": ([P, L, I, P, P, I, I, P, P], None),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes, fn.restype = args, res
        _lib = lib
        return lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return _load().oracle_num_threads()


# ------------------------------------------------------------ number formats

def bf16_round(v) -> np.ndarray:
    v = _c(v, np.float32)
    out = np.empty(v.shape, np.uint16)
    _load().oracle_bf16_round(_p(v), _p(out), v.size)
    return out


def bf16_to_f32(b) -> np.ndarray:
    b = _c(b, np.uint16)
    out = np.empty(b.shape, np.float32)
    _load().oracle_bf16_to_f32(_p(b), _p(out), b.size)
    return out


def e4m3_encode(v) -> np.ndarray:
    v = _c(v, np.float32)
    out = np.empty(v.shape, np.uint8)
    _load().oracle_e4m3_encode(_p(v), _p(out), v.size)
    return out


def e4m3_decode(b) -> np.ndarray:
    b = _c(b, np.uint8)
    out = np.empty(b.shape, np.float32)
    _load().oracle_e4m3_decode(_p(b), _p(out), b.size)
    return out


def quantize_rows(w, scale_ub: float | None = None):
    """Per-row FP8 quantisation over the last axis: (codes uint8, scales f32)."""
    w = _c(w, np.float32)
    cols = w.shape[-1]
    rows = w.size // cols if cols else 0
    q = np.empty(w.shape, np.uint8)
    s = np.empty(w.shape[:-1], np.float32)
    ub = None if scale_ub is None else np.array([scale_ub], np.float32)
    _load().oracle_quantize_rows(_p(w), rows, cols, _p(ub), _p(q), _p(s))
    return q, s


# -------------------------------------------------------------------- stages

def _scores_args(scores):
    if scores.dtype == np.uint16:
        dtype = BF16
    elif scores.dtype == np.float32:
        dtype = F32
    else:
        raise TypeError("scores must be bf16 bits (uint16) or float32")
    st, se = (s // scores.itemsize for s in scores.strides)
    return dtype, st, se


def route(scores, top_k: int, valid_tokens: int | None = None):
    """Top-k routing; returns dict(counts[E+1], offsets[E+1], expert_indices,
    token_indices, inv[Tv, k]) with the index arrays cut to Tv * k rows."""
    T, E = scores.shape
    Tv = T if valid_tokens is None else int(valid_tokens)
    dtype, st, se = _scores_args(scores)
    a = Tv * top_k
    counts = np.zeros(E + 1, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    ei = np.full(max(a, 1), -1, np.int32)
    ti = np.full(max(a, 1), -1, np.int32)
    inv = np.full(max(a, 1), -1, np.int32)
    rc = _load().oracle_route(_p(scores), dtype, st, se, T, E, top_k, Tv, _p(counts), _p(offsets),
                              _p(ei), _p(ti), _p(inv))
    if rc != 0:
        raise ValueError("oracle_route: top_k outside [1, E] or valid tokens outside [0, T]")
    return dict(counts=counts, offsets=offsets, expert_indices=ei[:a], token_indices=ti[:a],
                inv=inv[:a].reshape(Tv, top_k))


def gather_scale(x, token_indices, expert_indices, scores, valid_rows: int | None = None):
    x = _c(x, np.uint16)
    a = len(token_indices)
    v = a if valid_rows is None else int(valid_rows)
    ti, ei = _c(token_indices, np.int32), _c(expert_indices, np.int32)
    dtype, st, se = _scores_args(scores)
    out = np.zeros((a, x.shape[1]), np.uint16)
    _load().oracle_gather_scale(_p(x), x.shape[1], _p(ti), _p(ei), v, _p(scores), dtype, st, se, _p(out))
    return out


def gather_scale_quant(x, token_indices, expert_indices, scores, scale_ub: float | None = None,
                       valid_rows: int | None = None):
    x = _c(x, np.uint16)
    a = len(token_indices)
    v = a if valid_rows is None else int(valid_rows)
    ti, ei = _c(token_indices, np.int32), _c(expert_indices, np.int32)
    dtype, st, se = _scores_args(scores)
    ub = None if scale_ub is None else np.array([scale_ub], np.float32)
    out = np.zeros((a, x.shape[1]), np.uint8)
    scale = np.zeros(a, np.float32)
    _load().oracle_gather_scale_quant(_p(x), x.shape[1], _p(ti), _p(ei), v, _p(scores), dtype, st, se,
                                      _p(ub), _p(out), _p(scale))
    return out, scale


def grouped_gemm_bf16(x, w, counts):
    """x[a, K] bf16 bits, w[E, N, K] bf16 bits, counts[E] -> y[a, N] bf16 bits."""
    x, w = _c(x, np.uint16), _c(w, np.uint16)
    E, N, K = w.shape
    counts = _c(counts[:E], np.int32)
    y = np.zeros((x.shape[0], N), np.uint16)
    _load().oracle_grouped_gemm_bf16(_p(x), _p(w), _p(counts), E, N, K, _p(y))
    return y


def grouped_gemm_fp8(xq, wq, counts, x_scale, w_scale):
    """xq[a, K] e4m3, wq[E, N, K] e4m3, x_scale[a], w_scale[E, N] -> y[a, N] bf16 bits."""
    xq, wq = _c(xq, np.uint8), _c(wq, np.uint8)
    E, N, K = wq.shape
    counts = _c(counts[:E], np.int32)
    xs, ws = _c(x_scale, np.float32), _c(w_scale, np.float32)
    y = np.zeros((xq.shape[0], N), np.uint16)
    _load().oracle_grouped_gemm_fp8(_p(xq), _p(wq), _p(counts), _p(xs), _p(ws), E, N, K, _p(y))
    return y


def silu_mul(y, H: int, valid_rows: int | None = None):
    """y[a, 2H] bf16 bits -> z[a, H] = silu(y[:, :H]) * y[:, H:] (bf16 bits)."""
    y = _c(y, np.uint16)
    a = y.shape[0]
    v = a if valid_rows is None else int(valid_rows)
    z = np.zeros((a, H), np.uint16)
    _load().oracle_silu_mul(_p(y), ctypes.c_void_p(y.ctypes.data + 2 * H), y.shape[1], v, H, _p(z))
    return z


def silu_mul_quant(y, H: int, scale_ub: float | None = None, valid_rows: int | None = None, *,
                   z_bf16: bool = False):
    """y[a, 2H] bf16 bits -> (z[a, H] e4m3 codes, z_scale[a] f32): z = silu(y0) * y1
    quantised per row with the gathers' row rule (bound ``scale_ub``).

    z_bf16=False: the row rule acts on the fp32 value of z (silu_mul_quant of
    MetaShufflingMoE._fused_silu_mul, one rounding).  z_bf16=True: z is first
    rounded to bf16, as silu_mul writes it, and the row rule acts on those bf16
    values; this is the dense reference's order (BaselineMoE._forward forms
    routed_z as a bf16 tensor and _fake_quant quantises its rows) and the
    grouped GEMM's fused SiLU*mul + quantisation epilogue.  Rows >= valid_rows
    are zero.
    """
    if z_bf16:
        a = y.shape[0]
        v = a if valid_rows is None else int(valid_rows)
        zq = np.zeros((a, H), np.uint8)
        zs = np.zeros(a, np.float32)
        if v > 0:
            zb = silu_mul(y, H, v)
            zq[:v], zs[:v] = quantize_rows(bf16_to_f32(zb[:v]), scale_ub)
        return zq, zs
    y = _c(y, np.uint16)
    a = y.shape[0]
    v = a if valid_rows is None else int(valid_rows)
    ub = None if scale_ub is None else np.array([scale_ub], np.float32)
    z = np.zeros((a, H), np.uint8)
    zs = np.zeros(a, np.float32)
    _load().oracle_silu_mul_quant(_p(y), ctypes.c_void_p(y.ctypes.data + 2 * H), y.shape[1], v, H,
                                  _p(ub), _p(z), _p(zs))
    return z, zs


def scatter_add(out, rows, token_indices, valid_rows: int | None = None):
    """out[T, D] bf16 bits (updated in place and returned), rows[a, D] bf16 bits."""
    assert out.dtype == np.uint16 and out.flags.c_contiguous
    rows = _c(rows, np.uint16)
    ti = _c(token_indices, np.int32)
    v = len(ti) if valid_rows is None else int(valid_rows)
    _load().oracle_scatter_add(_p(out), out.shape[0], out.shape[1], _p(rows), _p(ti), v)
    return out


# ------------------------------------------------------------ router scores

def router_scores(x, w_router, valid_tokens: int | None = None, logits: bool = False):
    """x[T, D] bf16 bits, w_router[E, D] bf16 bits (router_DE transposed).

    Returns scores[T, E] bf16 bits (rows >= valid_tokens are zero), and the
    bf16 logits as well when ``logits``.
    """
    x = _c(x, np.uint16)
    w = _c(w_router, np.uint16)
    T, D = x.shape
    E = w.shape[0]
    assert w.shape[1] == D
    v = T if valid_tokens is None else int(valid_tokens)
    sc = np.zeros((T, E), np.uint16)
    lg = np.zeros((T, E), np.uint16) if logits else None
    _load().oracle_router_scores(_p(x), _p(w), T, D, E, v, _p(sc), _p(lg))
    return (sc, lg) if logits else sc


# ------------------------------------------------------------------- forward

def moe_forward(x, scores, top_k: int, weights, *, fp8: bool, valid_tokens: int | None = None,
                out_init=None, scale_ub: float | None = None, H: int | None = None, z_bf16: bool = False):
    """The routed-expert forward of MetaShufflingMoE._no_comm_forward (one GPU,
    no shared expert), on the CPU.

    x[T, D] bf16 bits; scores[T, E] bf16 bits or f32.  ``weights(ids)`` returns
    the weights of the experts ``ids`` (ascending) as (w13[n, 2H, D],
    w2[n, D, H]): bf16 bits, or fp32 when ``fp8`` (quantised per row here).
    out_init[T, D] (bf16 bits) is the tensor the routed rows are added into
    (zeros when None).  z_bf16: on the FP8 path, z is rounded to bf16 before its
    row quantisation (see silu_mul_quant).  Returns the final output and every
    intermediate.
    """
    T, D = x.shape
    E = scores.shape[1]
    r = route(scores, top_k, valid_tokens)
    a = int(r["counts"][E])
    counts = r["counts"][:E]
    used = [e for e in range(E) if counts[e] > 0]
    cu = counts[used] if used else np.zeros(0, np.int32)
    res = dict(route=r, used_experts=used)
    out = np.zeros((T, D), np.uint16) if out_init is None else np.array(out_init, np.uint16, copy=True)
    if a == 0:
        res["out"] = out
        return res
    w13, w2 = weights(used)
    Hd = w2.shape[2] if H is None else H
    if not fp8:
        xg = gather_scale(x, r["token_indices"], r["expert_indices"], scores)
        y = grouped_gemm_bf16(xg, w13, cu)
        z = silu_mul(y, Hd)
        o = grouped_gemm_bf16(z, w2, cu)
        res.update(x_routed=xg, y=y, z=z, o=o)
    else:
        w13q, w13s = quantize_rows(w13)
        w2q, w2s = quantize_rows(w2)
        xq, xs = gather_scale_quant(x, r["token_indices"], r["expert_indices"], scores, scale_ub)
        y = grouped_gemm_fp8(xq, w13q, cu, xs, w13s)
        zq, zs = silu_mul_quant(y, Hd, scale_ub, z_bf16=z_bf16)
        o = grouped_gemm_fp8(zq, w2q, cu, zs, w2s)
        res.update(x_routed=xq, x_scale=xs, y=y, z=zq, z_scale=zs, o=o,
                   w13q=w13q, w13s=w13s, w2q=w2q, w2s=w2s)
    scatter_add(out, o, r["token_indices"])
    res["out"] = out
    return res


def moe_forward_tokens(tokens, x, scores, top_k: int, weights, *, fp8: bool, out_init=None,
                       scale_ub: float | None = None, z_bf16: bool = False):
    """The forward's output rows for a sample of tokens only.

    Every stage of the forward works row by row (routing per token, gather and
    quantisation per routed row, GEMMs per row, the combine per token in
    ascending expert order), so running it on the sampled tokens alone gives
    exactly those tokens' rows of the full forward.  ``tokens`` must be valid
    token ids.  Returns (out[len(tokens), D], the sub-forward's dict).
    """
    tokens = np.asarray(tokens, np.int64)
    xs = np.ascontiguousarray(x[tokens])
    ss = np.ascontiguousarray(scores[tokens])
    oi = None if out_init is None else np.ascontiguousarray(out_init[tokens])
    res = moe_forward(xs, ss, top_k, weights, fp8=fp8, out_init=oi, scale_ub=scale_ub, z_bf16=z_bf16)
    return res["out"], res


# ----------------------------------------------------------- top-k finalize

def topk_weights(scores, r):
    """The routing weights in the order of the route's inverse permutation:
    w[t, j] = f32(scores[t, expert of row inv[t, j]]) (the top-k values)."""
    sc = np.asarray(scores)
    if sc.dtype == np.uint16:
        sc = bf16_to_f32(sc)
    inv = np.asarray(r["inv"])
    e = np.asarray(r["expert_indices"])[inv]
    t = np.arange(inv.shape[0])[:, None]
    return np.ascontiguousarray(sc[t, e], np.float32)


def topk_finalize(rows, weights, idx, shared=None):
    """rows[n, D] bf16 bits, weights fp32 [M, k], idx int32 [M, k] (-1: absent),
    shared bf16 bits [M, D] or None -> out[M, D] bf16 bits."""
    rows = _c(rows, np.uint16)
    w = _c(weights, np.float32)
    ix = _c(idx, np.int32)
    M, k = ix.shape
    D = rows.shape[1]
    sh = None if shared is None else _c(shared, np.uint16)
    out = np.zeros((M, D), np.uint16)
    _load().oracle_topk_finalize(_p(rows), rows.shape[0], D, _p(w), _p(ix), M, k, _p(sh), _p(out))
    return out


def moe_forward_output_weighted(x, scores, top_k: int, weights, *, fp8: bool, valid_tokens: int | None = None,
                                shared_out=None, scale_ub: float | None = None, z_bf16: bool = False):
    """The routed experts with the routing weights applied to the expert outputs
    (top-k finalize) instead of their inputs: route -> gather (unit scores) ->
    grouped GEMM w13 -> silu_mul(_quant) -> grouped GEMM w2 -> topk_finalize with
    the top-k values in inverse-permutation order, plus ``shared_out`` when given.
    Returns the dict of the stages; out[t] for t >= valid_tokens is zero."""
    T, D = x.shape
    E = scores.shape[1]
    v = T if valid_tokens is None else int(valid_tokens)
    r = route(scores, top_k, v)
    counts = r["counts"][:E]
    used = [e for e in range(E) if counts[e] > 0]
    out = np.zeros((T, D), np.uint16)
    res = dict(route=r, used_experts=used)
    if not used:
        if shared_out is not None:
            out[:v] = topk_finalize(np.zeros((0, D), np.uint16), np.zeros((v, top_k), np.float32),
                                    np.full((v, top_k), -1, np.int32), shared_out[:v])
        res["out"] = out
        return res
    cu = counts[used]
    w13, w2 = weights(used)
    Hd = w2.shape[2]
    unit = np.full((T, E), 0x3F80, np.uint16)       # bf16 1.0: the gather copies the row
    if not fp8:
        xg = gather_scale(x, r["token_indices"], r["expert_indices"], unit)
        z = silu_mul(grouped_gemm_bf16(xg, w13, cu), Hd)
        o = grouped_gemm_bf16(z, w2, cu)
    else:
        w13q, w13s = quantize_rows(w13)
        w2q, w2s = quantize_rows(w2)
        xq, xs = gather_scale_quant(x, r["token_indices"], r["expert_indices"], unit, scale_ub)
        zq, zs = silu_mul_quant(grouped_gemm_fp8(xq, w13q, cu, xs, w13s), Hd, scale_ub, z_bf16=z_bf16)
        o = grouped_gemm_fp8(zq, w2q, cu, zs, w2s)
    wts = topk_weights(scores, r)
    out[:v] = topk_finalize(o, wts, r["inv"], None if shared_out is None else shared_out[:v])
    res.update(o=o, topk_weights=wts, out=out)
    return res


# ------------------------------------------------------------ shared expert

def shared_expert(x, w13, w2, *, fp8: bool, scale_ub: float | None = None, valid_tokens: int | None = None,
                  z_bf16: bool = False):
    """The shared expert of MetaShufflingMoE._shared_expert_part1 / _part2 on
    the valid token rows: y = x @ w13.T, z = silu_mul(y0, y1), out = z @ w2.T.

    w13[2H, D], w2[D, H]: bf16 bits, or fp32 when ``fp8``.  On the FP8-rowwise
    path the weights are quantised per row here, x per row with the gathers'
    row rule at unit score (bound ``scale_ub``), and z by silu_mul_quant
    (``z_bf16`` as there).
    Returns out[T, D] bf16 bits; rows >= valid_tokens stay zero.
    """
    T, D = x.shape
    v = T if valid_tokens is None else int(valid_tokens)
    out = np.zeros((T, D), np.uint16)
    if v == 0:
        return out
    counts = np.array([v], np.int32)
    H = w2.shape[-1]
    if not fp8:
        y = grouped_gemm_bf16(x[:v], np.asarray(w13)[None], counts)
        z = silu_mul(y, H)
        out[:v] = grouped_gemm_bf16(z, np.asarray(w2)[None], counts)
    else:
        w13q, w13s = quantize_rows(w13)
        w2q, w2s = quantize_rows(w2)
        xq, xs = quantize_rows(bf16_to_f32(x[:v]), scale_ub)
        y = grouped_gemm_fp8(xq, w13q[None], counts, xs, w13s)
        zq, zs = silu_mul_quant(y, H, scale_ub, z_bf16=z_bf16)
        out[:v] = grouped_gemm_fp8(zq, w2q[None], counts, zs, w2s)
    return out


def moe_layer_forward(x, w_router, top_k: int, weights, *, fp8: bool, shared=None,
                      valid_tokens: int | None = None, scale_ub: float | None = None, weighting: str = "input",
                      z_bf16: bool = False):
    """The whole MoE layer of MetaShufflingMoE._no_comm_forward on one GPU:
    router scores, the shared expert (``shared`` = (w13, w2), or None for a
    layer without one), and the routed experts added into its output
    (``weighting`` "input": scores scale the expert inputs; "output": the top-k
    finalize weights the expert outputs and adds the shared output;
    ``z_bf16`` as in silu_mul_quant, for the routed and the shared expert).
    Returns the routed forward's dict plus ``scores`` and ``shared_out``.
    """
    scores = router_scores(x, w_router, valid_tokens)
    base = None
    if shared is not None:
        base = shared_expert(x, shared[0], shared[1], fp8=fp8, scale_ub=scale_ub, valid_tokens=valid_tokens,
                             z_bf16=z_bf16)
    if weighting == "output":
        res = moe_forward_output_weighted(x, scores, top_k, weights, fp8=fp8, valid_tokens=valid_tokens,
                                          shared_out=base, scale_ub=scale_ub, z_bf16=z_bf16)
    else:
        res = moe_forward(x, scores, top_k, weights, fp8=fp8, valid_tokens=valid_tokens, out_init=base,
                          scale_ub=scale_ub, z_bf16=z_bf16)
    res["scores"] = scores
    res["shared_out"] = base
    return res


def moe_layer_forward_tokens(tokens, x, w_router, top_k: int, weights, *, fp8: bool, shared=None,
                             scale_ub: float | None = None, weighting: str = "input", z_bf16: bool = False):
    """moe_layer_forward's output rows for a sample of valid tokens: every stage,
    the router and the shared expert included, works token by token."""
    tokens = np.asarray(tokens, np.int64)
    res = moe_layer_forward(np.ascontiguousarray(x[tokens]), w_router, top_k, weights, fp8=fp8, shared=shared,
                            scale_ub=scale_ub, weighting=weighting, z_bf16=z_bf16)
    return res["out"], res
