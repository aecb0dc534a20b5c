"""ctypes binding of libmoe_gb300 (include/moe.h), with the same entry-point names.

Argument marshalling only: tensors become device pointers and sizes, the
current PyTorch stream becomes the cudaStream_t, and a non-zero status raises
MoEError.  Output tensors may be passed in (pre-allocated, e.g. to keep rows
past the valid count untouched) or are allocated here with torch.empty.
Every computation runs in the library's CUDA kernels; loading fails loudly if
the library has not been built.
"""
from __future__ import annotations

import ctypes
import re
from pathlib import Path

import torch

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "libmoe_gb300.so"
HEADER = _PKG.parent / "include" / "moe.h"

MOE_OK, MOE_ERR_INVALID, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_WORKSPACE = 0, -1, -2, -3, -4
MOE_DTYPE_BF16, MOE_DTYPE_F32, MOE_DTYPE_E4M3 = 0, 1, 2
MOE_EPILOGUE_NONE, MOE_EPILOGUE_SILU_MUL, MOE_EPILOGUE_SILU_MUL_QUANT = 0, 1, 2
MOE_GEMM_CTA_PAIRS = 0x100
MOE_WEIGHTS_PACKED = 0x200
MOE_DEVERR_BAD_INDEX, MOE_DEVERR_BAD_COUNT, MOE_DEVERR_TIMEOUT = 1, 2, 4


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int, cuda_error: int = 0):
        self.status = status
        msg = f"{fn} failed: {_lib.moe_status_string(status).decode()} ({status})"
        if status == MOE_ERR_CUDA:
            msg += f", cudaError {cuda_error}"
        super().__init__(msg)


def _load() -> ctypes.CDLL:
    if not LIB_PATH.exists():
        raise ImportError(f"{LIB_PATH.name} is not built: run `python -m moe_token_routing_index_gb300.build` "
                          "(the CUDA library is required; there is no fallback)")
    lib = ctypes.CDLL(str(LIB_PATH))
    P, I, L, S, U = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.POINTER(ctypes.c_uint)
    sigs = {
        "moe_status_string": ([I], ctypes.c_char_p),
        "moe_last_cuda_error": ([], I),
        "moe_device_error": ([U, P], I),
        "moe_router_workspace_size": ([I, I, I, ctypes.POINTER(S)], I),
        "moe_router_scores": ([P, I, I, P, I, P, P, P, S, P], I),
        "moe_router_route_workspace_size": ([I, I, I, I, ctypes.POINTER(S)], I),
        "moe_router_route": ([P, I, I, P, I, I, P, P, P, P, P, P, P, P, P, S, P], I),
        "moe_dense_gemm": ([P, I, I, P, I, P, P, I, P], I),
        "moe_selftest_bounded_wait": ([I, L, P], I),
        "moe_route_workspace_size": ([I, I, I, ctypes.POINTER(S)], I),
        "moe_route": ([P, I, L, L, I, I, I, P, P, P, P, P, P, P, P, S, P], I),
        "moe_route_no_alloc": ([P, I, L, L, I, I, I, P, P, P, P, P, P, P], I),
        "moe_gather_scale": ([P, I, I, P, P, I, P, I, L, L, I, P, P, I, P, P], I),
        "moe_gather_scale_quant": ([P, I, I, P, P, I, P, I, L, L, I, P, P, I, P, P, P, P], I),
        "moe_quantize_rows": ([P, L, I, P, P, P, P], I),
        "moe_grouped_gemm": ([P, P, P, I, I, I, I, P, I, P, I, I, P, P, P, P], I),
        "moe_expert_mlp_workspace_size": ([I, ctypes.POINTER(S)], I),
        "moe_scatter_add_padded": ([P, P, P, I, P, P, I, I, I, I, I, P], I),
        "moe_topk_finalize": ([P, L, I, P, I, P, I, I, P, P, P, P], I),
        "moe_expert_mlp": ([P, P, P, P, I, I, I, I, P, P, P, I, I, P, S, I, P], I),
        "moe_pack_weights_size": ([I, I, I, I, ctypes.POINTER(S)], I),
        "moe_pack_weights": ([P, I, I, I, I, P, P], I),
        "moe_grouped_gemm_fp8_rowwise": ([P, P, P, P, P, I, I, I, I, P, I, P, I, I, P, P, P, P], I),
        "moe_silu_mul": ([P, P, L, I, I, P, P, P], I),
        "moe_silu_mul_quant": ([P, P, L, I, I, P, P, P, P, P], I),
        "moe_scatter_add": ([P, P, P, P, I, I, I, I, P, I, P], I),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes, fn.restype = args, res
    return lib


_lib = _load()


def header_symbols() -> list[str]:
    """Names of the functions include/moe.h declares."""
    text = HEADER.read_text()
    return sorted(set(re.findall(r"^(?:int|const char\*)\s+(moe_\w+)\s*\(", text, flags=re.M)))


def library() -> ctypes.CDLL:
    return _lib


def _check(fn: str, status: int):
    if status != MOE_OK:
        raise MoEError(fn, status, _lib.moe_last_cuda_error() if status == MOE_ERR_CUDA else 0)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return MOE_DTYPE_BF16
    if t.dtype == torch.float32:
        return MOE_DTYPE_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _need(t: torch.Tensor, dtype, name: str, contiguous: bool = True):
    """dtype, device and layout checks of a matrix argument: the C ABI reads it as a
    dense row-major array (contiguous=False: only the last dimension must be dense)."""
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if not contiguous and t.dim() > 0 and t.stride(-1) != 1:
        raise ValueError(f"{name} must be dense along its last dimension")


def device_error(stream=None) -> int:
    """Read and clear the device-side error bits (synchronises the stream)."""
    bits = ctypes.c_uint(0)
    _check("moe_device_error", _lib.moe_device_error(ctypes.byref(bits), _stream(stream)))
    return bits.value


# ------------------------------------------------------------------ routing

def moe_router_workspace_size(T: int, D: int, E: int) -> int:
    n = ctypes.c_size_t(0)
    _check("moe_router_workspace_size", _lib.moe_router_workspace_size(T, D, E, ctypes.byref(n)))
    return n.value


def moe_router_scores(x: torch.Tensor, w_router: torch.Tensor, num_valid_tokens: torch.Tensor | None = None, *,
                      out: torch.Tensor | None = None, workspace: torch.Tensor | None = None, stream=None):
    """scores[T, E] = bf16(sigmoid(bf16(x @ w_router.T))) for x[T, D] and w_router[E, D] (bf16)."""
    T, D = x.shape
    E = w_router.shape[0]
    _need(x, torch.bfloat16, "x")
    _need(w_router, torch.bfloat16, "w_router")
    if num_valid_tokens is not None:
        _need(num_valid_tokens, torch.int32, "num_valid_tokens")
    if out is None:
        out = torch.empty(T, E, dtype=torch.bfloat16, device=x.device)
    _need(out, out.dtype, "out")
    ws_bytes = moe_router_workspace_size(T, D, E)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=x.device)
    st = _lib.moe_router_scores(_ptr(x), T, D, _ptr(w_router), E, _ptr(num_valid_tokens), _ptr(out),
                                _ptr(workspace), workspace.numel(), _stream(stream))
    _check("moe_router_scores", st)
    return out


def moe_router_route_workspace_size(T: int, D: int, E: int, top_k: int) -> int:
    n = ctypes.c_size_t(0)
    _check("moe_router_route_workspace_size", _lib.moe_router_route_workspace_size(T, D, E, top_k, ctypes.byref(n)))
    return n.value


def moe_router_route(x: torch.Tensor, w_router: torch.Tensor, top_k: int, num_valid_tokens=None, *,
                     scores: torch.Tensor | None = None, with_weights: bool = False, out: dict | None = None,
                     workspace: torch.Tensor | None = None, stream=None):
    """Router scores and routing in two kernels (the top-k selection in the router's
    epilogue).  Returns (scores[T, E] bf16, the dict of moe_route)."""
    T, D = x.shape
    E = w_router.shape[0]
    _need(x, torch.bfloat16, "x")
    _need(w_router, torch.bfloat16, "w_router")
    if num_valid_tokens is not None:
        _need(num_valid_tokens, torch.int32, "num_valid_tokens")
    if scores is None:
        scores = torch.empty(T, E, dtype=torch.bfloat16, device=x.device)
    _need(scores, torch.bfloat16, "scores")
    dev = x.device
    o = dict(out or {})
    i32 = dict(dtype=torch.int32, device=dev)
    o.setdefault("counts", torch.empty(E + 1, **i32))
    o.setdefault("expert_offsets", torch.empty(E + 1, **i32))
    o.setdefault("expert_indices", torch.empty(T * top_k, **i32))
    o.setdefault("token_indices", torch.empty(T * top_k, **i32))
    o.setdefault("inv_rows", torch.empty(T * top_k, **i32))
    if with_weights:
        o.setdefault("topk_weights", torch.empty(T * top_k, dtype=torch.float32, device=dev))
    else:
        o["topk_weights"] = None
    ws_bytes = moe_router_route_workspace_size(T, D, E, top_k)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    st = _lib.moe_router_route(_ptr(x), T, D, _ptr(w_router), E, top_k, _ptr(num_valid_tokens), _ptr(scores),
                               _ptr(o["counts"]), _ptr(o["expert_offsets"]), _ptr(o["expert_indices"]),
                               _ptr(o["token_indices"]), _ptr(o["inv_rows"]), _ptr(o["topk_weights"]),
                               _ptr(workspace), workspace.numel(), _stream(stream))
    _check("moe_router_route", st)
    return scores, o


def moe_route_workspace_size(T: int, E: int, top_k: int) -> int:
    n = ctypes.c_size_t(0)
    _check("moe_route_workspace_size", _lib.moe_route_workspace_size(T, E, top_k, ctypes.byref(n)))
    return n.value


def moe_route(scores: torch.Tensor, top_k: int, num_valid_tokens: torch.Tensor | None = None, *,
              with_inv: bool = True, with_weights: bool = False, out: dict | None = None,
              workspace: torch.Tensor | None = None, stream=None):
    """Route scores[T, E]; returns dict(counts, expert_offsets, expert_indices,
    token_indices, inv_rows) of int32 device tensors (index arrays of T * top_k),
    plus topk_weights (fp32 [T * top_k], in inv_rows order) when with_weights."""
    T, E = scores.shape
    dev = scores.device
    o = dict(out or {})
    i32 = dict(dtype=torch.int32, device=dev)
    o.setdefault("counts", torch.empty(E + 1, **i32))
    o.setdefault("expert_offsets", torch.empty(E + 1, **i32))
    o.setdefault("expert_indices", torch.empty(T * top_k, **i32))
    o.setdefault("token_indices", torch.empty(T * top_k, **i32))
    if with_inv:
        o.setdefault("inv_rows", torch.empty(T * top_k, **i32))
    else:
        o["inv_rows"] = None
    if with_weights:
        o.setdefault("topk_weights", torch.empty(T * top_k, dtype=torch.float32, device=dev))
    else:
        o["topk_weights"] = None
    ws_bytes = moe_route_workspace_size(T, E, top_k)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    if num_valid_tokens is not None:
        _need(num_valid_tokens, torch.int32, "num_valid_tokens")
    st = _lib.moe_route(_ptr(scores), _dtype_code(scores), scores.stride(0), scores.stride(1), T, E, top_k,
                        _ptr(num_valid_tokens), _ptr(o["counts"]), _ptr(o["expert_offsets"]),
                        _ptr(o["expert_indices"]), _ptr(o["token_indices"]), _ptr(o["inv_rows"]),
                        _ptr(o["topk_weights"]), _ptr(workspace), workspace.numel(), _stream(stream))
    _check("moe_route", st)
    return o


def _scores_args(scores):
    """(pointer, dtype code, stride_t, stride_e, E) of a score tensor; None = unit scores."""
    if scores is None:
        return None, MOE_DTYPE_BF16, 0, 0, 1
    return _ptr(scores), _dtype_code(scores), scores.stride(0), scores.stride(1), scores.shape[1]


# ------------------------------------------------------------------- gather

def moe_gather_scale(x, token_indices, expert_indices, scores, valid_token_count=None, *, inv_rows=None,
                     top_k: int = 1, out=None, stream=None):
    T, D = x.shape
    a = token_indices.shape[0]
    _need(x, torch.bfloat16, "x")
    if out is None:
        out = torch.empty(a, D, dtype=x.dtype, device=x.device)
    _need(out, out.dtype, "out")
    st = _lib.moe_gather_scale(_ptr(x), T, D, _ptr(token_indices), _ptr(expert_indices), a, *_scores_args(scores),
                               _ptr(valid_token_count), _ptr(inv_rows), top_k, _ptr(out), _stream(stream))
    _check("moe_gather_scale", st)
    return out


def moe_gather_scale_quant(x, token_indices, expert_indices, scores, scale_ub=None, valid_token_count=None, *,
                           inv_rows=None, top_k: int = 1, out=None, out_scale=None, stream=None):
    T, D = x.shape
    a = token_indices.shape[0]
    _need(x, torch.bfloat16, "x")
    if out is None:
        out = torch.empty(a, D, dtype=torch.float8_e4m3fn, device=x.device)
    _need(out, out.dtype, "out")
    if out_scale is None:
        out_scale = torch.empty(a, dtype=torch.float32, device=x.device)
    _need(out_scale, out_scale.dtype, "out_scale")
    st = _lib.moe_gather_scale_quant(_ptr(x), T, D, _ptr(token_indices), _ptr(expert_indices), a,
                                     *_scores_args(scores),
                                     _ptr(valid_token_count), _ptr(inv_rows), top_k, _ptr(scale_ub), _ptr(out),
                                     _ptr(out_scale), _stream(stream))
    _check("moe_gather_scale_quant", st)
    return out, out_scale


def moe_quantize_rows(w: torch.Tensor, scale_ub=None, *, out=None, out_scale=None, stream=None):
    """Per-row FP8 quantisation over the last dim of an fp32 tensor."""
    _need(w, torch.float32, "w")
    cols = w.shape[-1]
    rows = w.numel() // cols if cols else 0
    if out is None:
        out = torch.empty(w.shape, dtype=torch.float8_e4m3fn, device=w.device)
    _need(out, out.dtype, "out")
    if out_scale is None:
        out_scale = torch.empty(w.shape[:-1], dtype=torch.float32, device=w.device)
    _need(out_scale, out_scale.dtype, "out_scale")
    st = _lib.moe_quantize_rows(_ptr(w), rows, cols, _ptr(scale_ub), _ptr(out), _ptr(out_scale), _stream(stream))
    _check("moe_quantize_rows", st)
    return out, out_scale


# ------------------------------------------------------------- grouped GEMM

def _scatter_args(scatter_indices, out, accumulate):
    if scatter_indices is None:
        return None, 0, 0
    if out is None:
        raise ValueError("the fused combine writes into a caller-provided out[T, N]")
    return scatter_indices, out.shape[0], int(accumulate)


class PackedWeights:
    """Weights [E, N, K] (bf16 or e4m3) in the tile-packed layout of moe_pack_weights:
    `data` holds the packed bytes on the device; `shape` and `dtype` are the logical
    ones.  Accepted wherever the grouped GEMMs and moe_expert_mlp take weights."""

    def __init__(self, data: torch.Tensor, shape, dtype):
        self.data, self.shape, self.dtype = data, tuple(shape), dtype

    @property
    def device(self):
        return self.data.device


def moe_pack_weights_size(E: int, N: int, K: int, dtype: int) -> int:
    n = ctypes.c_size_t(0)
    _check("moe_pack_weights_size", _lib.moe_pack_weights_size(E, N, K, dtype, ctypes.byref(n)))
    return n.value


def moe_pack_weights(w: torch.Tensor, stream=None) -> PackedWeights:
    """Tile-packed copy of w [E, N, K] bf16 or e4m3 (every 128-row x 128-byte box contiguous)."""
    E, N, K = w.shape
    if w.dtype not in (torch.bfloat16, torch.float8_e4m3fn):
        raise TypeError(f"w must be bf16 or e4m3, got {w.dtype}")
    _need(w, w.dtype, "w")
    dt = MOE_DTYPE_E4M3 if w.dtype == torch.float8_e4m3fn else MOE_DTYPE_BF16
    data = torch.empty(moe_pack_weights_size(E, N, K, dt), dtype=torch.uint8, device=w.device)
    _check("moe_pack_weights", _lib.moe_pack_weights(_ptr(w), E, N, K, dt, _ptr(data), _stream(stream)))
    return PackedWeights(data, (E, N, K), w.dtype)


def _weights_arg(w, dtype, name: str, flags: int):
    """Pointer and flags of a weights argument: a row-major [E, N, K] tensor or PackedWeights."""
    if isinstance(w, PackedWeights):
        if w.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}, got packed {w.dtype}")
        if not w.data.is_cuda:
            raise TypeError(f"{name} must be on a CUDA device")
        return _ptr(w.data), flags | MOE_WEIGHTS_PACKED
    _need(w, dtype, name)
    return _ptr(w), flags


def _gemm_outputs(x, N, epilogue, out, z_out, z_scale):
    """The bf16 output (y, or z for the SiLU epilogues) and, with SILU_MUL_QUANT,
    the e4m3 z and its row scales; allocated when not given."""
    a_max = x.shape[0]
    kind = epilogue & 0xFF
    n_out = N // 2 if kind in (MOE_EPILOGUE_SILU_MUL, MOE_EPILOGUE_SILU_MUL_QUANT) else N
    if out is None:
        out = torch.empty(a_max, n_out, dtype=torch.bfloat16, device=x.device)
    _need(out, out.dtype, "out")
    if kind != MOE_EPILOGUE_SILU_MUL_QUANT:
        return out, None, None
    if z_out is None:
        z_out = torch.empty(a_max, n_out, dtype=torch.float8_e4m3fn, device=x.device)
    _need(z_out, torch.float8_e4m3fn, "z_out")
    if z_scale is None:
        z_scale = torch.empty(a_max, dtype=torch.float32, device=x.device)
    _need(z_scale, torch.float32, "z_scale")
    return out, z_out, z_scale


def moe_grouped_gemm(x, w, counts, *, epilogue: int = MOE_EPILOGUE_NONE, out=None, scatter_indices=None,
                     accumulate: bool = True, scale_ub=None, z_out=None, z_scale=None, stream=None):
    """x[a_max, K] bf16, w[E, N, K] bf16, counts[>= E] int32 -> y[a_max, N or N/2].
    With scatter_indices (top_k = 1), routed row r lands in out[scatter_indices[r]].
    With MOE_EPILOGUE_SILU_MUL_QUANT, out receives the bf16 z and the call returns
    (z_out e4m3 [a_max, N/2], z_scale fp32 [a_max]) instead."""
    a_max, K = x.shape
    E, N, K2 = w.shape
    assert K == K2
    _need(x, torch.bfloat16, "x")
    w_ptr, epilogue = _weights_arg(w, torch.bfloat16, "w", epilogue)
    si, t_out, acc = _scatter_args(scatter_indices, out, accumulate)
    out, z_out, z_scale = _gemm_outputs(x, N, epilogue, out, z_out, z_scale)
    st = _lib.moe_grouped_gemm(_ptr(x), w_ptr, _ptr(counts), E, a_max, N, K, _ptr(out), epilogue, _ptr(si),
                               t_out, acc, _ptr(scale_ub), _ptr(z_out), _ptr(z_scale), _stream(stream))
    _check("moe_grouped_gemm", st)
    return out if z_out is None else (z_out, z_scale)


def moe_grouped_gemm_fp8_rowwise(x, w, counts, x_scale, w_scale, *, epilogue: int = MOE_EPILOGUE_NONE, out=None,
                                 scatter_indices=None, accumulate: bool = True, scale_ub=None, z_out=None,
                                 z_scale=None, stream=None):
    """As moe_grouped_gemm on e4m3 x[a_max, K] and w[E, N, K] with fp32 row scales
    x_scale[a_max] and w_scale[E, N]."""
    a_max, K = x.shape
    E, N, K2 = w.shape
    assert K == K2
    _need(x, torch.float8_e4m3fn, "x")
    w_ptr, epilogue = _weights_arg(w, torch.float8_e4m3fn, "w", epilogue)
    si, t_out, acc = _scatter_args(scatter_indices, out, accumulate)
    out, z_out, z_scale = _gemm_outputs(x, N, epilogue, out, z_out, z_scale)
    st = _lib.moe_grouped_gemm_fp8_rowwise(_ptr(x), w_ptr, _ptr(counts), _ptr(x_scale), _ptr(w_scale), E, a_max,
                                           N, K, _ptr(out), epilogue, _ptr(si), t_out, acc, _ptr(scale_ub),
                                           _ptr(z_out), _ptr(z_scale), _stream(stream))
    _check("moe_grouped_gemm_fp8_rowwise", st)
    return out if z_out is None else (z_out, z_scale)


def moe_expert_mlp_workspace_size(E: int) -> int:
    n = ctypes.c_size_t(0)
    _check("moe_expert_mlp_workspace_size", _lib.moe_expert_mlp_workspace_size(E, ctypes.byref(n)))
    return n.value


def moe_expert_mlp(x, w13, w2, counts, *, z=None, out=None, scatter_indices=None, accumulate: bool = True,
                   workspace=None, stream=None):
    """Both bf16 grouped GEMMs in one launch: z = silu_mul(x w13^T), out = z w2^T per expert
    (with scatter_indices, top_k = 1: row r lands in out[scatter_indices[r]])."""
    a_max, D = x.shape
    E, n2, D2 = w13.shape
    H = n2 // 2
    assert D == D2 and tuple(w2.shape) == (E, D, H)
    _need(x, torch.bfloat16, "x")
    if isinstance(w13, PackedWeights) != isinstance(w2, PackedWeights):
        raise TypeError("w13 and w2 must both be packed or both be row-major")
    w13_ptr, flags = _weights_arg(w13, torch.bfloat16, "w13", 0)
    w2_ptr, _ = _weights_arg(w2, torch.bfloat16, "w2", 0)
    if z is None:
        z = torch.empty(a_max, H, dtype=torch.bfloat16, device=x.device)
    _need(z, z.dtype, "z")
    si, t_out, acc = _scatter_args(scatter_indices, out, accumulate)
    if out is None:
        out = torch.empty(a_max, D, dtype=torch.bfloat16, device=x.device)
    _need(out, out.dtype, "out")
    if workspace is None:   # zero on first use; each call leaves it zero
        workspace = torch.zeros(moe_expert_mlp_workspace_size(E), dtype=torch.uint8, device=x.device)
    st = _lib.moe_expert_mlp(_ptr(x), w13_ptr, w2_ptr, _ptr(counts), E, a_max, D, H, _ptr(z), _ptr(out),
                             _ptr(si), t_out, acc, _ptr(workspace), workspace.numel(), flags, _stream(stream))
    _check("moe_expert_mlp", st)
    return out


# ----------------------------------------------------------------- silu_mul

def moe_silu_mul(y, H: int | None = None, valid_rows=None, *, out=None, stream=None):
    """y[a, 2H] bf16 -> z[a, H] = silu(y[:, :H]) * y[:, H:]."""
    a, n2 = y.shape
    H = n2 // 2 if H is None else H
    _need(y, torch.bfloat16, "y", contiguous=False)
    if out is None:
        out = torch.empty(a, H, dtype=torch.bfloat16, device=y.device)
    _need(out, out.dtype, "out")
    x1 = ctypes.c_void_p(y.data_ptr() + H * y.element_size())
    st = _lib.moe_silu_mul(_ptr(y), x1, y.stride(0), a, H, _ptr(valid_rows), _ptr(out), _stream(stream))
    _check("moe_silu_mul", st)
    return out


def moe_silu_mul_quant(y, H: int | None = None, scale_ub=None, valid_rows=None, *, out=None, out_scale=None,
                       stream=None):
    a, n2 = y.shape
    H = n2 // 2 if H is None else H
    _need(y, torch.bfloat16, "y", contiguous=False)
    if out is None:
        out = torch.empty(a, H, dtype=torch.float8_e4m3fn, device=y.device)
    _need(out, out.dtype, "out")
    if out_scale is None:
        out_scale = torch.empty(a, dtype=torch.float32, device=y.device)
    _need(out_scale, out_scale.dtype, "out_scale")
    x1 = ctypes.c_void_p(y.data_ptr() + H * y.element_size())
    st = _lib.moe_silu_mul_quant(_ptr(y), x1, y.stride(0), a, H, _ptr(valid_rows), _ptr(scale_ub), _ptr(out),
                                 _ptr(out_scale), _stream(stream))
    _check("moe_silu_mul_quant", st)
    return out, out_scale


# -------------------------------------------------------------- scatter-add

def moe_scatter_add(out, rows, token_indices, inv_rows=None, top_k: int = 1, valid_token_count=None, *,
                    accumulate: bool = True, stream=None):
    """out[T, D] += rows[a, D] by token, in place (deterministic); with
    accumulate=False the routed sum overwrites the valid tokens of out."""
    T, D = out.shape
    a = rows.shape[0]
    _need(out, torch.bfloat16, "out")
    _need(rows, torch.bfloat16, "rows")
    st = _lib.moe_scatter_add(_ptr(out), _ptr(rows), _ptr(token_indices), _ptr(inv_rows), top_k, a, T, D,
                              _ptr(valid_token_count), int(accumulate), _stream(stream))
    _check("moe_scatter_add", st)
    return out


def moe_scatter_add_padded(out, rows, token_counts, token_indices, inv_rows=None, top_k: int = 1, *,
                           accumulate: bool = True, stream=None):
    """scatter_add_padded_tokens on one GPU: the first sum(token_counts) rows of
    rows[T_K, D] (by-expert order) are added into out[T, D] by token."""
    T, D = out.shape
    T_K = rows.shape[0]
    E = token_counts.shape[0]
    _need(out, torch.bfloat16, "out")
    _need(rows, torch.bfloat16, "rows")
    _need(token_counts, torch.int32, "token_counts")
    st = _lib.moe_scatter_add_padded(_ptr(out), _ptr(rows), _ptr(token_counts), E, _ptr(token_indices),
                                     _ptr(inv_rows), top_k, T_K, T, D, int(accumulate), _stream(stream))
    _check("moe_scatter_add_padded", st)
    return out


def moe_topk_finalize(rows, expert_weights, expanded_idx_to_permuted_idx, shared_output=None,
                      valid_token_count=None, *, out=None, stream=None):
    """out[M, D] = bf16(sum_j w[t, j] * rows[idx[t, j]]) (-0 -> +0), plus the shared
    output (one more rounding); rows[n, D] bf16, weights fp32 or bf16 [M, k], idx int32 [M, k]."""
    n_rows, D = rows.shape
    M, k = expanded_idx_to_permuted_idx.shape
    _need(rows, torch.bfloat16, "rows")
    _need(expanded_idx_to_permuted_idx, torch.int32, "expanded_idx_to_permuted_idx")
    if shared_output is not None:
        _need(shared_output, torch.bfloat16, "shared_output")
    if out is None:
        out = torch.empty(M, D, dtype=torch.bfloat16, device=rows.device)
    _need(out, out.dtype, "out")
    st = _lib.moe_topk_finalize(_ptr(rows), n_rows, D, _ptr(expert_weights), _dtype_code(expert_weights),
                                _ptr(expanded_idx_to_permuted_idx), M, k, _ptr(valid_token_count),
                                _ptr(shared_output), _ptr(out), _stream(stream))
    _check("moe_topk_finalize", st)
    return out


def moe_dense_gemm(x, w, valid_rows=None, *, epilogue: int = MOE_EPILOGUE_NONE, out=None, stream=None):
    """y = x[M, K] @ w[N, K]^T (bf16, split-K over a cluster); with the SiLU*mul
    epilogue y[M, N/2] = silu_mul of the two halves."""
    M, K = x.shape
    N, K2 = w.shape
    assert K == K2
    _need(x, torch.bfloat16, "x")
    _need(w, torch.bfloat16, "w")
    if valid_rows is not None:
        _need(valid_rows, torch.int32, "valid_rows")
    n_out = N // 2 if epilogue == MOE_EPILOGUE_SILU_MUL else N
    if out is None:
        out = torch.empty(M, n_out, dtype=torch.bfloat16, device=x.device)
    _need(out, torch.bfloat16, "out")
    st = _lib.moe_dense_gemm(_ptr(x), M, K, _ptr(w), N, _ptr(valid_rows), _ptr(out), epilogue, _stream(stream))
    _check("moe_dense_gemm", st)
    return out


def moe_selftest_bounded_wait(which: int, limit_ns: int = 20_000_000, stream=None) -> int:
    """Run a bounded device wait that never succeeds (0: mbarrier, 1: grid barrier);
    returns the device error bits afterwards (MOE_DEVERR_TIMEOUT expected)."""
    _check("moe_selftest_bounded_wait", _lib.moe_selftest_bounded_wait(which, limit_ns, _stream(stream)))
    return device_error(stream)
