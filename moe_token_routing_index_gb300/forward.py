"""The single-GPU routed-expert forward, composed from the C-ABI stages.

Stage order of mslk/moe/layers.py, MetaShufflingMoE._no_comm_forward
(routed experts, no shared expert):

  bf16:  route -> gather*score -> grouped GEMM w13 with the SiLU*mul epilogue
         -> grouped GEMM w2 -> scatter-add (both GEMMs in one persistent launch,
         moe_expert_mlp, when the layer streams its weights: T*top_k <= 128*E)
  FP8:   route -> gather*score -> e4m3 rows -> grouped GEMM w13 (FP8 rowwise)
         -> silu_mul_quant -> grouped GEMM w2 (FP8 rowwise) -> scatter-add

With top_k = 1 the scatter-add is fused into the w2 GEMM's epilogue (each
routed row owns its token), as _routed_expert does with _scatter_add_indices.

Weights stay resident on the device; every buffer of the pipeline is
allocated once per token-buffer size, so a forward launches kernels only
(no allocation), and the valid-row count flows on the device from the router
(counts[E]) into every later stage.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import binding as mb
from .workloads import MoEConfig

__all__ = ["MoELayer"]


@dataclass
class _Buffers:
    T: int
    route: dict
    ws: torch.Tensor
    mlp_ws: torch.Tensor
    xr: torch.Tensor              # routed rows: bf16 [T*k, D] or e4m3 [T*k, D]
    xs: torch.Tensor | None       # FP8: row scales [T*k]
    y: torch.Tensor | None        # FP8: GEMM1 output bf16 [T*k, 2H]
    z: torch.Tensor               # bf16 [T*k, H] or e4m3 [T*k, H]
    zs: torch.Tensor | None       # FP8: row scales [T*k]
    o: torch.Tensor               # GEMM2 output bf16 [T*k, D]


class MoELayer:
    """Routed experts of one MoE layer on one GPU.

    w13 [E, 2H, D] and w2 [E, D, H]: bf16 (bf16 layer), or e4m3 with fp32
    per-row scales w13_scale [E, 2H], w2_scale [E, D] (FP8-rowwise layer).
    """

    def __init__(self, top_k: int, w13: torch.Tensor, w2: torch.Tensor, w13_scale: torch.Tensor | None = None,
                 w2_scale: torch.Tensor | None = None, scale_ub: float | None = None,
                 fused_mlp: bool | None = None, cta_pairs: bool | None = None):
        self.E, n2, self.D = w13.shape
        self.H = n2 // 2
        assert w2.shape == (self.E, self.D, self.H), "w2 must be [E, D, H]"
        self.top_k = top_k
        self.fp8 = w13.dtype == torch.float8_e4m3fn
        if self.fp8:
            assert w13_scale is not None and w2_scale is not None
        self.w13, self.w2 = w13.contiguous(), w2.contiguous()
        self.w13_scale = None if w13_scale is None else w13_scale.contiguous()
        self.w2_scale = None if w2_scale is None else w2_scale.contiguous()
        dev = w13.device
        self.scale_ub = None if scale_ub is None else torch.tensor([scale_ub], dtype=torch.float32, device=dev)
        # None: one launch for both bf16 GEMMs when the batch averages at most one
        # 128-row tile per expert (weight-streaming, HBM-bound), else two launches.
        self.fused_mlp = fused_mlp
        # None: 256-row tiles on CTA pairs for the bf16 GEMMs when the batch averages
        # at least one such tile per expert; 128-row tiles otherwise.  The FP8 GEMMs
        # keep 128-row tiles: on GB300 their pair tiles measured slower (prefill,
        # 512 rows per expert) or padded more rows (344 rows per expert).
        self.cta_pairs = cta_pairs
        self._bufs: _Buffers | None = None

    @classmethod
    def from_weights(cls, cfg: MoEConfig, w13: torch.Tensor, w2: torch.Tensor, **kw) -> "MoELayer":
        """bf16 weights as they are; fp32 weights of an FP8 layer are quantised
        per row on the device (moe_quantize_rows)."""
        if cfg.fp8:
            w13q, w13s = mb.moe_quantize_rows(w13.float().contiguous())
            w2q, w2s = mb.moe_quantize_rows(w2.float().contiguous())
            return cls(cfg.top_k, w13q, w2q, w13s, w2s, scale_ub=cfg.scale_ub, **kw)
        return cls(cfg.top_k, w13.to(torch.bfloat16), w2.to(torch.bfloat16), scale_ub=cfg.scale_ub, **kw)

    # ------------------------------------------------------------ buffers
    def buffers(self, T: int, device) -> _Buffers:
        if self._bufs is not None and self._bufs.T == T:
            return self._bufs
        k, E, D, H = self.top_k, self.E, self.D, self.H
        a = T * k
        i32 = dict(dtype=torch.int32, device=device)
        route = dict(counts=torch.zeros(E + 1, **i32), expert_offsets=torch.zeros(E + 1, **i32),
                     expert_indices=torch.zeros(a, **i32), token_indices=torch.zeros(a, **i32),
                     inv_rows=torch.zeros(a, **i32))
        ws = torch.empty(max(mb.moe_route_workspace_size(T, E, k), 256), dtype=torch.uint8, device=device)
        mlp_ws = torch.empty(mb.moe_expert_mlp_workspace_size(E), dtype=torch.uint8, device=device)
        if self.fp8:
            e4 = dict(dtype=torch.float8_e4m3fn, device=device)
            f32 = dict(dtype=torch.float32, device=device)
            b = _Buffers(T, route, ws, mlp_ws, torch.empty(a, D, **e4), torch.empty(a, **f32),
                         torch.empty(a, 2 * H, dtype=torch.bfloat16, device=device), torch.empty(a, H, **e4),
                         torch.empty(a, **f32), torch.empty(a, D, dtype=torch.bfloat16, device=device))
        else:
            bf = dict(dtype=torch.bfloat16, device=device)
            b = _Buffers(T, route, ws, mlp_ws, torch.empty(a, D, **bf), None, None, torch.empty(a, H, **bf), None,
                         torch.empty(a, D, **bf))
        self._bufs = b
        return b

    # ------------------------------------------------------------ forward
    def stages(self, x: torch.Tensor, scores: torch.Tensor, num_valid_tokens: torch.Tensor | None,
               out: torch.Tensor, accumulate: bool):
        """The forward as a list of (stage name, launch callable), in order."""
        T = x.shape[0]
        b = self.buffers(T, x.device)
        r = b.route
        counts = r["counts"]
        valid = counts[self.E:]                      # routed rows, written by the router on the device
        ti, ei = r["token_indices"], r["expert_indices"]
        inv = r["inv_rows"] if self.top_k > 1 else None
        k = self.top_k
        fuse_combine = k == 1
        pairs = mb.MOE_GEMM_CTA_PAIRS if self.use_cta_pairs(T) else 0
        # the w2 GEMM writes either the routed rows o, or (top_k = 1) the tokens' rows of out
        w2_out = dict(out=out, scatter_indices=ti, accumulate=accumulate) if fuse_combine else dict(out=b.o)
        st = [("route", lambda: mb.moe_route(scores, k, num_valid_tokens, out=r, workspace=b.ws))]
        if not self.fp8:
            st.append(("gather", lambda: mb.moe_gather_scale(x, ti, ei, scores, valid, inv_rows=inv, top_k=k,
                                                             out=b.xr)))
            if self.use_fused_mlp(T):
                st.append(("expert_mlp", lambda: mb.moe_expert_mlp(b.xr, self.w13, self.w2, counts, z=b.z,
                                                                   workspace=b.mlp_ws, **w2_out)))
            else:
                st += [
                    ("gemm_w13_silu", lambda: mb.moe_grouped_gemm(b.xr, self.w13, counts,
                                                                  epilogue=mb.MOE_EPILOGUE_SILU_MUL | pairs,
                                                                  out=b.z)),
                    ("gemm_w2", lambda: mb.moe_grouped_gemm(b.z, self.w2, counts, epilogue=pairs, **w2_out)),
                ]
        else:
            st += [
                ("gather_quant", lambda: mb.moe_gather_scale_quant(x, ti, ei, scores, self.scale_ub, valid,
                                                                   inv_rows=inv, top_k=k, out=b.xr,
                                                                   out_scale=b.xs)),
                ("gemm_w13", lambda: mb.moe_grouped_gemm_fp8_rowwise(b.xr, self.w13, counts, b.xs, self.w13_scale,
                                                                     epilogue=pairs, out=b.y)),
                ("silu_quant", lambda: mb.moe_silu_mul_quant(b.y, self.H, self.scale_ub, valid, out=b.z,
                                                             out_scale=b.zs)),
                ("gemm_w2", lambda: mb.moe_grouped_gemm_fp8_rowwise(b.z, self.w2, counts, b.zs, self.w2_scale,
                                                                    epilogue=pairs, **w2_out)),
            ]
        if not fuse_combine:
            st.append(("scatter", lambda: mb.moe_scatter_add(out, b.o, ti, inv, k, valid, accumulate=accumulate)))
        return st

    def __call__(self, x: torch.Tensor, scores: torch.Tensor, num_valid_tokens: torch.Tensor | None = None,
                 out: torch.Tensor | None = None, accumulate: bool = False) -> torch.Tensor:
        """x[T, D] bf16, scores[T, E] (bf16 or f32) on the device; num_valid_tokens:
        device int32 [1] (None: all T).  Returns out[T, D] bf16: for valid tokens
        the routed sum (added into out when accumulate), other rows untouched."""
        if out is None:
            out = torch.zeros(x.shape[0], self.D, dtype=torch.bfloat16, device=x.device)
        for _, launch in self.stages(x, scores, num_valid_tokens, out, accumulate):
            launch()
        return out

    def use_fused_mlp(self, T: int) -> bool:
        if self.fp8:
            return False
        if self.fused_mlp is not None:
            return self.fused_mlp
        return T * self.top_k <= 128 * self.E

    def use_cta_pairs(self, T: int) -> bool:
        if self.cta_pairs is not None:
            return self.cta_pairs
        return not self.fp8 and T * self.top_k >= 256 * self.E

    def kernel_launches(self, T: int | None = None) -> int:
        """Kernels one forward launches: routing (1 for small batches, else 3),
        gather, the GEMMs (1 fused, or 2), silu_mul_quant (FP8), scatter."""
        T = self._bufs.T if T is None and self._bufs is not None else (T or 0)
        route = 1 if (T <= 1024 and T * self.E <= 16384 and T * self.top_k <= 8192 and self.E <= 256) else 3
        scatter = 0 if self.top_k == 1 else 1
        if self.fp8:
            return route + 4 + scatter
        return route + 1 + (1 if self.use_fused_mlp(T) else 2) + scatter
