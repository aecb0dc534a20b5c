"""The single-GPU MoE layer forward, composed from the C-ABI stages.

Stage order of mslk/moe/layers.py, MetaShufflingMoE._no_comm_forward:

  router (optional): scores = sigmoid(tokens @ router_DE)        moe_router_scores
  routed experts, bf16:  route -> gather*score -> grouped GEMM w13 with the
         SiLU*mul epilogue -> grouped GEMM w2 -> scatter-add (both GEMMs in one
         persistent launch, moe_expert_mlp, when the layer streams its weights:
         T*top_k <= 128*E)
  routed experts, FP8:   route -> gather*score -> e4m3 rows -> grouped GEMM w13
         (FP8 rowwise) with the SiLU*mul + quantisation epilogue (bf16 z, then its
         rows to e4m3) -> grouped GEMM w2 (FP8 rowwise) -> scatter-add
  shared expert (optional): the same MLP over every valid token (one expert,
         unit scores) written into the output first; the routed combine then
         adds into it, as _routed_expert does with shared_output.  Small bf16
         batches use the split-K dense GEMMs (moe_dense_gemm), the others the
         grouped kernels with one expert.

With top_k = 1 the scatter-add is fused into the w2 GEMM's epilogue (each
routed row owns its token), as _routed_expert does with _scatter_add_indices.
The shared expert runs on a second stream while the router, routing and
gather run (overlap_router_and_shared_expert of _no_comm_forward); the
combine waits for it.

Weights stay resident on the device; every buffer of the pipeline is
allocated once per token-buffer size, so a forward launches kernels only
(no allocation), and the valid-row count flows on the device from the router
(counts[E]) into every later stage.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

from . import binding as mb
from .workloads import MoEConfig

__all__ = ["MoELayer"]

MAIN, SIDE = "main", "side"


@dataclass
class _Buffers:
    T: int
    route: dict
    ws: torch.Tensor
    mlp_ws: torch.Tensor
    xr: torch.Tensor              # routed rows: bf16 [T*k, D] or e4m3 [T*k, D]
    xs: torch.Tensor | None       # FP8: row scales [T*k]
    y: torch.Tensor | None        # FP8: the w13 epilogue's bf16 z [T*k, H], before its rows are quantised
    z: torch.Tensor               # bf16 [T*k, H] or e4m3 [T*k, H]
    zs: torch.Tensor | None       # FP8: row scales [T*k]
    o: torch.Tensor               # GEMM2 output bf16 [T*k, D]
    extra: dict = field(default_factory=dict)   # router and shared-expert buffers


class MoELayer:
    """One MoE layer on one GPU: routed experts, and optionally the router and
    a shared expert.

    w13 [E, 2H, D] and w2 [E, D, H]: bf16 (bf16 layer), or e4m3 with fp32
    per-row scales w13_scale [E, 2H], w2_scale [E, D] (FP8-rowwise layer).
    router: bf16 [E, D], router_DE transposed (None: the caller passes scores).
    shared_w13 [2Hs, D], shared_w2 [D, Hs]: the shared expert, in the layer's
    dtype (e4m3 with scales shared_w13_scale [2Hs], shared_w2_scale [D]).
    pack_weights: hold w13 and w2 in the tile-packed layout (moe_pack_weights), so
    that the grouped GEMMs stream them as contiguous boxes; None packs them when H
    and D are multiples of 128.  The output is the same bit for bit either way.
    """

    def __init__(self, top_k: int, w13: torch.Tensor, w2: torch.Tensor, w13_scale: torch.Tensor | None = None,
                 w2_scale: torch.Tensor | None = None, scale_ub: float | None = None,
                 fused_mlp: bool | None = None, cta_pairs: bool | None = None, *,
                 router: torch.Tensor | None = None, shared_w13: torch.Tensor | None = None,
                 shared_w2: torch.Tensor | None = None, shared_w13_scale: torch.Tensor | None = None,
                 shared_w2_scale: torch.Tensor | None = None, overlap_shared: bool = True,
                 weighting: str = "input", pack_weights: bool | None = None):
        self.E, n2, self.D = w13.shape
        self.H = n2 // 2
        assert w2.shape == (self.E, self.D, self.H), "w2 must be [E, D, H]"
        self.top_k = top_k
        self.fp8 = w13.dtype == torch.float8_e4m3fn
        if self.fp8:
            assert w13_scale is not None and w2_scale is not None
        # FP8 layers quantise z in the w13 GEMM's epilogue, after its bf16 rounding
        # (MOE_EPILOGUE_SILU_MUL_QUANT): the z_bf16 reading of the CPU oracle
        self.z_bf16 = self.fp8
        self.w13, self.w2 = w13.contiguous(), w2.contiguous()
        if pack_weights is None:
            pack_weights = self.H % 128 == 0 and self.D % 128 == 0 and w13.is_cuda
        if pack_weights:   # resident weights: packed once, the row-major copies are not kept
            self.w13, self.w2 = mb.moe_pack_weights(self.w13), mb.moe_pack_weights(self.w2)
        self.w13_scale = None if w13_scale is None else w13_scale.contiguous()
        self.w2_scale = None if w2_scale is None else w2_scale.contiguous()
        dev = w13.device
        self.scale_ub = None if scale_ub is None else torch.tensor([scale_ub], dtype=torch.float32, device=dev)
        # None: one launch for both bf16 GEMMs when the batch averages at most one
        # 128-row tile per expert (weight-streaming, HBM-bound), else two launches.
        self.fused_mlp = fused_mlp
        # None: 256-row tiles on CTA pairs for the bf16 GEMMs when they pad the expert
        # rows little more than 128-row tiles do (judged from the previous forward's
        # counts; before the first, when the batch averages at least 256 rows per
        # expert).  The output is the same bit for bit either way.  The FP8 GEMMs keep
        # 128-row tiles: inside a whole forward on GB300 their pair tiles ran slower
        # (prefill, 512 rows per expert: 0.953 against 0.890 ms per step, the clock
        # lower under the power cap) or padded more rows (344 rows per expert: 1.062
        # against 0.901 ms), although in isolation they keep the tensor pipe busier.
        self.cta_pairs = cta_pairs
        self._counts_host: torch.Tensor | None = None   # pinned copy of the last forward's counts
        self._counts_event: torch.cuda.Event | None = None
        self._capturing = False
        self.router = None if router is None else router.contiguous()
        if self.router is not None:
            assert self.router.shape == (self.E, self.D) and self.router.dtype == torch.bfloat16
        self.shared = shared_w13 is not None
        if self.shared:
            assert shared_w2 is not None and shared_w13.shape[1] == self.D
            self.Hs = shared_w13.shape[0] // 2
            assert shared_w2.shape == (self.D, self.Hs)
            assert (shared_w13.dtype == torch.float8_e4m3fn) == self.fp8
            # one expert of the grouped kernels: [1, 2Hs, D] and [1, D, Hs]
            self.sw13, self.sw2 = shared_w13.contiguous()[None], shared_w2.contiguous()[None]
            self.sw13_scale = None if shared_w13_scale is None else shared_w13_scale.contiguous()
            self.sw2_scale = None if shared_w2_scale is None else shared_w2_scale.contiguous()
            if self.fp8:
                assert self.sw13_scale is not None and self.sw2_scale is not None
        self.overlap_shared = overlap_shared
        # "input": the score scales each routed row before the experts (gather_scale_dense_tokens);
        # "output": the experts see the unscaled rows and the top-k finalize weights their outputs.
        if weighting not in ("input", "output"):
            raise ValueError("weighting must be 'input' or 'output'")
        self.weighting = weighting
        self._side: torch.cuda.Stream | None = None
        self._bufs: _Buffers | None = None

    @classmethod
    def from_weights(cls, cfg: MoEConfig, w13: torch.Tensor, w2: torch.Tensor, *,
                     router: torch.Tensor | None = None, shared: tuple | None = None, **kw) -> "MoELayer":
        """bf16 weights as they are; fp32 weights of an FP8 layer (routed and
        shared) are quantised per row on the device (moe_quantize_rows)."""
        if shared is not None:
            s13, s2 = shared
            if cfg.fp8:
                q13, sc13 = mb.moe_quantize_rows(s13.float().contiguous())
                q2, sc2 = mb.moe_quantize_rows(s2.float().contiguous())
                kw.update(shared_w13=q13, shared_w2=q2, shared_w13_scale=sc13, shared_w2_scale=sc2)
            else:
                kw.update(shared_w13=s13.to(torch.bfloat16), shared_w2=s2.to(torch.bfloat16))
        if router is not None:
            kw["router"] = router.to(torch.bfloat16)
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
        f32 = dict(dtype=torch.float32, device=device)
        bf = dict(dtype=torch.bfloat16, device=device)
        e4 = dict(dtype=torch.float8_e4m3fn, device=device)
        route = dict(counts=torch.zeros(E + 1, **i32), expert_offsets=torch.zeros(E + 1, **i32),
                     expert_indices=torch.zeros(a, **i32), token_indices=torch.zeros(a, **i32),
                     inv_rows=torch.zeros(a, **i32))
        if self.weighting == "output":
            route["topk_weights"] = torch.zeros(a, **f32)
        ws = torch.empty(max(mb.moe_route_workspace_size(T, E, k), 256), dtype=torch.uint8, device=device)
        # zero on first use; the expert MLP leaves it zero
        mlp_ws = torch.zeros(mb.moe_expert_mlp_workspace_size(max(E, 1)), dtype=torch.uint8, device=device)
        if self.fp8:
            b = _Buffers(T, route, ws, mlp_ws, torch.empty(a, D, **e4), torch.empty(a, **f32),
                         torch.empty(a, H, **bf), torch.empty(a, H, **e4), torch.empty(a, **f32),
                         torch.empty(a, D, **bf))
        else:
            b = _Buffers(T, route, ws, mlp_ws, torch.empty(a, D, **bf), None, None, torch.empty(a, H, **bf), None,
                         torch.empty(a, D, **bf))
        x = b.extra
        if self.router is not None:
            x["scores"] = torch.empty(T, E, **bf)
            x["router_ws"] = torch.empty(max(mb.moe_router_workspace_size(T, D, E), 256), dtype=torch.uint8,
                                         device=device)
        if self.shared:
            Hs = self.Hs
            x["all_tokens"] = torch.tensor([T], **i32)       # the shared expert's row count without a valid count
            x["ident"] = torch.arange(T, **i32)
            if self.weighting == "output":
                x["sh_out"] = torch.empty(T, D, **bf)           # the finalize adds it to the weighted sum
            x["sh_mlp_ws"] = torch.zeros(mb.moe_expert_mlp_workspace_size(1), dtype=torch.uint8, device=device)
            if self.fp8:
                x["zero"] = torch.zeros(T, **i32)
                x["unit"] = torch.ones(T, 1, **f32)           # unit scores: the gather's product is exact
                x["sh_xq"], x["sh_xs"] = torch.empty(T, D, **e4), torch.empty(T, **f32)
                x["sh_y"] = torch.empty(T, Hs, **bf)
                x["sh_zq"], x["sh_zs"] = torch.empty(T, Hs, **e4), torch.empty(T, **f32)
            else:
                x["sh_z"] = torch.empty(T, Hs, **bf)
        self._bufs = b
        return b

    # ------------------------------------------------------------ forward
    def stages(self, x: torch.Tensor, scores: torch.Tensor | None, num_valid_tokens: torch.Tensor | None,
               out: torch.Tensor, accumulate: bool):
        """The forward as a list of (stage name, launch callable, lane), in a valid
        serial order.  Lane SIDE holds the shared expert, which only reads x and
        writes out; the first MAIN stage after it that touches out is the combine."""
        T = x.shape[0]
        b = self.buffers(T, x.device)
        ex = b.extra
        st = []
        routed_by_router = scores is None
        if routed_by_router:
            # the router's epilogue selects the experts; one more kernel emits the routing
            if self.router is None:
                raise ValueError("scores are required for a layer without a router")
            scores = ex["scores"]
            st.append(("router_route", lambda: mb.moe_router_route(
                x, self.router, self.top_k, num_valid_tokens, scores=ex["scores"],
                with_weights=self.weighting == "output", out=b.route, workspace=b.ws), MAIN))
        if self.weighting == "output":
            if accumulate:
                raise ValueError("the top-k finalize writes the output; accumulate is not supported with it")
            sh_out = None
            if self.shared:
                sh_out = ex["sh_out"]
                st += [(n, f, SIDE) for n, f in self._shared_stages(x, num_valid_tokens, sh_out, False)]
            st += [(n, f, MAIN) for n, f in self._routed_stages(x, scores, num_valid_tokens, out, False, sh_out,
                                                                routed=routed_by_router)]
            return st
        if self.shared:
            st += [(n, f, SIDE) for n, f in self._shared_stages(x, num_valid_tokens, out, accumulate)]
            accumulate = True       # the routed rows are added into the shared expert's output
        st += [(n, f, MAIN) for n, f in self._routed_stages(x, scores, num_valid_tokens, out, accumulate,
                                                            routed=routed_by_router)]
        return st

    def _shared_stages(self, x, num_valid_tokens, out, accumulate):
        T = x.shape[0]
        ex = self.buffers(T, x.device).extra
        rows = num_valid_tokens if num_valid_tokens is not None else ex["all_tokens"]   # counts of one expert
        # accumulate: the shared rows are added into out (row t to token t)
        add = dict(scatter_indices=ex["ident"], accumulate=True) if accumulate else {}
        if not self.fp8:
            if T <= 256 and not accumulate:
                # few row tiles: split the weights' K dimension over clusters so that every SM streams
                return [
                    ("shared_w13_silu", lambda: mb.moe_dense_gemm(x, self.sw13[0], rows,
                                                                  epilogue=mb.MOE_EPILOGUE_SILU_MUL, out=ex["sh_z"])),
                    ("shared_w2", lambda: mb.moe_dense_gemm(ex["sh_z"], self.sw2[0], rows, out=out)),
                ]
            if T <= 128:
                return [("shared_mlp", lambda: mb.moe_expert_mlp(x, self.sw13, self.sw2, rows, z=ex["sh_z"], out=out,
                                                                 workspace=ex["sh_mlp_ws"], **add))]
            return [
                ("shared_w13_silu", lambda: mb.moe_grouped_gemm(x, self.sw13, rows, epilogue=mb.MOE_EPILOGUE_SILU_MUL,
                                                                out=ex["sh_z"])),
                ("shared_w2", lambda: mb.moe_grouped_gemm(ex["sh_z"], self.sw2, rows, out=out, **add)),
            ]
        return [
            ("shared_quant", lambda: mb.moe_gather_scale_quant(x, ex["ident"], ex["zero"], ex["unit"], self.scale_ub,
                                                               rows, out=ex["sh_xq"], out_scale=ex["sh_xs"])),
            ("shared_w13_silu_quant", lambda: mb.moe_grouped_gemm_fp8_rowwise(
                ex["sh_xq"], self.sw13, rows, ex["sh_xs"], self.sw13_scale, epilogue=mb.MOE_EPILOGUE_SILU_MUL_QUANT,
                out=ex["sh_y"], scale_ub=self.scale_ub, z_out=ex["sh_zq"], z_scale=ex["sh_zs"])),
            ("shared_w2", lambda: mb.moe_grouped_gemm_fp8_rowwise(ex["sh_zq"], self.sw2, rows, ex["sh_zs"],
                                                                  self.sw2_scale, out=out, **add)),
        ]

    def _routed_stages(self, x, scores, num_valid_tokens, out, accumulate, shared_out=None, routed=False):
        T = x.shape[0]
        b = self.buffers(T, x.device)
        r = b.route
        counts = r["counts"]
        valid = counts[self.E:]                      # routed rows, written by the router on the device
        ti, ei = r["token_indices"], r["expert_indices"]
        inv = r["inv_rows"] if self.top_k > 1 else None
        k = self.top_k
        out_w = self.weighting == "output"
        fuse_combine = k == 1 and not out_w
        pairs = mb.MOE_GEMM_CTA_PAIRS if self.use_cta_pairs(T) else 0
        # the w2 GEMM writes either the routed rows o, or (top_k = 1) the tokens' rows of out
        w2_out = dict(out=out, scatter_indices=ti, accumulate=accumulate) if fuse_combine else dict(out=b.o)
        # routed: the router stage has routed the tokens already (moe_router_route)
        st = [] if routed else [("route", lambda: mb.moe_route(scores, k, num_valid_tokens, with_weights=out_w,
                                                                out=r, workspace=b.ws))]
        gscores = None if out_w else scores    # output weighting: the gathers copy the rows
        if not self.fp8:
            st.append(("gather", lambda: mb.moe_gather_scale(x, ti, ei, gscores, valid, inv_rows=inv, top_k=k,
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
                ("gather_quant", lambda: mb.moe_gather_scale_quant(x, ti, ei, gscores, self.scale_ub, valid,
                                                                   inv_rows=inv, top_k=k, out=b.xr,
                                                                   out_scale=b.xs)),
                ("gemm_w13_silu_quant", lambda: mb.moe_grouped_gemm_fp8_rowwise(
                    b.xr, self.w13, counts, b.xs, self.w13_scale, epilogue=mb.MOE_EPILOGUE_SILU_MUL_QUANT | pairs,
                    out=b.y, scale_ub=self.scale_ub, z_out=b.z, z_scale=b.zs)),
                ("gemm_w2", lambda: mb.moe_grouped_gemm_fp8_rowwise(b.z, self.w2, counts, b.zs, self.w2_scale,
                                                                    epilogue=pairs, **w2_out)),
            ]
        if out_w:
            idx = r["inv_rows"].view(T, k)
            wts = r["topk_weights"].view(T, k)
            st.append(("finalize", lambda: mb.moe_topk_finalize(b.o, wts, idx, shared_out, num_valid_tokens,
                                                                out=out)))
        elif not fuse_combine:
            st.append(("scatter", lambda: mb.moe_scatter_add(out, b.o, ti, inv, k, valid, accumulate=accumulate)))
        return st

    @staticmethod
    def combine_stage(names) -> str:
        """The first routed stage that writes the layer output."""
        for n in ("finalize", "scatter", "expert_mlp", "gemm_w2"):   # else the w2 GEMM's epilogue (top_k = 1)
            if n in names:
                return n
        raise ValueError("no combine stage")

    def run(self, stages, overlap: bool | None = None, events=None):
        """Launch the stages; with overlap the SIDE lane runs on a second stream
        from the start and the combine stage waits for it.  events: optional
        {name: (start, end)} CUDA events recorded around each MAIN-lane stage
        (and SIDE-lane stages on their stream)."""
        overlap = self.overlap_shared if overlap is None else overlap
        side = [s for s in stages if s[2] == SIDE]
        if not side or not overlap:
            for n, f, _ in stages:
                self._launch(n, f, events)
            return
        main = torch.cuda.current_stream()
        if self._side is None:
            self._side = torch.cuda.Stream(device=main.device)
            self._fork, self._join = torch.cuda.Event(), torch.cuda.Event()
        fork, join = self._fork, self._join
        fork.record(main)
        with torch.cuda.stream(self._side):
            self._side.wait_event(fork)
            for n, f, _ in side:
                self._launch(n, f, events)
            join.record(self._side)
        comb = self.combine_stage([s[0] for s in stages if s[2] == MAIN])
        for n, f, lane in stages:
            if lane != MAIN:
                continue
            if n == comb:
                main.wait_event(join)
            self._launch(n, f, events)

    @staticmethod
    def _launch(name, f, events):
        if events is None or name not in events:
            f()
            return
        s, e = events[name]
        s.record()
        f()
        e.record()

    def __call__(self, x: torch.Tensor, scores: torch.Tensor | None = None,
                 num_valid_tokens: torch.Tensor | None = None, out: torch.Tensor | None = None,
                 accumulate: bool = False) -> torch.Tensor:
        """x[T, D] bf16 and scores[T, E] (bf16 or f32; None: the layer's router
        computes them) on the device; num_valid_tokens: device int32 [1] (None:
        all T).  Returns out[T, D] bf16: for valid tokens the shared expert's
        output (if any) plus the routed sum, added into out when accumulate;
        other rows untouched."""
        if out is None:
            out = torch.zeros(x.shape[0], self.D, dtype=torch.bfloat16, device=x.device)
        self.run(self.stages(x, scores, num_valid_tokens, out, accumulate))
        if not self.use_fused_mlp(x.shape[0]):
            self._note_counts(self.buffers(x.shape[0], x.device).route["counts"])
        return out

    def capture(self, x: torch.Tensor, scores: torch.Tensor | None = None,
                num_valid_tokens: torch.Tensor | None = None, out: torch.Tensor | None = None,
                accumulate: bool = False):
        """Record one forward on these device tensors into a CUDA graph (stages,
        the second stream of the shared expert and its events included).  Returns
        (graph, out): graph.replay() reruns the forward on the tensors' current
        contents with no host-side launch work."""
        if out is None:
            out = torch.zeros(x.shape[0], self.D, dtype=torch.bfloat16, device=x.device)
        stages = self.stages(x, scores, num_valid_tokens, out, accumulate)
        self.run(stages)              # resolves the per-device lookups and kernel attributes outside the capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        self._capturing = True
        try:
            with torch.cuda.graph(graph):
                self.run(stages)
        finally:
            self._capturing = False
        return graph, out

    def use_fused_mlp(self, T: int) -> bool:
        if self.fp8:
            return False
        if self.fused_mlp is not None:
            return self.fused_mlp
        return T * self.top_k <= 128 * self.E

    # Rows per useful row that 256-row pair tiles may pad beyond 128-row tiles and
    # still win: on the bf16 fine_grained GEMMs pairs took 9% less time per row.
    PAIR_PADDING_MARGIN = 1.09

    @staticmethod
    def prefer_pairs(counts) -> bool:
        """256-row tiles for these per-expert row counts: when they pad at most
        PAIR_PADDING_MARGIN times the rows that 128-row tiles pad to."""
        c = np.asarray(counts, np.int64)
        c = c[c > 0]
        if c.size == 0:
            return False
        pair_rows = int(np.sum((c + 255) // 256 * 256))
        single_rows = int(np.sum((c + 127) // 128 * 128))
        return pair_rows <= MoELayer.PAIR_PADDING_MARGIN * single_rows

    def use_cta_pairs(self, T: int) -> bool:
        if self.cta_pairs is not None:
            return self.cta_pairs
        if self.fp8:
            return False
        last = self._last_counts()
        if last is not None:
            return self.prefer_pairs(last)
        return T * self.top_k >= 256 * self.E

    def _last_counts(self):
        """The previous forward's per-expert counts, if their copy to the host has landed."""
        if self._counts_event is None or not self._counts_event.query():
            return None
        return self._counts_host[: self.E].numpy()

    def _note_counts(self, counts: torch.Tensor):
        """Start a copy of this forward's counts to pinned host memory (for the tile choice)."""
        if self._capturing or self.fp8 or self.cta_pairs is not None:
            return
        if self._counts_host is None:
            self._counts_host = torch.empty(self.E + 1, dtype=torch.int32).pin_memory()
            self._counts_event = torch.cuda.Event()
        self._counts_host.copy_(counts, non_blocking=True)
        self._counts_event.record()

    def kernel_launches(self, T: int | None = None, with_router: bool = False) -> int:
        """Kernels one forward launches: the router (if used), routing (one
        kernel: single-block or cooperative), gather, the GEMMs (1 fused, or 2),
        the row pass of the FP8 w13 GEMM's quantising epilogue, scatter, and the
        shared expert's."""
        T = self._bufs.T if T is None and self._bufs is not None else (T or 0)
        route = 1                 # with the router: its emit kernel
        scatter = 0 if (self.top_k == 1 and self.weighting == "input") else 1   # scatter or finalize
        n = (route + 4 + scatter) if self.fp8 else (route + 1 + (1 if self.use_fused_mlp(T) else 2) + scatter)
        if with_router:
            n += 1
        if self.shared:
            n += 4 if self.fp8 else 2
        return n
