"""Seeded synthetic workloads for the routed-expert MoE forward.

This module only draws inputs: token activations, router scores and expert
weights, with the shapes and value distributions of the five MoE layer
workloads below.  It holds none of the forward's arithmetic (no routing,
scaling, quantisation, GEMM, activation or combine), so both the CUDA path
and the CPU oracle can take their inputs from it.

Shapes follow the layouts of ``mslk/moe/layers.py`` (RoutedExperts.build):
``x[T, D]``, ``scores[T, E]`` (the sigmoid of router logits, as in
MetaShufflingMoE._route), ``w13[E, 2H, D]`` whose rows ``[0, H)`` are the
SiLU-input projection and rows ``[H, 2H)`` the gate multiplier, and
``w2[E, D, H]``.  For FP8-rowwise workloads the weights are drawn in fp32 and
each side quantises them per row with its own code.

Seeding: every tensor gets its own stream from ``numpy.random.SeedSequence``
(seed 0 unless stated), so adding a tensor never shifts another one.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

__all__ = ["MoEConfig", "CONFIGS", "make_tokens", "make_logits", "make_scores",
           "make_weights", "make_router", "make_shared_weights", "tensor_seed"]


@dataclass(frozen=True)
class MoEConfig:
    """One MoE layer workload.

    T: token-buffer rows; Tv: tokens that are valid (routed), ``None`` = T;
    D: model dim; H: expert hidden dim; E: experts; top_k: experts per token;
    fp8: FP8-rowwise activations and weights (else bf16);
    scale_ub: upper bound on activation row max for FP8 quantisation;
    skew: router-logit structure: "uniform", "zipf" (per-expert bias
    ln(k_e), k_e ~ Zipf(1.1)), or "zero_experts" (experts in
    ``zero_experts`` get logits shifted by -30, so they receive no token);
    weight_std: standard deviation of the N(0, std) expert weights.
    """

    name: str
    T: int
    D: int
    H: int
    E: int
    top_k: int
    fp8: bool = False
    Tv: int | None = None
    scale_ub: float | None = None
    skew: str = "uniform"
    zero_experts: tuple[int, ...] = field(default=())
    weight_std: float = 0.02

    @property
    def valid_tokens(self) -> int:
        return self.T if self.Tv is None else self.Tv

    @property
    def routed_rows(self) -> int:
        return self.valid_tokens * self.top_k

    def gemm_flops(self) -> float:
        """Multiply-adds x2 of both grouped GEMMs over the routed rows."""
        a = self.routed_rows
        return 2.0 * a * (2 * self.H) * self.D + 2.0 * a * self.D * self.H


CONFIGS: dict[str, MoEConfig] = {
    # Tiny MoE layer, the correctness case.
    "tiny": MoEConfig("tiny", T=64, D=256, H=512, E=8, top_k=1),
    # Decode-shaped, uniform routing.
    "decode": MoEConfig("decode", T=128, D=5120, H=8192, E=16, top_k=1),
    # Decode-shaped with four experts that receive no token.
    "decode_zero": MoEConfig("decode_zero", T=128, D=5120, H=8192, E=16, top_k=1,
                             skew="zero_experts", zero_experts=(1, 5, 9, 13)),
    # Prefill with FP8-rowwise activations and weights, activation scale bound 1200.
    "prefill_fp8": MoEConfig("prefill_fp8", T=8192, D=5120, H=8192, E=16, top_k=1,
                             fp8=True, scale_ub=1200.0),
    # Fine-grained experts with a Zipf-skewed expert load.
    "fine_grained": MoEConfig("fine_grained", T=4096, D=7168, H=2048, E=128, top_k=8,
                              skew="zipf"),
    # Padded batch: 16384-row buffer of which 11000 tokens are valid, FP8 rowwise.
    "padded_fp8": MoEConfig("padded_fp8", T=16384, D=4096, H=1536, E=128, top_k=4,
                            fp8=True, Tv=11000),
}

# Stream indices inside the SeedSequence spawn (child i does not depend on how many are spawned).
(_STREAM_TOKENS, _STREAM_LOGITS, _STREAM_W13, _STREAM_W2, _STREAM_BIAS, _STREAM_ROUTER, _STREAM_SHARED13,
 _STREAM_SHARED2) = range(8)
_NSTREAMS = 8


def tensor_seed(seed: int, stream: int) -> int:
    """A 63-bit seed for one tensor's stream, derived from the workload seed."""
    child = np.random.SeedSequence(seed).spawn(_NSTREAMS)[stream]
    return int(child.generate_state(2, dtype=np.uint64)[0] >> np.uint64(1))


def _cpu_gen(seed: int, stream: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(tensor_seed(seed, stream))
    return g


def make_tokens(cfg: MoEConfig, seed: int = 0) -> torch.Tensor:
    """x[T, D] bf16 with entries N(0, 1), drawn on the CPU."""
    g = _cpu_gen(seed, _STREAM_TOKENS)
    return torch.randn(cfg.T, cfg.D, generator=g, dtype=torch.float32).to(torch.bfloat16)


def make_logits(cfg: MoEConfig, seed: int = 0) -> torch.Tensor:
    """Router logits[T, E] fp32: N(0, 1) plus the workload's per-expert structure."""
    g = _cpu_gen(seed, _STREAM_LOGITS)
    logits = torch.randn(cfg.T, cfg.E, generator=g, dtype=torch.float32)
    if cfg.skew == "zipf":
        ss = np.random.SeedSequence(seed).spawn(_NSTREAMS)[_STREAM_BIAS]
        k = np.random.Generator(np.random.PCG64(ss)).zipf(1.1, cfg.E)
        logits += torch.from_numpy(np.log(k.astype(np.float64))).to(torch.float32)[None, :]
    elif cfg.skew == "zero_experts":
        logits[:, list(cfg.zero_experts)] -= 30.0
    elif cfg.skew != "uniform":
        raise ValueError(f"unknown skew {cfg.skew!r}")
    return logits


def make_scores(cfg: MoEConfig, seed: int = 0) -> torch.Tensor:
    """scores[T, E] bf16: the fp32 sigmoid of the logits rounded to bf16.

    The router's own projection is not part of this workload; its output
    distribution is what the generator reproduces.
    """
    return torch.sigmoid(make_logits(cfg, seed)).to(torch.bfloat16)


def make_weights(cfg: MoEConfig, seed: int = 0, device: str | torch.device = "cpu",
                 experts: list[int] | None = None) -> tuple[torch.Tensor, torch.Tensor]:
    """Expert weights (w13[E, 2H, D], w2[E, D, H]) with entries N(0, weight_std).

    bf16 for bf16 workloads, fp32 for FP8 workloads (each side quantises them
    per row itself).  Drawn on ``device`` with that device's generator, one
    expert at a time from a per-expert seed, so ``experts`` (a subset of
    expert ids) reproduces exactly those experts' slices on the same device.
    """
    dev = torch.device(device)
    dtype = torch.float32 if cfg.fp8 else torch.bfloat16
    ids = list(range(cfg.E)) if experts is None else list(experts)
    w13 = torch.empty(len(ids), 2 * cfg.H, cfg.D, dtype=dtype, device=dev)
    w2 = torch.empty(len(ids), cfg.D, cfg.H, dtype=dtype, device=dev)
    g = torch.Generator(device=dev)
    base13, base2 = tensor_seed(seed, _STREAM_W13), tensor_seed(seed, _STREAM_W2)
    mask = (1 << 63) - 1
    for i, e in enumerate(ids):
        g.manual_seed((base13 + 0x9E3779B97F4A7C15 * (e + 1)) & mask)
        w13[i] = (torch.randn(2 * cfg.H, cfg.D, generator=g, device=dev) * cfg.weight_std).to(dtype)
        g.manual_seed((base2 + 0x9E3779B97F4A7C15 * (e + 1)) & mask)
        w2[i] = (torch.randn(cfg.D, cfg.H, generator=g, device=dev) * cfg.weight_std).to(dtype)
    return w13, w2


def make_router(cfg: MoEConfig, seed: int = 0, device: str | torch.device = "cpu") -> torch.Tensor:
    """Router weight, transposed: w_router[E, D] = router_DE[D, E], bf16 with
    entries N(0, 1/D), so that with N(0, 1) tokens the logits are about N(0, 1)
    (the logit distribution of the uniform workloads).  Drawn on the CPU."""
    g = _cpu_gen(seed, _STREAM_ROUTER)
    w = torch.randn(cfg.E, cfg.D, generator=g, dtype=torch.float32) / float(np.sqrt(cfg.D))
    return w.to(torch.bfloat16).to(device)


def make_shared_weights(cfg: MoEConfig, seed: int = 0,
                        device: str | torch.device = "cpu") -> tuple[torch.Tensor, torch.Tensor]:
    """Shared-expert weights (w13[2H, D], w2[D, H]) with entries N(0, weight_std):
    bf16, or fp32 for FP8 workloads.  Drawn on ``device``."""
    dev = torch.device(device)
    dtype = torch.float32 if cfg.fp8 else torch.bfloat16
    g = torch.Generator(device=dev)
    g.manual_seed(tensor_seed(seed, _STREAM_SHARED13))
    w13 = (torch.randn(2 * cfg.H, cfg.D, generator=g, device=dev) * cfg.weight_std).to(dtype)
    g.manual_seed(tensor_seed(seed, _STREAM_SHARED2))
    w2 = (torch.randn(cfg.D, cfg.H, generator=g, device=dev) * cfg.weight_std).to(dtype)
    return w13, w2
