"""The seeded workload generators: determinism, shapes and the routing structure
each workload promises (zero-token experts, Zipf skew, padding)."""
import numpy as np
import torch

import oracle
from moe_token_routing_index_gb300 import workloads
from tests.helpers import bits


def test_generators_are_deterministic_and_shaped():
    cfg = workloads.CONFIGS["tiny"]
    x1, x2 = workloads.make_tokens(cfg), workloads.make_tokens(cfg)
    assert x1.shape == (64, 256) and x1.dtype == torch.bfloat16 and torch.equal(x1, x2)
    s = workloads.make_scores(cfg)
    assert s.shape == (64, 8) and torch.all((s >= 0) & (s <= 1))
    w13, w2 = workloads.make_weights(cfg)
    assert w13.shape == (8, 1024, 256) and w2.shape == (8, 256, 512)
    assert abs(float(w13.float().std()) - 0.02) < 1e-3
    sub13, sub2 = workloads.make_weights(cfg, experts=[2, 5])
    assert torch.equal(sub13, w13[[2, 5]]) and torch.equal(sub2, w2[[2, 5]])
    assert not torch.equal(workloads.make_tokens(cfg, seed=1), x1)


def test_fp8_workloads_draw_fp32_weights():
    cfg = workloads.MoEConfig("small_fp8", T=8, D=32, H=16, E=2, top_k=1, fp8=True)
    w13, w2 = workloads.make_weights(cfg)
    assert w13.dtype == torch.float32 and w2.dtype == torch.float32


def test_zero_expert_workload_leaves_experts_empty():
    cfg = workloads.CONFIGS["decode_zero"]
    r = oracle.route(bits(workloads.make_scores(cfg)), cfg.top_k)
    counts = r["counts"][:cfg.E]
    assert all(counts[e] == 0 for e in cfg.zero_experts)
    assert counts.sum() == cfg.T


def test_zipf_workload_is_skewed():
    cfg = workloads.CONFIGS["fine_grained"]
    r = oracle.route(bits(workloads.make_scores(cfg)), cfg.top_k)
    counts = r["counts"][:cfg.E]
    mean = cfg.routed_rows / cfg.E
    assert (counts == 0).any(), "some experts receive no token"
    assert (counts > 4 * mean).any(), "some experts receive more than four times the mean load"


def test_padded_workload_routes_only_valid_tokens():
    cfg = workloads.CONFIGS["padded_fp8"]
    r = oracle.route(bits(workloads.make_scores(cfg)), cfg.top_k, cfg.valid_tokens)
    assert r["counts"][cfg.E] == 44000 and r["token_indices"].max() == 10999
