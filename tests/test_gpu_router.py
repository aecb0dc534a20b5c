"""moe_router_scores (tcgen05 router GEMM + sigmoid) against the oracle.

The GPU accumulates each logit in fp32 (split over CTAs in a fixed order), the
oracle in fp64; both round the logit to bf16 and take the sigmoid of that.
The fp32 sum is within about 1e-5 of the exact one, so the two bf16 logits
are at most one bf16 step apart, and a score may land on the sigmoid of the
neighbouring logit.  Bound, per element: the GPU score lies between
bf16(sigmoid(l - delta)) and bf16(sigmoid(l + delta)) (one more score step
either way for the fp32 sigmoid), with l the oracle's logit and delta = one
bf16 step of l plus 1e-3; and at least 99.5% of the scores are bit-identical.
Routing is an integer decision taken on the bf16 scores: moe_route on the
GPU's scores must equal the oracle's routing of those same scores bit for bit.
Rows past the valid tokens keep their sentinel bytes.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_token_routing_index_gb300 import workloads
from tests.helpers import bits, f64, is_sentinel, sentinel_like

pytestmark = pytest.mark.gpu


def _mb():
    from moe_token_routing_index_gb300 import binding

    return binding


def _bf16_bits(v: np.ndarray) -> np.ndarray:
    return bits(torch.from_numpy(np.asarray(v, np.float64)).to(torch.float32).to(torch.bfloat16))


def _bf16_step(v: np.ndarray) -> np.ndarray:
    a = np.abs(v)
    return np.exp2(np.floor(np.log2(np.where(a > 0, a, 2.0 ** -126))) - 7)


def _check_scores(got_bits: np.ndarray, x_bits, w_bits, Tv: int):
    ref, lg = oracle.router_scores(x_bits, w_bits, Tv, logits=True)
    got, ref, l = got_bits[:Tv], ref[:Tv], f64(lg[:Tv])
    delta = _bf16_step(l) + 1e-3
    lo = _bf16_bits(1.0 / (1.0 + np.exp(-(l - delta)))).astype(np.int32) - 1
    hi = _bf16_bits(1.0 / (1.0 + np.exp(-(l + delta)))).astype(np.int32) + 1
    g = got.astype(np.int32)          # scores are >= 0: bf16 bit order is value order
    bad = (g < lo) | (g > hi)
    assert not bad.any(), f"{bad.sum()} scores outside the bound, first at {np.argwhere(bad)[0]}"
    exact = (got == ref).mean()
    assert exact >= 0.995, f"only {exact:.5f} of the scores bit-identical"
    return ref


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill_fp8", "fine_grained", "padded_fp8"])
def test_router_scores_workloads(name):
    mb = _mb()
    cfg = workloads.CONFIGS[name]
    x = workloads.make_tokens(cfg)
    w = workloads.make_router(cfg)
    Tv = cfg.valid_tokens
    nv = torch.tensor([Tv], dtype=torch.int32, device="cuda")
    out = sentinel_like((cfg.T, cfg.E), torch.bfloat16)
    mb.moe_router_scores(x.cuda(), w.cuda(), nv, out=out)
    assert mb.device_error() == 0
    _check_scores(bits(out), bits(x), bits(w), Tv)
    assert is_sentinel(out[Tv:])
    # the routing decision on the GPU's scores
    r = mb.moe_route(out, cfg.top_k, nv)
    r_ref = oracle.route(bits(out), cfg.top_k, Tv)
    np.testing.assert_array_equal(r["counts"].cpu().numpy(), r_ref["counts"])
    a = Tv * cfg.top_k
    np.testing.assert_array_equal(r["token_indices"][:a].cpu().numpy(), r_ref["token_indices"])
    np.testing.assert_array_equal(r["expert_indices"][:a].cpu().numpy(), r_ref["expert_indices"])


@pytest.mark.parametrize("T,D,E,Tv", [(1, 16, 1, 1), (130, 48, 8, 129), (300, 1040, 24, 300), (257, 64, 256, 200),
                                      (1000, 7168, 100, 999), (5, 16384, 200, 5), (4096, 256, 16, 0),
                                      (40000, 128, 64, 39999)])
def test_router_scores_ragged_shapes(T, D, E, Tv):
    mb = _mb()
    g = torch.Generator().manual_seed(T * 7 + D + E)
    x = torch.randn(T, D, generator=g).to(torch.bfloat16)
    w = (torch.randn(E, D, generator=g) / D ** 0.5).to(torch.bfloat16)
    out = sentinel_like((T, E), torch.bfloat16)
    nv = torch.tensor([Tv], dtype=torch.int32, device="cuda")
    mb.moe_router_scores(x.cuda(), w.cuda(), nv, out=out)
    assert mb.device_error() == 0
    if Tv:
        _check_scores(bits(out), bits(x), bits(w), Tv)
    assert is_sentinel(out[Tv:])


def test_router_scores_deterministic_and_count_clamped():
    mb = _mb()
    cfg = workloads.CONFIGS["fine_grained"]
    x = workloads.make_tokens(cfg).cuda()
    w = workloads.make_router(cfg).cuda()
    o1 = mb.moe_router_scores(x, w).clone()
    o2 = mb.moe_router_scores(x, w)
    assert torch.equal(o1, o2)
    # a count above T is clamped to T and flagged
    nv = torch.tensor([cfg.T + 5], dtype=torch.int32, device="cuda")
    o3 = mb.moe_router_scores(x, w, nv)
    assert mb.device_error() & mb.MOE_DEVERR_BAD_COUNT
    assert torch.equal(o1, o3)


ROUTE_KEYS = ("counts", "expert_offsets", "expert_indices", "token_indices", "inv_rows", "topk_weights")


def _router_route_case(x, w, top_k, Tv):
    """moe_router_route against moe_router_scores followed by moe_route, bit for bit, and
    against the oracle's routing of the GPU's scores; nothing written past Tv."""
    mb = _mb()
    T, E = x.shape[0], w.shape[0]
    nv = torch.tensor([Tv], dtype=torch.int32, device="cuda")
    a_max = T * top_k
    out = {k: sentinel_like((E + 1,) if k in ("counts", "expert_offsets") else (max(a_max, 1),),
                            torch.float32 if k == "topk_weights" else torch.int32) for k in ROUTE_KEYS}
    scores = sentinel_like((T, E), torch.bfloat16)
    mb.moe_router_route(x, w, top_k, nv, scores=scores, with_weights=True, out=out)
    ref_scores = mb.moe_router_scores(x, w, nv, out=sentinel_like((T, E), torch.bfloat16))
    ref = mb.moe_route(ref_scores, top_k, nv, with_weights=True)
    torch.cuda.synchronize()
    assert mb.device_error() == 0
    assert torch.equal(scores.view(torch.int16), ref_scores.view(torch.int16))
    assert is_sentinel(scores[Tv:])
    a = Tv * top_k
    assert torch.equal(out["counts"], ref["counts"]) and torch.equal(out["expert_offsets"], ref["expert_offsets"])
    for k in ROUTE_KEYS[2:]:
        assert torch.equal(out[k][:a].view(torch.int32), ref[k][:a].view(torch.int32)), k
        assert is_sentinel(out[k][a:a_max]), f"{k} written past the routed rows"
    r_ref = oracle.route(bits(scores), top_k, Tv)
    np.testing.assert_array_equal(out["counts"].cpu().numpy(), r_ref["counts"])
    np.testing.assert_array_equal(out["token_indices"][:a].cpu().numpy(), r_ref["token_indices"])
    np.testing.assert_array_equal(out["expert_indices"][:a].cpu().numpy(), r_ref["expert_indices"])
    np.testing.assert_array_equal(out["inv_rows"][:a].cpu().numpy().reshape(Tv, top_k), r_ref["inv"])
    np.testing.assert_array_equal(out["topk_weights"][:a].cpu().numpy().reshape(Tv, top_k),
                                  oracle.topk_weights(bits(scores)[:Tv], r_ref))
    return scores


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill_fp8", "fine_grained", "padded_fp8"])
def test_router_route_workloads(name):
    """The top-k selection in the router's epilogue, on every workload's router."""
    cfg = workloads.CONFIGS[name]
    x = workloads.make_tokens(cfg).cuda()
    w = workloads.make_router(cfg).cuda()
    scores = _router_route_case(x, w, cfg.top_k, cfg.valid_tokens)
    _check_scores(bits(scores), bits(x), bits(w), cfg.valid_tokens)


@pytest.mark.parametrize("T,D,E,top_k,Tv", [(1, 16, 1, 1, 1), (130, 48, 8, 8, 129), (300, 1040, 24, 3, 300),
                                            (257, 64, 256, 6, 200), (1000, 7168, 100, 4, 999),
                                            (5, 16384, 200, 2, 5), (4096, 256, 16, 2, 0),
                                            (40000, 128, 64, 8, 39999), (16384, 4096, 128, 4, 11000)])
def test_router_route_ragged_shapes(T, D, E, top_k, Tv):
    """Ragged token counts (chunks cut by the valid count, tiles split over clusters of
    1-8 CTAs), E up to 256 (two column groups per lane), top_k = E, no valid token."""
    g = torch.Generator().manual_seed(T * 5 + D + E)
    x = torch.randn(T, D, generator=g).to(torch.bfloat16).cuda()
    w = (torch.randn(E, D, generator=g) / D ** 0.5).to(torch.bfloat16).cuda()
    _router_route_case(x, w, top_k, Tv)


def test_router_route_ties_go_to_the_lower_expert():
    """A router with equal rows gives equal scores for those experts: the lower index wins."""
    g = torch.Generator().manual_seed(3)
    T, D, E, k = 200, 128, 32, 4
    x = torch.randn(T, D, generator=g).to(torch.bfloat16).cuda()
    w = (torch.randn(E, D, generator=g) / D ** 0.5).to(torch.bfloat16)
    w[5] = w[20]
    w[6] = w[20]
    w[31] = w[0]
    _router_route_case(x, w.cuda(), k, T)
