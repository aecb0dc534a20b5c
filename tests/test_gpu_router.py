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
