"""moe_route (CUDA) against the oracle: bit-exact counts, offsets, permutation
and inverse permutation, on every workload and on the edge cases."""
import numpy as np
import pytest
import torch

import oracle
from moe_token_routing_index_gb300 import workloads
from tests.helpers import bits

pytestmark = pytest.mark.gpu


def _compare(scores_t: torch.Tensor, top_k: int, Tv: int | None = None):
    from moe_token_routing_index_gb300 import binding as mb

    T, E = scores_t.shape
    nv = None if Tv is None else torch.tensor([Tv], dtype=torch.int32, device="cuda")
    sentinel = -12345
    out = {n: torch.full((T * top_k,), sentinel, dtype=torch.int32, device="cuda")
           for n in ("expert_indices", "token_indices", "inv_rows")}
    got = mb.moe_route(scores_t.cuda(), top_k, nv, out=out)
    assert mb.device_error() == 0
    sc = scores_t.cpu()
    ref = oracle.route(bits(sc) if sc.dtype == torch.bfloat16 else sc.numpy(), top_k, Tv)
    a = int(ref["counts"][E])
    np.testing.assert_array_equal(got["counts"].cpu().numpy(), ref["counts"])
    np.testing.assert_array_equal(got["expert_offsets"].cpu().numpy(), ref["offsets"])
    np.testing.assert_array_equal(got["expert_indices"][:a].cpu().numpy(), ref["expert_indices"])
    np.testing.assert_array_equal(got["token_indices"][:a].cpu().numpy(), ref["token_indices"])
    np.testing.assert_array_equal(got["inv_rows"][:a].cpu().numpy(), ref["inv"].ravel())
    for n in ("expert_indices", "token_indices", "inv_rows"):
        assert torch.all(got[n][a:] == sentinel), f"{n} written past Tv * top_k"
    return got


@pytest.mark.parametrize("name", list(workloads.CONFIGS))
def test_route_workloads_bit_exact(name):
    cfg = workloads.CONFIGS[name]
    _compare(workloads.make_scores(cfg), cfg.top_k, cfg.Tv)


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (5, 3, 3), (37, 5, 2), (33, 32, 4), (70, 33, 1), (257, 64, 8),
                                   (100, 130, 6), (65, 1024, 2), (64, 1024, 1)])
def test_route_shapes(T, E, k):
    g = torch.Generator().manual_seed(T * 1000 + E * 10 + k)
    s = torch.randn(T, E, generator=g).to(torch.bfloat16)
    _compare(s, k)


def test_route_ties_and_signed_zeros():
    g = torch.Generator().manual_seed(7)
    palette = torch.tensor([0.0, -0.0, 0.5, 0.5, 1.0, -1.0])
    s = palette[torch.randint(0, 6, (300, 40), generator=g)].to(torch.bfloat16)
    _compare(s, 5)
    _compare(torch.zeros(64, 16, dtype=torch.bfloat16), 3)          # all tied
    _compare(-torch.zeros(64, 16, dtype=torch.bfloat16), 16)        # -0 everywhere, k = E


def test_route_f32_and_strided_scores():
    g = torch.Generator().manual_seed(8)
    s = torch.randn(150, 24, generator=g)
    _compare(s, 3)                                                   # f32 scores
    sb = torch.randn(24, 150, generator=g).to(torch.bfloat16)
    st = sb.cuda().t()                                               # stride_t = 1, stride_e = 150
    assert st.stride() == (1, 150)
    _compare(st, 2)


@pytest.mark.parametrize("Tv", [0, 1, 31, 32, 33, 500])
def test_route_valid_tokens(Tv):
    g = torch.Generator().manual_seed(Tv)
    s = torch.randn(500, 20, generator=g).to(torch.bfloat16)
    _compare(s, 3, Tv)


def test_route_deterministic():
    from moe_token_routing_index_gb300 import binding as mb

    cfg = workloads.CONFIGS["fine_grained"]
    s = workloads.make_scores(cfg).cuda()
    r1 = mb.moe_route(s, cfg.top_k)
    r2 = mb.moe_route(s, cfg.top_k)
    for n in ("counts", "expert_offsets", "expert_indices", "token_indices", "inv_rows"):
        assert torch.equal(r1[n], r2[n])


def test_route_out_of_range_valid_count_is_clamped_and_flagged():
    from moe_token_routing_index_gb300 import binding as mb

    s = torch.randn(40, 8).to(torch.bfloat16).cuda()
    got = mb.moe_route(s, 2, torch.tensor([1000], dtype=torch.int32, device="cuda"))
    assert mb.device_error() & mb.MOE_DEVERR_BAD_COUNT
    assert int(got["counts"][8]) == 80


@pytest.mark.parametrize("T,E,k,Tv", [(131072, 64, 2, 131072), (200000, 8, 1, 199999), (65536, 256, 6, 40001)])
def test_route_large_batches(T, E, k, Tv):
    """Far more 32-token chunks than resident blocks (each block loops over many),
    the largest expert counts per chunk, and a valid count inside a chunk."""
    g = torch.Generator().manual_seed(T + E)
    s = torch.randn(T, E, generator=g).to(torch.bfloat16)
    _compare(s, k, Tv)
