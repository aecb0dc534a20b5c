"""moe_route_no_alloc, the routing entry point for callers that cannot allocate
device memory (it uses a fixed scratch array inside the library instead of a
caller workspace), called through the C ABI.

Two calls in a row, with different workload sizes so the second runs over the
first one's leftover scratch, must each give exactly what moe_route (with a
caller workspace) gives for the same inputs; sizes past the fixed scratch are
rejected without launching anything.  This file is collected last so a
stop-at-first-failure run has already run every other test.
"""
import ctypes

import pytest
import torch

from moe_token_routing_index_gb300 import workloads

pytestmark = pytest.mark.gpu

NAMES = ("counts", "expert_offsets", "expert_indices", "token_indices", "inv_rows")


def _no_alloc_route(scores, top_k, num_valid):
    from moe_token_routing_index_gb300 import binding as mb

    T, E = scores.shape
    i32 = dict(dtype=torch.int32, device=scores.device)
    out = {n: torch.full((E + 1,) if n in ("counts", "expert_offsets") else (T * top_k,), -7, **i32)
           for n in NAMES}
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    st = mb.library().moe_route_no_alloc(
        p(scores), mb.MOE_DTYPE_BF16, scores.stride(0), scores.stride(1), T, E, top_k, p(num_valid),
        p(out["counts"]), p(out["expert_offsets"]), p(out["expert_indices"]), p(out["token_indices"]),
        p(out["inv_rows"]), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, out


def test_no_alloc_route_matches_moe_route_twice_in_a_row():
    from moe_token_routing_index_gb300 import binding as mb

    for name in ("padded_fp8", "fine_grained"):
        cfg = workloads.CONFIGS[name]
        s = workloads.make_scores(cfg).cuda()
        nv = None if cfg.Tv is None else torch.tensor([cfg.Tv], dtype=torch.int32, device="cuda")
        st, got = _no_alloc_route(s, cfg.top_k, nv)
        assert st == mb.MOE_OK, mb.library().moe_status_string(st)
        ref = mb.moe_route(s, cfg.top_k, nv)
        torch.cuda.synchronize()
        assert mb.device_error() == 0
        a = cfg.routed_rows
        assert torch.equal(got["counts"], ref["counts"]) and torch.equal(got["expert_offsets"], ref["expert_offsets"])
        for n in ("expert_indices", "token_indices", "inv_rows"):
            assert torch.equal(got[n][:a], ref[n][:a]), f"{name}: {n}"
            assert torch.all(got[n][a:] == -7), f"{name}: {n} written past the routed rows"


def test_no_alloc_route_rejects_sizes_past_its_scratch():
    from moe_token_routing_index_gb300 import binding as mb

    s = torch.zeros(65536, 128, dtype=torch.bfloat16, device="cuda")    # needs 1.25 MiB of scratch
    st, out = _no_alloc_route(s, 1, None)
    torch.cuda.synchronize()
    assert st == mb.MOE_ERR_WORKSPACE
    assert all(torch.all(out[n] == -7) for n in NAMES), "nothing may be launched"
