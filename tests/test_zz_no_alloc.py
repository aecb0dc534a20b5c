"""moe_route_no_alloc, the routing entry point for callers that cannot allocate
device memory (it uses a fixed scratch array inside the library instead of a
caller workspace), called through the C ABI.

Two calls in a row, with different workload sizes so the second runs over the
first one's leftover scratch, must each give exactly what moe_route (with a
caller workspace) gives for the same inputs; once set up, calls change neither
the device's free memory nor PyTorch's allocations; sizes past the fixed
scratch are rejected without launching anything.  This file is collected last so a
stop-at-first-failure run has already run every other test.
"""
import ctypes

import pytest
import torch

from moe_token_routing_index_gb300 import workloads

pytestmark = pytest.mark.gpu

NAMES = ("counts", "expert_offsets", "expert_indices", "token_indices", "inv_rows")


def _no_alloc_out(scores, top_k):
    """Output tensors for one call, every entry -7 (to see what the call writes)."""
    T, E = scores.shape
    i32 = dict(dtype=torch.int32, device=scores.device)
    return {n: torch.full((E + 1,) if n in ("counts", "expert_offsets") else (max(T * top_k, 1),), -7, **i32)
            for n in NAMES}


def _call_no_alloc(scores, top_k, num_valid, out):
    from moe_token_routing_index_gb300 import binding as mb

    T, E = scores.shape
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    return mb.library().moe_route_no_alloc(
        p(scores), mb.MOE_DTYPE_BF16, scores.stride(0), scores.stride(1), T, E, top_k, p(num_valid),
        p(out["counts"]), p(out["expert_offsets"]), p(out["expert_indices"]), p(out["token_indices"]),
        p(out["inv_rows"]), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _no_alloc_route(scores, top_k, num_valid):
    out = _no_alloc_out(scores, top_k)
    return _call_no_alloc(scores, top_k, num_valid, out), out


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


def test_no_alloc_route_allocates_nothing_after_its_set_up():
    """After the set-up call (T = 0: the scratch address is looked up and the routing
    code loaded, nothing routed), routing calls change neither the device's free memory
    nor PyTorch's allocated bytes."""
    from moe_token_routing_index_gb300 import binding as mb

    cfg = workloads.CONFIGS["padded_fp8"]
    s = workloads.make_scores(cfg).cuda()
    nv = torch.tensor([cfg.Tv], dtype=torch.int32, device="cuda")
    st, setup = _no_alloc_route(s[:0], cfg.top_k, None)
    torch.cuda.synchronize()
    assert st == mb.MOE_OK and int(setup["counts"].abs().sum()) == 0
    outs = [_no_alloc_out(s, cfg.top_k) for _ in range(2)]       # outputs allocated before measuring
    torch.cuda.synchronize()
    free0, torch0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    for out in outs:
        assert _call_no_alloc(s, cfg.top_k, nv, out) == mb.MOE_OK
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0, "a routing call changed the device's free memory"
    assert torch.cuda.memory_allocated() == torch0
    assert torch.equal(outs[0]["token_indices"], outs[1]["token_indices"])
    assert mb.device_error() == 0


def test_no_alloc_route_rejects_sizes_past_its_scratch():
    from moe_token_routing_index_gb300 import binding as mb

    s = torch.zeros(65536, 128, dtype=torch.bfloat16, device="cuda")    # needs 1.25 MiB of scratch
    st, out = _no_alloc_route(s, 1, None)
    torch.cuda.synchronize()
    assert st == mb.MOE_ERR_WORKSPACE
    assert all(torch.all(out[n] == -7) for n in NAMES), "nothing may be launched"
