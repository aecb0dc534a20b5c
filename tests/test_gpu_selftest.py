"""The bounded device-side waits give up and report instead of hanging: each
wait of moe_selftest_bounded_wait never succeeds (an mbarrier nobody arrives
at; a grid barrier one block skips), must record MOE_DEVERR_TIMEOUT after its
limit, and leave the context usable for the next correct call."""
import time

import numpy as np
import pytest
import torch

import oracle
from moe_token_routing_index_gb300 import workloads
from tests.helpers import bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("which", [0, 1])
def test_bounded_wait_times_out_and_context_stays_usable(which):
    from moe_token_routing_index_gb300 import binding as mb

    assert mb.device_error() == 0
    t0 = time.perf_counter()
    err = mb.moe_selftest_bounded_wait(which, 20_000_000)       # 20 ms
    dt = time.perf_counter() - t0
    assert err & mb.MOE_DEVERR_TIMEOUT
    assert 0.015 < dt < 5.0, dt                                   # it waited about its limit, then returned
    cfg = workloads.CONFIGS["tiny"]
    s = workloads.make_scores(cfg)
    r = mb.moe_route(s.cuda(), cfg.top_k)
    assert mb.device_error() == 0
    np.testing.assert_array_equal(r["token_indices"].cpu().numpy(), oracle.route(bits(s), cfg.top_k)["token_indices"])
