"""Edge cases of the whole layer on the GPU: no valid token at all (every stage
sees zero rows; the output stays untouched, no device error), and every token
routed to a single expert (one expert holds all rows of both GEMMs), checked
against the oracle on sampled tokens."""
import numpy as np
import pytest
import torch

import oracle
from moe_token_routing_index_gb300 import workloads
from tests.helpers import bits, f64, is_sentinel, rms, sentinel_like

pytestmark = pytest.mark.gpu


def _mb():
    from moe_token_routing_index_gb300 import binding

    return binding


@pytest.mark.parametrize("name", ["tiny", "padded_fp8", "fine_grained"])
@pytest.mark.parametrize("weighting", ["input", "output"])
def test_zero_valid_tokens_touch_nothing(name, weighting):
    from moe_token_routing_index_gb300.forward import MoELayer

    mb = _mb()
    cfg = workloads.CONFIGS[name]
    x = workloads.make_tokens(cfg).cuda()
    w13, w2 = workloads.make_weights(cfg, device="cuda")
    layer = MoELayer.from_weights(cfg, w13, w2, router=workloads.make_router(cfg).cuda(),
                                  shared=workloads.make_shared_weights(cfg, device="cuda"), weighting=weighting)
    nv = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = sentinel_like((cfg.T, cfg.D), torch.bfloat16)
    layer(x, None, nv, out=out)
    torch.cuda.synchronize()
    assert mb.device_error() == 0
    assert is_sentinel(out)
    assert int(layer.buffers(cfg.T, "cuda").route["counts"][cfg.E]) == 0


@pytest.mark.parametrize("name", ["prefill_fp8", "fine_grained"])
def test_all_tokens_on_one_expert(name):
    from moe_token_routing_index_gb300.forward import MoELayer

    mb = _mb()
    cfg = workloads.CONFIGS[name]
    k = cfg.top_k
    x = workloads.make_tokens(cfg)
    # experts 3 .. 3+k-1 score highest for every token: they take every routed row
    s = torch.full((cfg.T, cfg.E), 0.25)
    s[:, 3:3 + k] = torch.linspace(0.9, 0.5, k)
    s = s.to(torch.bfloat16)
    w13, w2 = workloads.make_weights(cfg, device="cuda")
    layer = MoELayer.from_weights(cfg, w13, w2)
    out = sentinel_like((cfg.T, cfg.D), torch.bfloat16)
    layer(x.cuda(), s.cuda(), out=out)
    torch.cuda.synchronize()
    assert mb.device_error() == 0
    counts = layer.buffers(cfg.T, "cuda").route["counts"].cpu().numpy()
    assert all(counts[3 + j] == cfg.T for j in range(k)) and counts[:cfg.E].sum() == cfg.T * k
    sample = np.unique(np.concatenate([[0, cfg.T - 1], np.random.default_rng(5).integers(0, cfg.T, 8)]))
    if cfg.fp8:
        wf = lambda ids: (w13[ids].float().cpu().numpy(), w2[ids].float().cpu().numpy())
    else:
        wf = lambda ids: (bits(w13[ids]), bits(w2[ids]))
    ref, _ = oracle.moe_forward_tokens(sample, bits(x), bits(s), k, wf, fp8=cfg.fp8, z_bf16=cfg.fp8,
                                       scale_ub=cfg.scale_ub)
    got, exp = f64(bits(out[torch.from_numpy(sample).cuda()])), f64(ref)
    tol = 6e-2 if cfg.fp8 else 2e-2
    a = np.abs(exp)
    step = np.exp2(np.floor(np.log2(np.where(a > 0, a, 1e-38))) - 7)
    err = np.abs(got - exp)
    assert np.all(err <= tol * rms(exp) + step), err.max() / rms(exp)
