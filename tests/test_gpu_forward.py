"""The whole routed-expert forward (MoELayer over the C ABI) against the oracle.

Tolerance (end to end, over the compared output rows): |gpu - oracle| <=
tol * rms(oracle) with tol = 2e-2 for bf16 layers and 6e-2 for FP8-rowwise
layers, plus one bf16 step of the oracle value at that element.  The output
is itself rounded to bf16, and the two sides sum in different orders and
precisions (fp32 tensor-core accumulation vs fp64), so near a rounding
boundary they can land one bf16 step apart; for an element larger than about
2.6 * rms that single step alone exceeds 2e-2 * rms.  Without the allowance
the bound must still hold on at least 99.9% of the elements.  The tiny workload is compared in full; the full-size workloads on a
sample of tokens (the oracle computes those tokens' rows exactly as its full
forward would).  Routing is compared bit for bit on the full workload, and
padding tokens must keep their sentinel bytes.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_token_routing_index_gb300 import workloads
from tests.helpers import assert_forward_close, bits, f64, is_sentinel, rms, sentinel_like

pytestmark = pytest.mark.gpu


def _run(cfg, seed=0):
    from moe_token_routing_index_gb300 import binding as mb
    from moe_token_routing_index_gb300.forward import MoELayer

    x = workloads.make_tokens(cfg, seed)
    s = workloads.make_scores(cfg, seed)
    w13, w2 = workloads.make_weights(cfg, seed, device="cuda")
    layer = MoELayer.from_weights(cfg, w13, w2)
    nv = None if cfg.Tv is None else torch.tensor([cfg.Tv], dtype=torch.int32, device="cuda")
    out = sentinel_like((cfg.T, cfg.D), torch.bfloat16)
    layer(x.cuda(), s.cuda(), nv, out=out)
    torch.cuda.synchronize()
    assert mb.device_error() == 0
    return x, s, w13, w2, layer, out


def _weights_fn(cfg, w13, w2):
    if cfg.fp8:
        return lambda ids: (w13[ids].float().cpu().numpy(), w2[ids].float().cpu().numpy())
    return lambda ids: (bits(w13[ids]), bits(w2[ids]))


def _tol(cfg):
    return 6e-2 if cfg.fp8 else 2e-2


def _assert_close(got, exp, tol, label=""):
    assert_forward_close(got, exp, tol, label)


def test_forward_tiny_full():
    cfg = workloads.CONFIGS["tiny"]
    x, s, w13, w2, layer, out = _run(cfg)
    ref = oracle.moe_forward(bits(x), bits(s), cfg.top_k, _weights_fn(cfg, w13, w2), fp8=False)
    exp = f64(ref["out"])
    got = f64(bits(out))
    _assert_close(got, exp, _tol(cfg), "forward tiny (all tokens)")
    # stage by stage: routing and the gathered rows are bit-exact
    r = layer.buffers(cfg.T, "cuda").route
    np.testing.assert_array_equal(r["token_indices"].cpu().numpy(), ref["route"]["token_indices"])
    np.testing.assert_array_equal(bits(layer.buffers(cfg.T, "cuda").xr), ref["x_routed"])


@pytest.mark.parametrize("name", ["decode", "decode_zero", "prefill_fp8", "fine_grained", "padded_fp8"])
def test_forward_workloads_sampled(name):
    cfg = workloads.CONFIGS[name]
    x, s, w13, w2, layer, out = _run(cfg)
    Tv = cfg.valid_tokens
    # routing over the whole workload, bit-exact
    r_ref = oracle.route(bits(s), cfg.top_k, Tv)
    r = layer.buffers(cfg.T, "cuda").route
    np.testing.assert_array_equal(r["counts"].cpu().numpy(), r_ref["counts"])
    a = Tv * cfg.top_k
    np.testing.assert_array_equal(r["token_indices"][:a].cpu().numpy(), r_ref["token_indices"])
    # the output rows of sampled tokens
    rng = np.random.default_rng(1)
    sample = np.unique(np.concatenate([[0, Tv - 1], rng.integers(0, Tv, 30)]))
    ref_rows, _ = oracle.moe_forward_tokens(sample, bits(x), bits(s), cfg.top_k, _weights_fn(cfg, w13, w2),
                                            fp8=cfg.fp8, z_bf16=cfg.fp8, scale_ub=cfg.scale_ub)
    exp = f64(ref_rows)
    got = f64(bits(out[torch.from_numpy(sample).cuda()]))
    _assert_close(got, exp, _tol(cfg), f"forward {name} ({len(sample)} sampled tokens)")
    if Tv < cfg.T:
        assert is_sentinel(out[Tv:]), "padding tokens must stay untouched"


def test_forward_is_deterministic():
    from moe_token_routing_index_gb300.forward import MoELayer

    cfg = workloads.CONFIGS["fine_grained"]
    x = workloads.make_tokens(cfg).cuda()
    s = workloads.make_scores(cfg).cuda()
    w13, w2 = workloads.make_weights(cfg, device="cuda")
    layer = MoELayer.from_weights(cfg, w13, w2)
    o1 = layer(x, s).clone()
    o2 = layer(x, s)
    assert torch.equal(o1, o2)


@pytest.mark.parametrize("name", ["fine_grained", "tiny", "prefill_fp8"])
def test_forward_cta_pair_tiles_change_no_bit(name):
    """256-row tiles on CTA pairs accumulate each output element in the same order
    as 128-row tiles, so the whole forward is identical either way."""
    from moe_token_routing_index_gb300 import binding as mb
    from moe_token_routing_index_gb300.forward import MoELayer

    cfg = workloads.CONFIGS[name]
    x = workloads.make_tokens(cfg).cuda()
    s = workloads.make_scores(cfg).cuda()
    w13, w2 = workloads.make_weights(cfg, device="cuda")
    outs = []
    for pairs in (False, True):
        layer = MoELayer.from_weights(cfg, w13, w2, cta_pairs=pairs, fused_mlp=False)
        outs.append(layer(x, s).clone())
    torch.cuda.synchronize()
    assert mb.device_error() == 0
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("name,with_shared", [("tiny", False), ("tiny", True), ("decode", False),
                                              ("fine_grained", False), ("padded_fp8", True)])
def test_forward_accumulates_into_existing_output(name, with_shared):
    """accumulate=True adds the layer into out (a residual, say): the shared rows are added
    into out first (fp32 sum, one rounding), then the routed rows, as the oracle's combine
    adds them into its starting output."""
    from moe_token_routing_index_gb300 import binding as mb
    from moe_token_routing_index_gb300.forward import MoELayer

    cfg = workloads.CONFIGS[name]
    x = workloads.make_tokens(cfg)
    s = workloads.make_scores(cfg)
    w13, w2 = workloads.make_weights(cfg, device="cuda")
    sh = workloads.make_shared_weights(cfg, device="cuda") if with_shared else None
    layer = MoELayer.from_weights(cfg, w13, w2, shared=sh)
    g = torch.Generator().manual_seed(11)
    init = torch.randn(cfg.T, cfg.D, generator=g).to(torch.bfloat16)
    out = init.cuda()
    nv = None if cfg.Tv is None else torch.tensor([cfg.Tv], dtype=torch.int32, device="cuda")
    layer(x.cuda(), s.cuda(), nv, out=out, accumulate=True)
    torch.cuda.synchronize()
    assert mb.device_error() == 0
    Tv = cfg.valid_tokens
    rng = np.random.default_rng(6)
    sample = np.arange(Tv) if Tv <= 64 else np.unique(np.concatenate([[0, Tv - 1], rng.integers(0, Tv, 10)]))
    base = bits(init)[sample]
    if sh is not None:
        conv = (lambda t: t.float().cpu().numpy()) if cfg.fp8 else bits
        shared = oracle.shared_expert(np.ascontiguousarray(bits(x)[sample]), conv(sh[0]), conv(sh[1]), fp8=cfg.fp8,
                                      z_bf16=cfg.fp8, scale_ub=cfg.scale_ub)
        base = bits((torch.from_numpy(f64(base)).float() + torch.from_numpy(f64(shared)).float()).to(torch.bfloat16))
    ref, _ = oracle.moe_forward_tokens(sample, bits(x), bits(s), cfg.top_k, _weights_fn(cfg, w13, w2), fp8=cfg.fp8,
                                       z_bf16=cfg.fp8, out_init=None, scale_ub=cfg.scale_ub)
    res = oracle.moe_forward(np.ascontiguousarray(bits(x)[sample]), np.ascontiguousarray(bits(s)[sample]), cfg.top_k,
                             _weights_fn(cfg, w13, w2), fp8=cfg.fp8, z_bf16=cfg.fp8,
                             out_init=np.ascontiguousarray(base), scale_ub=cfg.scale_ub)
    got = f64(bits(out[torch.from_numpy(sample).cuda()]))
    _assert_close(got, f64(res["out"]), _tol(cfg), f"forward {name} accumulate (shared {with_shared})")
    assert rms(f64(res["out"]) - f64(ref)) > 0              # the starting output did take part
    if Tv < cfg.T:
        assert torch.equal(out[Tv:].cpu(), init[Tv:]), "padding tokens keep their values"


@pytest.mark.parametrize("name", ["decode", "fine_grained", "padded_fp8"])
def test_layer_with_packed_weights_equals_row_major(name):
    """MoELayer packs its resident weights by default (H and D multiples of 128); the
    forward equals the row-major layer's bit for bit."""
    from moe_token_routing_index_gb300 import binding as mb
    from moe_token_routing_index_gb300.forward import MoELayer

    cfg = workloads.CONFIGS[name]
    x = workloads.make_tokens(cfg).cuda()
    s = workloads.make_scores(cfg).cuda()
    nv = None if cfg.Tv is None else torch.tensor([cfg.Tv], dtype=torch.int32, device="cuda")
    w13, w2 = workloads.make_weights(cfg, device="cuda")
    packed = MoELayer.from_weights(cfg, w13, w2)
    plain = MoELayer.from_weights(cfg, w13, w2, pack_weights=False)
    assert isinstance(packed.w13, mb.PackedWeights) and not isinstance(plain.w13, mb.PackedWeights)
    o1 = packed(x, s, nv).clone()
    o2 = plain(x, s, nv)
    torch.cuda.synchronize()
    assert mb.device_error() == 0
    assert torch.equal(o1, o2)
