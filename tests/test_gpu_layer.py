"""The whole MoE layer (router scores, shared expert, routed experts) against the oracle.

Routing is an integer decision taken on bf16 scores, and the GPU router's
scores may differ from the oracle's by rounding (their bound is checked in
test_gpu_router.py).  So the oracle takes the routing decision on the GPU's
own scores: the expected output is the oracle's shared expert plus the
oracle's routed forward from those scores, compared with the same derived
tolerance as the routed forward (tol * rms plus one bf16 step of the
element; the strict bound on at least 99.9% of the elements).  Padding
tokens keep their sentinel bytes, and the overlapped (two-stream) forward
equals the serial one bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_token_routing_index_gb300 import workloads
from tests.helpers import assert_forward_close, bits, f64, is_sentinel, rms, sentinel_like

pytestmark = pytest.mark.gpu


def _assert_close(got, exp, tol, label=""):
    assert_forward_close(got, exp, tol, label)


def _host_weights(cfg, w13, w2):
    if cfg.fp8:
        return lambda ids: (w13[ids].float().cpu().numpy(), w2[ids].float().cpu().numpy())
    return lambda ids: (bits(w13[ids]), bits(w2[ids]))


def _host_shared(cfg, sh):
    if sh is None:
        return None
    if cfg.fp8:
        return sh[0].float().cpu().numpy(), sh[1].float().cpu().numpy()
    return bits(sh[0]), bits(sh[1])


def _layer(cfg, with_router=True, with_shared=True, overlap=True):
    from moe_token_routing_index_gb300.forward import MoELayer

    x = workloads.make_tokens(cfg)
    w13, w2 = workloads.make_weights(cfg, device="cuda")
    router = workloads.make_router(cfg).cuda() if with_router else None
    sh = workloads.make_shared_weights(cfg, device="cuda") if with_shared else None
    layer = MoELayer.from_weights(cfg, w13, w2, router=router, shared=sh, overlap_shared=overlap)
    return x, w13, w2, router, sh, layer


def _forward(cfg, layer, x, scores=None):
    from moe_token_routing_index_gb300 import binding as mb

    nv = None if cfg.Tv is None else torch.tensor([cfg.Tv], dtype=torch.int32, device="cuda")
    out = sentinel_like((cfg.T, cfg.D), torch.bfloat16)
    layer(x.cuda(), None if scores is None else scores.cuda(), nv, out=out)
    torch.cuda.synchronize()
    assert mb.device_error() == 0
    return out


def _tol(cfg):
    return 6e-2 if cfg.fp8 else 2e-2


@pytest.mark.parametrize("with_router,with_shared", [(True, True), (False, True), (True, False)])
def test_layer_tiny_full(with_router, with_shared):
    cfg = workloads.CONFIGS["tiny"]
    x, w13, w2, router, sh, layer = _layer(cfg, with_router, with_shared)
    given = None if with_router else workloads.make_scores(cfg)
    out = _forward(cfg, layer, x, given)
    scores = bits(layer.buffers(cfg.T, "cuda").extra["scores"]) if with_router else bits(given)
    base = None
    if with_shared:
        base = oracle.shared_expert(bits(x), *_host_shared(cfg, sh), fp8=cfg.fp8, z_bf16=cfg.fp8,
                                    scale_ub=cfg.scale_ub)
    ref = oracle.moe_forward(bits(x), scores, cfg.top_k, _host_weights(cfg, w13, w2), fp8=cfg.fp8, z_bf16=cfg.fp8,
                             out_init=base, scale_ub=cfg.scale_ub)
    _assert_close(f64(bits(out)), f64(ref["out"]), _tol(cfg),
                  f"layer tiny (router {with_router}, shared {with_shared})")


@pytest.mark.parametrize("name", ["decode", "prefill_fp8", "fine_grained", "padded_fp8"])
def test_layer_workloads_sampled(name):
    cfg = workloads.CONFIGS[name]
    x, w13, w2, router, sh, layer = _layer(cfg)
    out = _forward(cfg, layer, x)
    Tv = cfg.valid_tokens
    scores = bits(layer.buffers(cfg.T, "cuda").extra["scores"])
    rng = np.random.default_rng(2)
    sample = np.unique(np.concatenate([[0, Tv - 1], rng.integers(0, Tv, 30)]))
    xb = bits(x)
    base = oracle.shared_expert(np.ascontiguousarray(xb[sample]), *_host_shared(cfg, sh), fp8=cfg.fp8,
                                z_bf16=cfg.fp8, scale_ub=cfg.scale_ub)
    ref, _ = oracle.moe_forward_tokens(sample, xb, scores, cfg.top_k, _host_weights(cfg, w13, w2), fp8=cfg.fp8,
                                       z_bf16=cfg.fp8, out_init=None, scale_ub=cfg.scale_ub)
    # the routed rows of the sample, added into the shared rows (fp32 sum, one rounding per element)
    res = oracle.moe_forward(np.ascontiguousarray(xb[sample]), np.ascontiguousarray(scores[sample]), cfg.top_k,
                             _host_weights(cfg, w13, w2), fp8=cfg.fp8, z_bf16=cfg.fp8, out_init=base,
                             scale_ub=cfg.scale_ub)
    got = f64(bits(out[torch.from_numpy(sample).cuda()]))
    _assert_close(got, f64(res["out"]), _tol(cfg), f"layer {name} ({len(sample)} sampled tokens)")
    # the shared part alone is what the routed part was added to
    assert rms(f64(res["out"]) - f64(ref)) > 0
    if Tv < cfg.T:
        assert is_sentinel(out[Tv:]), "padding tokens must stay untouched"


@pytest.mark.parametrize("name", ["tiny", "fine_grained", "padded_fp8", "decode"])
def test_layer_overlap_equals_serial(name):
    cfg = workloads.CONFIGS[name]
    x, w13, w2, router, sh, layer = _layer(cfg, overlap=True)
    o1 = _forward(cfg, layer, x).clone()
    layer.overlap_shared = False
    o2 = _forward(cfg, layer, x)
    assert torch.equal(o1, o2)
    layer.overlap_shared = True
    o3 = _forward(cfg, layer, x)
    assert torch.equal(o1, o3)


@pytest.mark.parametrize("name,full", [("tiny", True), ("decode", False), ("decode", True), ("padded_fp8", True),
                                       ("fine_grained", False), ("prefill_fp8", False)])
def test_cuda_graph_replay_equals_eager(name, full):
    """A captured forward (CUDA graph, with the shared expert's second stream) replays to
    the eager forward's bytes, and follows new input contents."""
    from moe_token_routing_index_gb300 import binding as mb
    from moe_token_routing_index_gb300.forward import MoELayer

    cfg = workloads.CONFIGS[name]
    x = workloads.make_tokens(cfg).cuda()
    s = None if full else workloads.make_scores(cfg).cuda()
    w13, w2 = workloads.make_weights(cfg, device="cuda")
    kw = dict(router=workloads.make_router(cfg).cuda(), shared=workloads.make_shared_weights(cfg, device="cuda")) \
        if full else {}
    layer = MoELayer.from_weights(cfg, w13, w2, **kw)
    nv = None if cfg.Tv is None else torch.tensor([cfg.Tv], dtype=torch.int32, device="cuda")
    eager = layer(x, s, nv).clone()
    graph, out = layer.capture(x, s, nv)
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert mb.device_error() == 0
    assert torch.equal(out, eager)
    x2 = workloads.make_tokens(cfg, seed=1).cuda()
    eager2 = layer(x2, s, nv).clone()
    x.copy_(x2)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager2)


def test_two_layers_on_two_streams_match_sequential_runs():
    """Independent layers (own buffers and workspaces) may run concurrently on separate
    streams: cooperative routes, persistent GEMMs and cluster launches of both share
    the device, and each output equals its sequential run bit for bit."""
    from moe_token_routing_index_gb300 import binding as mb
    from moe_token_routing_index_gb300.forward import MoELayer

    layers, inputs = [], []
    for name, full in (("padded_fp8", True), ("fine_grained", False)):
        cfg = workloads.CONFIGS[name]
        w13, w2 = workloads.make_weights(cfg, device="cuda")
        kw = dict(router=workloads.make_router(cfg).cuda(), shared=workloads.make_shared_weights(cfg, device="cuda")) \
            if full else {}
        layers.append(MoELayer.from_weights(cfg, w13, w2, **kw))
        nv = None if cfg.Tv is None else torch.tensor([cfg.Tv], dtype=torch.int32, device="cuda")
        inputs.append((workloads.make_tokens(cfg).cuda(), None if full else workloads.make_scores(cfg).cuda(), nv))
    ref = [layer(*inp).clone() for layer, inp in zip(layers, inputs)]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [torch.zeros_like(r) for r in ref]
    for _ in range(3):
        for layer, inp, st, o in zip(layers, inputs, streams, outs):
            with torch.cuda.stream(st):
                layer(*inp, out=o)
    torch.cuda.synchronize()
    assert mb.device_error() == 0
    for o, r in zip(outs, ref):
        assert torch.equal(o, r)
