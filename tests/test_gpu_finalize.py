"""Output-side weighting on the GPU against the oracle: the top-k weights the
router emits (bit-exact), unit-score gathers (bit-exact), moe_topk_finalize
(bit-exact: fp32 products and sums in slot order on both sides),
moe_scatter_add_padded (bit-exact, = the dense scatter over sum(counts) rows),
and the output-weighted layer forward (the derived forward tolerance)."""
import numpy as np
import pytest
import torch

import oracle
from moe_token_routing_index_gb300 import workloads
from tests.helpers import assert_forward_close, bits, f64, is_sentinel, rms, sentinel_like

pytestmark = pytest.mark.gpu


def _mb():
    from moe_token_routing_index_gb300 import binding

    return binding


def _i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()


@pytest.mark.parametrize("name", ["tiny", "decode", "fine_grained", "padded_fp8"])
def test_route_topk_weights_bit_exact(name):
    mb = _mb()
    cfg = workloads.CONFIGS[name]
    s = workloads.make_scores(cfg)
    Tv = cfg.valid_tokens
    nv = torch.tensor([Tv], dtype=torch.int32, device="cuda")
    r = mb.moe_route(s.cuda(), cfg.top_k, nv, with_weights=True)
    assert mb.device_error() == 0
    ref = oracle.route(bits(s), cfg.top_k, Tv)
    got = r["topk_weights"].view(cfg.T, cfg.top_k)[:Tv].cpu().numpy()
    np.testing.assert_array_equal(got, oracle.topk_weights(bits(s), ref))


@pytest.mark.parametrize("name", ["padded_fp8", "tiny"])
@pytest.mark.parametrize("quant", [False, True])
def test_unit_score_gathers_copy_rows(quant, name):
    mb = _mb()
    cfg = workloads.CONFIGS[name]
    x = workloads.make_tokens(cfg)
    r = oracle.route(bits(workloads.make_scores(cfg)), cfg.top_k, cfg.valid_tokens)
    a = len(r["token_indices"])
    ti, ei = _i32(r["token_indices"]), _i32(r["expert_indices"])
    unit = np.full((cfg.T, cfg.E), 0x3F80, np.uint16)
    if quant:
        q, sc = mb.moe_gather_scale_quant(x.cuda(), ti, ei, None)
        q_ref, sc_ref = oracle.gather_scale_quant(bits(x), r["token_indices"], r["expert_indices"], unit)
        np.testing.assert_array_equal(bits(q), q_ref)
        np.testing.assert_array_equal(sc.cpu().numpy(), sc_ref)
    else:
        out = mb.moe_gather_scale(x.cuda(), ti, ei, None)
        np.testing.assert_array_equal(bits(out), bits(x)[r["token_indices"]])
        # token-major (staged) path with the inverse permutation
        out2 = mb.moe_gather_scale(x.cuda(), ti, ei, None, inv_rows=_i32(r["inv"].ravel()), top_k=cfg.top_k)
        np.testing.assert_array_equal(bits(out2), bits(x)[r["token_indices"]])
    assert mb.device_error() == 0 and a > 0


@pytest.mark.parametrize("n,D,M,k,Mv,wdt,with_shared",
                         [(500, 256, 300, 4, 300, "f32", True), (44000, 4096, 11000, 4, 11000, "f32", False),
                          (70, 7168, 40, 8, 33, "bf16", True), (9, 16, 5, 1, 5, "f32", False),
                          (64, 2064, 64, 2, 60, "bf16", False), (120, 512, 50, 3, 47, "f32", True),
                          (300, 272, 90, 5, 90, "bf16", False), (200, 128, 12, 40, 11, "f32", True)])
def test_topk_finalize_bit_exact(n, D, M, k, Mv, wdt, with_shared):
    mb = _mb()
    g = torch.Generator().manual_seed(n + D + M)
    rows = (torch.randn(n, D, generator=g) * 2).to(torch.bfloat16)
    w = torch.rand(M, k, generator=g) * 2 - 0.5
    if wdt == "bf16":
        w = w.to(torch.bfloat16)
    idx = torch.randint(-1, n, (M, k), generator=g, dtype=torch.int32)
    shared = torch.randn(M, D, generator=g).to(torch.bfloat16) if with_shared else None
    out = sentinel_like((M, D), torch.bfloat16)
    nv = torch.tensor([Mv], dtype=torch.int32, device="cuda")
    mb.moe_topk_finalize(rows.cuda(), w.cuda(), idx.cuda(), None if shared is None else shared.cuda(), nv, out=out)
    assert mb.device_error() == 0
    ref = oracle.topk_finalize(bits(rows), w.float().numpy(), idx.numpy(), None if shared is None else bits(shared))
    np.testing.assert_array_equal(bits(out[:Mv]), ref[:Mv])
    assert is_sentinel(out[Mv:])


def test_topk_finalize_flags_bad_index():
    mb = _mb()
    rows = torch.ones(4, 32, dtype=torch.bfloat16, device="cuda")
    idx = torch.tensor([[0, 7], [1, -1]], dtype=torch.int32, device="cuda")
    w = torch.ones(2, 2, device="cuda")
    out = mb.moe_topk_finalize(rows, w, idx)
    assert mb.device_error() & mb.MOE_DEVERR_BAD_INDEX
    assert torch.equal(out, torch.ones(2, 32, dtype=torch.bfloat16, device="cuda"))   # the bad route is skipped


@pytest.mark.parametrize("name", ["fine_grained", "padded_fp8", "decode"])
def test_scatter_add_padded_equals_dense_scatter(name):
    mb = _mb()
    cfg = workloads.CONFIGS[name]
    s = workloads.make_scores(cfg)
    r = oracle.route(bits(s), cfg.top_k, cfg.valid_tokens)
    a = len(r["token_indices"])
    T_K = cfg.T * cfg.top_k
    g = torch.Generator().manual_seed(a)
    rows = torch.randn(T_K, cfg.D, generator=g).to(torch.bfloat16)    # padding rows past a hold noise
    init = torch.randn(cfg.T, cfg.D, generator=g).to(torch.bfloat16)
    out = init.cuda()
    inv = None
    if cfg.top_k > 1:
        inv = torch.zeros(T_K, dtype=torch.int32)
        inv[:a] = torch.from_numpy(r["inv"].ravel())
        inv = inv.cuda()
    ti = torch.zeros(T_K, dtype=torch.int32)
    ti[:a] = torch.from_numpy(r["token_indices"])
    mb.moe_scatter_add_padded(out, rows.cuda(), _i32(r["counts"][:cfg.E]), ti.cuda(), inv, cfg.top_k)
    assert mb.device_error() == 0
    ref = oracle.scatter_add(bits(init).copy(), bits(rows[:a]), r["token_indices"])
    np.testing.assert_array_equal(bits(out), ref)


def _host_weights(cfg, w13, w2):
    if cfg.fp8:
        return lambda ids: (w13[ids].float().cpu().numpy(), w2[ids].float().cpu().numpy())
    return lambda ids: (bits(w13[ids]), bits(w2[ids]))


@pytest.mark.parametrize("name,with_shared", [("tiny", False), ("tiny", True), ("fine_grained", True),
                                              ("padded_fp8", True), ("decode", False)])
def test_output_weighted_layer(name, with_shared):
    from moe_token_routing_index_gb300.forward import MoELayer

    mb = _mb()
    cfg = workloads.CONFIGS[name]
    x = workloads.make_tokens(cfg)
    s = workloads.make_scores(cfg)
    w13, w2 = workloads.make_weights(cfg, device="cuda")
    sh = workloads.make_shared_weights(cfg, device="cuda") if with_shared else None
    layer = MoELayer.from_weights(cfg, w13, w2, shared=sh, weighting="output")
    Tv = cfg.valid_tokens
    nv = None if cfg.Tv is None else torch.tensor([Tv], dtype=torch.int32, device="cuda")
    out = sentinel_like((cfg.T, cfg.D), torch.bfloat16)
    layer(x.cuda(), s.cuda(), nv, out=out)
    torch.cuda.synchronize()
    assert mb.device_error() == 0
    rng = np.random.default_rng(3)
    sample = np.arange(Tv) if Tv <= 64 else np.unique(np.concatenate([[0, Tv - 1], rng.integers(0, Tv, 10)]))
    xs, ss = np.ascontiguousarray(bits(x)[sample]), np.ascontiguousarray(bits(s)[sample])
    base = None
    if sh is not None:
        conv = (lambda t: t.float().cpu().numpy()) if cfg.fp8 else bits
        base = oracle.shared_expert(xs, conv(sh[0]), conv(sh[1]), fp8=cfg.fp8, z_bf16=cfg.fp8,
                                    scale_ub=cfg.scale_ub)
    ref = oracle.moe_forward_output_weighted(xs, ss, cfg.top_k, _host_weights(cfg, w13, w2), fp8=cfg.fp8,
                                             z_bf16=cfg.fp8, shared_out=base, scale_ub=cfg.scale_ub)["out"]
    got = f64(bits(out[torch.from_numpy(sample).cuda()]))
    exp = f64(ref)
    tol = 6e-2 if cfg.fp8 else 2e-2
    assert_forward_close(got, exp, tol, f"output-weighted forward {name} (shared {with_shared})")
    if Tv < cfg.T:
        assert is_sentinel(out[Tv:])


@pytest.mark.parametrize("name", ["tiny", "padded_fp8"])
def test_output_weighted_layer_with_router(name):
    """Router scores, the shared expert and output-side weighting together: the
    routing decision is taken on the GPU's own scores on both sides."""
    from moe_token_routing_index_gb300.forward import MoELayer

    mb = _mb()
    cfg = workloads.CONFIGS[name]
    x = workloads.make_tokens(cfg)
    w13, w2 = workloads.make_weights(cfg, device="cuda")
    router = workloads.make_router(cfg).cuda()
    sh = workloads.make_shared_weights(cfg, device="cuda")
    layer = MoELayer.from_weights(cfg, w13, w2, router=router, shared=sh, weighting="output")
    Tv = cfg.valid_tokens
    nv = None if cfg.Tv is None else torch.tensor([Tv], dtype=torch.int32, device="cuda")
    out = sentinel_like((cfg.T, cfg.D), torch.bfloat16)
    layer(x.cuda(), None, nv, out=out)
    torch.cuda.synchronize()
    assert mb.device_error() == 0
    scores = bits(layer.buffers(cfg.T, "cuda").extra["scores"])
    rng = np.random.default_rng(4)
    sample = np.arange(Tv) if Tv <= 64 else np.unique(np.concatenate([[0, Tv - 1], rng.integers(0, Tv, 10)]))
    xs, ss = np.ascontiguousarray(bits(x)[sample]), np.ascontiguousarray(scores[sample])
    conv = (lambda t: t.float().cpu().numpy()) if cfg.fp8 else bits
    base = oracle.shared_expert(xs, conv(sh[0]), conv(sh[1]), fp8=cfg.fp8, z_bf16=cfg.fp8, scale_ub=cfg.scale_ub)
    ref = oracle.moe_forward_output_weighted(xs, ss, cfg.top_k, _host_weights(cfg, w13, w2), fp8=cfg.fp8,
                                             z_bf16=cfg.fp8, shared_out=base, scale_ub=cfg.scale_ub)["out"]
    got = f64(bits(out[torch.from_numpy(sample).cuda()]))
    exp = f64(ref)
    tol = 6e-2 if cfg.fp8 else 2e-2
    assert_forward_close(got, exp, tol, f"output-weighted layer {name}")
    if Tv < cfg.T:
        assert is_sentinel(out[Tv:])
