"""The row-wise CUDA stages against the oracle: gather*score and the FP8
quantising gather (bit-exact), silu_mul (within one bf16 step), silu_mul_quant
(codes within one e4m3 step) and the scatter-add combine (bit-exact), at the
workloads' full sizes and on ragged small cases; rows past the valid count
must keep their sentinel bytes."""
import numpy as np
import pytest
import torch

import oracle
from moe_token_routing_index_gb300 import workloads
from tests.helpers import bits, dev_bf16, e4m3_step_diff, is_sentinel, sentinel_like

pytestmark = pytest.mark.gpu


def _mb():
    from moe_token_routing_index_gb300 import binding

    return binding


def _routed(cfg):
    """Inputs of the gather stage: x, scores and the oracle's routing (int32 on device)."""
    x = workloads.make_tokens(cfg)
    s = workloads.make_scores(cfg)
    r = oracle.route(bits(s), cfg.top_k, cfg.valid_tokens)
    return x, s, r


def _idx(a, n=None):
    t = torch.from_numpy(np.ascontiguousarray(a, np.int32))
    if n is not None and n > len(a):      # pad the buffer like the router's T * top_k arrays
        t = torch.cat([t, torch.zeros(n - len(a), dtype=torch.int32)])
    return t.cuda()


GATHER_CASES = ["tiny", "decode", "decode_zero", "fine_grained"]
QUANT_CASES = ["prefill_fp8", "padded_fp8"]


@pytest.mark.parametrize("name", GATHER_CASES + QUANT_CASES)
def test_gather_scale_bit_exact(name):
    mb = _mb()
    cfg = workloads.CONFIGS[name]
    x, s, r = _routed(cfg)
    a_buf = cfg.T * cfg.top_k
    valid = torch.tensor([r["counts"][cfg.E]], dtype=torch.int32, device="cuda")
    out = sentinel_like((a_buf, cfg.D), torch.bfloat16)
    mb.moe_gather_scale(x.cuda(), _idx(r["token_indices"], a_buf), _idx(r["expert_indices"], a_buf), s.cuda(),
                        valid, out=out)
    assert mb.device_error() == 0
    ref = oracle.gather_scale(bits(x), r["token_indices"], r["expert_indices"], bits(s))
    a = len(r["token_indices"])
    np.testing.assert_array_equal(bits(out[:a]), ref)
    assert is_sentinel(out[a:])


@pytest.mark.parametrize("name", QUANT_CASES + ["tiny", "fine_grained"])
@pytest.mark.parametrize("ub", [None, 1200.0, 0.5])
def test_gather_scale_quant_bit_exact(name, ub):
    mb = _mb()
    cfg = workloads.CONFIGS[name]
    x, s, r = _routed(cfg)
    a_buf = cfg.T * cfg.top_k
    valid = torch.tensor([r["counts"][cfg.E]], dtype=torch.int32, device="cuda")
    ub_t = None if ub is None else torch.tensor([ub], dtype=torch.float32, device="cuda")
    out = sentinel_like((a_buf, cfg.D), torch.float8_e4m3fn)
    osc = sentinel_like((a_buf,), torch.float32)
    mb.moe_gather_scale_quant(x.cuda(), _idx(r["token_indices"], a_buf), _idx(r["expert_indices"], a_buf),
                              s.cuda(), ub_t, valid, out=out, out_scale=osc)
    assert mb.device_error() == 0
    q, sc = oracle.gather_scale_quant(bits(x), r["token_indices"], r["expert_indices"], bits(s), ub)
    a = len(r["token_indices"])
    np.testing.assert_array_equal(bits(out[:a]), q)
    np.testing.assert_array_equal(osc[:a].cpu().numpy(), sc)
    assert is_sentinel(out[a:]) and is_sentinel(osc[a:])


@pytest.mark.parametrize("T,D,a,E", [(5, 16, 7, 3), (40, 272, 33, 6), (9, 2064, 13, 2), (3, 16384, 4, 2)])
def test_gather_ragged_shapes(T, D, a, E):
    mb = _mb()
    g = torch.Generator().manual_seed(T + D + a)
    x = torch.randn(T, D, generator=g).to(torch.bfloat16)
    s = torch.rand(T, E, generator=g)                      # f32 scores this time
    ti = torch.randint(0, T, (a,), generator=g, dtype=torch.int32)
    ei = torch.randint(0, E, (a,), generator=g, dtype=torch.int32)
    out = mb.moe_gather_scale(x.cuda(), ti.cuda(), ei.cuda(), s.cuda())
    np.testing.assert_array_equal(bits(out), oracle.gather_scale(bits(x), ti.numpy(), ei.numpy(), s.numpy()))
    q, sc = mb.moe_gather_scale_quant(x.cuda(), ti.cuda(), ei.cuda(), s.cuda())
    q_ref, sc_ref = oracle.gather_scale_quant(bits(x), ti.numpy(), ei.numpy(), s.numpy())
    np.testing.assert_array_equal(bits(q), q_ref)
    np.testing.assert_array_equal(sc.cpu().numpy(), sc_ref)


def test_gather_bad_index_is_skipped_and_flagged():
    mb = _mb()
    x = torch.randn(4, 32).to(torch.bfloat16).cuda()
    s = torch.rand(4, 2).cuda()
    ti = torch.tensor([0, 9, 1], dtype=torch.int32, device="cuda")
    ei = torch.tensor([0, 1, 5], dtype=torch.int32, device="cuda")
    out = sentinel_like((3, 32), torch.bfloat16)
    mb.moe_gather_scale(x, ti, ei, s, out=out)
    assert mb.device_error() & mb.MOE_DEVERR_BAD_INDEX
    assert is_sentinel(out[1:]) and not is_sentinel(out[:1])


def _y_rows(a, H, seed, scale=2.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(a, 2 * H, generator=g) * scale).to(torch.bfloat16)


@pytest.mark.parametrize("a,H,valid", [(64, 512, 64), (8192, 8192, 8192), (32768, 2048, 30000), (7, 16, 5),
                                       (33, 1552, 20)])
def test_silu_mul_within_one_bf16_step(a, H, valid):
    mb = _mb()
    y = _y_rows(a, H, a + H)
    out = sentinel_like((a, H), torch.bfloat16)
    mb.moe_silu_mul(y.cuda(), H, torch.tensor([valid], dtype=torch.int32, device="cuda"), out=out)
    ref = oracle.silu_mul(bits(y), H, valid)
    got = bits(out[:valid]).astype(np.int32)
    diff = np.abs(got - ref[:valid].astype(np.int32))
    assert diff.max() <= 1 and (diff == 0).mean() > 0.999
    assert is_sentinel(out[valid:])


@pytest.mark.parametrize("a,H,valid,ub", [(8192, 8192, 8192, 1200.0), (65536, 1536, 44000, None), (9, 48, 9, 0.25),
                                          (20, 16384, 17, None)])
def test_silu_mul_quant_within_one_e4m3_step(a, H, valid, ub):
    mb = _mb()
    y = _y_rows(a, H, a + 3 * H)
    ub_t = None if ub is None else torch.tensor([ub], dtype=torch.float32, device="cuda")
    out = sentinel_like((a, H), torch.float8_e4m3fn)
    osc = sentinel_like((a,), torch.float32)
    mb.moe_silu_mul_quant(y.cuda(), H, ub_t, torch.tensor([valid], dtype=torch.int32, device="cuda"), out=out,
                          out_scale=osc)
    q_ref, s_ref = oracle.silu_mul_quant(bits(y), H, ub, valid)
    steps = e4m3_step_diff(bits(out[:valid]), q_ref[:valid])
    assert steps.max() <= 1 and (steps == 0).mean() > 0.999
    np.testing.assert_allclose(osc[:valid].cpu().numpy(), s_ref[:valid], rtol=1e-6)
    assert is_sentinel(out[valid:]) and is_sentinel(osc[valid:])


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill_fp8", "fine_grained", "padded_fp8"])
@pytest.mark.parametrize("use_inv", [True, False])
def test_scatter_add_bit_exact(name, use_inv):
    mb = _mb()
    cfg = workloads.CONFIGS[name]
    if cfg.top_k > 1 and not use_inv:
        pytest.skip("top_k > 1 needs the inverse permutation")
    s = workloads.make_scores(cfg)
    r = oracle.route(bits(s), cfg.top_k, cfg.valid_tokens)
    a = len(r["token_indices"])
    g = torch.Generator().manual_seed(a)
    rows = torch.randn(a, cfg.D, generator=g).to(torch.bfloat16)
    init = torch.randn(cfg.T, cfg.D, generator=g).to(torch.bfloat16)
    out = init.cuda()
    valid = torch.tensor([a], dtype=torch.int32, device="cuda")
    inv = _idx(r["inv"].ravel()) if use_inv else None
    mb.moe_scatter_add(out, rows.cuda(), _idx(r["token_indices"]), inv, cfg.top_k, valid)
    assert mb.device_error() == 0
    ref = oracle.scatter_add(bits(init).copy(), bits(rows), r["token_indices"])
    np.testing.assert_array_equal(bits(out), ref)
    Tv = cfg.valid_tokens
    assert torch.equal(out[Tv:].cpu(), init[Tv:]), "tokens past the valid count stay as they were"
    # overwrite mode: the same as adding into zeros, and still leaves the padding tokens alone
    out2 = init.cuda()
    mb.moe_scatter_add(out2, rows.cuda(), _idx(r["token_indices"]), inv, cfg.top_k, valid, accumulate=False)
    ref0 = oracle.scatter_add(np.zeros_like(bits(init)), bits(rows), r["token_indices"])
    np.testing.assert_array_equal(bits(out2[:Tv]), ref0[:Tv])
    assert torch.equal(out2[Tv:].cpu(), init[Tv:])


@pytest.mark.parametrize("T,D,E,k", [(300, 256, 8, 2), (97, 2064, 12, 3), (64, 512, 16, 5), (13, 144, 48, 40)])
@pytest.mark.parametrize("accumulate", [False, True])
def test_scatter_add_inverse_any_top_k(T, D, E, k, accumulate):
    """The inverse-permutation combine for top_k values with and without a specialised
    kernel (2, and 3, 5, 40 on the generic one): bit-exact against the oracle, in both
    the overwrite and the accumulate mode."""
    mb = _mb()
    g = torch.Generator().manual_seed(T + D + k)
    s = torch.rand(T, E, generator=g).to(torch.bfloat16)
    r = oracle.route(bits(s), k)
    a = T * k
    rows = (torch.randn(a, D, generator=g) * 3).to(torch.bfloat16)
    init = torch.randn(T, D, generator=g).to(torch.bfloat16)
    out = init.cuda()
    mb.moe_scatter_add(out, rows.cuda(), _idx(r["token_indices"]), _idx(r["inv"].ravel()), k,
                       torch.tensor([a], dtype=torch.int32, device="cuda"), accumulate=accumulate)
    assert mb.device_error() == 0
    base = bits(init).copy() if accumulate else np.zeros((T, D), np.uint16)   # overwrite = adding into zeros
    ref = oracle.scatter_add(base, bits(rows), r["token_indices"])
    np.testing.assert_array_equal(bits(out), ref)


@pytest.mark.parametrize("name", ["fine_grained", "padded_fp8", "tiny"])
@pytest.mark.parametrize("quant", [False, True])
def test_token_major_gather_equals_row_major(name, quant):
    """With the router's inverse permutation the gathers read each x row once per token;
    the output equals the row-major gather (and so the oracle) bit for bit."""
    mb = _mb()
    cfg = workloads.CONFIGS[name]
    x, s, r = _routed(cfg)
    a_buf = cfg.T * cfg.top_k
    a = len(r["token_indices"])
    valid = torch.tensor([a], dtype=torch.int32, device="cuda")
    ti, ei = _idx(r["token_indices"], a_buf), _idx(r["expert_indices"], a_buf)
    inv = _idx(r["inv"].ravel(), a_buf)
    xd, sd = x.cuda(), s.cuda()
    if quant:
        q1 = sentinel_like((a_buf, cfg.D), torch.float8_e4m3fn)
        s1 = sentinel_like((a_buf,), torch.float32)
        mb.moe_gather_scale_quant(xd, ti, ei, sd, None, valid, inv_rows=inv, top_k=cfg.top_k, out=q1, out_scale=s1)
        q_ref, s_ref = oracle.gather_scale_quant(bits(x), r["token_indices"], r["expert_indices"], bits(s))
        np.testing.assert_array_equal(bits(q1[:a]), q_ref)
        np.testing.assert_array_equal(s1[:a].cpu().numpy(), s_ref)
        assert is_sentinel(q1[a:]) and is_sentinel(s1[a:])
    else:
        o1 = sentinel_like((a_buf, cfg.D), torch.bfloat16)
        mb.moe_gather_scale(xd, ti, ei, sd, valid, inv_rows=inv, top_k=cfg.top_k, out=o1)
        ref = oracle.gather_scale(bits(x), r["token_indices"], r["expert_indices"], bits(s))
        np.testing.assert_array_equal(bits(o1[:a]), ref)
        assert is_sentinel(o1[a:])
    assert mb.device_error() == 0


@pytest.mark.parametrize("T,D,E,k", [(37, 16, 8, 3), (50, 272, 12, 5), (29, 2064, 9, 7), (40, 7168, 40, 32),
                                     (21, 1024, 64, 40), (13, 8192, 6, 2), (20000, 64, 8, 3), (12000, 2048, 16, 5)])
@pytest.mark.parametrize("quant", [False, True])
def test_token_major_gather_ragged(T, D, E, k, quant):
    """Token-major gathers on ragged shapes: top_k that does not divide the 32-row
    metadata window, top_k = 32 and above it (row-major fallback), rows of 8 and 16
    staging warps and rows too wide to stage, many tokens per warp (the slot ring
    wraps), f32 and bf16 scores, and values whose products are subnormal or
    saturate the e4m3 range: bit-exact against the oracle."""
    mb = _mb()
    g = torch.Generator().manual_seed(T * 7 + D + k)
    x = torch.randn(T, D, generator=g)
    x[0, : min(D, 8)] = torch.tensor([1e-39, -3e-40, 2e-38, 0.0, -0.0, 5e-41, 1e-38, -1e-39])[: min(D, 8)]
    x[min(1, T - 1)] *= 1e30
    x = x.to(torch.bfloat16)
    s = torch.rand(T, E, generator=g)
    s[min(2, T - 1)] *= 1e-30
    s = s.to(torch.bfloat16)
    r = oracle.route(bits(s), k)
    a = T * k
    ti, ei, inv = _idx(r["token_indices"]), _idx(r["expert_indices"]), _idx(r["inv"].ravel())
    sd = s.cuda() if T % 2 == 0 else s.float().cuda()
    s_ref = bits(s) if T % 2 == 0 else s.float().numpy()
    valid = torch.tensor([a], dtype=torch.int32, device="cuda")
    if quant:
        q = sentinel_like((a, D), torch.float8_e4m3fn)
        sc = sentinel_like((a,), torch.float32)
        mb.moe_gather_scale_quant(x.cuda(), ti, ei, sd, None, valid, inv_rows=inv, top_k=k, out=q, out_scale=sc)
        q_ref, sc_ref = oracle.gather_scale_quant(bits(x), r["token_indices"], r["expert_indices"], s_ref)
        np.testing.assert_array_equal(bits(q), q_ref)
        np.testing.assert_array_equal(sc.cpu().numpy(), sc_ref)
    else:
        o = sentinel_like((a, D), torch.bfloat16)
        mb.moe_gather_scale(x.cuda(), ti, ei, sd, valid, inv_rows=inv, top_k=k, out=o)
        np.testing.assert_array_equal(bits(o), oracle.gather_scale(bits(x), r["token_indices"], r["expert_indices"],
                                                                   s_ref))
    assert mb.device_error() == 0


def test_binding_rejects_strided_matrices():
    mb = _mb()
    x = torch.randn(64, 32, device="cuda").to(torch.bfloat16).t()        # a transposed view: not row-major
    ti = torch.zeros(4, dtype=torch.int32, device="cuda")
    s = torch.rand(32, 2, device="cuda")
    with pytest.raises(ValueError):
        mb.moe_gather_scale(x, ti, ti, s)
    y = torch.randn(8, 64, device="cuda").to(torch.bfloat16)
    with pytest.raises(ValueError):
        mb.moe_silu_mul(y, 16, out=torch.empty(16, 8, dtype=torch.bfloat16, device="cuda").t())
    # rows of y may be strided (the ABI takes the row stride): a column slice is accepted
    z = mb.moe_silu_mul(torch.randn(8, 96, device="cuda").to(torch.bfloat16)[:, :64], 32)
    assert z.shape == (8, 32) and mb.device_error() == 0


@pytest.mark.parametrize("staged", [False, True])
@pytest.mark.parametrize("quant", [False, True])
def test_gather_sees_inputs_of_a_slow_preceding_kernel(staged, quant):
    """The gathers are launched with programmatic stream serialization: they may start
    before the previous kernel ends when that kernel signals (the routing kernels do;
    every forward's parity test covers that case), and must otherwise wait for it as any
    launch does.  Here the inputs come from torch kernels that never signal, queued
    behind a reduction over 1 GiB that feeds every input (token indices, expert indices,
    scores, valid count), so the GPU is busy when the gather is enqueued.  In three
    rounds with changing inputs, each result equals the oracle's gather of the final
    inputs bit for bit."""
    mb = _mb()
    T, D, E, k = 512, 2048, 16, (4 if staged else 1)
    a = T * k
    g = torch.Generator(device="cuda").manual_seed(3)
    x = torch.randn(T, D, device="cuda", generator=g).to(torch.bfloat16)
    big = torch.ones(1 << 28, device="cuda")                     # 1 GiB of fp32 ones
    for rnd in range(3):
        zero = (big.sum() * 0.0).to(torch.int32)                 # 0, produced by a slow kernel
        perm = torch.randperm(T, device="cuda", generator=g).to(torch.int32)
        tok = (perm.repeat_interleave(k) + zero).contiguous()    # routed row -> token
        exp = ((torch.arange(a, device="cuda", dtype=torch.int32) * 7 + rnd) % E + zero).contiguous()
        scores = (torch.rand(T, E, device="cuda", generator=g) + zero.float()).to(torch.bfloat16)
        valid = (torch.tensor([a - 3 * rnd], device="cuda", dtype=torch.int32) + zero).contiguous()
        inv = None
        if staged:   # token-major: token t's k rows are rows t*k .. t*k+k-1 of the buffer, in order
            order = torch.argsort(perm.long())
            inv = ((order.view(T, 1) * k + torch.arange(k, device="cuda").view(1, k)).reshape(-1)
                   .to(torch.int32) + zero).contiguous()
            tok = perm.repeat_interleave(k).to(torch.int32)
            tok = (tok + zero).contiguous()
            valid = (torch.tensor([a], device="cuda", dtype=torch.int32) + zero).contiguous()
        kw = dict(inv_rows=inv, top_k=k) if staged else {}
        if quant:
            out, sc = mb.moe_gather_scale_quant(x, tok, exp, scores, None, valid, **kw)
        else:
            out = mb.moe_gather_scale(x, tok, exp, scores, valid, **kw)
        torch.cuda.synchronize()
        assert mb.device_error() == 0
        n = int(valid.item())
        ti, ei, sb = tok.cpu().numpy(), exp.cpu().numpy(), bits(scores.cpu())
        if quant:   # bit-exact against the oracle: codes and scales
            q_ref, s_ref = oracle.gather_scale_quant(bits(x.cpu()), ti, ei, sb, None, n)
            assert np.array_equal(out[:n].view(torch.uint8).cpu().numpy(), q_ref[:n]), f"round {rnd}"
            assert np.array_equal(sc[:n].cpu().numpy(), s_ref[:n]), f"round {rnd}"
        else:
            ref = oracle.gather_scale(bits(x.cpu()), ti, ei, sb, n)
            assert np.array_equal(bits(out[:n].cpu()), ref[:n]), f"round {rnd}"
