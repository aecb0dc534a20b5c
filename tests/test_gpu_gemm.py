"""The tcgen05 grouped GEMMs (bf16 and FP8 rowwise) against the oracle.

Tolerance: the kernel accumulates in fp32 on the tensor cores, the oracle in
fp64; both round once to bf16.  So an output may differ from the oracle by one
bf16 step of the result plus the fp32 accumulation error, bounded by
2^-20 * sum_k |x_k w_k| (K terms, each addition off by at most 2^-24 relative,
with ample slack).  The fused SiLU*mul epilogue must equal the unfused GEMM
followed by moe_silu_mul bit for bit (same accumulators, same arithmetic).
"""
import numpy as np
import pytest
import torch

import oracle
from moe_token_routing_index_gb300 import workloads
from tests.helpers import bits, dev_bf16, dev_e4m3, f64, is_sentinel, sentinel_like

pytestmark = pytest.mark.gpu


def _mb():
    from moe_token_routing_index_gb300 import binding

    return binding


def _bf16_ulp(v: np.ndarray) -> np.ndarray:
    a = np.abs(v).astype(np.float64)
    e = np.floor(np.log2(np.where(a > 0, a, 1e-38)))
    return np.exp2(e - 7)


def _check_close(got_bits, ref_bits, abs_bound, min_exact=0.9):
    got, ref = f64(got_bits), f64(ref_bits)
    err = np.abs(got - ref)
    tol = _bf16_ulp(ref) + abs_bound
    bad = err > tol
    assert not bad.any(), f"{bad.sum()} of {bad.size} outside tolerance; worst {err[bad].max():.3e}"
    assert (err == 0).mean() >= min_exact, f"only {(err == 0).mean():.4f} bit-exact"


def _abs_bound_bf16(x_bits, w_bits, counts, rows=None):
    """2^-20 * sum_k |x_rk w_enk| for every output (r, n), per expert segment."""
    xa, wa = np.abs(f64(x_bits)), np.abs(f64(w_bits))
    out = np.zeros((x_bits.shape[0], w_bits.shape[1]))
    off = 0
    for e, c in enumerate(counts):
        out[off:off + c] = xa[off:off + c] @ wa[e].T
        off += c
    return 2.0 ** -20 * out


def _problem(E, counts, N, K, a_max=None, seed=0, std=0.05):
    g = torch.Generator().manual_seed(seed)
    a = int(sum(counts))
    a_max = a if a_max is None else a_max
    x = torch.randn(a_max, K, generator=g).to(torch.bfloat16)
    w = (torch.randn(E, N, K, generator=g) * std).to(torch.bfloat16)
    return x, w, np.array(counts, np.int32), a


SHAPES = [
    # E, counts, N, K, a_max
    (1, [128], 256, 64, None),          # one tile, one K block
    (3, [5, 0, 130], 256, 64, None),    # ragged experts, an empty expert
    (2, [77, 200], 512, 320, None),     # several N tiles and K blocks
    (4, [1, 0, 0, 129], 48, 80, 300),   # partial N tile, K tail, rows past the counts
    (5, [300, 17, 0, 64, 250], 1040, 272, 700),
    # the largest expert count: 1024 experts, most of them empty or with a few rows
    (1024, [int(c) for c in np.random.default_rng(1024).choice([0, 0, 0, 1, 3, 130], 1024)], 64, 64, None),
]


@pytest.mark.parametrize("E,counts,N,K,a_max", SHAPES)
def test_grouped_gemm_bf16(E, counts, N, K, a_max):
    mb = _mb()
    x, w, cnt, a = _problem(E, counts, N, K, a_max, seed=N + K)
    y = sentinel_like((x.shape[0], N), torch.bfloat16)
    mb.moe_grouped_gemm(x.cuda(), w.cuda(), torch.from_numpy(cnt).cuda(), out=y)
    assert mb.device_error() == 0
    ref = oracle.grouped_gemm_bf16(bits(x[:a]), bits(w), cnt)
    _check_close(bits(y[:a]), ref, _abs_bound_bf16(bits(x[:a]), bits(w), cnt))
    assert is_sentinel(y[a:])


@pytest.mark.parametrize("E,counts,N,K,a_max", SHAPES)
def test_fused_silu_mul_equals_unfused(E, counts, N, K, a_max):
    if N % 32:
        pytest.skip("SiLU*mul needs N = 2H with H a multiple of 16")
    mb = _mb()
    x, w, cnt, a = _problem(E, counts, N, K, a_max, seed=3 * N + K, std=0.2)
    xd, wd, cd = x.cuda(), w.cuda(), torch.from_numpy(cnt).cuda()
    H = N // 2
    y = mb.moe_grouped_gemm(xd, wd, cd)
    z_unfused = mb.moe_silu_mul(y[:a].contiguous(), H)
    z = sentinel_like((x.shape[0], H), torch.bfloat16)
    mb.moe_grouped_gemm(xd, wd, cd, epilogue=mb.MOE_EPILOGUE_SILU_MUL, out=z)
    assert mb.device_error() == 0
    assert torch.equal(z[:a], z_unfused)
    assert is_sentinel(z[a:])


def test_all_experts_empty_is_a_no_op():
    mb = _mb()
    x, w, cnt, a = _problem(3, [0, 0, 0], 64, 64, 50)
    y = sentinel_like((50, 64), torch.bfloat16)
    mb.moe_grouped_gemm(x.cuda(), w.cuda(), torch.from_numpy(cnt).cuda(), out=y)
    assert mb.device_error() == 0 and is_sentinel(y)


@pytest.mark.parametrize("E,counts,N,K,a_max", SHAPES)
def test_grouped_gemm_fp8(E, counts, N, K, a_max):
    mb = _mb()
    x, w, cnt, a = _problem(E, counts, N, K, a_max, seed=5 * N + K)
    xq, xs = oracle.gather_scale_quant(bits(x), np.arange(x.shape[0], dtype=np.int32),
                                       np.zeros(x.shape[0], np.int32), bits(torch.ones(x.shape[0], 1,
                                                                                       dtype=torch.bfloat16)))
    wq, ws = oracle.quantize_rows(w.float().numpy())
    y = sentinel_like((x.shape[0], N), torch.bfloat16)
    mb.moe_grouped_gemm_fp8_rowwise(dev_e4m3(xq), dev_e4m3(wq), torch.from_numpy(cnt).cuda(),
                                    torch.from_numpy(xs).cuda(), torch.from_numpy(ws).cuda(), out=y)
    assert mb.device_error() == 0
    ref = oracle.grouped_gemm_fp8(xq[:a], wq, cnt, xs[:a], ws)
    dx = oracle.e4m3_decode(xq[:a]).astype(np.float64)
    dw = oracle.e4m3_decode(wq).astype(np.float64)
    bound = np.zeros((a, N))
    off = 0
    for e, c in enumerate(cnt):
        bound[off:off + c] = (np.abs(dx[off:off + c]) @ np.abs(dw[e]).T) * xs[off:off + c, None] * ws[e][None, :]
        off += c
    _check_close(bits(y[:a]), ref, 2.0 ** -20 * bound)
    assert is_sentinel(y[a:])
    if N % 32 == 0:
        z = mb.moe_grouped_gemm_fp8_rowwise(dev_e4m3(xq), dev_e4m3(wq), torch.from_numpy(cnt).cuda(),
                                            torch.from_numpy(xs).cuda(), torch.from_numpy(ws).cuda(),
                                            epilogue=mb.MOE_EPILOGUE_SILU_MUL)
        assert torch.equal(z[:a], mb.moe_silu_mul(y[:a].contiguous(), N // 2))


def _sample_rows(cnt, rng, per_expert=3):
    """First, last and a few random rows of every non-empty expert (sorted)."""
    rows, off = [], 0
    for c in cnt:
        if c:
            rows += [off, off + c - 1] + list(rng.integers(off, off + c, per_expert))
        off += c
    return np.unique(np.array(rows, np.int64))


@pytest.mark.parametrize("name", ["decode", "decode_zero", "fine_grained"])
def test_grouped_gemm_bf16_workloads_sampled(name):
    """Full-size w13 and w2 GEMMs of the bf16 workloads; oracle on sampled rows."""
    mb = _mb()
    cfg = workloads.CONFIGS[name]
    s = workloads.make_scores(cfg)
    r = oracle.route(bits(s), cfg.top_k, cfg.valid_tokens)
    cnt = r["counts"][:cfg.E]
    a = int(cnt.sum())
    g = torch.Generator().manual_seed(11)
    x = torch.randn(a, cfg.D, generator=g).to(torch.bfloat16)
    w13, w2 = workloads.make_weights(cfg, device="cuda")
    cd = torch.from_numpy(cnt).cuda()
    y = mb.moe_grouped_gemm(x.cuda(), w13, cd)
    z = mb.moe_grouped_gemm(x.cuda(), w13, cd, epilogue=mb.MOE_EPILOGUE_SILU_MUL)
    o = mb.moe_grouped_gemm(z, w2, cd)
    assert mb.device_error() == 0
    rows = _sample_rows(cnt, np.random.default_rng(0))
    exp_of_row = np.repeat(np.arange(cfg.E), cnt)[rows]
    used = sorted(set(exp_of_row.tolist()))
    sub_cnt = np.array([(exp_of_row == e).sum() for e in used], np.int32)
    w13_u, w2_u = bits(w13[used]), bits(w2[used])
    y_ref = oracle.grouped_gemm_bf16(bits(x)[rows], w13_u, sub_cnt)
    _check_close(bits(y[rows]), y_ref, _abs_bound_bf16(bits(x)[rows], w13_u, sub_cnt))
    assert torch.equal(z, mb.moe_silu_mul(y, cfg.H))
    o_ref = oracle.grouped_gemm_bf16(bits(z)[rows], w2_u, sub_cnt)
    _check_close(bits(o[rows]), o_ref, _abs_bound_bf16(bits(z)[rows], w2_u, sub_cnt))


def _sample_rows_with_tail(cnt, rng, per_expert=3, tile=128):
    """First, last, the first row of the last (partial) tile, and a few random rows of
    every non-empty expert (sorted)."""
    rows, off = [], 0
    for c in cnt:
        if c:
            rows += [off, off + c - 1, off + (c - 1) // tile * tile] + list(rng.integers(off, off + c, per_expert))
        off += c
    return np.unique(np.array(rows, np.int64))


def _fp8_bound(xq_rows, xs_rows, wq, ws, sub_cnt):
    """2^-20 * sum_k |x_k w_k| * xs * ws for the sampled rows (per expert segment)."""
    dx = oracle.e4m3_decode(xq_rows).astype(np.float64)
    out = np.zeros((xq_rows.shape[0], wq.shape[1]))
    off = 0
    for i, c in enumerate(sub_cnt):
        dw = oracle.e4m3_decode(wq[i]).astype(np.float64)
        out[off:off + c] = (np.abs(dx[off:off + c]) @ np.abs(dw).T) * xs_rows[off:off + c, None] * ws[i][None, :]
        off += c
    return 2.0 ** -20 * out


@pytest.mark.parametrize("variant", ["single", "pairs", "packed"])
@pytest.mark.parametrize("name", ["prefill_fp8", "padded_fp8"])
def test_grouped_gemm_fp8_workloads_sampled(name, variant):
    """Full-size FP8-rowwise w13 and w2 GEMMs of the FP8 workloads, with the workload's
    weights quantised per row on the device: every non-empty expert's first, last,
    last-tile and random rows against the oracle (fp32 accumulation bound), for 128-row
    tiles, CTA-pair tiles and packed weights; the SILU_MUL_QUANT epilogue on the full
    problem equal to silu_mul of the plain output and to the oracle's row rule on its
    bf16 z (codes and scales bit for bit)."""
    mb = _mb()
    cfg = workloads.CONFIGS[name]
    r = oracle.route(bits(workloads.make_scores(cfg)), cfg.top_k, cfg.valid_tokens)
    cnt = r["counts"][:cfg.E]
    a = int(cnt.sum())
    cd = torch.from_numpy(cnt.copy()).cuda()
    w13f, w2f = workloads.make_weights(cfg, device="cuda")
    w13q, w13s = mb.moe_quantize_rows(w13f)
    w2q, w2s = mb.moe_quantize_rows(w2f)
    del w13f, w2f
    g = torch.Generator().manual_seed(17)
    # codes across the range (clamped: PyTorch's e4m3fn cast turns values past 448 into NaN)
    xq = (torch.randn(a, cfg.D, generator=g) * 60).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).cuda()
    xs = (torch.rand(a, generator=g) * 0.02 + 0.001).cuda()
    flags = mb.MOE_GEMM_CTA_PAIRS if variant == "pairs" else 0
    a13 = mb.moe_pack_weights(w13q) if variant == "packed" else w13q
    a2 = mb.moe_pack_weights(w2q) if variant == "packed" else w2q
    ub = torch.tensor([cfg.scale_ub or 1200.0], dtype=torch.float32, device="cuda")
    y = mb.moe_grouped_gemm_fp8_rowwise(xq, a13, cd, xs, w13s, epilogue=flags)
    zb = torch.empty(a, cfg.H, dtype=torch.bfloat16, device="cuda")
    zq, zs = mb.moe_grouped_gemm_fp8_rowwise(xq, a13, cd, xs, w13s, epilogue=mb.MOE_EPILOGUE_SILU_MUL_QUANT | flags,
                                             out=zb, scale_ub=ub)
    o = mb.moe_grouped_gemm_fp8_rowwise(zq, a2, cd, zs, w2s, epilogue=flags)
    torch.cuda.synchronize()
    assert mb.device_error() == 0
    assert torch.equal(zb, mb.moe_silu_mul(y, cfg.H))
    zq_ref, zs_ref = oracle.quantize_rows(oracle.bf16_to_f32(bits(zb)), float(ub.item()))
    np.testing.assert_array_equal(bits(zq), zq_ref)
    np.testing.assert_array_equal(zs.cpu().numpy(), zs_ref)
    rows = _sample_rows_with_tail(cnt, np.random.default_rng(0))
    exp_of_row = np.repeat(np.arange(cfg.E), cnt)[rows]
    used = sorted(set(exp_of_row.tolist()))
    sub_cnt = np.array([(exp_of_row == e).sum() for e in used], np.int32)
    xq_h, xs_h = bits(xq)[rows], xs.cpu().numpy()[rows]
    w13_h, w13s_h = bits(w13q[used]), w13s[used].cpu().numpy()
    y_ref = oracle.grouped_gemm_fp8(xq_h, w13_h, sub_cnt, xs_h, w13s_h)
    _check_close(bits(y[rows]), y_ref, _fp8_bound(xq_h, xs_h, w13_h, w13s_h, sub_cnt))
    zq_h, zs_h = bits(zq)[rows], zs.cpu().numpy()[rows]
    w2_h, w2s_h = bits(w2q[used]), w2s[used].cpu().numpy()
    o_ref = oracle.grouped_gemm_fp8(zq_h, w2_h, sub_cnt, zs_h, w2s_h)
    _check_close(bits(o[rows]), o_ref, _fp8_bound(zq_h, zs_h, w2_h, w2s_h, sub_cnt))


@pytest.mark.parametrize("fp8", [False, True])
def test_banded_tile_order_long_k(fp8):
    """A reduction long enough that the tile order splits each expert's row tiles into
    bands (bf16: 2 row tiles per band of 128-row tiles, 1 per band of pair tiles; FP8: 4
    and 2), with every other band walking N backwards and a partial last band: pairs ==
    single-CTA tiles bit for bit, and every expert's first, last, last-tile and random
    rows within the oracle bound."""
    mb = _mb()
    E, counts, N, K = 3, [700, 0, 300], 512, 61440
    g = torch.Generator().manual_seed(123)
    a = sum(counts)
    x = torch.randn(a, K, generator=g).to(torch.bfloat16)
    w = (torch.randn(E, N, K, generator=g) * 0.01).to(torch.bfloat16)
    cnt = np.array(counts, np.int32)
    cd = torch.from_numpy(cnt).cuda()
    rows = _sample_rows_with_tail(cnt, np.random.default_rng(3))
    exp_of_row = np.repeat(np.arange(E), cnt)[rows]
    used = sorted(set(exp_of_row.tolist()))
    sub_cnt = np.array([(exp_of_row == e).sum() for e in used], np.int32)
    if fp8:
        xq, xs = mb.moe_quantize_rows(x.float().cuda())
        wq, ws = mb.moe_quantize_rows(w.float().cuda())
        y1 = mb.moe_grouped_gemm_fp8_rowwise(xq, wq, cd, xs, ws)
        y2 = mb.moe_grouped_gemm_fp8_rowwise(xq, wq, cd, xs, ws, epilogue=mb.MOE_GEMM_CTA_PAIRS)
        xq_h, xs_h = bits(xq)[rows], xs.cpu().numpy()[rows]
        wq_h, ws_h = bits(wq[used]), ws[used].cpu().numpy()
        ref = oracle.grouped_gemm_fp8(xq_h, wq_h, sub_cnt, xs_h, ws_h)
        bound = _fp8_bound(xq_h, xs_h, wq_h, ws_h, sub_cnt)
    else:
        y1 = mb.moe_grouped_gemm(x.cuda(), w.cuda(), cd)
        y2 = mb.moe_grouped_gemm(x.cuda(), w.cuda(), cd, epilogue=mb.MOE_GEMM_CTA_PAIRS)
        ref = oracle.grouped_gemm_bf16(bits(x)[rows], bits(w[used]), sub_cnt)
        bound = _abs_bound_bf16(bits(x)[rows], bits(w[used]), sub_cnt)
    torch.cuda.synchronize()
    assert mb.device_error() == 0
    assert torch.equal(y1, y2)
    _check_close(bits(y1[rows]), ref, bound)


SILU_QUANT_SHAPES = [s for s in SHAPES if s[2] % 32 == 0] + [
    (2, [77, 300], 2 * 8192, 64, 400),       # z rows of 8192 elements (8 warps per row, 4 vectors each)
    (1, [33], 2 * 16384, 32, None),          # the largest H the row pass takes
]


@pytest.mark.parametrize("pairs", [False, True])
@pytest.mark.parametrize("ub", [None, 0.75])
@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("E,counts,N,K,a_max", SILU_QUANT_SHAPES)
def test_silu_mul_quant_epilogue(E, counts, N, K, a_max, fp8, ub, pairs):
    """MOE_EPILOGUE_SILU_MUL_QUANT: y holds the SILU_MUL epilogue's bf16 z bit for bit, and
    (z_out, z_scale) equal the quantising gather of that z with identity indices and unit
    scores, and the oracle's row rule on it, bit for bit; rows past the counts untouched.
    ub = 0.75 makes the bound bind on most rows."""
    mb = _mb()
    x, w, cnt, a = _problem(E, counts, N, K, a_max, seed=11 * N + K, std=0.2)
    cd = torch.from_numpy(cnt).cuda()
    H = N // 2
    if fp8:
        xq, xs = mb.moe_quantize_rows(x.float().cuda())
        wq, ws = mb.moe_quantize_rows(w.float().cuda())
        gemm = lambda **kw: mb.moe_grouped_gemm_fp8_rowwise(xq, wq, cd, xs, ws, **kw)
    else:
        gemm = lambda **kw: mb.moe_grouped_gemm(x.cuda(), w.cuda(), cd, **kw)
    flags = mb.MOE_GEMM_CTA_PAIRS if pairs else 0
    ubt = None if ub is None else torch.tensor([ub], dtype=torch.float32, device="cuda")
    z_ref = gemm(epilogue=mb.MOE_EPILOGUE_SILU_MUL | flags)
    rows = x.shape[0]
    zb = sentinel_like((rows, H), torch.bfloat16)
    zq = sentinel_like((rows, H), torch.float8_e4m3fn)
    zs = sentinel_like((rows,), torch.float32)
    got = gemm(epilogue=mb.MOE_EPILOGUE_SILU_MUL_QUANT | flags, out=zb, scale_ub=ubt, z_out=zq, z_scale=zs)
    assert got[0] is zq and got[1] is zs
    torch.cuda.synchronize()
    assert mb.device_error() == 0
    assert torch.equal(zb[:a], z_ref[:a])
    ident = torch.arange(a, dtype=torch.int32, device="cuda")
    q2, s2 = mb.moe_gather_scale_quant(zb[:a].contiguous(), ident, torch.zeros_like(ident), None, ubt)
    assert torch.equal(zq[:a].view(torch.uint8), q2.view(torch.uint8))
    assert torch.equal(zs[:a], s2)
    q_ref, s_ref = oracle.quantize_rows(oracle.bf16_to_f32(bits(zb[:a])), ub)
    np.testing.assert_array_equal(bits(zq[:a]), q_ref)
    np.testing.assert_array_equal(zs[:a].cpu().numpy(), s_ref)
    assert is_sentinel(zb[a:]) and is_sentinel(zq[a:]) and is_sentinel(zs[a:])


@pytest.mark.parametrize("E,counts,D,H,a_max", [(1, [128], 64, 128, None), (3, [5, 0, 130], 256, 512, None),
                                                (5, [300, 17, 0, 64, 250], 272, 528, 700),
                                                (16, [8] * 12 + [0] * 4, 512, 1024, 130)])
def test_expert_mlp_one_launch_equals_two(E, counts, D, H, a_max):
    """moe_expert_mlp (both GEMMs in one persistent launch) equals the two calls bit for bit."""
    mb = _mb()
    g = torch.Generator().manual_seed(D + H)
    a = int(sum(counts))
    a_max = a if a_max is None else a_max
    x = torch.randn(a_max, D, generator=g).to(torch.bfloat16).cuda()
    w13 = (torch.randn(E, 2 * H, D, generator=g) * 0.1).to(torch.bfloat16).cuda()
    w2 = (torch.randn(E, D, H, generator=g) * 0.1).to(torch.bfloat16).cuda()
    cd = torch.tensor(counts, dtype=torch.int32, device="cuda")
    z_ref = mb.moe_grouped_gemm(x, w13, cd, epilogue=mb.MOE_EPILOGUE_SILU_MUL)
    y_ref = mb.moe_grouped_gemm(z_ref, w2, cd)
    y = sentinel_like((a_max, D), torch.bfloat16)
    z = torch.empty(a_max, H, dtype=torch.bfloat16, device="cuda")
    for _ in range(2):   # the workspace is reused as it is left
        mb.moe_expert_mlp(x, w13, w2, cd, z=z, out=y)
    assert mb.device_error() == 0
    assert torch.equal(y[:a], y_ref[:a]) and torch.equal(z[:a], z_ref[:a])
    assert is_sentinel(y[a:])


def test_expert_mlp_leaves_its_workspace_zero():
    """The per-expert counters of moe_expert_mlp start at zero and every call leaves them
    zero (the last block to finish resets them): three route -> gather -> MLP passes on one
    workspace agree bit for bit, and the workspace reads zero after each."""
    mb = _mb()
    g = torch.Generator().manual_seed(11)
    E, D, H, T = 16, 512, 1024, 128
    x = torch.randn(T, D, generator=g).to(torch.bfloat16).cuda()
    s = torch.rand(T, E, generator=g).to(torch.bfloat16).cuda()
    w13 = (torch.randn(E, 2 * H, D, generator=g) * 0.1).to(torch.bfloat16).cuda()
    w2 = (torch.randn(E, D, H, generator=g) * 0.1).to(torch.bfloat16).cuda()
    ws = torch.zeros(mb.moe_expert_mlp_workspace_size(E), dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(3):
        r = mb.moe_route(s, 1)
        xr = mb.moe_gather_scale(x, r["token_indices"], r["expert_indices"], s)
        outs.append(mb.moe_expert_mlp(xr, w13, w2, r["counts"], workspace=ws).clone())
        torch.cuda.synchronize()
        assert int(ws.count_nonzero()) == 0
    assert mb.device_error() == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    cnt = r["counts"][:E]
    z_ref = mb.moe_grouped_gemm(xr, w13, cnt, epilogue=mb.MOE_EPILOGUE_SILU_MUL)
    assert torch.equal(outs[0], mb.moe_grouped_gemm(z_ref, w2, cnt))


@pytest.mark.parametrize("name", ["decode", "fine_grained"])
def test_expert_mlp_workloads_equal_two_launches(name):
    mb = _mb()
    cfg = workloads.CONFIGS[name]
    r = oracle.route(bits(workloads.make_scores(cfg)), cfg.top_k, cfg.valid_tokens)
    cnt = torch.from_numpy(r["counts"][:cfg.E].copy()).cuda()
    a = cfg.routed_rows
    g = torch.Generator().manual_seed(5)
    x = torch.randn(a, cfg.D, generator=g).to(torch.bfloat16).cuda()
    w13, w2 = workloads.make_weights(cfg, device="cuda")
    z_ref = mb.moe_grouped_gemm(x, w13, cnt, epilogue=mb.MOE_EPILOGUE_SILU_MUL)
    y_ref = mb.moe_grouped_gemm(z_ref, w2, cnt)
    y = mb.moe_expert_mlp(x, w13, w2, cnt)
    assert mb.device_error() == 0
    assert torch.equal(y, y_ref)


@pytest.mark.parametrize("accumulate", [True, False])
@pytest.mark.parametrize("fp8", [False, True])
def test_fused_combine_equals_gemm_then_scatter(accumulate, fp8):
    """top_k = 1: the w2 GEMM writing out[token] directly equals GEMM + moe_scatter_add bit for bit."""
    mb = _mb()
    E, counts, N, K, T = 5, [70, 0, 33, 129, 1], 272, 192, 300
    x, w, cnt, a = _problem(E, counts, N, K, None, seed=77)
    perm = torch.randperm(T, generator=torch.Generator().manual_seed(1))[:a].to(torch.int32).cuda()  # token of each row
    cd = torch.from_numpy(cnt).cuda()
    init = torch.randn(T, N, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16).cuda()
    if fp8:
        xq, xs = mb.moe_quantize_rows(x.float().cuda())
        wq, ws = mb.moe_quantize_rows(w.float().cuda())
        gemm = lambda **kw: mb.moe_grouped_gemm_fp8_rowwise(xq, wq, cd, xs, ws, **kw)
    else:
        gemm = lambda **kw: mb.moe_grouped_gemm(x.cuda(), w.cuda(), cd, **kw)
    o = gemm()
    ref = init.clone()
    mb.moe_scatter_add(ref, o, perm, None, 1, accumulate=accumulate)
    got = init.clone()
    gemm(out=got, scatter_indices=perm, accumulate=accumulate)
    assert mb.device_error() == 0
    assert torch.equal(got, ref)


def test_expert_mlp_fused_combine_equals_unfused():
    mb = _mb()
    E, counts, D, H, T = 4, [40, 0, 90, 17], 256, 384, 200
    g = torch.Generator().manual_seed(9)
    a = sum(counts)
    x = torch.randn(a, D, generator=g).to(torch.bfloat16).cuda()
    w13 = (torch.randn(E, 2 * H, D, generator=g) * 0.1).to(torch.bfloat16).cuda()
    w2 = (torch.randn(E, D, H, generator=g) * 0.1).to(torch.bfloat16).cuda()
    cd = torch.tensor(counts, dtype=torch.int32, device="cuda")
    perm = torch.randperm(T, generator=g)[:a].to(torch.int32).cuda()
    o = mb.moe_expert_mlp(x, w13, w2, cd)
    ref = sentinel_like((T, D), torch.bfloat16)
    mb.moe_scatter_add(ref, o, perm, None, 1, accumulate=False)
    got = sentinel_like((T, D), torch.bfloat16)
    mb.moe_expert_mlp(x, w13, w2, cd, out=got, scatter_indices=perm, accumulate=False)
    assert mb.device_error() == 0
    assert torch.equal(got, ref)


PAIR_SHAPES = [
    # E, counts, N, K, a_max: row tiles of 256 on CTA pairs; odd 128-row tile counts, empty experts
    (1, [256], 256, 64, None),
    (2, [512, 256], 512, 320, None),
    (3, [5, 0, 130], 256, 64, None),
    (4, [1, 0, 0, 383], 48, 80, 500),
    (5, [300, 17, 0, 640, 250], 1040, 272, 1300),
    (1024, [int(c) for c in np.random.default_rng(1025).choice([0, 0, 0, 2, 257], 1024)], 64, 64, None),
]


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("E,counts,N,K,a_max", PAIR_SHAPES)
def test_grouped_gemm_cta_pairs(E, counts, N, K, a_max, fp8):
    """256-row tiles on CTA pairs (cta_group::2): within the oracle bound, bit-identical to the
    single-CTA tiles (the same per-element accumulation), and the SiLU*mul epilogue equal to
    silu_mul of the plain output."""
    mb = _mb()
    x, w, cnt, a = _problem(E, counts, N, K, a_max, seed=7 * N + K)
    cd = torch.from_numpy(cnt).cuda()
    y = sentinel_like((x.shape[0], N), torch.bfloat16)
    if fp8:
        xq, xs = mb.moe_quantize_rows(x.float().cuda())
        wq, ws = mb.moe_quantize_rows(w.float().cuda())
        gemm = lambda **kw: mb.moe_grouped_gemm_fp8_rowwise(xq, wq, cd, xs, ws, **kw)
    else:
        gemm = lambda **kw: mb.moe_grouped_gemm(x.cuda(), w.cuda(), cd, **kw)
    gemm(epilogue=mb.MOE_GEMM_CTA_PAIRS, out=y)
    assert mb.device_error() == 0
    assert is_sentinel(y[a:])
    y1 = gemm()   # single-CTA tiles
    if fp8:
        ref = oracle.grouped_gemm_fp8(bits(xq.cpu())[:a], bits(wq.cpu()), cnt, xs.cpu().numpy()[:a],
                                      ws.cpu().numpy())
        dx = oracle.e4m3_decode(bits(xq.cpu())[:a]).astype(np.float64)
        dw = oracle.e4m3_decode(bits(wq.cpu())).astype(np.float64)
        bound = np.zeros((a, N))
        off = 0
        for e, c in enumerate(cnt):
            bound[off:off + c] = ((np.abs(dx[off:off + c]) @ np.abs(dw[e]).T) * xs.cpu().numpy()[off:off + c, None]
                                  * ws.cpu().numpy()[e][None, :])
            off += c
        _check_close(bits(y[:a]), ref, 2.0 ** -20 * bound)
    else:
        ref = oracle.grouped_gemm_bf16(bits(x[:a]), bits(w), cnt)
        _check_close(bits(y[:a]), ref, _abs_bound_bf16(bits(x[:a]), bits(w), cnt))
    assert torch.equal(y[:a], y1[:a])
    if N % 32 == 0:
        z = sentinel_like((x.shape[0], N // 2), torch.bfloat16)
        gemm(epilogue=mb.MOE_EPILOGUE_SILU_MUL | mb.MOE_GEMM_CTA_PAIRS, out=z)
        assert mb.device_error() == 0
        assert torch.equal(z[:a], mb.moe_silu_mul(y[:a].contiguous(), N // 2))
        assert is_sentinel(z[a:])


@pytest.mark.parametrize("M,K,N,valid", [(128, 5120, 16384, 128), (128, 8192, 5120, 128), (200, 1024, 512, 170),
                                         (1, 256, 64, 1), (300, 4096, 2048, 300), (64, 16, 48, 64)])
def test_dense_splitk_gemm(M, K, N, valid):
    """moe_dense_gemm (K split over a cluster, partials added in rank order): the plain
    output within the oracle bound on sampled columns; the SiLU*mul epilogue equal to
    moe_silu_mul of the plain output bit for bit (same tiles, same split, same sums)."""
    mb = _mb()
    g = torch.Generator().manual_seed(M + K + N)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    w = (torch.randn(N, K, generator=g) * 0.05).to(torch.bfloat16)
    vr = torch.tensor([valid], dtype=torch.int32, device="cuda")
    y = sentinel_like((M, N), torch.bfloat16)
    mb.moe_dense_gemm(x.cuda(), w.cuda(), vr, out=y)
    assert mb.device_error() == 0
    cols = np.unique(np.random.default_rng(N).integers(0, N, min(N, 384)))
    ref = oracle.grouped_gemm_bf16(bits(x[:valid]), bits(w)[cols][None], np.array([valid], np.int32))
    _check_close(bits(y[:valid])[:, cols], ref, _abs_bound_bf16(bits(x[:valid]), bits(w)[cols][None], [valid]))
    assert is_sentinel(y[valid:])
    if N % 32 == 0:
        H = N // 2
        z = sentinel_like((M, H), torch.bfloat16)
        mb.moe_dense_gemm(x.cuda(), w.cuda(), vr, epilogue=mb.MOE_EPILOGUE_SILU_MUL, out=z)
        z_ref = mb.moe_silu_mul(y[:valid].contiguous(), H)
        assert mb.device_error() == 0
        assert torch.equal(z[:valid], z_ref)
        assert is_sentinel(z[valid:])


def _ref_pack(w: torch.Tensor) -> torch.Tensor:
    """The tile-packed layout written out with reshapes: rows cut into 128-row blocks and
    bytes into 128-byte blocks (zero-padded), boxes in (row block, byte block) order."""
    E, N, K = w.shape
    rb = w.contiguous().view(torch.uint8).reshape(E * N, -1)
    R, B = rb.shape
    nr, nc = (R + 127) // 128, (B + 127) // 128
    pad = torch.zeros(nr * 128, nc * 128, dtype=torch.uint8, device=w.device)
    pad[:R, :B] = rb
    return pad.view(nr, 128, nc, 128).permute(0, 2, 1, 3).contiguous().view(-1)


@pytest.mark.parametrize("E,N,K,fp8", [(3, 256, 208, False), (2, 384, 256, True), (3, 100, 64, False),
                                       (1, 128, 4096, True), (5, 256, 5120, False)])
def test_pack_weights_layout(E, N, K, fp8):
    mb = _mb()
    g = torch.Generator().manual_seed(E * N + K)
    w = torch.randn(E, N, K, generator=g)
    w = (w * 0.5).to(torch.float8_e4m3fn) if fp8 else w.to(torch.bfloat16)
    p = mb.moe_pack_weights(w.cuda())
    torch.cuda.synchronize()
    assert p.shape == (E, N, K) and p.dtype == w.dtype
    assert torch.equal(p.data, _ref_pack(w.cuda()))


@pytest.mark.parametrize("E,counts,N,K,fp8,silu,pairs", [
    (4, [130, 0, 257, 64], 512, 256, False, True, False),
    (4, [130, 0, 257, 64], 512, 256, False, False, True),
    (3, [300, 17, 256], 256, 208, False, False, False),      # a partial last K block (416 bytes)
    (3, [300, 17, 256], 768, 512, True, True, False),
    (2, [600, 90], 384, 256, True, False, True),
    (16, [512] * 16, 1024, 5120, True, False, False),
])
def test_packed_weights_gemm_equals_row_major(E, counts, N, K, fp8, silu, pairs):
    """Packed weights give the grouped GEMMs bit-identical results (the same boxes land in
    shared memory), over bf16 and FP8, plain and SiLU*mul epilogues, single-CTA and
    CTA-pair tiles, ragged counts and a partial K block."""
    mb = _mb()
    g = torch.Generator().manual_seed(N + K + E)
    a = int(sum(counts))
    cd = torch.tensor(counts, dtype=torch.int32, device="cuda")
    epi = (mb.MOE_EPILOGUE_SILU_MUL if silu else mb.MOE_EPILOGUE_NONE) | (mb.MOE_GEMM_CTA_PAIRS if pairs else 0)
    if fp8:
        x = (torch.randn(a, K, generator=g) * 0.5).to(torch.float8_e4m3fn).cuda()
        w = (torch.randn(E, N, K, generator=g) * 0.5).to(torch.float8_e4m3fn).cuda()
        xs = (torch.rand(a, generator=g) + 0.5).cuda()
        ws = (torch.rand(E * N, generator=g) + 0.5).cuda()
        y0 = mb.moe_grouped_gemm_fp8_rowwise(x, w, cd, xs, ws, epilogue=epi)
        y1 = mb.moe_grouped_gemm_fp8_rowwise(x, mb.moe_pack_weights(w), cd, xs, ws, epilogue=epi)
    else:
        x = torch.randn(a, K, generator=g).to(torch.bfloat16).cuda()
        w = (torch.randn(E, N, K, generator=g) * 0.1).to(torch.bfloat16).cuda()
        y0 = mb.moe_grouped_gemm(x, w, cd, epilogue=epi)
        y1 = mb.moe_grouped_gemm(x, mb.moe_pack_weights(w), cd, epilogue=epi)
    torch.cuda.synchronize()
    assert mb.device_error() == 0
    assert torch.equal(y0, y1)


@pytest.mark.parametrize("accumulate", [False, True])
def test_packed_weights_fused_combine_and_expert_mlp(accumulate):
    """The fused top_k = 1 combine and the one-launch expert MLP with packed weights equal
    their row-major runs bit for bit."""
    mb = _mb()
    g = torch.Generator().manual_seed(21)
    E, D, H, T = 16, 512, 1024, 128
    x = torch.randn(T, D, generator=g).to(torch.bfloat16).cuda()
    w13 = (torch.randn(E, 2 * H, D, generator=g) * 0.1).to(torch.bfloat16).cuda()
    w2 = (torch.randn(E, D, H, generator=g) * 0.1).to(torch.bfloat16).cuda()
    cd = torch.tensor([8] * 12 + [0, 20, 12, 0], dtype=torch.int32, device="cuda")
    perm = torch.randperm(T, generator=g).to(torch.int32).cuda()
    init = torch.randn(T, D, generator=g).to(torch.bfloat16).cuda()
    outs = []
    for pack in (False, True):
        a13 = mb.moe_pack_weights(w13) if pack else w13
        a2 = mb.moe_pack_weights(w2) if pack else w2
        o = init.clone()
        mb.moe_expert_mlp(x, a13, a2, cd, out=o, scatter_indices=perm, accumulate=accumulate)
        z = mb.moe_grouped_gemm(x, a13, cd, epilogue=mb.MOE_EPILOGUE_SILU_MUL)
        o2 = init.clone()
        mb.moe_grouped_gemm(z, a2, cd, out=o2, scatter_indices=perm, accumulate=accumulate)
        outs.append((o, o2, z))
    torch.cuda.synchronize()
    assert mb.device_error() == 0
    for u, v in zip(outs[0], outs[1]):
        assert torch.equal(u, v)
    assert torch.equal(outs[1][0], outs[1][1])
