"""Pins for the oracle's top-k finalize and the output-weighted routed forward.

topk_finalize (the routing weights applied to unweighted GEMM2 rows, in slot
order, fp32, one bf16 rounding, negative zero written as +0, then the shared
output added with one more rounding): pinned by hand-worked values, a case
that separates the two-rounding reading from a single rounding, the
negative-zero rule, an independent float32 brute force in numpy, and the
permutation special case.  The output-weighted forward is pinned to the dense
formula sum_e w_te * MLP_e(x_t) in fp64.
"""
import numpy as np
import torch

import oracle
from tests.helpers import bits, f64, rms


def _bf16(a) -> np.ndarray:
    return bits(torch.as_tensor(np.asarray(a, np.float64)).to(torch.float32).to(torch.bfloat16))


def test_finalize_hand_worked():
    rows = _bf16([[1.0, -2.0, 3.0, 0.5], [4.0, 8.0, -1.0, 2.0], [100.0, 100.0, 100.0, 100.0]])
    w = np.array([[0.5, 0.25, 7.0], [2.0, 0.0, 1.0]], np.float32)
    idx = np.array([[0, 1, -1], [1, 2, 0]], np.int32)          # -1: an absent route
    out = f64(oracle.topk_finalize(rows, w, idx))
    np.testing.assert_array_equal(out[0], [1.5, 1.0, 1.25, 0.75])
    np.testing.assert_array_equal(out[1], [9.0, 14.0, 1.0, 4.5])


def test_finalize_rounds_routed_sum_before_adding_shared():
    # routed sum 1 + 2^-9 rounds to 1.0 in bf16; 1.0 + 2^-8 is a tie that goes to even (1.0).
    # One rounding of 1 + 2^-9 + 2^-8 would give 1 + 2^-7 instead.
    rows = _bf16([[1.0], [2.0 ** -9]])
    w = np.array([[1.0, 1.0]], np.float32)
    idx = np.array([[0, 1]], np.int32)
    shared = _bf16([[2.0 ** -8]])
    assert oracle.topk_finalize(rows, w, idx)[0, 0] == 0x3F80
    assert oracle.topk_finalize(rows, w, idx, shared)[0, 0] == 0x3F80
    assert _bf16([1 + 2.0 ** -9 + 2.0 ** -8])[0] == 0x3F81


def test_finalize_writes_negative_zero_as_positive_zero():
    rows = _bf16([[2.0 ** -133, 0.0]])                          # the smallest bf16 subnormal
    w = np.array([[-(2.0 ** -10)]], np.float32)                  # product -2^-143: bf16 rounds it to -0
    out = oracle.topk_finalize(rows, w, np.array([[0]], np.int32))
    assert out[0, 0] == 0x0000 and out[0, 1] == 0x0000
    assert _bf16([-(2.0 ** -143)])[0] == 0x8000                 # what the sum rounds to before the rule


def test_finalize_float32_brute_force():
    rng = np.random.default_rng(40)
    n, D, M, k = 30, 24, 12, 4
    rows = _bf16(rng.standard_normal((n, D)) * 3)
    w = rng.uniform(-1, 1, (M, k)).astype(np.float32)
    idx = rng.integers(-1, n, (M, k)).astype(np.int32)
    shared = _bf16(rng.standard_normal((M, D)))
    got = oracle.topk_finalize(rows, w, idx, shared)
    rv = f64(rows).astype(np.float32)
    sv = f64(shared).astype(np.float32)
    for t in range(M):
        for d in range(D):
            acc = np.float32(0.0)
            for j in range(k):
                if idx[t, j] >= 0:
                    acc = np.float32(acc + np.float32(w[t, j] * rv[idx[t, j], d]))
            r = _bf16([acc])[0]
            r = np.uint16(0) if r == 0x8000 else r
            want = _bf16([np.float32(f64(np.array([r], np.uint16))[0]) + sv[t, d]])[0]
            assert got[t, d] == want, (t, d)


def test_finalize_one_route_unit_weight_is_a_permutation():
    rng = np.random.default_rng(41)
    rows = _bf16(rng.standard_normal((9, 16)))
    perm = rng.permutation(9).astype(np.int32)[:, None]
    out = oracle.topk_finalize(rows, np.ones((9, 1), np.float32), perm)
    np.testing.assert_array_equal(out, rows[perm[:, 0]])


def test_topk_weights_follow_the_inverse_permutation():
    rng = np.random.default_rng(42)
    T, E, k = 20, 6, 3
    s = _bf16(rng.uniform(0, 1, (T, E)))
    r = oracle.route(s, k)
    w = oracle.topk_weights(s, r)
    sv = f64(s)
    for t in range(T):
        es = r["expert_indices"][r["inv"][t]]
        assert list(es) == sorted(es)                            # ascending expert = ascending row
        np.testing.assert_array_equal(w[t], sv[t, es].astype(np.float32))
        assert set(es) == set(np.argsort(-sv[t], kind="stable")[:k])


def test_output_weighted_forward_against_dense_formula():
    rng = np.random.default_rng(43)
    T, D, H, E, k, Tv = 24, 64, 32, 5, 2, 21
    x = _bf16(rng.standard_normal((T, D)))
    s = _bf16(rng.uniform(0, 1, (T, E)))
    w13 = _bf16(rng.standard_normal((E, 2 * H, D)) * 0.05)
    w2 = _bf16(rng.standard_normal((E, D, H)) * 0.05)
    sh = _bf16(rng.standard_normal((T, D)) * 0.1)
    res = oracle.moe_forward_output_weighted(x, s, k, lambda ids: (w13[ids], w2[ids]), fp8=False, valid_tokens=Tv,
                                             shared_out=sh)
    xf, sf = f64(x), f64(s)
    ref = np.zeros((Tv, D))
    for t in range(Tv):
        for e in np.argsort(-sf[t], kind="stable")[:k]:
            y = f64(w13[e]) @ xf[t]
            z = y[:H] / (1 + np.exp(-y[:H])) * y[H:]
            ref[t] += sf[t, e] * (f64(w2[e]) @ z)
    ref += f64(sh[:Tv])
    got = f64(res["out"][:Tv])
    assert np.linalg.norm(got - ref) <= 1e-2 * np.linalg.norm(ref)
    assert np.abs(got - ref).max() <= 0.1 * rms(ref)
    assert np.all(res["out"][Tv:] == 0)
    # the weights act on the output: scaling every weight by 2 doubles the routed part exactly
    s2 = _bf16(f64(s) * 2)
    r2 = oracle.moe_forward_output_weighted(x, s2, k, lambda ids: (w13[ids], w2[ids]), fp8=False, valid_tokens=Tv)
    r1 = oracle.moe_forward_output_weighted(x, s, k, lambda ids: (w13[ids], w2[ids]), fp8=False, valid_tokens=Tv)
    np.testing.assert_array_equal(f64(r2["out"][:Tv]), 2 * f64(r1["out"][:Tv]))


def test_layer_forward_with_output_weighting_composes_the_stages():
    rng = np.random.default_rng(44)
    T, D, H, E, k = 16, 64, 32, 4, 2
    x = _bf16(rng.standard_normal((T, D)))
    wr = _bf16(rng.standard_normal((E, D)) * 0.125)
    w13 = _bf16(rng.standard_normal((E, 2 * H, D)) * 0.05)
    w2 = _bf16(rng.standard_normal((E, D, H)) * 0.05)
    sh = (_bf16(rng.standard_normal((2 * H, D)) * 0.05), _bf16(rng.standard_normal((D, H)) * 0.05))
    wf = lambda ids: (w13[ids], w2[ids])
    got = oracle.moe_layer_forward(x, wr, k, wf, fp8=False, shared=sh, weighting="output")["out"]
    base = oracle.shared_expert(x, *sh, fp8=False)
    want = oracle.moe_forward_output_weighted(x, oracle.router_scores(x, wr), k, wf, fp8=False, shared_out=base)
    np.testing.assert_array_equal(got, want["out"])
    part, _ = oracle.moe_layer_forward_tokens(np.array([1, 5, 9]), x, wr, k, wf, fp8=False, shared=sh,
                                              weighting="output")
    np.testing.assert_array_equal(part, got[[1, 5, 9]])
