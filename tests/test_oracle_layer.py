"""Pins for the oracle's router scores, shared expert and whole-layer forward.

Router scores (MetaShufflingMoE._route: sigmoid of the linear router, bf16):
pinned by closed forms (a zero router gives sigmoid(0) = 1/2 exactly, one-hot
routers copy scaled token entries, integer inputs give exact integer logits),
the identity sigmoid(-l) = 1 - sigmoid(l), and a pure-Python brute force on a
tiny case.  The shared expert is pinned to the routed path it must equal (one
expert, every token routed to it with score 1) and to a dense float64 SwiGLU;
the layer forward to its two limiting cases (no routed contribution, no
shared contribution).
"""
import math

import numpy as np
import torch

import oracle
from tests.helpers import bf16_from_bits, bits, f64, rms


def _bf16(a) -> np.ndarray:
    return bits(torch.as_tensor(np.asarray(a, np.float64)).to(torch.float32).to(torch.bfloat16))


def _rand_bf16(rng, *shape, scale=1.0):
    return _bf16(rng.standard_normal(shape) * scale)


# ------------------------------------------------------------ router scores

def test_zero_router_scores_are_one_half():
    rng = np.random.default_rng(30)
    x = _rand_bf16(rng, 7, 48)
    sc, lg = oracle.router_scores(x, np.zeros((5, 48), np.uint16), logits=True)
    assert np.all(sc == 0x3F00)            # bf16(0.5)
    assert np.all(f64(lg) == 0.0)


def test_one_hot_router_copies_scaled_token_entries():
    # w[e, d] = 2 when d = perm[e]: logit[t, e] = 2 x[t, perm[e]] exactly, which
    # fixes both the operand order and the expert/feature indexing
    rng = np.random.default_rng(31)
    T, D, E = 9, 40, 6
    x = _rand_bf16(rng, T, D)
    perm = rng.permutation(D)[:E]
    w = np.zeros((E, D), np.uint16)
    w[np.arange(E), perm] = _bf16([2.0])[0]
    _, lg = oracle.router_scores(x, w, logits=True)
    np.testing.assert_array_equal(f64(lg), 2.0 * f64(x)[:, perm])


def test_integer_logits_and_sigmoid_closed_forms():
    rng = np.random.default_rng(32)
    T, D, E = 6, 64, 5
    xi = rng.integers(-3, 4, (T, D))
    wi = rng.integers(-2, 3, (E, D))
    sc, lg = oracle.router_scores(_bf16(xi), _bf16(wi), logits=True)
    exact = xi @ wi.T                       # |logit| <= 384 < 2^9: some are not bf16-representable
    np.testing.assert_array_equal(lg, _bf16(exact))
    # sigmoid at integer points, from math.exp of the bf16 logit
    want = [[1.0 / (1.0 + math.exp(-v)) for v in row] for row in f64(lg)]
    np.testing.assert_array_equal(sc, _bf16(want))
    # saturation: a logit of 64 gives exactly 1.0, one of -64 a tiny positive score
    x1 = _bf16(np.full((1, 16), 4.0))
    s_hi = oracle.router_scores(x1, _bf16(np.ones((1, 16))))
    s_lo = oracle.router_scores(x1, _bf16(-np.ones((1, 16))))
    assert f64(s_hi)[0, 0] == 1.0
    assert 0.0 < f64(s_lo)[0, 0] < 1e-27


def test_sigmoid_reads_the_bf16_rounded_logit():
    # logits a + b that bf16 cannot hold: the score is the sigmoid of the rounded
    # logit (the linear's bf16 output), and for some of them that differs from
    # the sigmoid of the exact sum
    a = f64(_bf16(np.linspace(-4, 4, 257)))
    b = 3 * 2.0 ** -10
    x = _bf16(np.ones((1, 2)))
    w = _bf16(np.stack([a, np.full_like(a, b)], 1))
    sc, lg = oracle.router_scores(x, w, logits=True)
    exact = a + b
    np.testing.assert_array_equal(lg[0], _bf16(exact))
    from_rounded = _bf16(1.0 / (1.0 + np.exp(-f64(lg[0]))))
    from_exact = _bf16(1.0 / (1.0 + np.exp(-exact)))
    np.testing.assert_array_equal(sc[0], from_rounded)
    assert np.any(from_rounded != from_exact)


def test_sigmoid_reflection_identity():
    rng = np.random.default_rng(33)
    T, D, E = 50, 128, 16
    x = _rand_bf16(rng, T, D)
    w = _rand_bf16(rng, E, D, scale=1.0 / math.sqrt(D))
    wneg = w ^ np.uint16(0x8000)            # negate every weight (sign bit)
    s_pos = f64(oracle.router_scores(x, w))
    s_neg = f64(oracle.router_scores(x, wneg))
    # sigmoid(-l) = 1 - sigmoid(l); each score is within half a bf16 step (<= 2^-9) of its exact value
    assert np.all(np.abs(s_pos + s_neg - 1.0) <= 2.0 ** -8)
    lg = f64(oracle.router_scores(x, w, logits=True)[1])
    assert np.all(s_pos[lg > 0] >= 0.5) and np.all(s_pos[lg < 0] <= 0.5)


def test_router_brute_force_tiny_and_valid_rows():
    rng = np.random.default_rng(34)
    T, D, E, Tv = 5, 24, 6, 4
    x = _rand_bf16(rng, T, D)
    w = _rand_bf16(rng, E, D, scale=0.3)
    sc = oracle.router_scores(x, w, valid_tokens=Tv)
    xf, wf = f64(x), f64(w)
    for t in range(Tv):
        for e in range(E):
            logit = f64(_bf16([math.fsum(float(a) * float(b) for a, b in zip(xf[t], wf[e]))]))[0]
            assert sc[t, e] == _bf16([1.0 / (1.0 + math.exp(-logit))])[0], (t, e)
    assert np.all(sc[Tv:] == 0), "rows past the valid tokens are not written"


# ------------------------------------------------------------ shared expert

def _expert(rng, D, H, fp8):
    w13 = rng.standard_normal((2 * H, D)) * 0.05
    w2 = rng.standard_normal((D, H)) * 0.05
    if fp8:
        return w13.astype(np.float32), w2.astype(np.float32)
    return _bf16(w13), _bf16(w2)


def test_shared_expert_equals_one_expert_with_unit_scores():
    rng = np.random.default_rng(35)
    T, D, H = 12, 64, 48
    x = _rand_bf16(rng, T, D)
    ones = _bf16(np.ones((T, 1)))
    for fp8, z_bf16 in ((False, False), (True, False), (True, True)):
        w13, w2 = _expert(rng, D, H, fp8)
        got = oracle.shared_expert(x, w13, w2, fp8=fp8, scale_ub=30.0, z_bf16=z_bf16)
        ref = oracle.moe_forward(x, ones, 1, lambda ids: (w13[None], w2[None]), fp8=fp8, scale_ub=30.0,
                                 z_bf16=z_bf16)["out"]
        np.testing.assert_array_equal(got, ref)


def test_shared_expert_fp8_input_rule_is_the_gathers_at_unit_score():
    rng = np.random.default_rng(36)
    T, D = 10, 96
    x = _rand_bf16(rng, T, D, scale=3.0)
    q1, s1 = oracle.quantize_rows(oracle.bf16_to_f32(x), 5.0)
    q2, s2 = oracle.gather_scale_quant(x, np.arange(T, dtype=np.int32), np.zeros(T, np.int32),
                                       _bf16(np.ones((T, 1))), 5.0)
    np.testing.assert_array_equal(q1, q2)
    np.testing.assert_array_equal(s1, s2)


def test_shared_expert_against_dense_swiglu_and_valid_rows():
    rng = np.random.default_rng(37)
    T, D, H, Tv = 16, 128, 64, 13
    x = _rand_bf16(rng, T, D)
    w13, w2 = _expert(rng, D, H, False)
    got = oracle.shared_expert(x, w13, w2, fp8=False, valid_tokens=Tv)
    y = f64(x) @ f64(w13).T
    z = y[:, :H] / (1 + np.exp(-y[:, :H])) * y[:, H:]
    ref = z @ f64(w2).T
    err = np.abs(f64(got[:Tv]) - ref[:Tv])
    assert err.max() <= 2e-2 * rms(ref[:Tv])
    assert np.all(got[Tv:] == 0)


# ------------------------------------------------------------- layer forward

def test_layer_forward_limits():
    rng = np.random.default_rng(38)
    T, D, H, E, k = 24, 64, 32, 4, 2
    x = _rand_bf16(rng, T, D)
    wr = _rand_bf16(rng, E, D, scale=0.125)
    w13 = _bf16(rng.standard_normal((E, 2 * H, D)) * 0.05)
    w2 = _bf16(rng.standard_normal((E, D, H)) * 0.05)
    sh = _expert(rng, D, H, False)
    routed = lambda ids: (w13[ids], w2[ids])
    # no routed contribution (w2 = 0): the output is the shared expert's, unchanged
    zero_w2 = lambda ids: (w13[ids], np.zeros_like(w2[ids]))
    res = oracle.moe_layer_forward(x, wr, k, zero_w2, fp8=False, shared=sh)
    np.testing.assert_array_equal(res["out"], res["shared_out"])
    np.testing.assert_array_equal(res["shared_out"], oracle.shared_expert(x, *sh, fp8=False))
    # no shared expert: the routed forward on the router's scores
    res = oracle.moe_layer_forward(x, wr, k, routed, fp8=False)
    np.testing.assert_array_equal(res["out"], oracle.moe_forward(x, oracle.router_scores(x, wr), k, routed,
                                                                 fp8=False)["out"])
    # both: every token's output is the shared row plus its routed rows (fp32 sum, one rounding)
    full = oracle.moe_layer_forward(x, wr, k, routed, fp8=False, shared=sh)
    o, ti = full["o"], full["route"]["token_indices"]
    acc = f64(full["shared_out"]).astype(np.float32)
    for r in range(len(ti)):
        acc[ti[r]] += f64(o[r : r + 1])[0].astype(np.float32)
    np.testing.assert_array_equal(full["out"], bits(torch.from_numpy(acc).to(torch.bfloat16)))


def test_layer_forward_tokens_equals_full_rows():
    rng = np.random.default_rng(39)
    T, D, H, E, k = 20, 64, 32, 6, 2
    x = _rand_bf16(rng, T, D)
    wr = _rand_bf16(rng, E, D, scale=0.125)
    w13 = rng.standard_normal((E, 2 * H, D)).astype(np.float32) * 0.05
    w2 = rng.standard_normal((E, D, H)).astype(np.float32) * 0.05
    sh = _expert(rng, D, H, True)
    wf = lambda ids: (w13[ids], w2[ids])
    tok = np.array([0, 3, 7, 19])
    for z_bf16 in (False, True):
        full = oracle.moe_layer_forward(x, wr, k, wf, fp8=True, shared=sh, scale_ub=20.0, z_bf16=z_bf16)["out"]
        part, _ = oracle.moe_layer_forward_tokens(tok, x, wr, k, wf, fp8=True, shared=sh, scale_ub=20.0,
                                                  z_bf16=z_bf16)
        np.testing.assert_array_equal(part, full[tok])
