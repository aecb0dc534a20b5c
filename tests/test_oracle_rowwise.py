"""Pins for the oracle's row-wise stages: gather*score, gather + FP8 quantise,
silu_mul(_quant) and the scatter-add combine.

Pinned by identities of the arithmetic (unit and power-of-two scores, integer
sums), hand-worked quantised rows, closed-form error bounds of the e4m3 grid,
and PyTorch's independent bf16 casts and SiLU.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import bf16_from_bits, bits, e4m3_step_diff, f64, parse_golden


def _rand_bf16(rng, *shape, scale=1.0):
    return bits((torch.from_numpy(rng.standard_normal(shape).astype(np.float32)) * scale).to(torch.bfloat16))


def _scores(vals):
    return bits(torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16))


# ------------------------------------------------------------------ gather

def test_gather_unit_and_power_of_two_scores_are_exact():
    rng = np.random.default_rng(10)
    T, D, E = 12, 48, 3
    x = _rand_bf16(rng, T, D)
    ti = np.array([3, 0, 11, 5, 3], np.int32)
    ei = np.array([0, 1, 2, 1, 2], np.int32)
    ones = _scores(np.ones((T, E)))
    np.testing.assert_array_equal(oracle.gather_scale(x, ti, ei, ones), x[ti])
    halves = _scores(np.full((T, E), 0.5))
    np.testing.assert_array_equal(f64(oracle.gather_scale(x, ti, ei, halves)), f64(x[ti]) / 2)


def test_gather_matches_torch_product_and_respects_valid_rows():
    rng = np.random.default_rng(11)
    T, D, E = 20, 64, 6
    x = _rand_bf16(rng, T, D)
    s = _scores(1 / (1 + np.exp(-rng.standard_normal((T, E)))))
    ti = rng.integers(0, T, 30).astype(np.int32)
    ei = rng.integers(0, E, 30).astype(np.int32)
    out = oracle.gather_scale(x, ti, ei, s, valid_rows=22)
    sv = bf16_from_bits(s).float()
    ref = (bf16_from_bits(x).float()[ti] * sv[ti, ei][:, None]).to(torch.bfloat16)
    np.testing.assert_array_equal(out[:22], bits(ref)[:22])
    assert np.all(out[22:] == 0), "rows at or past the valid count are not written"


# ------------------------------------------------------- gather + quantise

def _parse_case(ln):
    kv = dict(f.split("=") for f in ln.split()[1:])
    x = [float(v) for v in kv["x"].split(",")]
    ub = None if kv["ub"] == "none" else float(kv["ub"])
    return x, float(kv["score"]), ub, np.float32(kv["scale"]), [int(c, 16) for c in kv["codes"].split(",")]


def test_gather_quant_golden_rows(golden_dir):
    for ln in parse_golden(golden_dir / "quant_rows.txt"):
        xv, score, ub, scale, codes = _parse_case(ln)
        x = _scores(np.array([xv]))
        s = _scores(np.array([[score]]))
        q, sc = oracle.gather_scale_quant(x, np.array([0], np.int32), np.array([0], np.int32), s, ub)
        assert [hex(c) for c in q[0]] == [hex(c) for c in codes], ln
        assert sc[0] == scale, ln


def test_gather_quant_error_bounds_and_extremes():
    rng = np.random.default_rng(12)
    T, D, E, a = 16, 256, 4, 24
    x = _rand_bf16(rng, T, D)
    s = _scores(rng.uniform(0.1, 1.0, (T, E)))
    ti = rng.integers(0, T, a).astype(np.int32)
    ei = rng.integers(0, E, a).astype(np.int32)
    q, sc = oracle.gather_scale_quant(x, ti, ei, s)
    v = f64(x)[ti] * bf16_from_bits(s).double().numpy()[ti, ei][:, None]
    deq = oracle.e4m3_decode(q).astype(np.float64) * sc[:, None]
    m = np.abs(v).max(axis=1)
    # the row's largest magnitude maps to the largest code 448 (ub and EPS inactive)
    big = np.abs(v) == m[:, None]
    assert np.all(np.abs(oracle.e4m3_decode(q))[big] == 448.0)
    # relative error of a normal e4m3 value is at most half a step: 2^-4
    normal = np.abs(v) * (448.0 / m[:, None]) >= 2.0 ** -6
    assert np.all(np.abs(deq - v)[normal] <= 2.0 ** -4 * np.abs(v)[normal] * (1 + 1e-6))
    # subnormal range: absolute error at most half the subnormal step 2^-9, in scaled units
    sub = ~normal
    assert np.all(np.abs(deq - v)[sub] <= (2.0 ** -10) * (m[:, None] / 448.0).repeat(D, 1)[sub] * (1 + 1e-6))


def test_gather_quant_scale_bound_and_zero_row():
    x = _scores(np.array([[100.0, -50.0, 0.0, 1.0], [0.0, 0.0, 0.0, 0.0]]))
    s = _scores(np.ones((2, 1)))
    ti, ei = np.array([0, 1], np.int32), np.array([0, 0], np.int32)
    q, sc = oracle.gather_scale_quant(x, ti, ei, s, scale_ub=10.0)
    # m = min(100, 10) = 10: s = 44.8; values past the bound saturate
    assert sc[0] == np.float32(1) / (np.float32(448) / np.float32(10))
    assert q[0, 0] == 0x7E and q[0, 1] == 0xFE and q[0, 2] == 0x00
    # an all-zero row takes m = EPS and quantises to zeros
    assert np.all(q[1] == 0) and sc[1] == np.float32(1) / (np.float32(448) / np.float32(1e-12))


# ---------------------------------------------------------------- silu_mul

def test_silu_mul_identities():
    rng = np.random.default_rng(13)
    a, H = 8, 32
    y0 = rng.standard_normal((a, H)).astype(np.float32) * 3
    y0[0] = 0.0
    y0[1] = np.abs(y0[1]) + 40.0            # sigmoid = 1 to far below fp32 precision
    y1 = rng.standard_normal((a, H)).astype(np.float32)
    y = bits(torch.from_numpy(np.concatenate([y0, y1], 1)).to(torch.bfloat16))
    z = oracle.silu_mul(y, H)
    assert np.all(f64(z[0]) == 0.0)
    y0b, y1b = bf16_from_bits(y[:, :H]).float(), bf16_from_bits(y[:, H:]).float()
    np.testing.assert_array_equal(z[1], bits((y0b[1] * y1b[1]).to(torch.bfloat16)))
    # against torch's own SiLU in float64, rounded to bf16: equal up to one bf16 step
    ref = bits((torch.nn.functional.silu(y0b.double()) * y1b.double()).to(torch.bfloat16))
    diff = np.abs(z.astype(np.int32) - ref.astype(np.int32))
    assert diff.max() <= 1 and (diff == 0).mean() > 0.99


def test_silu_odd_identity():
    # silu(a) - silu(-a) = a  (y1 = 1)
    a_vals = np.linspace(-6, 6, 64, dtype=np.float32)
    y = bits(torch.from_numpy(np.stack([np.concatenate([a_vals, -a_vals]),
                                        np.ones(128, np.float32)]).reshape(1, 256)).to(torch.bfloat16))
    z = f64(oracle.silu_mul(y.reshape(1, 256), 128))[0]
    a_b = f64(y[0, :64])
    # each z is within half a bf16 step (at most 2^-8 relative) of silu, and |silu(a)| <= |a|
    assert np.all(np.abs(z[:64] - z[64:128] - a_b) <= 2 * 2.0 ** -8 * np.abs(a_b))


def test_silu_mul_quant_consistent_with_silu_and_quant_rule():
    rng = np.random.default_rng(14)
    a, H = 10, 96
    y = _rand_bf16(rng, a, 2 * H, scale=2.0)
    zq, zs = oracle.silu_mul_quant(y, H, scale_ub=1200.0, valid_rows=9)
    y0, y1 = f64(y[:, :H]), f64(y[:, H:])
    z = y0 / (1 + np.exp(-y0)) * y1
    m = np.abs(z).max(axis=1)
    np.testing.assert_allclose(zs[:9], m[:9] / 448.0, rtol=2e-7)
    deq = oracle.e4m3_decode(zq[:9]).astype(np.float64) * zs[:9, None]
    err = np.abs(deq - z[:9])
    assert np.all(err <= 2.0 ** -4 * np.abs(z[:9]) + 2.0 ** -10 * m[:9, None] / 448 * 1.01)
    assert np.all(zq[9] == 0) and zs[9] == 0


def test_silu_mul_quant_of_bf16_z_is_the_row_rule_on_silu_mul_output():
    """z_bf16=True quantises the bf16 z that silu_mul writes: here the row rule is
    applied by PyTorch (fp32 max, IEEE division and reciprocal, its own e4m3 cast)
    to the oracle's silu_mul output, and codes and scales must match exactly."""
    rng = np.random.default_rng(16)
    a, H, v = 12, 160, 11
    y = _rand_bf16(rng, a, 2 * H, scale=2.5)
    y[3, :H] = bits(torch.full((H,), 40.0, dtype=torch.bfloat16))      # a large row: the bound 1200 binds
    y[3, H:] = bits(torch.full((H,), 64.0, dtype=torch.bfloat16))
    y[5] = 0                                                             # an all-zero row: m = EPS
    zq, zs = oracle.silu_mul_quant(y, H, scale_ub=1200.0, valid_rows=v, z_bf16=True)
    zb = bf16_from_bits(oracle.silu_mul(y, H, v)[:v]).float()
    m = torch.clamp(zb.abs().amax(dim=1), min=1e-12)
    m = torch.minimum(m, torch.tensor(1200.0))
    s = torch.tensor(448.0) / m
    q = (zb * s[:, None]).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    np.testing.assert_array_equal(zq[:v], q.view(torch.uint8).numpy())
    np.testing.assert_array_equal(zs[:v], (1.0 / s).numpy())
    assert zs[3] == np.float32(1) / (np.float32(448) / np.float32(1200))
    assert np.all(zq[v:] == 0) and np.all(zs[v:] == 0)
    # the fp32-z reading differs on a few codes (double rounding), by one step at most
    zq32, zs32 = oracle.silu_mul_quant(y, H, scale_ub=1200.0, valid_rows=v)
    diff = e4m3_step_diff(zq[:v], zq32[:v])
    assert diff.max() <= 1 and 0 < (diff > 0).mean() < 0.05


# ------------------------------------------------------------- scatter-add

def test_scatter_add_integer_rows_sum_exactly():
    rng = np.random.default_rng(15)
    T, D, k = 10, 16, 3
    ti = np.repeat(np.arange(T, dtype=np.int32), k)
    rng.shuffle(ti)
    rows_i = rng.integers(-20, 20, (T * k, D))
    init_i = rng.integers(-20, 20, (T, D))
    out = bits(torch.from_numpy(init_i.astype(np.float32)).to(torch.bfloat16))
    rows = bits(torch.from_numpy(rows_i.astype(np.float32)).to(torch.bfloat16))
    oracle.scatter_add(out, rows, ti)
    expect = init_i.copy()
    np.add.at(expect, ti, rows_i)
    np.testing.assert_array_equal(f64(out), expect.astype(np.float64))


def test_scatter_add_k1_is_a_permutation_and_leaves_other_tokens():
    rng = np.random.default_rng(16)
    T, D = 12, 24
    perm = rng.permutation(10).astype(np.int32)    # tokens 10, 11 receive nothing
    rows = _rand_bf16(rng, 10, D)
    out = np.zeros((T, D), np.uint16)
    out[10:] = 0x3F80                               # 1.0, must stay
    oracle.scatter_add(out, rows, perm, valid_rows=8)
    np.testing.assert_array_equal(out[perm[:8]], rows[:8])
    assert np.all(out[perm[8:]] == 0) and np.all(out[10:] == 0x3F80)


def test_gather_then_scatter_with_identity_expert_gives_score_times_x():
    # top_k = 1, E = 1 and an identity expert: the combine returns score * x.
    rng = np.random.default_rng(17)
    T, D = 14, 40
    x = _rand_bf16(rng, T, D)
    s = _scores(rng.uniform(0, 1, (T, 1)))
    r = oracle.route(s, 1)
    g = oracle.gather_scale(x, r["token_indices"], r["expert_indices"], s)
    out = np.zeros((T, D), np.uint16)
    oracle.scatter_add(out, g, r["token_indices"])
    ref = (bf16_from_bits(x).float() * bf16_from_bits(s).float()).to(torch.bfloat16)
    np.testing.assert_array_equal(out, bits(ref))
