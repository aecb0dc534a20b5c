"""Pins for the oracle's grouped GEMMs (bf16 and FP8 rowwise).

Pinned by identity weights, by integer-valued operands whose products sum
exactly (so numpy's matmul gives the exact answer), by numpy's matmul per
expert segment, and by power-of-two scales.
"""
import numpy as np
import torch

import oracle
from tests.helpers import bits, f64


def _bf16(a):
    return bits(torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16))


def test_identity_weights_copy_rows():
    rng = np.random.default_rng(20)
    E, K = 3, 16
    counts = np.array([5, 0, 7], np.int32)
    x = _bf16(rng.standard_normal((12, K)))
    w = _bf16(np.stack([np.eye(K)] * E))
    np.testing.assert_array_equal(oracle.grouped_gemm_bf16(x, w, counts), x)


def test_integer_operands_match_numpy_per_expert():
    rng = np.random.default_rng(21)
    E, N, K = 4, 24, 40
    counts = np.array([3, 0, 9, 5], np.int32)
    a = counts.sum()
    xi = rng.integers(-8, 8, (a, K))
    wi = rng.integers(-8, 8, (E, N, K))
    y = oracle.grouped_gemm_bf16(_bf16(xi), _bf16(wi), counts)
    off = 0
    for e in range(E):
        seg = slice(off, off + counts[e])
        ref = xi[seg] @ wi[e].T            # exact integers
        np.testing.assert_array_equal(y[seg], _bf16(ref), err_msg=f"expert {e}")
        off += counts[e]


def test_random_single_expert_is_a_plain_gemm():
    rng = np.random.default_rng(22)
    a, N, K = 17, 33, 72
    x = _bf16(rng.standard_normal((a, K)))
    w = _bf16(rng.standard_normal((1, N, K)) * 0.05)
    y = oracle.grouped_gemm_bf16(x, w, np.array([a], np.int32))
    ref = _bf16((f64(x) @ f64(w[0]).T).astype(np.float32))
    diff = np.abs(y.astype(np.int32) - ref.astype(np.int32))
    assert diff.max() <= 1 and (diff == 0).mean() > 0.999


def test_rows_past_the_experts_are_not_written():
    x = _bf16(np.ones((6, 16)))
    w = _bf16(np.ones((2, 8, 16)))
    y = oracle.grouped_gemm_bf16(x, w, np.array([2, 1], np.int32))
    assert np.all(f64(y[:3]) == 16.0) and np.all(y[3:] == 0)


def test_fp8_unit_and_power_of_two_scales():
    rng = np.random.default_rng(23)
    E, N, K = 2, 16, 32
    counts = np.array([4, 6], np.int32)
    xi = rng.integers(-6, 7, (10, K)).astype(np.float32)   # small integers are exact e4m3 values
    wi = rng.integers(-6, 7, (E, N, K)).astype(np.float32)
    xq, wq = oracle.e4m3_encode(xi), oracle.e4m3_encode(wi)
    np.testing.assert_array_equal(oracle.e4m3_decode(xq), xi)
    xs = np.exp2(rng.integers(-3, 3, 10)).astype(np.float32)
    ws = np.exp2(rng.integers(-3, 3, (E, N))).astype(np.float32)
    y = oracle.grouped_gemm_fp8(xq, wq, counts, xs, ws)
    off = 0
    for e in range(E):
        seg = slice(off, off + counts[e])
        ref = (xi[seg].astype(np.float64) @ wi[e].T.astype(np.float64)) * xs[seg, None] * ws[e][None, :]
        np.testing.assert_array_equal(y[seg], _bf16(ref))
        off += counts[e]


def test_quantize_rows_matches_gather_quant_rule():
    # quantize_rows is the same row rule as the gather quantiser (score 1).
    rng = np.random.default_rng(24)
    w = rng.standard_normal((5, 64)).astype(np.float32) * 0.02
    wb = torch.from_numpy(w).to(torch.bfloat16)
    q, s = oracle.quantize_rows(wb.float().numpy())
    one = _bf16(np.ones((5, 1)))
    idx = np.arange(5, dtype=np.int32)
    q2, s2 = oracle.gather_scale_quant(bits(wb), idx, np.zeros(5, np.int32), one)
    np.testing.assert_array_equal(q, q2)
    np.testing.assert_array_equal(s, s2)
