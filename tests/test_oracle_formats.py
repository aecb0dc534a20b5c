"""Pins for the oracle's number formats: bf16 rounding and OCP E4M3 encode/decode.

Pinned against the format definitions (hand-worked codes in
tests/golden/e4m3_codes.txt) and against PyTorch's own, independent casts.
"""
import numpy as np
import torch

import oracle
from tests.helpers import parse_golden


def test_e4m3_golden_codes(golden_dir):
    vals, codes = [], []
    for ln in parse_golden(golden_dir / "e4m3_codes.txt"):
        v, c = ln.split()[:2]
        vals.append(float(v))
        codes.append(int(c, 16))
    got = oracle.e4m3_encode(np.array(vals, np.float32))
    assert [hex(c) for c in got] == [hex(c) for c in codes]


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    nan = (codes & 0x7F) == 0x7F
    assert np.isnan(ours[nan]).all() and np.isnan(ref[nan]).all()
    np.testing.assert_array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(1)
    v = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * 50,
        rng.uniform(-448, 448, 20000).astype(np.float32),
        (rng.standard_normal(5000) * 1e-3).astype(np.float32),  # subnormal range
        oracle.e4m3_decode(np.arange(256, dtype=np.uint8)),       # every code value
    ])
    v = v[np.isfinite(v)]
    # exact midpoints between neighbouring codes exercise ties-to-even
    grid = np.unique(np.abs(oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))))
    mids = ((grid[1:].astype(np.float64) + grid[:-1]) / 2).astype(np.float32)
    v = np.concatenate([v, mids, -mids])
    ours = oracle.e4m3_encode(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, ref)


def test_e4m3_roundtrip_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    np.testing.assert_array_equal(oracle.e4m3_encode(oracle.e4m3_decode(codes)), codes)


def test_bf16_round_matches_torch_including_ties():
    rng = np.random.default_rng(2)
    v = rng.standard_normal(100000).astype(np.float32) * rng.choice([1e-3, 1.0, 1e3], 100000).astype(np.float32)
    u = v.view(np.uint32)
    ties = (u[:5000] & np.uint32(0xFFFF0000)) | np.uint32(0x8000)   # exactly halfway
    v = np.concatenate([v, ties.view(np.float32), np.array([0.0, -0.0, 3.4e38, -3.4e38], np.float32)])
    ours = oracle.bf16_round(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    np.testing.assert_array_equal(oracle.bf16_to_f32(ours),
                                  torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())
