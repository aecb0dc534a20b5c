"""Pins for the oracle's top-k routing and by-expert permutation.

Pinned by a hand-worked example, by brute force over all k-subsets on tiny
inputs, by a library sort, and by the invariants of the permutation.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle
from moe_token_routing_index_gb300 import workloads
from tests.helpers import bits, parse_golden


def _bf16_scores(vals, T, E):
    return bits(torch.tensor(vals, dtype=torch.float32).reshape(T, E).to(torch.bfloat16))


def test_route_golden_tiny(golden_dir):
    kv = {}
    for ln in parse_golden(golden_dir / "route_tiny.txt"):
        key, *rest = ln.split()
        kv[key] = rest
    T, E, k, Tv = (int(kv[n][0]) for n in ("T", "E", "top_k", "valid_tokens"))
    scores = _bf16_scores([float(v) for v in kv["scores"]], T, E)
    r = oracle.route(scores, k, Tv)
    for name in ("counts", "offsets", "expert_indices", "token_indices"):
        np.testing.assert_array_equal(r[name], np.array(kv[name], np.int32), err_msg=name)
    np.testing.assert_array_equal(r["inv"].ravel(), np.array(kv["inv"], np.int32))


def _check_invariants(r, T, E, k, Tv, chosen_sets):
    a = Tv * k
    counts, offsets = r["counts"], r["offsets"]
    ei, ti, inv = r["expert_indices"], r["token_indices"], r["inv"]
    assert counts[E] == a and counts[:E].sum() == a
    np.testing.assert_array_equal(offsets[:E], np.concatenate([[0], np.cumsum(counts[:E])[:-1]]))
    assert offsets[E] == a
    assert np.all(np.diff(ei) >= 0)
    for e in range(E):
        seg = ti[offsets[e]:offsets[e] + counts[e]]
        assert np.all(np.diff(seg) > 0), "tokens within an expert must be strictly increasing"
        assert np.all(ei[offsets[e]:offsets[e] + counts[e]] == e)
    assert np.all((ti >= 0) & (ti < Tv))
    per_tok = np.bincount(ti, minlength=Tv)
    assert np.all(per_tok == k)
    pairs = set(zip(ei.tolist(), ti.tolist()))
    assert len(pairs) == a, "each (token, expert) pair appears once"
    for t in range(Tv):
        rows = inv[t]
        assert np.all(np.diff(rows) > 0)
        assert np.all(ti[rows] == t)
        assert set(ei[rows].tolist()) == chosen_sets[t]


@pytest.mark.parametrize("E,k", [(1, 1), (2, 1), (2, 2), (3, 2), (4, 3), (5, 2), (6, 3)])
def test_route_brute_force_subsets(E, k):
    # A top-k set with ties to the lower index is the k-subset with the largest
    # score sum that is lexicographically smallest among all such subsets.
    rng = np.random.default_rng(E * 10 + k)
    T = 40
    palette = np.array([0.0, -0.0, 0.25, 0.5, 0.5, 0.75, 1.0], np.float32)  # many ties
    vals = rng.choice(palette, size=(T, E))
    scores = _bf16_scores(vals.ravel().tolist(), T, E)
    sv = torch.from_numpy(scores.view(np.int16)).view(torch.bfloat16).double().numpy()
    r = oracle.route(scores, k)
    chosen = []
    for t in range(T):
        best = None
        for sub in itertools.combinations(range(E), k):   # ascending tuples, lexicographic order
            s = sum(sv[t, e] for e in sub)
            if best is None or s > best[0]:
                best = (s, sub)
        chosen.append(set(best[1]))
    _check_invariants(r, T, E, k, T, chosen)


@pytest.mark.parametrize("name", ["tiny", "decode_zero", "fine_grained", "padded_fp8"])
def test_route_matches_stable_sort_on_workloads(name):
    cfg = workloads.CONFIGS[name]
    scores = bits(workloads.make_scores(cfg))
    Tv = cfg.valid_tokens
    r = oracle.route(scores, cfg.top_k, Tv)
    sv = torch.from_numpy(scores.view(np.int16)).view(torch.bfloat16).float().numpy()
    # numpy's stable sort on the negated score keeps equal scores in ascending expert order
    order = np.argsort(-sv[:Tv], axis=1, kind="stable")[:, :cfg.top_k]
    chosen = [set(row.tolist()) for row in order]
    _check_invariants(r, cfg.T, cfg.E, cfg.top_k, Tv, chosen)


def test_route_special_cases():
    rng = np.random.default_rng(3)
    T, E = 9, 5
    scores = _bf16_scores(rng.standard_normal(T * E).tolist(), T, E)
    # k = E: every token goes to every expert
    r = oracle.route(scores, E)
    assert np.all(r["counts"][:E] == T)
    np.testing.assert_array_equal(r["token_indices"], np.tile(np.arange(T), E))
    # E = 1: one expert, rows are the tokens in order
    r1 = oracle.route(scores[:, :1].copy(), 1)
    np.testing.assert_array_equal(r1["token_indices"], np.arange(T))
    assert r1["counts"].tolist() == [T, T]
    # no valid token: empty routing
    r0 = oracle.route(scores, 2, 0)
    assert r0["counts"].tolist() == [0] * (E + 1) and len(r0["token_indices"]) == 0
    with pytest.raises(ValueError):
        oracle.route(scores, E + 1)
    with pytest.raises(ValueError):
        oracle.route(scores, 1, T + 1)


def test_route_f32_and_strided_scores_agree():
    rng = np.random.default_rng(4)
    T, E, k = 33, 12, 3
    sb = _bf16_scores(rng.standard_normal(T * E).tolist(), T, E)
    sf = torch.from_numpy(sb.view(np.int16)).view(torch.bfloat16).float().numpy()
    strided = np.ascontiguousarray(sb.T).T            # stride_t = 1, stride_e = T
    assert strided.strides != sb.strides
    r_b, r_f, r_s = oracle.route(sb, k), oracle.route(sf, k), oracle.route(strided, k)
    for key in ("counts", "expert_indices", "token_indices", "inv"):
        np.testing.assert_array_equal(r_b[key], r_f[key])
        np.testing.assert_array_equal(r_b[key], r_s[key])
