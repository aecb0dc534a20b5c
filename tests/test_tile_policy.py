"""The host-side choice between 256-row (CTA pair) and 128-row GEMM tiles:
pairs when they pad the experts' rows at most 9% more than 128-row tiles."""
from moe_token_routing_index_gb300.forward import MoELayer


def test_pairs_for_large_experts():
    assert MoELayer.prefer_pairs([4096, 4096, 0, 0, 8])       # Zipf-like: a few big experts
    assert MoELayer.prefer_pairs([512] * 16)                   # exact multiples of 256


def test_single_tiles_for_experts_just_past_a_pair_tile():
    assert not MoELayer.prefer_pairs([257] * 128)              # 512 against 384 rows per expert
    assert not MoELayer.prefer_pairs([100, 120, 64])           # everything fits one 128-row tile
    assert not MoELayer.prefer_pairs([0, 0, 0])                # nothing routed


def test_margin_boundary():
    # pairs 512 rows, single 384 rows: 1.33 > 1.09
    assert not MoELayer.prefer_pairs([300])
    # pairs 768 rows, single 768 rows: equal padding
    assert MoELayer.prefer_pairs([700])
