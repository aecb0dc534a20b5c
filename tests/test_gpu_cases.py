"""The timing cases of the package (python -m moe_token_routing_index_gb300.cases ...)
run end to end and report every row kernel of the boundary."""
import pytest

pytestmark = pytest.mark.gpu


def test_rowwise_case_times_every_row_kernel():
    from moe_token_routing_index_gb300 import cases

    res = cases.case_rowwise("tiny", 2)
    assert set(res["kernels"]) == {"moe_router_scores", "moe_router_route", "moe_route", "moe_gather_scale", "moe_gather_scale_quant", "moe_silu_mul",
                                   "moe_silu_mul_quant", "moe_scatter_add", "moe_scatter_add_padded",
                                   "moe_topk_finalize"}
    for d in res["kernels"].values():
        assert d["us"] > 0 and d["bytes"] > 0


def test_w13_case_runs_the_layer_gemm():
    """`cases w13 <workload>` (the source of the committed traffic figures) runs the
    workload's w13 GEMM on the active experts and reports its rows and rate."""
    from moe_token_routing_index_gb300 import cases, workloads

    res = cases.case_w13("tiny", "single", 2)
    cfg = workloads.CONFIGS["tiny"]
    assert res["rows"] == cfg.valid_tokens * cfg.top_k
    assert 1 <= res["experts"] <= cfg.E and res["us"] > 0 and res["TFLOP/s"] > 0
