"""The traffic figures bench.py reports: each names a kernel source that exists and a
(workload, stage) pair the bench can report, and the source hash covers the code of every
local header the source includes, so a code change in any of them retires the figure
while an edit of comments does not."""
import re

import bench
from moe_token_routing_index_gb300 import workloads

CSRC = bench.ROOT / "moe_token_routing_index_gb300" / "csrc"
STAGES = {"route", "gather", "gather_quant", "expert_mlp", "gemm_w13_silu_quant", "gemm_w13_silu", "gemm_w2",
          "scatter", "finalize", "router_route"}


def test_traffic_entries_name_existing_sources_and_stages():
    for (workload, stage), (nbytes, src, digest) in bench.TRAFFIC.items():
        assert workload in workloads.CONFIGS, workload
        assert stage in STAGES, stage
        for f in ((src,) if isinstance(src, str) else src):
            assert (CSRC / f).is_file(), f
        assert nbytes > 0 and re.fullmatch(r"[0-9a-f]{12}", digest)


def test_source_hash_follows_includes(tmp_path, monkeypatch):
    # a private copy of a source tree: editing a header two includes deep changes the hash
    pkg = tmp_path / "moe_token_routing_index_gb300" / "csrc"
    pkg.mkdir(parents=True)
    (tmp_path / "include").mkdir()
    (pkg / "k.cu").write_text('#include "a.cuh"\nint k;\n')
    (pkg / "a.cuh").write_text('#pragma once\n#include "../../include/x.h"\nint a;\n')
    (tmp_path / "include" / "x.h").write_text("int x;\n")
    (pkg / "unrelated.cuh").write_text("int u;\n")
    monkeypatch.setattr(bench, "ROOT", tmp_path)
    h0 = bench.kernel_source_hash("k.cu")
    (pkg / "unrelated.cuh").write_text("int u2;\n")
    assert bench.kernel_source_hash("k.cu") == h0
    (tmp_path / "include" / "x.h").write_text("// a comment\nint   x; /* and another */\n")
    assert bench.kernel_source_hash("k.cu") == h0          # comments and layout do not count
    (tmp_path / "include" / "x.h").write_text("int x2;\n")
    assert bench.kernel_source_hash("k.cu") != h0


def test_traffic_is_reported_only_for_matching_sources(monkeypatch):
    key = next(iter(bench.TRAFFIC))
    nbytes, src, digest = bench.TRAFFIC[key]
    monkeypatch.setitem(bench.TRAFFIC, key, (nbytes, src, bench.kernel_source_hash(src)))
    assert bench.traffic_for(*key) == nbytes
    monkeypatch.setitem(bench.TRAFFIC, key, (nbytes, src, "000000000000"))
    assert bench.traffic_for(*key) is None
