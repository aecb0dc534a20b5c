"""The benchmark's multi-rank logic on CPU with the gloo backend, world size 2:
the max-over-ranks step time, the whole-job throughput, and the reference arm's
rule that only rank 0 does work."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [1.5, 4.0][rank]                          # rank 1 is the slow one
        got = bench.max_over_ranks(ms, torch.device("cpu"))
        tps = bench.job_tokens_per_s(128, world, got)
        dist.barrier()
        q.put((rank, got, tps))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, tps in res:
        assert got == 4.0, "every rank sees the slowest rank's time"
        assert tps == pytest.approx(2 * 128 / 4.0e-3)


def test_single_process_is_its_own_max():
    import torch

    assert bench.max_over_ranks(2.5, torch.device("cpu")) == 2.5


def test_reference_arm_runs_on_rank_0_only(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    args = bench.argparse.Namespace(steps=3, warmup=3)
    from moe_token_routing_index_gb300 import workloads

    assert bench.run_reference(args, workloads.CONFIGS["tiny"]) is None


def test_reference_arm_prints_its_line(capsys, monkeypatch):
    import json

    monkeypatch.delenv("RANK", raising=False)
    bench.main(["--impl", "reference", "--config", "tiny", "--steps", "3", "--warmup", "3"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
