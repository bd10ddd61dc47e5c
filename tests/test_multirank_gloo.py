"""Multi-rank host logic of bench.py on CPU: two gloo ranks.

Each rank drafts its own batch (weak scaling); the only cross-rank traffic is
the barrier and the max of the step time.  No GPU is used.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    bench.dist_init(w, "gloo")
    bench.barrier(w)
    step_s = 0.010 + 0.005 * rank          # rank 1 is the slow one
    slowest = bench.reduce_scalar(step_s, w, "max")
    total_units = bench.reduce_scalar(512.0, w, "sum")
    value = bench.aggregate(512, slowest, w)
    # seeds of the ranks' batches differ: independent problems per rank
    seed = bench.workload("tiny_f32", r).seed
    out.put((rank, slowest, total_units, value, seed))
    import torch.distributed as dist
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_aggregate_weak_scaling():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=90) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    (r0, s0, u0, v0, seed0), (r1, s1, u1, v1, seed1) = res
    assert s0 == s1 == pytest.approx(0.015)          # max over ranks
    assert u0 == u1 == 1024.0
    assert v0 == v1 == pytest.approx(2 * 512 / 0.015)
    assert seed0 != seed1


def test_reference_arm_runs_on_rank_zero_only(capsys, monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.run_reference(bench.parse_args(["--impl", "reference", "--workload", "tiny_f32"]), 1, 2)
    assert capsys.readouterr().out == ""


def test_reference_arm_prints_one_json_line(capsys):
    import json

    import bench
    bench.run_reference(bench.parse_args(["--impl", "reference", "--workload", "tiny_f32", "--steps", "2",
                                          "--warmup", "1"]), 0, 1)
    lines = capsys.readouterr().out.strip().splitlines()
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "block-tokens/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
