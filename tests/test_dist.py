"""The N>1 path of the benchmark on CPU ranks (gloo, world size 2).

Each rank runs an independent replica of the step (the MX GEMM shards by
problem: no collective touches the data path), so the only cross-rank
steps are the barrier and taking the slowest rank's time.  These tests run
that host logic with two gloo ranks and check the aggregate, and that the
reference arm does its work on rank 0 only."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, local_ms, out):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms = bench.max_over_ranks(local_ms[rank], world)
        tf = bench.job_throughput(2.0 * 8192 ** 3, world, ms)
        dist.barrier()
        out[rank] = (ms, tf)
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_throughput():
    world = 2
    local_ms = [0.61, 0.47]
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), local_ms, out), nprocs=world,
             join=True)
    for r in range(world):
        ms, tf = out[r]
        assert ms == pytest.approx(0.61)                 # slowest rank
        assert tf == pytest.approx(2 * 2.0 * 8192 ** 3 / 0.61e-3 / 1e12)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.5, 1) == 0.5
    assert bench.job_throughput(1e12, 1, 1.0) == pytest.approx(1000.0)


def test_reference_arm_only_on_rank_zero(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    called = []
    monkeypatch.setattr(bench, "run_reference",
                        lambda args: called.append(1) or {"impl": "reference"})
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.main(["--impl", "reference"])
    assert not called and capsys.readouterr().out == ""
    monkeypatch.setenv("RANK", "0")
    bench.main(["--impl", "reference"])
    assert called == [1] and '"impl": "reference"' in capsys.readouterr().out


def test_both_arms_print_the_same_metric():
    """The driver divides our line by the reference arm's only when metric,
    unit and direction agree; the reference line also carries ms_per_step so
    that its timing can be checked against the run's wall clock."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    args = bench.parse_args(["--impl", "reference", "--workload", "mx256",
                             "--steps", "2", "--warmup", "0",
                             "--ref-budget", "2"])
    ref = bench.run_reference(args)
    c = workloads.case("mx256")
    assert ref["metric"] == bench.metric_name(c)
    assert ref["unit"] == "TFLOP/s" and ref["higher_is_better"] is True
    assert ref["steps"] == 2 and ref["ms_per_step"] > 0
    assert ref["step"] == bench.step_description(c)
    assert ref["cpu_baseline"]["value"] == ref["value"]
