"""The multi-rank path of bench.py on CPU: two gloo ranks (the replicas of
--gpus 2 share nothing but the timing reduction), and the reference arm, which
only rank 0 runs."""
import os
import socket

import pytest

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r measured (r + 1) ms device time and (10 - r) ms end to end
        got = bench.max_over_ranks([rank + 1.0, 10.0 - rank], dist, "cpu")
        dist.barrier()
    finally:
        dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(" ".join(str(v) for v in got))


def test_max_over_ranks_gloo_world_size_2(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    for r in range(2):
        vals = [float(v) for v in (tmp_path / f"rank{r}.txt").read_text().split()]
        assert vals == [2.0, 10.0]  # every rank sees the slowest rank's times


def test_max_over_ranks_without_a_group():
    assert bench.max_over_ranks([3, 4.5]) == [3.0, 4.5]


def test_replica_value_is_all_ranks_work_over_the_slowest_time():
    class W(bench.Workload):
        def groups(self):
            return [("g", None, 2e12, 0, "tensor")]  # 2 TFLOP per step and rank
    # 4 ranks, slowest 10 ms per step: 4 x 2e12 / 0.010 s = 800 TFLOP/s
    assert W().value(10.0) * 4 == pytest.approx(800.0)


def test_reference_arm_runs_on_rank_0_only(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")

    class Args:
        workload = "resnet3x3"
        steps = 3
        warmup = 3
    assert bench.run_reference(Args()) == 0
    assert capsys.readouterr().out == ""
