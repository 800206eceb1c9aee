"""The bench's N > 1 path on CPU: two gloo ranks (replicas only: the layer has no
data-path collective, the job's time is the slowest rank's), and the reference
arm runs on rank 0 alone."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_path):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    got = bench.max_over_ranks([10.0 + rank, 5.0 - rank, 3.0], torch.device("cpu"))
    dist.barrier()
    dist.destroy_process_group()
    with open(f"{out_path}.{rank}", "w") as f:
        f.write(repr(got))


def test_max_over_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    out = str(tmp_path / "res")
    mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    for r in range(2):
        assert eval(open(f"{out}.{r}").read()) == [11.0, 5.0, 3.0]   # every rank sees the slowest rank's time


def test_max_over_ranks_without_a_process_group():
    import bench
    assert bench.max_over_ranks([1.5, 2.5], torch.device("cpu")) == [1.5, 2.5]


def test_reference_arm_prints_nothing_on_other_ranks(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")

    class A:
        steps, warmup, ref_calls_per_step = 1, 3, 1
    bench.run_reference(A())
    assert capsys.readouterr().out == ""
