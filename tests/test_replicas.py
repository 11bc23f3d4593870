"""CPU: the multi-GPU path of the benchmark is N independent replicas (one
process per GPU, no data exchange); its whole-job figures are the slowest
rank's time and the sum of every rank's units. Checked here with two gloo
processes on the host, and the reference arm's non-zero ranks do no work."""

import json
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir, secs, units):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        t, u = bench.aggregate_over_ranks(world, secs[rank], units[rank], "cpu")
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"t": t, "u": u}, f)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_replica_aggregation_over_gloo(tmp_path, world):
    secs = [0.25, 1.5, 0.75][:world]
    units = [1000, 2500, 40][:world]
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path), secs, units), nprocs=world,
             join=True)
    for r in range(world):
        got = json.load(open(tmp_path / f"r{r}.json"))
        assert got["t"] == max(secs)           # the slowest rank sets the time
        assert got["u"] == float(sum(units))   # units of every rank count


def test_single_rank_is_identity():
    import bench
    assert bench.aggregate_over_ranks(1, 0.5, 7, "cpu") == (0.5, 7)


def test_reference_arm_nonzero_rank_does_nothing(capsys):
    import bench

    class Args:
        pass

    assert bench.run_reference(Args(), 1, 2) is None
    assert capsys.readouterr().out == ""
