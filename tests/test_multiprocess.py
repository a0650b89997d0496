"""The N > 1 host path of bench.py on CPU: two gloo ranks on 127.0.0.1.

Each rank holds its own step times; the whole job's time is the slowest
rank's (max over ranks), which every rank must receive.  The reference arm
runs on rank 0 only; other ranks return without work.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = [1e-3 * (rank + 1), 2e-3 * (world - rank)]
    got = bench.max_over_ranks(mine, "cpu")
    out[rank] = got
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_gloo(world):
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    want = [1e-3 * world, 2e-3 * world]
    for r in range(world):
        assert out[r] == pytest.approx(want)


def test_reference_arm_other_ranks_do_no_work(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    args = type("A", (), {"steps": 1, "warmup": 0, "gpus": 2})()
    bench.run_reference(args)
    assert capsys.readouterr().out == ""
