"""The N > 1 host path of the benchmark, on CPU with gloo and two ranks: the
whole-job time is the max over ranks and the bytes are summed, so the value
is the aggregate over independent replicas."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        sec, nbytes = bench.aggregate_ranks(1.0 + rank, 1000.0 * (rank + 1))
        q.put((rank, sec, nbytes, bench.dist_env()))
    finally:
        dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, sec, nbytes, env in got:
        assert sec == 2.0            # max over ranks
        assert nbytes == 3000.0      # sum over ranks
        assert env[0] == rank and env[1] == 2


def test_single_process_is_identity():
    import bench
    assert bench.aggregate_ranks(1.5, 10.0) == (1.5, 10.0)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"]) == 0
    assert capsys.readouterr().out == ""
