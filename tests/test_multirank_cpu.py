"""The bench's multi-GPU path runs independent replicas that meet only at the
timing barriers: check its max-over-ranks timing reduction and the replica
token accounting with two gloo ranks on the CPU, and that the reference arm
does no work on ranks other than 0."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [10.0 + rank, 5.0 * (rank + 1), 1.0]  # per-rank timings
        got = bench.reduce_max(ms, dist, device="cpu")
        dist.barrier()
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [11.0, 10.0, 1.0]


def test_replica_throughput_counts_every_rank():
    import bench
    # 2 replicas x 4096 tokens x 10 steps in the slowest rank's 20 ms
    assert bench.replica_throughput(4096, 10, 2, 20.0) == pytest.approx(4096 * 10 * 2 / 0.020)


def test_reference_arm_does_nothing_off_rank_zero(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps, warmup = 1, 1
    assert bench.run_reference(Args(), bench.WL.TINY) is None
    assert capsys.readouterr().out == ""
