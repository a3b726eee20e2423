"""Multi-rank bench logic on CPU (gloo, world_size 2): the ranks are
independent replicas; the whole-job value uses the slowest rank's time and
counts the tokens of every rank."""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    bench.barrier(ws)
    ms = 100.0 if rank == 0 else 250.0  # the slower rank decides
    value, ms_max = bench.whole_job_tokens_per_s(ms, ws, steps=10, tokens_per_step=64, device="cpu")
    bench.barrier(ws)
    q.put((rank, value, ms_max))
    dist.destroy_process_group()


def test_whole_job_value_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, value, ms_max in got:
        assert ms_max == pytest.approx(250.0)
        assert value == pytest.approx(2 * 10 * 64 / 0.25)


def test_single_rank_value():
    import bench
    value, ms = bench.whole_job_tokens_per_s(50.0, 1, steps=4, tokens_per_step=8, device="cpu")
    assert ms == 50.0 and value == pytest.approx(4 * 8 / 0.05)
