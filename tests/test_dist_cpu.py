"""The bench's N > 1 path on CPU: two gloo ranks, each with its own timed
region, aggregated as the slowest rank's time (MAX all-reduce) and whole-job
tokens/s = ranks x steps over it (weak scaling: independent token streams per
rank, no collective on the data path)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, dev_ms, e2e_ms, K, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        res = bench.aggregate_over_ranks(dev_ms[rank], e2e_ms[rank], K, world, "cpu")
        out.put((rank, res))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("with_e2e", [True, False])
def test_two_ranks_take_the_slowest(with_e2e):
    world, K = 2, 448
    dev_ms = [600.0, 655.5]
    e2e_ms = [1.40, 1.55] if with_e2e else [None, None]
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, dev_ms, e2e_ms, K, out)) for r in range(world)]
    for p in procs:
        p.start()
    results = dict(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(world):
        dev_max, value, e2e_value = results[r]
        assert dev_max == 655.5
        assert value == pytest.approx(world * K / 0.6555)
        if with_e2e:
            assert e2e_value == pytest.approx(world * 1e3 / 1.55)
        else:
            assert e2e_value is None


def test_one_rank_needs_no_process_group():
    assert not dist.is_initialized()
    dev_max, value, e2e_value = bench.aggregate_over_ranks(700.0, 1.5, 448, 1, "cpu")
    assert dev_max == 700.0 and value == pytest.approx(640.0) and e2e_value == pytest.approx(1e3 / 1.5)
