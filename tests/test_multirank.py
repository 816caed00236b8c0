"""The N > 1 host path on CPU: world size 2 over gloo (no GPU)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

from diffusion_transformer_elementwise_gb300.replicas import aggregate_gbs, max_over_ranks, row_block


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = [3.5, 7.25][rank]          # per-rank timed region, ms
        m = max_over_ranks(elapsed)
        blk = row_block(32640, rank, world)
        q.put((rank, m, blk))
    finally:
        dist.destroy_process_group()


def test_two_ranks_max_and_row_blocks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [m for _, m, _ in res] == [7.25, 7.25]
    (_, _, b0), (_, _, b1) = res
    assert b0 == (0, 16320) and b1 == (16320, 32640)


@pytest.mark.parametrize("rows,world", [(10, 3), (7, 7), (3, 5), (0, 2), (32640, 8)])
def test_row_blocks_partition(rows, world):
    blocks = [row_block(rows, r, world) for r in range(world)]
    assert blocks[0][0] == 0 and blocks[-1][1] == rows
    for (a0, a1), (b0, b1) in zip(blocks, blocks[1:]):
        assert a1 == b0
    sizes = [b - a for a, b in blocks]
    assert max(sizes) - min(sizes) <= 1


def test_aggregate_and_single_process():
    assert max_over_ranks(2.0) == 2.0  # no process group
    assert aggregate_gbs(1_000_000_000, 10, 2, 1000.0) == pytest.approx(20.0)
    with pytest.raises(ValueError):
        aggregate_gbs(1, 1, 1, 0.0)
    with pytest.raises(ValueError):
        row_block(10, 2, 2)
