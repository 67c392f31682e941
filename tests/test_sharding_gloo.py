"""The multi-rank path on CPU: two gloo ranks each take a row shard, produce
its dropout mask with their own elem_base (through the oracle), and the
gathered shards equal the unsharded mask; the benchmark's max-over-ranks
timing reduction is checked the same way."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from elementwise_epilogues_transformer_gb300.sharding import row_shard, shard_elem_base


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, rows, cols, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle as O
        import bench
        r0, r1 = row_shard(rows, world, rank)
        base = shard_elem_base(r0, cols, global_base=12345)
        mask = O.keep_mask(1234, 7, base, (r1 - r0) * cols, 0.3)
        sizes = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(sizes, torch.tensor([mask.size], dtype=torch.int64))
        maxn = int(max(s.item() for s in sizes))
        buf = torch.zeros(maxn, dtype=torch.uint8)
        buf[:mask.size] = torch.from_numpy(mask)
        bufs = [torch.zeros(maxn, dtype=torch.uint8) for _ in range(world)]
        dist.all_gather(bufs, buf)
        t = bench.max_over_ranks(float(rank + 1) * 1.5, world)
        if rank == 0:
            gathered = np.concatenate([b[:int(s.item())].numpy() for b, s in zip(bufs, sizes)])
            q.put((gathered, t))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("rows", [7, 16])
def test_two_rank_row_shards_reproduce_unsharded_mask(rows):
    import oracle as O
    O.lib()  # build before forking workers
    world, cols = 2, 40
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, rows, cols, q)) for r in range(world)]
    for p in procs:
        p.start()
    gathered, tmax = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    full = O.keep_mask(1234, 7, 12345, rows * cols, 0.3)
    assert np.array_equal(gathered, full)
    assert tmax == 3.0


def test_row_shard_partition():
    for rows in range(0, 20):
        for world in range(1, 5):
            spans = [row_shard(rows, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == rows
            for (a, b), (c, d) in zip(spans, spans[1:]):
                assert b == c and b - a >= d - c >= b - a - 1
    with pytest.raises(ValueError):
        row_shard(4, 2, 2)
