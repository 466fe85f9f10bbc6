"""The N > 1 path on CPU: two gloo ranks (world size 2).

Each rank takes its shard of the rows (modulation_bit_exact_gb300.shard),
runs the operation on it (the CPU oracle stands in for the device here; the
sharding is what is tested), and the gathered shards must equal the
unsharded result bit for bit: rows are independent, so there is no
collective on the data path.  The benchmark's max-over-ranks timing
reduction is checked the same way.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from modulation_bit_exact_gb300.shard import row_shard


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _case(rows, D, mod_rows, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, D, generator=g).to(torch.bfloat16)
    sc = (0.1 * torch.randn(mod_rows, D, generator=g)).to(torch.bfloat16)
    sh = (0.1 * torch.randn(mod_rows, D, generator=g)).to(torch.bfloat16)
    u = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    return u(x), u(sc), u(sh)


def _worker(rank, world, port, rows, D, mod_rows, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        X, SC, SH = _case(rows, D, mod_rows, seed=5)
        lo, hi, mlo, mhi = row_shard(rows, mod_rows, world, rank)
        mine = oracle.ln_modulate(X[lo:hi], SC[mlo:mhi], SH[mlo:mhi], 1e-6)
        # gather (for the check only): pad to the largest shard
        n = torch.tensor([hi - lo])
        ns = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(ns, n)
        cap = int(max(t.item() for t in ns))
        buf = torch.zeros(cap, D, dtype=torch.int32)  # gloo moves 32-bit integers
        buf[:hi - lo] = torch.from_numpy(mine.astype(np.int32))
        parts = [torch.zeros(cap, D, dtype=torch.int32) for _ in range(world)]
        dist.all_gather(parts, buf)
        import bench
        t_max = bench.max_over_ranks(10.0 + rank, dist, "cpu")
        if rank == 0:
            got = np.concatenate([p[:int(c.item())].numpy() for p, c in zip(parts, ns)]).astype(np.uint16)
            q.put((got, t_max))
        else:
            q.put((None, t_max))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("rows,mod_rows", [(64, 64), (96, 4), (70, 1)])
def test_two_rank_shards_equal_the_whole(rows, mod_rows):
    world, D = 2, 256
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, rows, D, mod_rows, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=90) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    import oracle
    X, SC, SH = _case(rows, D, mod_rows, seed=5)
    want = oracle.ln_modulate(X, SC, SH, 1e-6)
    got = [r[0] for r in results if r[0] is not None][0]
    assert np.array_equal(got, want)
    assert all(r[1] == 11.0 for r in results)  # the slowest rank's time, on every rank


def test_row_shard_rules():
    # per-token: any contiguous split, the first ranks one row more
    assert [row_shard(10, 10, 3, r) for r in range(3)] == [(0, 4, 0, 4), (4, 7, 4, 7), (7, 10, 7, 10)]
    # whole samples
    assert [row_shard(40, 4, 2, r) for r in range(2)] == [(0, 20, 0, 2), (20, 40, 2, 4)]
    # inside one sample
    assert [row_shard(40, 2, 4, r) for r in range(4)] == [(0, 10, 0, 1), (10, 20, 0, 1), (20, 30, 1, 2),
                                                          (30, 40, 1, 2)]
    with pytest.raises(ValueError):
        row_shard(30, 3, 2, 0)
    # every split covers the rows exactly once, in order
    for rows, mod_rows, world in ((8704, 2, 8), (8704, 2, 1), (32760, 32760, 8), (4352 * 4, 4, 2)):
        spans = [row_shard(rows, mod_rows, world, r) for r in range(world)]
        assert spans[0][0] == 0 and spans[-1][1] == rows
        assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
        seq = rows // mod_rows
        for lo, hi, mlo, mhi in spans:
            assert mlo == lo // seq and mhi == (hi - 1) // seq + 1
