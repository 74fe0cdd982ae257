"""The multi-rank logic of bench.py on CPU ranks (gloo, world size 2).

Each rank owns a contiguous slab of rows and needs no exchange for y, rstd
and dx.  The only cross-rank quantities are the timing (maximum over ranks)
and, when one dW over all ranks' rows is wanted, one sum of [hidden]
vectors.  Both are checked here without a GPU: the timing reductions of
bench.py, the row sharding, and that per-rank oracle dW partials summed in
rank order give the single-rank dW.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    os.environ["RANK"] = str(rank)
    os.environ["WORLD_SIZE"] = str(world)
    import bench
    import workloads as W
    from oracle import rms_norm as orm

    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, _ = bench.dist_env()
    assert (r, w) == (rank, world)
    # timing: the maximum over ranks, and the aggregate rate
    t = bench.reduce_max(1.0 + rank, world)
    rate = bench.reduce_max_rate(100.0 / (1 + rank), world, None)
    bench.barrier(world)
    # rows: contiguous slabs
    wl = W.FP32_256x1024.with_(rows=37, hidden=24)
    lo, hi = bench.shard_rows(wl.rows, rank, world)
    inp = W.make_inputs(wl)
    xd, gd, dyd = (W.as_float64(inp[k]) for k in ("x", "gamma", "dy"))
    rstd = orm.rstd_exact(xd[lo:hi], wl.eps)
    _, dw_part = orm.backward_exact(dyd[lo:hi], xd[lo:hi], gd, rstd, 0)
    parts = [torch.zeros(wl.hidden, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(parts, torch.from_numpy(dw_part))
    dw = sum(p.numpy() for p in parts)   # fixed rank order
    np.save(os.path.join(out_dir, f"rank{rank}.npy"),
            np.array([t, rate, lo, hi] + list(dw), dtype=np.float64))
    dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_cpu_ranks(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [np.load(tmp_path / f"rank{r}.npy") for r in range(world)]
    for r in res:
        assert r[0] == 2.0                       # max over ranks of 1 + rank
        assert abs(r[1] - 2 * 50.0) < 1e-9       # world / max(1/rate)
    # the slabs tile the rows exactly
    assert res[0][2] == 0 and res[0][3] == res[1][2] and res[1][3] == 37
    # per-rank partials summed in rank order give the single-rank dW
    import workloads as W
    from oracle import rms_norm as orm
    wl = W.FP32_256x1024.with_(rows=37, hidden=24)
    inp = W.make_inputs(wl)
    xd, gd, dyd = (W.as_float64(inp[k]) for k in ("x", "gamma", "dy"))
    _, dw_all = orm.backward_exact(dyd, xd, gd, orm.rstd_exact(xd, wl.eps), 0)
    for r in res:
        np.testing.assert_allclose(r[4:], dw_all, rtol=1e-12, atol=1e-12)
        assert np.array_equal(r[4:], res[0][4:])   # every rank holds the same dW


def test_shard_rows_cover_every_row():
    import bench
    for rows in (0, 1, 7, 4096, 16385):
        for world in (1, 2, 3, 8):
            spans = [bench.shard_rows(rows, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == rows
            for a, b in zip(spans, spans[1:]):
                assert a[1] == b[0]
