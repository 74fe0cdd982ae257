"""The multi-rank logic on CPU ranks (gloo, world size 2 and 3).

Each rank owns a contiguous slab of rows and needs no exchange for y, rstd
and dx.  The cross-rank quantities are the timing (maximum over ranks) and
the weight gradient over all ranks' rows.  Checked here without a GPU: the
timing reductions of bench.py, the row sharding, and the library's own
partition of the weight gradient -- each rank takes its slab from
rms_norm_rank_rows (the C library's host function), forms the fp32 block
partials and chunk sums of its rows in the order the kernels use
(sequential over a block's rows, a fixed order over a chunk's 32 blocks),
the ranks all-gather their chunk sums, and every rank adds them in chunk
order.  That dW must equal, bit for bit, one rank doing all rows, and the
float64 oracle's dW within the dw tolerance.  (The GPU kernels' own order is
pinned against the same splits in tests/test_blocked_gpu.py.)
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


def _chunk_sums_f32(dy, x_hat, block_rows):
    """fp32 chunk sums of dy * x_hat over rows, in the kernels' order: each
    block's rows added in row order (one fp32 multiply-add per row); a
    chunk of 32 block partials p_k summed as ((s_0 + s_1) + ...) + s_15 with
    s_t = p_t + p_(t+16)."""
    rows = dy.shape[0]
    prod_terms = [(dy[r].astype(np.float32), x_hat[r].astype(np.float32)) for r in range(rows)]
    blocks = []
    for b0 in range(0, rows, block_rows):
        acc = np.zeros(dy.shape[1], np.float32)
        for d, xh in prod_terms[b0:b0 + block_rows]:
            # fma(d, xh, acc): the product is exact in float64; the sum is
            # rounded to fp32 (through float64, which an fma's single
            # rounding matches but for rare double roundings -- both sides of
            # every comparison here use this same emulation)
            acc = (d.astype(np.float64) * xh.astype(np.float64) + acc).astype(np.float32)
        blocks.append(acc)
    chunks = []
    for c0 in range(0, len(blocks), 32):
        p = blocks[c0:c0 + 32]
        p = p + [np.zeros_like(blocks[0])] * (32 - len(p))   # a missing block counts as +0
        s = [(p[t] + p[t + 16]).astype(np.float32) for t in range(16)]
        acc = s[0]
        for t in range(1, 16):
            acc = (acc + s[t]).astype(np.float32)
        chunks.append(acc)
    return chunks


def _sum_in_chunk_order(chunks):
    t = chunks[0].copy()
    for c in chunks[1:]:
        t = (t + c).astype(np.float32)
    return t


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

    # the library's partition of the weight gradient: rank slabs of whole
    # chunks, fp32 chunk sums all-gathered, added in chunk order
    import bwd_rms_norm_gb300 as L
    wb = W.LLAMA_BF16_4096x4096.with_(rows=211, hidden=48)
    brows = 2
    inp = W.make_inputs(wb)
    xd, gd, dyd = (W.as_float64(inp[k]) for k in ("x", "gamma", "dy"))
    rstd = np.float32(orm.rstd_exact(xd, wb.eps)).astype(np.float64)
    x_hat = (xd.astype(np.float32) * rstd.astype(np.float32)[:, None]).astype(np.float32)
    lo, hi = L.rms_norm_rank_rows(wb.rows, brows, world, rank)
    mine = _chunk_sums_f32(dyd[lo:hi], x_hat[lo:hi], brows) if hi > lo else []
    counts = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
    dist.all_gather(counts, torch.tensor([len(mine)], dtype=torch.int64))
    width = max(int(c.item()) for c in counts)
    pad = np.zeros((width, wb.hidden), np.float32)
    if mine:
        pad[:len(mine)] = np.stack(mine)
    gathered = [torch.zeros(width, wb.hidden, dtype=torch.float32) for _ in range(world)]
    dist.all_gather(gathered, torch.from_numpy(pad))
    chunks = [g.numpy()[i] for g, c in zip(gathered, counts) for i in range(int(c.item()))]
    dw32 = _sum_in_chunk_order(chunks)
    np.save(os.path.join(out_dir, f"blocked{rank}.npy"), np.concatenate([[lo, hi], dw32]))
    dist.destroy_process_group()


@pytest.mark.timeout(300)
@pytest.mark.parametrize("world", [2, 3])
def test_cpu_ranks(tmp_path, world):
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [np.load(tmp_path / f"rank{r}.npy") for r in range(world)]
    for r in res:
        assert r[0] == float(world)              # max over ranks of 1 + rank
        assert abs(r[1] - world * 100.0 / world) < 1e-9   # world / max(1/rate)
    # the slabs tile the rows exactly
    assert res[0][2] == 0 and res[-1][3] == 37
    for a, b in zip(res, res[1:]):
        assert a[3] == b[2]
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

    # the library's partition: slabs of whole chunks from the C library, and
    # the all-gathered fp32 chunk sums give the one-rank dW bit for bit
    import bwd_rms_norm_gb300 as L
    blk = [np.load(tmp_path / f"blocked{r}.npy") for r in range(world)]
    wb = W.LLAMA_BF16_4096x4096.with_(rows=211, hidden=48)
    spans = [(int(b[0]), int(b[1])) for b in blk]
    assert spans == [L.rms_norm_rank_rows(211, 2, world, r) for r in range(world)]
    assert spans[0][0] == 0 and spans[-1][1] == 211
    assert all(a % 64 == 0 for a, _ in spans)           # whole chunks of 32 blocks of 2 rows
    inp = W.make_inputs(wb)
    xd, gd, dyd = (W.as_float64(inp[k]) for k in ("x", "gamma", "dy"))
    rstd = np.float32(orm.rstd_exact(xd, wb.eps)).astype(np.float64)
    x_hat = (xd.astype(np.float32) * rstd.astype(np.float32)[:, None]).astype(np.float32)
    one_rank = _sum_in_chunk_order(_chunk_sums_f32(dyd, x_hat, 2))
    for b in blk:
        assert np.array_equal(b[2:].astype(np.float32), one_rank)
    _, dw_exact = orm.backward_exact(dyd, xd, gd, rstd, 0)
    scale = np.maximum(np.abs(dw_exact), np.sqrt(np.mean(dw_exact ** 2)))
    assert np.max(np.abs(one_rank - dw_exact) / scale) <= 1e-3


def test_shard_rows_cover_every_row():
    import bench
    for rows in (0, 1, 7, 4096, 16385):
        for world in (1, 2, 3, 8):
            spans = [bench.shard_rows(rows, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == rows
            for a, b in zip(spans, spans[1:]):
                assert a[1] == b[0]
