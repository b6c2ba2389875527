"""The N>1 host path on CPU with torch.distributed (gloo, world size 2): column-tile shards cover the
output exactly once, each rank's slice of the tiled weight is a valid tiled weight whose product is
the matching columns of the full product (computed here by the oracle), and the benchmark's
max-over-ranks timing reduction."""
import os
import socket

import numpy as np
import pytest

from block_quantized_matmul_gb300 import shard, synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, type_, K, N, M, out):
    import torch.distributed as dist

    import oracle

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = synth.weights(N, K, seed=11)
        x = synth.activations(M, K, seed=12)
        tiled = oracle.repack(type_, oracle.quantize_rows(type_, w), K, N)
        a_q, a_d = oracle.quantize_act(x)
        sh = shard.shard(type_, K, N, rank, world)
        part = None
        if sh.n_local:
            sl = tiled[sh.byte_offset:sh.byte_offset + sh.byte_len]
            part, _ = oracle.matmul(type_, sl, K, sh.n_local, a_q, a_d)
        parts = [None] * world
        dist.all_gather_object(parts, (sh.n0, sh.n_local, part))
        # the benchmark's aggregation: each rank's time, max over ranks
        import torch

        t = torch.tensor([1.0 + rank], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        if rank == 0:
            full, _ = oracle.matmul(type_, tiled, K, N, a_q, a_d)
            y = np.full((M, N), np.nan)
            covered = np.zeros(N, int)
            for n0, nl, p in parts:
                if nl:
                    y[:, n0:n0 + nl] = p
                    covered[n0:n0 + nl] += 1
            out.put((bool((covered == 1).all()), bool(np.array_equal(y, full)), float(t.item())))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("type_,K,N,M", [("q4_0", 64, 100, 3), ("q8_0", 96, 33, 2), ("iq4_nl", 32, 31, 1),
                                         ("mxfp4", 64, 70, 2)])
def test_two_rank_column_shards_reassemble_the_product(type_, K, N, M):
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, type_, K, N, M, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    covered_once, equal, tmax = q.get()
    assert covered_once and equal and tmax == 2.0


def test_shard_ranges():
    for nct in (0, 1, 5, 448, 4008):
        for world in (1, 2, 3, 8):
            rs = [shard.col_tile_range(nct, r, world) for r in range(world)]
            assert rs[0][0] == 0 and rs[-1][1] == nct
            assert all(rs[i][1] == rs[i + 1][0] for i in range(world - 1))
            sizes = [b - a for a, b in rs]
            assert max(sizes) - min(sizes) <= 1
    s = shard.shard("q8_0", 4096, 128256, 3, 8)
    assert s.byte_offset == s.ct0 * 128 * 1088 and s.byte_len == (s.ct1 - s.ct0) * 128 * 1088
    last = shard.shard("q4_0", 64, 70, 1, 2)     # 3 column tiles: 2 + 1, the last one ragged
    assert (last.ct0, last.ct1, last.n0, last.n_local) == (2, 3, 64, 6)
    with pytest.raises(ValueError):
        shard.shard("q4_0", 48, 10, 0, 1)
    for t in ("q4_0", "q8_0", "iq4_nl", "mxfp4", "q4_1"):
        assert shard.tile_bytes(t) == orc_tile_bytes(t)


def orc_tile_bytes(t):
    import oracle

    return oracle.tile_bytes(t)
