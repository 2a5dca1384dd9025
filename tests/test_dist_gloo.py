"""World-size-2 gloo tests of the multi-rank host logic, on CPU: the weight-sync
sharding plans keep the quantized bytes identical to the unsharded quantization
("End-to-End MXFP8 RL on Blackwell", section "The grid, byte for byte"), and the
benchmark's max-over-ranks timing reduction. The per-rank quantizer here is the CPU
oracle standing in for the GPU kernel (no GPU on this path)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from mxfp8_block_scaled_05_gb300.sharding import assign_weights, row_shards


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _weights():
    g = np.random.default_rng(0)
    shapes = [(300, 64), (128, 96), (64, 32), (512, 128), (96, 256)]
    out = []
    for r, c in shapes:
        f = (g.standard_normal((r, c)) * 0.02).astype(np.float32).view(np.uint32)
        out.append(((f + 0x7FFF + ((f >> 16) & 1)) >> 16).astype(np.uint16))
    return out


def _worker(rank, world, port, results):
    import oracle.mxfp8_oracle as O
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws = _weights()
        # whole-weight plan: each rank quantizes its weights, rank 0 gathers
        plan = assign_weights([w.size for w in ws], world)
        mine = {i: O.quantize(ws[i], O.ROW) for i in plan[rank]}
        gathered = [None] * world
        dist.all_gather_object(gathered, mine)
        # row-shard plan of the largest weight, swizzled scales
        big = ws[0]
        lo, hi = row_shards(big.shape[0], world)[rank]
        c, s = O.quantize(big[lo:hi], O.ROW)
        part = (c, O.swizzle_scales(s) if hi > lo else np.zeros(0, np.uint8))
        parts = [None] * world
        dist.all_gather_object(parts, part)
        # timing reduction used by the benchmark
        slowest = bench.max_over_ranks(1.0 + rank, world)
        if rank == 0:
            merged = {}
            for d in gathered:
                merged.update(d)
            ok_whole = sorted(merged) == list(range(len(ws))) and all(
                np.array_equal(merged[i][0], O.quantize(ws[i], O.ROW)[0]) and
                np.array_equal(merged[i][1], O.quantize(ws[i], O.ROW)[1]) for i in merged)
            cw, sw = O.quantize(big, O.ROW)
            ok_rows = (np.array_equal(np.concatenate([p[0] for p in parts]), cw) and
                       np.array_equal(np.concatenate([p[1] for p in parts]), O.swizzle_scales(sw)))
            results.put((ok_whole, ok_rows, slowest))
    finally:
        dist.destroy_process_group()


def test_sharded_sync_pass_world2():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    ok_whole, ok_rows, slowest = q.get()
    assert ok_whole and ok_rows
    assert slowest == 2.0


def test_row_shards_and_assignment():
    assert row_shards(300, 2) == [(0, 256), (256, 300)]
    assert row_shards(128, 3) == [(0, 128), (128, 128), (128, 128)]
    assert row_shards(0, 2) == [(0, 0), (0, 0)]
    for rows in (1, 127, 129, 4096, 24576, 1000):
        for world in (1, 2, 3, 8):
            sh = row_shards(rows, world)
            assert sh[0][0] == 0 and sh[-1][1] == rows
            assert all(a[1] == b[0] for a, b in zip(sh, sh[1:]))
            assert all(lo % 128 == 0 or lo == rows for lo, _ in sh)
    plan = assign_weights([10, 7, 7, 3, 1], 2)
    assert sorted(sum(plan, [])) == [0, 1, 2, 3, 4]
    loads = [sum([10, 7, 7, 3, 1][i] for i in p) for p in plan]
    assert max(loads) - min(loads) <= 3
    with pytest.raises(ValueError):
        row_shards(10, 0)
