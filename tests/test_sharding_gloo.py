"""The multi-rank path on the CPU: two gloo ranks. Head sharding is exact (each rank runs
the oracle on its block of heads; the gathered blocks equal the unsharded run) and needs
no collective on the data path; the bench's rank helpers (barrier, max over ranks) work
on gloo. CPU only."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from linear_attention_serving_02_gb300 import inputs, sharding


def test_head_range_partitions():
    for H in (0, 1, 5, 12, 96):
        for world in (1, 2, 3, 8):
            blocks = [sharding.head_range(H, r, world) for r in range(world)]
            assert blocks[0][0] == 0 and blocks[-1][1] == H
            for (a0, a1), (b0, b1) in zip(blocks, blocks[1:]):
                assert a1 == b0
            sizes = [h1 - h0 for h0, h1 in blocks]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        sharding.head_range(4, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, result_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        import bench

        T, H, N = 40, 5, 2
        full = inputs.prefill_inputs(T, H, N, seed=3, init_state=True, batch_rows=N)
        mine = sharding.shard_heads(full, rank, world, H)
        o, S = oracle.kda_forward(mine["q"], mine["k"], mine["v"], mine["z"], mine["A"], mine["b"], S0=mine["S0"])
        # gather the blocks on every rank (test side only: the data path has no collective)
        h0, h1 = sharding.head_range(H, rank, world)
        blocks_o = [None] * world
        blocks_s = [None] * world
        dist.all_gather_object(blocks_o, (h0, h1, o))
        dist.all_gather_object(blocks_s, (h0, h1, S))
        # the bench's rank helpers on gloo
        bench.barrier(world)
        m = bench.max_over_ranks(float(rank + 1), world)
        if rank == 0:
            o_ref, S_ref = oracle.kda_forward(full["q"], full["k"], full["v"], full["z"], full["A"], full["b"],
                                              S0=full["S0"])
            o_cat = np.concatenate([b[2] for b in sorted(blocks_o, key=lambda x: x[0])], axis=-2)
            S_cat = np.concatenate([b[2] for b in sorted(blocks_s, key=lambda x: x[0])], axis=1)
            ok = bool(np.array_equal(o_cat, o_ref) and np.array_equal(S_cat, S_ref) and m == float(world))
            with open(os.path.join(result_dir, "ok"), "w") as f:
                f.write("1" if ok else "0")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_head_shards_match_unsharded(tmp_path):
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, str(tmp_path))) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0, "rank exited with %s" % p.exitcode
    assert (tmp_path / "ok").read_text() == "1"
