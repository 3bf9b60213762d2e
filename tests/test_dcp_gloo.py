"""The sequence-sharded path on the host: two gloo ranks, no GPU.

Each rank lays out its shard of the cache with ``dcp.shard_cache``, computes
its partial (output + log-sum-exp) with the fp64 oracle, the ranks exchange
the partials with ``dcp.exchange_partials`` (one all-gather), and each merges
them with the oracle's merge: the result must equal the oracle's unsharded
decode. This checks the shard layout (every cached row on exactly one rank, in
position order) and the exchange protocol; the GPU kernels of the same steps
are checked on one GPU as virtual ranks.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LENS = [1, 17, 300, 0, 64]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _layer(kv_shared):
    from paged_gqa_decode_global_gb300 import inputs as synth
    pool = sum((L + 15) // 16 for L in LENS) + 4
    return synth.make_layer("dcp", LENS, 8, 2, 64, kv_shared=kv_shared, pool_pages=pool, seed=7)


def _rank_main(rank, world, port, mode, kv_shared, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import oracle
    from paged_gqa_decode_global_gb300 import dcp
    from paged_gqa_decode_global_gb300 import inputs as synth
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        li = _layer(kv_shared)
        k, v, table, lens = dcp.shard_cache(li.k_pool, li.v_pool, li.block_tables, LENS, world, rank, mode)
        o, lse = oracle.decode(synth.bits_u16(li.q), synth.bits_u16(k), None if v is None else synth.bits_u16(v),
                               table.numpy(), lens.numpy(), li.scale, 0, return_lse=True)
        o_all, lse_all = dcp.exchange_partials(torch.from_numpy(o), torch.from_numpy(lse))
        merged = oracle.merge(np.moveaxis(o_all.numpy(), 0, -2), np.moveaxis(lse_all.numpy(), 0, -1))
        full = oracle.decode(synth.bits_u16(li.q), synth.bits_u16(li.k_pool),
                             None if li.v_pool is None else synth.bits_u16(li.v_pool), li.block_tables.numpy(),
                             li.seq_lens.numpy(), li.scale, 0)
        q.put((rank, float(np.abs(merged - full).max()), int(lens.sum())))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("mode,kv_shared", [("interleaved", False), ("contiguous", False), ("interleaved", True)])
def test_two_ranks_reassemble_the_unsharded_decode(mode, kv_shared):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, mode, kv_shared, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, err, held in res:
        assert err <= 1e-12, (rank, err)
    assert sum(h for _, _, h in res) == sum(LENS)  # every cached row on exactly one rank


@pytest.mark.parametrize("R", [1, 2, 3, 5])
@pytest.mark.parametrize("mode", ["interleaved", "contiguous"])
def test_shards_partition_each_request_in_order(R, mode):
    from paged_gqa_decode_global_gb300 import dcp
    li = _layer(False)
    seen = {b: [] for b in range(len(LENS))}
    for r in range(R):
        k, v, table, lens = dcp.shard_cache(li.k_pool, li.v_pool, li.block_tables, LENS, R, r, mode)
        for b, L in enumerate(LENS):
            pos = dcp.shard_positions(L, R, r, mode)
            assert int(lens[b]) == len(pos)
            for i, t in enumerate(pos):
                src = li.k_pool[int(li.block_tables[b, t // 16]), :, t % 16, :]
                dst = k[int(table[b, i // 16]), :, i % 16, :]
                assert torch.equal(src, dst)
                assert torch.equal(li.v_pool[int(li.block_tables[b, t // 16]), :, t % 16, :],
                                   v[int(table[b, i // 16]), :, i % 16, :])
            seen[b] += pos
    for b, L in enumerate(LENS):
        assert sorted(seen[b]) == list(range(L))
