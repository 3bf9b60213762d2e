"""Sequence-sharded decode on one GPU, as virtual ranks, through the C ABI.

Each virtual rank holds one shard of the cache (dcp.shard_cache), runs
paged_decode_global_partial over it, and paged_decode_combine merges the
stacked partials -- the data an all-gather would hand every rank. Compared
with the fp64 oracle's unsharded decode at the decode bar (max |err| <= 2e-2,
cosine > 0.9995); one rank's partial (fp32 output and log-sum-exp) is compared
with the oracle on that shard alone.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_global_gb300 import binding as b
from paged_gqa_decode_global_gb300 import dcp
from paged_gqa_decode_global_gb300 import inputs as synth

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
MIN_COS = 0.9995


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _desc(li, num_pages, max_pages):
    return b.layer_desc(li.num_q_heads, li.num_kv_heads, li.head_dim, li.page_size, num_pages, max_pages, 0,
                        li.v_pool is None)


def _partial(li, k, v, table, lens, early_kv=False):
    step = dcp.PartialStep(_desc(li, k.shape[0], table.shape[1]), lens.tolist(), _sms(), "cuda", early_kv=early_kv)
    o, lse = step(li.q, k, v, table, lens, li.scale)
    torch.cuda.synchronize()
    return o, lse


def _full_oracle(li):
    return oracle.decode(synth.bits_u16(li.q), synth.bits_u16(li.k_pool),
                         None if li.v_pool is None else synth.bits_u16(li.v_pool), li.block_tables.cpu().numpy(),
                         li.seq_lens.cpu().numpy(), li.scale, 0)


def _compare(got, exp, tag):
    got = got.float().cpu().double().numpy()
    assert np.isfinite(got).all(), tag
    err = np.abs(got - exp).max()
    g, r = got.ravel(), exp.ravel()
    cos = float(g @ r / (np.linalg.norm(g) * np.linalg.norm(r)))
    assert err <= MAX_ABS, f"{tag}: max abs {err:.3e}"
    assert cos > MIN_COS, f"{tag}: cosine {cos:.7f}"


CASES = [(512, 16, 4, False), (512, 16, 4, True), (256, 16, 8, False)]
LENS = [1, 17, 300, 0, 2000, 4096]


@pytest.mark.parametrize("d,Hq,Hkv,kvs", CASES, ids=["d512-KneV", "d512-K=V", "d256-KneV"])
@pytest.mark.parametrize("R", [1, 2, 3, 4])
@pytest.mark.parametrize("mode", dcp.MODES)
def test_virtual_ranks_reassemble_the_decode(d, Hq, Hkv, kvs, R, mode):
    pool = sum((L + 15) // 16 for L in LENS) + 3
    li = synth.make_layer("dcp", LENS, Hq, Hkv, d, kv_shared=kvs, pool_pages=pool, seed=d + R, device="cuda")
    os_, lses = [], []
    for r in range(R):
        k, v, table, lens = dcp.shard_cache(li.k_pool, li.v_pool, li.block_tables, LENS, R, r, mode)
        o, lse = _partial(li, k, v, table, lens)
        os_.append(o)
        lses.append(lse)
    out = dcp.combine(torch.stack(os_), torch.stack(lses))
    torch.cuda.synchronize()
    _compare(out, _full_oracle(li), f"R={R} {mode}")
    assert (out[3].float() == 0).all()  # the empty request


def test_partial_matches_the_oracle_on_one_shard():
    pool = sum((L + 15) // 16 for L in LENS) + 3
    li = synth.make_layer("dcp", LENS, 16, 4, 512, pool_pages=pool, seed=3, device="cuda")
    k, v, table, lens = dcp.shard_cache(li.k_pool, li.v_pool, li.block_tables, LENS, 2, 1, "interleaved")
    o, lse = _partial(li, k, v, table, lens)
    exp_o, exp_lse = oracle.decode(synth.bits_u16(li.q), synth.bits_u16(k), synth.bits_u16(v), table.cpu().numpy(),
                                   lens.cpu().numpy(), li.scale, 0, return_lse=True)
    _compare(o, exp_o, "partial o")
    got_lse = lse.cpu().double().numpy()
    empty = ~np.isfinite(exp_lse)
    assert (np.isneginf(got_lse) == empty).all()  # request 0 (one token, on rank 0) and request 3 hold none here
    assert np.abs(got_lse[~empty] - exp_lse[~empty]).max() <= 5e-3 + 1e-3 * np.abs(exp_lse[~empty]).max()
    assert (o[torch.from_numpy(empty).cuda()] == 0).all()


def test_partial_plan_rules():
    desc = b.layer_desc(16, 4, 512, 16, 100, 64)
    pl = b.paged_decode_plan_partial(desc, [16], _sms())
    assert pl.partial == 1 and pl.merge_mode == 1 and pl.num_splits == 1  # fp32 pieces even for one piece
    win = b.layer_desc(16, 4, 512, 16, 100, 64, window=128)
    with pytest.raises(b.PagedDecodeError) as e:
        b.paged_decode_plan_partial(win, [16], _sms())
    assert e.value.status == b.PD_ERR_UNSUPPORTED


def test_early_kv_ranks_back_to_back():
    """The virtual ranks' partials with early_kv, queued back to back with no
    host sync (each rank's stage 1 copying while the previous rank's launches
    drain), then combined: equal to the unsharded oracle."""
    R = 3
    pool = sum((L + 15) // 16 for L in LENS) + 3
    li = synth.make_layer("dcp", LENS, 16, 4, 512, pool_pages=pool, seed=41, device="cuda")
    shards = [dcp.shard_cache(li.k_pool, li.v_pool, li.block_tables, LENS, R, r, "interleaved") for r in range(R)]
    steps = [dcp.PartialStep(_desc(li, k.shape[0], t.shape[1]), n.tolist(), _sms(), "cuda", early_kv=True)
             for k, _, t, n in shards]
    outs = [step(li.q, k, v, t, n, li.scale) for step, (k, v, t, n) in zip(steps, shards)]
    out = dcp.combine(torch.stack([o for o, _ in outs]), torch.stack([lse for _, lse in outs]))
    torch.cuda.synchronize()
    _compare(out, _full_oracle(li), "early_kv ranks")
