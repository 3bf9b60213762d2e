"""Pins the multi-token oracle (T new tokens per request, causal over the
paged cache) to things other than itself (CPU only):

* a library routine: torch's scaled_dot_product_attention in float64 on a
  dense, de-paged copy of K/V with an explicit boolean causal (and window)
  mask and explicit GQA head expansion;
* a special case that reduces to the pinned decode oracle: query token j
  equals single-token decode at length L - T + 1 + j, bit for bit; T = 1 is
  decode.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_global_gb300 import inputs as synth


def _multi_layer(lens, T, Hq, Hkv, d, window=0, kv_shared=False, P=16, seed=0):
    pool = sum((L + P - 1) // P for L in lens) + 3
    li = synth.make_layer("m", lens, Hq, Hkv, d, window=window, kv_shared=kv_shared, pool_pages=pool,
                          page_size=P, seed=seed)
    g = torch.Generator().manual_seed(seed + 5)
    q = torch.randn(len(lens), T, Hq, d, generator=g).to(torch.bfloat16)
    return li, q


def _multi(li, q):
    return oracle.decode_multi(synth.bits_u16(q), synth.bits_u16(li.k_pool),
                               None if li.v_pool is None else synth.bits_u16(li.v_pool), li.block_tables.numpy(),
                               li.seq_lens.numpy(), li.scale, li.window)


def _dense(li, pool, b):
    L = int(li.seq_lens[b])
    P = li.page_size
    rows = [pool[int(li.block_tables[b, t // P]), :, t % P, :].to(torch.float64) for t in range(L)]
    return torch.stack(rows, dim=1)  # [Hkv, L, d]


@pytest.mark.parametrize("d,G,W,T,P,kvs", [(8, 2, 0, 4, 16, False), (8, 4, 5, 3, 2, False), (256, 1, 17, 5, 16, True),
                                           (8, 8, 0, 1, 16, False), (16, 2, 3, 6, 1, False)])
def test_multi_matches_library_sdpa_with_causal_mask(d, G, W, T, P, kvs):
    lens = [T, T + 9, 40, 3 * T + 1]
    li, q = _multi_layer(lens, T, 2 * G, 2, d, window=W, kv_shared=kvs, P=P, seed=d + G + W + T)
    got = _multi(li, q)
    vpool = li.k_pool if li.v_pool is None else li.v_pool
    for b, L in enumerate(lens):
        K = _dense(li, li.k_pool, b).repeat_interleave(G, dim=0)
        V = _dense(li, vpool, b).repeat_interleave(G, dim=0)
        pos = torch.arange(L - T, L)[:, None]
        t = torch.arange(L)[None, :]
        allowed = t <= pos
        if W > 0:
            allowed &= t > pos - W
        qd = q[b].to(torch.float64).transpose(0, 1)  # [Hq, T, d]
        ref = torch.nn.functional.scaled_dot_product_attention(qd, K, V, attn_mask=allowed, scale=li.scale)
        np.testing.assert_allclose(got[b], ref.transpose(0, 1).numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("W", [0, 7])
def test_token_j_is_decode_at_its_own_length(W):
    T = 5
    lens = [5, 12, 33]
    li, q = _multi_layer(lens, T, 8, 2, 64, window=W, seed=3)
    got = _multi(li, q)
    for j in range(T):
        lens_j = np.array([L - T + 1 + j for L in lens], dtype=np.int32)
        ref = oracle.decode(synth.bits_u16(q[:, j]), synth.bits_u16(li.k_pool), synth.bits_u16(li.v_pool),
                            li.block_tables.numpy(), lens_j, li.scale, W)
        np.testing.assert_array_equal(got[:, j], ref)


def test_one_token_is_decode():
    li, q = _multi_layer([17, 40], 1, 4, 2, 32, seed=9)
    ref = oracle.decode(synth.bits_u16(q[:, 0]), synth.bits_u16(li.k_pool), synth.bits_u16(li.v_pool),
                        li.block_tables.numpy(), li.seq_lens.numpy(), li.scale, 0)
    np.testing.assert_array_equal(_multi(li, q)[:, 0], ref)


def test_length_below_token_count_is_refused():
    li, q = _multi_layer([3, 10], 4, 4, 2, 8)
    with pytest.raises(oracle.OracleError):
        _multi(li, q)
