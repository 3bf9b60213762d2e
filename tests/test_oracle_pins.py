"""Pins the fp64 oracle to things other than itself (CPU only).

* a library routine: torch's scaled_dot_product_attention in float64 over a
  dense, de-paged copy of K/V with an explicit boolean mask and explicit GQA
  head expansion;
* closed forms (L = 1, q = 0, equal keys, one dominant key) and hand-derived
  examples stored under tests/golden;
* invariants: window mask, page permutation, split + log-sum-exp merge,
  log-sum-exp of the scores.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_global_gb300 import inputs as synth

HERE = os.path.dirname(os.path.abspath(__file__))


def _layer(lens, Hq, Hkv, d, window=0, kv_shared=False, P=16, seed=0, extra_pages=3, q_std=1.0):
    pool = sum((L + P - 1) // P for L in lens) + extra_pages
    return synth.make_layer("t", lens, Hq, Hkv, d, window=window, kv_shared=kv_shared,
                            pool_pages=pool, page_size=P, seed=seed, q_std=q_std)


def _oracle(ly, **kw):
    return oracle.decode(synth.bits_u16(ly.q), synth.bits_u16(ly.k_pool),
                         None if ly.v_pool is None else synth.bits_u16(ly.v_pool),
                         ly.block_tables.numpy(), ly.seq_lens.numpy(), ly.scale, ly.window, **kw)


def _dense_kv(ly, pool, b):
    """Contiguous [Hkv, L, d] float64 copy of request b's cached rows."""
    L = int(ly.seq_lens[b])
    P = ly.page_size
    rows = []
    for t in range(L):
        page = int(ly.block_tables[b, t // P])
        rows.append(pool[page, :, t % P, :].to(torch.float64))
    if not rows:
        return torch.zeros(ly.num_kv_heads, 0, ly.head_dim, dtype=torch.float64)
    return torch.stack(rows, dim=1)


def _sdpa_reference(ly):
    """Library attention in float64 with an explicit window mask."""
    out = torch.zeros(ly.batch, ly.num_q_heads, ly.head_dim, dtype=torch.float64)
    G = ly.num_q_heads // ly.num_kv_heads
    vpool = ly.k_pool if ly.v_pool is None else ly.v_pool
    for b in range(ly.batch):
        L = int(ly.seq_lens[b])
        if L == 0:
            continue
        K = _dense_kv(ly, ly.k_pool, b).repeat_interleave(G, dim=0)  # [Hq, L, d]
        V = _dense_kv(ly, vpool, b).repeat_interleave(G, dim=0)
        q = ly.q[b].to(torch.float64).unsqueeze(1)                    # [Hq, 1, d]
        pos = torch.arange(L)
        keep = pos >= (L - ly.window) if ly.window > 0 else torch.ones(L, dtype=torch.bool)
        mask = keep.view(1, 1, L).expand(ly.num_q_heads, 1, L)
        o = torch.nn.functional.scaled_dot_product_attention(q, K, V, attn_mask=mask, scale=ly.scale)
        out[b] = o[:, 0, :]
    return out.numpy()


CASES = []
for d in (8, 256):
    for G in (1, 2, 4):
        for W in (0, 5, 16, 17):
            CASES.append((d, G, W))


@pytest.mark.parametrize("d,G,W", CASES)
def test_matches_library_sdpa(d, G, W):
    Hkv = 2
    ly = _layer([37, 64], Hkv * G, Hkv, d, window=W, seed=d * 100 + G * 10 + W)
    got = _oracle(ly)
    ref = _sdpa_reference(ly)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("P", [1, 2, 16, 32])
@pytest.mark.parametrize("kv_shared", [False, True])
def test_page_sizes_and_shared_kv(P, kv_shared):
    ly = _layer([5, 50, 33], 4, 2, 16, window=0, kv_shared=kv_shared, P=P, seed=P + 5 * kv_shared)
    np.testing.assert_allclose(_oracle(ly), _sdpa_reference(ly), rtol=1e-12, atol=1e-12)


def test_single_token_returns_its_value_row():
    ly = _layer([1, 1], 8, 2, 64, seed=3)
    got = _oracle(ly)
    G = 4
    for b in range(2):
        page = int(ly.block_tables[b, 0])
        for h in range(8):
            want = ly.v_pool[page, h // G, 0].to(torch.float64).numpy()
            assert np.array_equal(got[b, h], want)


def test_zero_query_gives_mean_of_values():
    ly = _layer([40, 17], 4, 2, 32, window=9, seed=4)
    ly.q.zero_()
    got = _oracle(ly)
    for b in range(2):
        L = int(ly.seq_lens[b])
        V = _dense_kv(ly, ly.v_pool, b)[:, max(0, L - 9):L]  # [Hkv, n, d]
        mean = V.mean(dim=1).repeat_interleave(2, dim=0).numpy()
        np.testing.assert_allclose(got[b], mean, rtol=1e-13, atol=1e-14)


def test_equal_keys_give_mean_of_values():
    ly = _layer([48], 2, 1, 16, seed=5)
    ly.k_pool[:] = ly.k_pool[int(ly.block_tables[0, 0]), 0, 0]
    got = _oracle(ly)
    mean = _dense_kv(ly, ly.v_pool, 0).mean(dim=1).repeat_interleave(2, dim=0).numpy()
    np.testing.assert_allclose(got[0], mean, rtol=1e-13, atol=1e-14)


def test_one_dominant_key_selects_its_value():
    ly = _layer([30], 1, 1, 16, seed=6)
    ly.k_pool.mul_(1e-3)
    ly.q[:] = 1.0
    page = int(ly.block_tables[0, 17 // 16])
    ly.k_pool[page, 0, 17 % 16] = 64.0
    got = _oracle(ly)
    want = ly.v_pool[page, 0, 17 % 16].to(torch.float64).numpy()
    np.testing.assert_allclose(got[0, 0], want, rtol=0, atol=1e-12)


def _scale(tag):
    return {"ln3": math.log(3.0), "ln7": math.log(7.0), "ln4": math.log(4.0),
            "ln8": math.log(8.0)}[tag] if isinstance(tag, str) else float(tag)


def test_hand_examples():
    with open(os.path.join(HERE, "golden", "hand_examples.json")) as f:
        data = json.load(f)
    for case in data["cases"]:
        P, d = case["page_size"], case["head_dim"]
        Hq, Hkv = case["num_q_heads"], case["num_kv_heads"]
        L = case["seq_len"]
        n_pages = (L + P - 1) // P
        pool_k = np.zeros((n_pages + 1, Hkv, P, d), dtype=np.float32)
        pool_v = np.zeros_like(pool_k)
        # logical page i lives in physical page n_pages - i (a reversed table)
        table = np.array([[n_pages - i for i in range(n_pages)]], dtype=np.int32)
        for t, (k, v) in enumerate(zip(case["k_tokens"], case["v_tokens"])):
            pool_k[table[0, t // P], 0, t % P] = k
            pool_v[table[0, t // P], 0, t % P] = v
        to_bits = lambda a: synth.bits_u16(torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16))
        out, lse = oracle.decode(to_bits(case["q"]), to_bits(pool_k), to_bits(pool_v), table,
                                 np.array([L], dtype=np.int32), _scale(case["scale"]), case["window"],
                                 return_lse=True)
        np.testing.assert_allclose(out, np.array(case["expected_out"]), rtol=0, atol=1e-14,
                                   err_msg=case["name"])
        if case["expected_lse"] is not None:
            assert abs(lse[0, 0] - _scale(case["expected_lse"])) < 1e-14, case["name"]


def test_window_mask_invariant():
    W = 24
    ly = _layer([100, 77], 8, 2, 32, window=W, seed=7)
    base = _oracle(ly)
    # rewrite every row before the window: output must not move by one bit
    ly2 = _layer([100, 77], 8, 2, 32, window=W, seed=7)
    g = torch.Generator().manual_seed(99)
    for b in range(2):
        L = int(ly2.seq_lens[b])
        for t in range(L - W):
            page = int(ly2.block_tables[b, t // 16])
            ly2.k_pool[page, :, t % 16] = torch.randn(2, 32, generator=g).to(torch.bfloat16) * 8
            ly2.v_pool[page, :, t % 16] = torch.randn(2, 32, generator=g).to(torch.bfloat16) * 8
    assert np.array_equal(base, _oracle(ly2))
    # rewriting position L - W (the oldest attended one) must change it
    L = int(ly2.seq_lens[0])
    t = L - W
    page = int(ly2.block_tables[0, t // 16])
    ly2.v_pool[page, :, t % 16] += 1.0
    assert not np.array_equal(base[0], _oracle(ly2)[0])
    # a window at least as long as the sequence is the global layer
    ly3 = _layer([100, 77], 8, 2, 32, window=100, seed=7)
    ly3_global = _layer([100, 77], 8, 2, 32, window=0, seed=7)
    assert np.array_equal(_oracle(ly3), _oracle(ly3_global))


def test_page_permutation_invariance():
    ly = _layer([70, 33, 16], 4, 2, 32, window=0, seed=8, extra_pages=9)
    base = _oracle(ly)
    g = torch.Generator().manual_seed(5)
    perm = torch.randperm(ly.num_pages, generator=g)  # new physical slot of each old page
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(ly.num_pages)
    k2 = ly.k_pool[inv].clone()
    v2 = ly.v_pool[inv].clone()
    t2 = ly.block_tables.clone()
    valid = t2 >= 0
    t2[valid] = perm[t2[valid].long()].to(torch.int32)
    out2 = oracle.decode(synth.bits_u16(ly.q), synth.bits_u16(k2), synth.bits_u16(v2), t2.numpy(),
                         ly.seq_lens.numpy(), ly.scale, 0)
    assert np.array_equal(base, out2)


@pytest.mark.parametrize("S,chunk", [(1, 1000), (2, 60), (3, 41), (7, 17), (7, 5), (9, 16)])
@pytest.mark.parametrize("window", [0, 29])
def test_split_merge_equals_unsplit(S, chunk, window):
    ly = _layer([100, 64, 1, 0], 8, 4, 16, window=window, seed=9 + S)
    full = _oracle(ly)
    o_part, lse_part = oracle.decode_split(
        synth.bits_u16(ly.q), synth.bits_u16(ly.k_pool), synth.bits_u16(ly.v_pool),
        ly.block_tables.numpy(), ly.seq_lens.numpy(), ly.scale, window, S, chunk)
    # with too few pieces the tail is simply not covered: only compare rows whose
    # attended range fits in S * chunk
    merged = oracle.merge(o_part, lse_part)
    for b, n in enumerate(ly.attended()):
        if n <= S * chunk:
            np.testing.assert_allclose(merged[b], full[b], rtol=1e-12, atol=1e-13)
    # empty pieces carry -inf and do not disturb the merge
    assert np.isneginf(lse_part[3]).all() and (o_part[3] == 0).all()


def test_lse_matches_scores():
    ly = _layer([45, 3], 4, 2, 16, window=0, seed=11)
    _, lse = _oracle(ly, return_lse=True)
    from scipy.special import logsumexp
    for b in range(2):
        K = _dense_kv(ly, ly.k_pool, b).repeat_interleave(2, dim=0)
        s = torch.einsum("hd,hld->hl", ly.q[b].to(torch.float64), K) * ly.scale
        np.testing.assert_allclose(lse[b], logsumexp(s.numpy(), axis=1), rtol=1e-13)


def test_empty_sequence_is_zero():
    ly = _layer([0, 5], 4, 2, 16, seed=12)
    out, lse = _oracle(ly, return_lse=True)
    assert (out[0] == 0).all() and np.isneginf(lse[0]).all()


def test_rejects_bad_page_and_length():
    ly = _layer([20], 2, 1, 16, seed=13)
    bt = ly.block_tables.numpy().copy()
    bt[0, 1] = ly.num_pages  # one past the pool
    with pytest.raises(oracle.OracleError):
        oracle.decode(synth.bits_u16(ly.q), synth.bits_u16(ly.k_pool), synth.bits_u16(ly.v_pool),
                      bt, ly.seq_lens.numpy(), ly.scale)
    with pytest.raises(oracle.OracleError):
        oracle.decode(synth.bits_u16(ly.q), synth.bits_u16(ly.k_pool), synth.bits_u16(ly.v_pool),
                      ly.block_tables.numpy(), np.array([10 ** 6], dtype=np.int32), ly.scale)


def test_row_subset_matches_full():
    ly = _layer([90, 31], 8, 2, 32, window=40, seed=14)
    full = _oracle(ly)
    rows = [3, 9, 15]
    part = _oracle(ly, rows=rows)
    for r in rows:
        b, h = divmod(r, 8)
        assert np.array_equal(part[b, h], full[b, h])
    assert (part[0, 0] == 0).all()


# ---- FP8 KV cache ---------------------------------------------------------------

def test_e4m3_decoder_matches_torch_for_every_code():
    """The oracle's e4m3 decoder against torch's float8_e4m3fn for all 256 codes."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_f64(c) for c in range(256)])
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all() and nan.sum() == 2  # S.1111.111 for both signs
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6


def _fp8_layer(lens, Hq, Hkv, d, window=0, kv_shared=False, seed=0):
    ly = _layer(lens, Hq, Hkv, d, window=window, kv_shared=kv_shared, seed=seed)
    return synth.quantize_kv_fp8(ly)


def _dequant(pool8, scale):
    return pool8.view(torch.float8_e4m3fn).to(torch.float64) * scale.to(torch.float64)[:, :, None, None]


@pytest.mark.parametrize("kv_shared,window", [(False, 0), (True, 9), (False, 20)])
def test_fp8_decode_matches_sdpa_on_dequantized_kv(kv_shared, window):
    """FP8 decode equals library attention over the explicitly dequantized cache."""
    f = _fp8_layer([37, 64, 5], 8, 2, 16, window=window, kv_shared=kv_shared, seed=40 + window)
    got = oracle.decode_fp8(synth.bits_u16(f.q), f.k8.numpy(), None if f.v8 is None else f.v8.numpy(),
                            f.k_scale.numpy(), None if f.v_scale is None else f.v_scale.numpy(),
                            f.block_tables.numpy(), f.seq_lens.numpy(), f.scale, window)
    K = _dequant(f.k8, f.k_scale)
    V = K if f.v8 is None else _dequant(f.v8, f.v_scale)
    dense = synth.make_layer("dq", [37, 64, 5], 8, 2, 16, window=window, pool_pages=f.num_pages, seed=0,
                             block_tables=f.block_tables)
    ref = _sdpa_reference_pools(dense, K, V, f.q)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def _sdpa_reference_pools(ly, K_pool, V_pool, q):
    """Library attention over float64 pools (any values), explicit window mask."""
    out = torch.zeros(ly.batch, q.shape[1], ly.head_dim, dtype=torch.float64)
    G = q.shape[1] // ly.num_kv_heads
    for b in range(ly.batch):
        L = int(ly.seq_lens[b])
        if L == 0:
            continue
        P = ly.page_size
        pages = [int(ly.block_tables[b, t // P]) for t in range(L)]
        K = torch.stack([K_pool[pages[t], :, t % P] for t in range(L)], dim=1).repeat_interleave(G, dim=0)
        V = torch.stack([V_pool[pages[t], :, t % P] for t in range(L)], dim=1).repeat_interleave(G, dim=0)
        qq = q[b].to(torch.float64).unsqueeze(1)
        pos = torch.arange(L)
        keep = pos >= (L - ly.window) if ly.window > 0 else torch.ones(L, dtype=torch.bool)
        mask = keep.view(1, 1, L).expand(q.shape[1], 1, L)
        out[b] = torch.nn.functional.scaled_dot_product_attention(qq, K, V, attn_mask=mask, scale=ly.scale)[:, 0]
    return out.numpy()


def test_fp8_single_token_is_its_scaled_value_row():
    f = _fp8_layer([1, 1], 4, 2, 32, seed=41)
    got = oracle.decode_fp8(synth.bits_u16(f.q), f.k8.numpy(), f.v8.numpy(), f.k_scale.numpy(), f.v_scale.numpy(),
                            f.block_tables.numpy(), f.seq_lens.numpy(), f.scale)
    for b in range(2):
        page = int(f.block_tables[b, 0])
        want = (f.v8[page, :, 0].view(torch.float8_e4m3fn).to(torch.float64)
                * f.v_scale[page].to(torch.float64)[:, None]).repeat_interleave(2, dim=0).numpy()
        assert np.array_equal(got[b], want)


def test_fp8_key_scale_is_a_logit_scale():
    """Doubling every K scale is the same as doubling the softmax scale."""
    f = _fp8_layer([50, 23], 4, 2, 16, seed=42)
    args = (f.k8.numpy(), f.v8.numpy())
    a = oracle.decode_fp8(synth.bits_u16(f.q), *args, (f.k_scale * 2).numpy(), f.v_scale.numpy(),
                          f.block_tables.numpy(), f.seq_lens.numpy(), f.scale)
    b_ = oracle.decode_fp8(synth.bits_u16(f.q), *args, f.k_scale.numpy(), f.v_scale.numpy(),
                           f.block_tables.numpy(), f.seq_lens.numpy(), 2 * f.scale)
    np.testing.assert_allclose(a, b_, rtol=1e-13, atol=1e-15)
