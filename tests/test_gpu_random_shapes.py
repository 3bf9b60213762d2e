"""Seeded random layer shapes through the C ABI against the fp64 oracle.

Each case draws a head_dim, a GQA group (1..16), a number of KV heads, K=V or
separate K and V, a bf16 or e4m3 cache, 1..8 query tokens per request, a
window (none or 37..1024 positions), a ragged batch (lengths log-uniform, some
shorter than the window or a page, some empty when decoding one token) and
the SM count the planner sizes the launch for, so that one-piece, cluster and
merge-kernel plans, one- and two-tile column CTAs and every producer form come
up. Bar: max |gpu - oracle| <= 2e-2, cosine > 0.9995 over the output, rows with
no attended position exactly zero. A multi-token case over an e4m3 cache is
compared token by token with the single-token e4m3 oracle at the token's own
length (the reduction the multi-token pins establish).
"""
import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_global_gb300 import binding as b
from paged_gqa_decode_global_gb300 import inputs as synth

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
MIN_COS = 0.9995


def _cases(n=120, seed=20261203):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        d = int(rng.choice([128, 256, 512]))
        fp8 = d != 128 and rng.random() < 0.35
        T = 1 if d == 128 or rng.random() < 0.5 else int(rng.choice([2, 3, 4, 8]))
        G = int(rng.choice([1, 2, 4, 8] if d == 128 else [1, 2, 3, 4, 8, 12, 16]))
        Hkv = int(rng.choice([1, 2, 4]))
        kvs = bool(rng.random() < 0.4)
        window = int(rng.choice([0, 0, 37, 256, 1024]))
        B = int(rng.integers(1, 7))
        lens = [int(x) for x in np.exp(rng.uniform(np.log(max(T, 1)), np.log(6000), B))]
        lens = [max(L, T) for L in lens]
        if T == 1 and rng.random() < 0.3:
            lens[int(rng.integers(B))] = 0
        sms = int(rng.choice([3, 20, 40, 152, 400, 1000]))
        if B * T * G * Hkv * max(lens) > 3_000_000:  # keeps the fp64 oracle to seconds
            continue
        out.append((d, G, Hkv, kvs, fp8, T, window, lens, sms))
    return out


CASES = _cases()


def _cases_pages(n=80, seed=20261204):
    """The same draws plus the page size (16..64 tokens: pages of one to four
    16-token blocks, an e4m3 scale per page) and the plan's early_kv flag."""
    rng = np.random.default_rng(seed)
    base = _cases(n, seed)
    return [c + (int(rng.choice([16, 32, 48, 64])), bool(rng.integers(2))) for c in base]


CASES_PAGES = _cases_pages()


def _compare(got, ref, empty_rows, tag):
    got = got.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all(), f"{tag}: non-finite output"
    if empty_rows.any():
        assert (got[empty_rows] == 0).all(), f"{tag}: rows with nothing attended are not zero"
    err = np.abs(got - ref).max()
    g, r = got.ravel(), ref.ravel()
    nr = np.linalg.norm(r)
    cos = float(g @ r / (np.linalg.norm(g) * nr)) if nr > 0 else 1.0
    assert err <= MAX_ABS, f"{tag}: max abs {err:.3e}"
    assert cos > MIN_COS, f"{tag}: cosine {cos:.7f}"


def _cases_big_batch(n=20, seed=20261207):
    """Batches of 16..256 short requests: many (request, KV head) pairs, the
    planner's few-pieces end, a launch grid deep in its third dimension."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        d = int(rng.choice([256, 512]))
        fp8 = rng.random() < 0.3
        T = 1 if rng.random() < 0.6 else int(rng.choice([2, 4]))
        G = int(rng.choice([1, 2, 4, 8, 16]))
        Hkv = int(rng.choice([1, 2, 4]))
        kvs = bool(rng.random() < 0.4)
        window = int(rng.choice([0, 0, 256]))
        B = int(rng.integers(16, 257))
        lens = [max(T, int(x)) for x in np.exp(rng.uniform(0.0, np.log(2000), B))]
        sms = int(rng.choice([40, 152, 1000]))
        if B * T * G * Hkv * max(lens) > 6_000_000:
            continue
        out.append((d, G, Hkv, kvs, fp8, T, window, lens, sms))
    return out


CASES_BIG_BATCH = _cases_big_batch()


def _case_id(c):
    d, G, Hkv, kvs, fp8, T, window, lens, sms = c
    return f"d{d}-G{G}-Hkv{Hkv}-{'kvs' if kvs else 'kv'}-{'fp8' if fp8 else 'bf16'}-T{T}-W{window}-B{len(lens)}-sm{sms}"


@pytest.mark.parametrize("case", CASES, ids=[_case_id(c) for c in CASES])
def test_random_shape_matches_oracle(case):
    _run_case(*case)


@pytest.mark.parametrize("case", CASES_PAGES,
                         ids=[_case_id(c[:9]) + f"-P{c[9]}-early{int(c[10])}" for c in CASES_PAGES])
def test_random_shape_with_page_size_and_early_kv_matches_oracle(case):
    _run_case(*case)


@pytest.mark.parametrize("case", CASES_BIG_BATCH, ids=[_case_id(c) for c in CASES_BIG_BATCH])
def test_random_big_batch_matches_oracle(case):
    _run_case(*case)


def _run_case(d, G, Hkv, kvs, fp8, T, window, lens, sms, P=16, early=False):
    Hq = G * Hkv
    li = synth.make_layer("rnd", lens, Hq, Hkv, d, window=window, kv_shared=kvs,
                          pool_pages=sum((L + P - 1) // P for L in lens) + 3, page_size=P,
                          seed=d + 7 * G + 31 * T + window + len(lens), device="cuda")
    g = torch.Generator(device="cuda").manual_seed(sms + T)
    q = li.q if T == 1 else (torch.randn(len(lens), T, Hq, d, generator=g, device="cuda")).to(torch.bfloat16)
    kv_dtype = b.PD_KV_FP8_E4M3 if fp8 else b.PD_KV_BF16
    desc = b.layer_desc(Hq, Hkv, d, li.page_size, li.num_pages, li.block_tables.shape[1], window, kvs, kv_dtype)
    plan = b.paged_decode_plan_multi(desc, T, lens, sms) if T > 1 else b.paged_decode_plan(desc, lens, sms)
    plan.early_kv = int(early)
    ws = torch.zeros(max(256, int(plan.workspace_bytes)), dtype=torch.uint8, device="cuda")
    out = torch.full_like(q, float("nan"))
    if fp8:
        f8 = synth.quantize_kv_fp8(li)
        fn = b.paged_decode_window_fp8 if window > 0 else b.paged_decode_global_fp8
        args = (plan, q, f8.k8, f8.v8, f8.k_scale, f8.v_scale, li.block_tables, li.seq_lens)
        fn(*args, *((window,) if window > 0 else ()), li.scale, ws, out)
    else:
        fn = b.paged_decode_window if window > 0 else b.paged_decode_global
        args = (plan, q, li.k_pool, li.v_pool, li.block_tables, li.seq_lens)
        fn(*args, *((window,) if window > 0 else ()), li.scale, ws, out)
    b.paged_decode_merge(plan, ws, out)
    assert b.paged_decode_check_device_error(plan, ws) == 0
    tag = f"S={plan.num_splits} mode={plan.merge_mode} P={P}"

    tables, seq = li.block_tables.cpu().numpy(), li.seq_lens.cpu().numpy()
    if fp8:
        k8, v8 = f8.k8.cpu().numpy(), None if f8.v8 is None else f8.v8.cpu().numpy()
        ks, vs = f8.k_scale.cpu().numpy(), None if f8.v_scale is None else f8.v_scale.cpu().numpy()
        if T == 1:
            ref = oracle.decode_fp8(synth.bits_u16(q), k8, v8, ks, vs, tables, seq, li.scale, window)
        else:
            qh = q.cpu()
            ref = np.zeros(tuple(q.shape), dtype=np.float64)
            for j in range(T):
                lens_j = np.array([L - T + 1 + j for L in lens], dtype=np.int32)
                ref[:, j] = oracle.decode_fp8(synth.bits_u16(qh[:, j].contiguous()), k8, v8, ks, vs, tables,
                                              lens_j, li.scale, window)
    else:
        kp = synth.bits_u16(li.k_pool)
        vp = None if li.v_pool is None else synth.bits_u16(li.v_pool)
        if T == 1:
            ref = oracle.decode(synth.bits_u16(q), kp, vp, tables, seq, li.scale, window)
        else:
            ref = oracle.decode_multi(synth.bits_u16(q.cpu()), kp, vp, tables, seq, li.scale, window)
    empty = np.zeros(tuple(q.shape[:-1]), dtype=bool)
    if T == 1:
        empty[np.array(lens) == 0] = True
    _compare(out, ref, empty, tag)


def _cases_sharded(n=40, seed=20261205):
    """Sequence-sharded decode: R virtual ranks each run the partial decode over
    their shard of the cache; the kernel combines the stacked partials."""
    from paged_gqa_decode_global_gb300 import dcp
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        d = int(rng.choice([256, 512]))
        G = int(rng.choice([1, 2, 3, 4, 8, 12, 16]))
        Hkv = int(rng.choice([1, 2, 4]))
        kvs = bool(rng.random() < 0.4)
        B = int(rng.integers(1, 6))
        lens = [int(x) for x in np.exp(rng.uniform(0.0, np.log(8000), B))]
        if rng.random() < 0.3:
            lens[int(rng.integers(B))] = 0
        R = int(rng.integers(1, 5))
        mode = str(rng.choice(dcp.MODES))
        sms = int(rng.choice([3, 40, 152, 1000]))
        if B * G * Hkv * max(lens) > 3_000_000:
            continue
        out.append((d, G, Hkv, kvs, lens, R, mode, sms))
    return out


CASES_SHARDED = _cases_sharded()


def _sharded_id(c):
    d, G, Hkv, kvs, lens, R, mode, sms = c
    return f"d{d}-G{G}-Hkv{Hkv}-{'kvs' if kvs else 'kv'}-B{len(lens)}-R{R}-{mode}-sm{sms}"


@pytest.mark.parametrize("case", CASES_SHARDED, ids=[_sharded_id(c) for c in CASES_SHARDED])
def test_random_sharded_decode_matches_oracle(case):
    from paged_gqa_decode_global_gb300 import dcp
    d, G, Hkv, kvs, lens, R, mode, sms = case
    li = synth.make_layer("rsh", lens, G * Hkv, Hkv, d, kv_shared=kvs,
                          pool_pages=sum((L + 15) // 16 for L in lens) + 3,
                          seed=d + G + 13 * R + len(lens), device="cuda")
    os_, lses = [], []
    for r in range(R):
        k, v, table, shard_lens = dcp.shard_cache(li.k_pool, li.v_pool, li.block_tables, lens, R, r, mode)
        desc = b.layer_desc(li.num_q_heads, Hkv, d, li.page_size, k.shape[0], table.shape[1], 0, kvs)
        step = dcp.PartialStep(desc, shard_lens.tolist(), sms, "cuda")
        o, lse = step(li.q, k, v, table, shard_lens, li.scale)
        os_.append(o)
        lses.append(lse)
    out = dcp.combine(torch.stack(os_), torch.stack(lses))
    torch.cuda.synchronize()
    ref = oracle.decode(synth.bits_u16(li.q), synth.bits_u16(li.k_pool),
                        None if li.v_pool is None else synth.bits_u16(li.v_pool), li.block_tables.cpu().numpy(),
                        li.seq_lens.cpu().numpy(), li.scale, 0)
    empty = np.zeros(tuple(li.q.shape[:-1]), dtype=bool)
    empty[np.array(lens) == 0] = True
    _compare(out, ref, empty, f"R={R} {mode}")
