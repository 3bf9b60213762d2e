"""Several query tokens per request (speculative-decode verification / a chunk
of prefill) on the GPU, through the C ABI, against the fp64 multi-token oracle.

Bar as for decode: max |gpu - oracle| <= 2e-2 and cosine > 0.9995 over each
output tensor (bf16 output, fp32 accumulation); a token whose causal range is
one position returns that value row bit for bit.
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


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _layer(lens, T, Hq, Hkv, d, window=0, kvs=False, P=16, seed=0, q_std=1.0):
    pool = sum((L + P - 1) // P for L in lens) + 3
    li = synth.make_layer("mt", lens, Hq, Hkv, d, window=window, kv_shared=kvs, pool_pages=pool, page_size=P,
                          seed=seed, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(seed + 77)
    q = (q_std * torch.randn(len(lens), T, Hq, d, generator=g, device="cuda")).to(torch.bfloat16)
    return li, q


def _desc(li):
    return b.layer_desc(li.num_q_heads, li.num_kv_heads, li.head_dim, li.page_size, li.num_pages,
                        li.block_tables.shape[1], li.window, li.v_pool is None)


def run_gpu(li, q, T, seq=None, sms=None):
    plan = b.paged_decode_plan_multi(_desc(li), T, li.seq_lens.tolist(), sms or _sms())
    ws = torch.zeros(max(256, plan.workspace_bytes), dtype=torch.uint8, device="cuda")
    out = torch.full_like(q, float("nan"))
    seq = li.seq_lens if seq is None else seq
    if li.window > 0:
        b.paged_decode_window(plan, q, li.k_pool, li.v_pool, li.block_tables, seq, li.window, li.scale, ws, out)
    else:
        b.paged_decode_global(plan, q, li.k_pool, li.v_pool, li.block_tables, seq, li.scale, ws, out)
    b.paged_decode_merge(plan, ws, out)
    flags = ctypes_flags(plan, ws)
    return out, plan, flags


def ctypes_flags(plan, ws):
    import ctypes
    f = ctypes.c_uint32(0)
    st = b.load_library().paged_decode_check_device_error(ctypes.byref(plan), ws.data_ptr(), ws.numel(), None,
                                                          ctypes.byref(f))
    assert st in (b.PD_OK, b.PD_ERR_DEVICE_FAULT)
    return int(f.value)


def run_oracle(li, q):
    return oracle.decode_multi(synth.bits_u16(q.cpu()), synth.bits_u16(li.k_pool.cpu()),
                               None if li.v_pool is None else synth.bits_u16(li.v_pool.cpu()),
                               li.block_tables.cpu().numpy(), li.seq_lens.cpu().numpy(), li.scale, li.window)


def compare(out, ref, tag):
    got = out.float().cpu().double().numpy()
    assert np.isfinite(got).all(), f"{tag}: non-finite output"
    err = np.abs(got - ref).max()
    g, r = got.ravel(), ref.ravel()
    cos = float(g @ r / (np.linalg.norm(g) * np.linalg.norm(r)))
    assert err <= MAX_ABS, f"{tag}: max abs {err:.3e}"
    assert cos > MIN_COS, f"{tag}: cosine {cos:.7f}"


CASES = [
    # d, Hq, Hkv, kvs, window, T, lens
    (512, 16, 4, False, 0, 2, [2, 17, 300, 1000]),         # T * G = 8: one column tile
    (512, 16, 4, True, 0, 4, [4, 33, 1024, 517]),          # two tiles
    (256, 16, 8, False, 1024, 4, [4100, 4200, 5, 1030]),   # sliding, windows cut per token
    (256, 8, 8, True, 37, 7, [7, 60, 200]),                # G = 1
    (512, 16, 2, False, 0, 3, [3, 100, 2000]),             # G = 8: one token per tile
    (256, 12, 4, False, 5, 6, [6, 40, 97]),                # G = 3: pairs straddle tiles
    (512, 8, 4, False, 16, 5, [5, 16, 17, 48]),            # window shorter than T's span
    (512, 16, 4, False, 0, 8, [8, 100, 1024, 3000]),       # four tiles: two CTAs of two
    (256, 16, 8, True, 1024, 6, [4100, 6, 1500]),          # two tiles, K=V, window
    (512, 12, 4, False, 37, 7, [7, 300, 2000]),            # three tiles: the last CTA's second tile unused
    (256, 64, 4, False, 0, 2, [2, 900, 33]),               # G = 16, two query tokens: four tiles
]


@pytest.mark.parametrize("case", CASES, ids=[f"d{c[0]}-G{c[1] // c[2]}-kvs{int(c[3])}-W{c[4]}-T{c[5]}"
                                             for c in CASES])
def test_multi_matches_oracle(case):
    d, Hq, Hkv, kvs, W, T, lens = case
    li, q = _layer(lens, T, Hq, Hkv, d, window=W, kvs=kvs, seed=d + T + W)
    out, plan, flags = run_gpu(li, q, T)
    assert flags == 0
    compare(out, run_oracle(li, q), f"S={plan.num_splits} mode={plan.merge_mode}")


# (lengths, SM count, query tokens): each merge mode, for one-tile CTAs (T = 2:
# 8 columns) and two-tile CTAs (T = 4, 8: 16 and 32 columns)
MODE_CASES = [([64, 64], 4, 8), ([1024] * 8, 152, 8), ([60000], 152, 4), ([64, 64], 4, 2), ([1024] * 8, 152, 2),
              ([60000], 152, 2)]
MODE_IDS = ["one-piece-2tiles", "cluster-merge-2tiles", "merge-kernel-2tiles", "one-piece", "cluster-merge",
            "merge-kernel"]


def _mode_plan(lens, sms, T):
    desc = b.layer_desc(16, 4, 512, 16, sum((L + 15) // 16 for L in lens) + 3, max((L + 15) // 16 for L in lens))
    return b.paged_decode_plan_multi(desc, T, lens, sms)


@pytest.mark.parametrize("lens,sms,T", MODE_CASES, ids=MODE_IDS)
def test_multi_merge_modes(lens, sms, T):
    """Lengths and SM counts that lead the planner to each of its merge modes."""
    li, q = _layer(lens, T, 16, 4, 512, seed=len(lens) + sms + T, q_std=0.5)
    out, plan, flags = run_gpu(li, q, T, sms=sms)
    assert flags == 0
    compare(out, run_oracle(li, q), f"S={plan.num_splits} mode={plan.merge_mode}")


def test_merge_modes_are_all_reached():
    for tiles in ((4, 8), (2,)):
        modes = {int(_mode_plan(lens, sms, T).merge_mode) for lens, sms, T in MODE_CASES if T in tiles}
        assert modes == {0, 1, 2}, (tiles, modes)


def test_first_token_of_a_fresh_sequence_returns_its_value_row():
    """T tokens with L = T: token 0 attends only position 0 -> its V row exactly."""
    T = 3
    li, q = _layer([T, T], T, 8, 2, 256, seed=4)
    out, _, flags = run_gpu(li, q, T)
    assert flags == 0
    G = 4
    for bi in range(2):
        page = int(li.block_tables[bi, 0])
        v0 = li.v_pool[page, :, 0, :]  # [Hkv, d]
        assert torch.equal(out[bi, 0], v0.repeat_interleave(G, dim=0))


def test_one_query_token_plan_is_the_decode_plan():
    desc = b.layer_desc(16, 4, 512, 16, 100, 64)
    a = b.paged_decode_plan(desc, [1000, 20], 152)
    m = b.paged_decode_plan_multi(desc, 1, [1000, 20], 152)
    assert bytes(a) == bytes(m)


def test_device_length_below_token_count_is_flagged():
    T = 4
    li, q = _layer([10, 30], T, 8, 2, 256, seed=8)
    seq = torch.tensor([2, 30], dtype=torch.int32, device="cuda")
    out, _, flags = run_gpu(li, q, T, seq=seq)
    assert flags & b.PD_DEVFLAG_BAD_SEQLEN
    # request 0: tokens at positions -2 and -1 attend nothing (zero rows)
    assert (out[0, :2].float() == 0).all()
    assert torch.isfinite(out.float()).all()


def test_plan_rejections():
    desc = b.layer_desc(16, 4, 512, 16, 100, 64)
    for T, lens, status in ((0, [10], b.PD_ERR_INVALID_ARG), (257, [300], b.PD_ERR_INVALID_ARG),
                            (4, [3], b.PD_ERR_INVALID_ARG)):
        with pytest.raises(b.PagedDecodeError) as e:
            b.paged_decode_plan_multi(desc, T, lens, 152)
        assert e.value.status == status
    d128 = b.layer_desc(16, 4, 128, 16, 100, 64)
    with pytest.raises(b.PagedDecodeError) as e:
        b.paged_decode_plan_multi(d128, 2, [10], 152)
    assert e.value.status == b.PD_ERR_UNSUPPORTED


FP8_CASES = [
    # d, Hq, Hkv, kvs, window, T, lens
    (512, 16, 4, False, 0, 2, [2, 17, 300, 1000]),
    (512, 16, 4, True, 0, 3, [3, 64, 700]),
    (256, 16, 8, False, 1024, 4, [4100, 4200, 5, 1030]),
    (256, 8, 4, True, 37, 5, [5, 60, 333]),
]


@pytest.mark.parametrize("case", FP8_CASES, ids=[f"d{c[0]}-kvs{int(c[3])}-W{c[4]}-T{c[5]}" for c in FP8_CASES])
def test_multi_over_fp8_cache_matches_per_token_oracle(case):
    """Over an e4m3 cache, token j of T must equal the (pinned) single-token
    FP8 oracle at length L - T + 1 + j."""
    d, Hq, Hkv, kvs, W, T, lens = case
    li, q = _layer(lens, T, Hq, Hkv, d, window=W, kvs=kvs, seed=d + T + W + 5)
    f8 = synth.quantize_kv_fp8(li)
    desc = b.layer_desc(Hq, Hkv, d, li.page_size, li.num_pages, li.block_tables.shape[1], W, kvs, b.PD_KV_FP8_E4M3)
    plan = b.paged_decode_plan_multi(desc, T, lens, _sms())
    ws = torch.zeros(max(256, plan.workspace_bytes), dtype=torch.uint8, device="cuda")
    out = torch.full_like(q, float("nan"))
    if W > 0:
        b.paged_decode_window_fp8(plan, q, f8.k8, f8.v8, f8.k_scale, f8.v_scale, li.block_tables, li.seq_lens, W,
                                  li.scale, ws, out)
    else:
        b.paged_decode_global_fp8(plan, q, f8.k8, f8.v8, f8.k_scale, f8.v_scale, li.block_tables, li.seq_lens,
                                  li.scale, ws, out)
    b.paged_decode_merge(plan, ws, out)
    assert ctypes_flags(plan, ws) == 0
    qh = q.cpu()
    ref = np.zeros(tuple(q.shape), dtype=np.float64)
    k8, v8 = f8.k8.cpu().numpy(), None if f8.v8 is None else f8.v8.cpu().numpy()
    ks, vs = f8.k_scale.cpu().numpy(), None if f8.v_scale is None else f8.v_scale.cpu().numpy()
    for j in range(T):
        lens_j = np.array([L - T + 1 + j for L in lens], dtype=np.int32)
        ref[:, j] = oracle.decode_fp8(synth.bits_u16(qh[:, j].contiguous()), k8, v8, ks, vs,
                                      li.block_tables.cpu().numpy(), lens_j, li.scale, W)
    compare(out, ref, f"fp8 S={plan.num_splits} mode={plan.merge_mode}")
