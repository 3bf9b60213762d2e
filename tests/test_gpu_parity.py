"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Bar (bf16 output, fp32 accumulation): max |gpu - oracle| <= 2e-2 and cosine
similarity > 0.9995 over each output tensor; rows with nothing attended must be
exactly zero; a one-token sequence must return its value row bit for bit.
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


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_gqa_decode_global_gb300 import build
    build.build()
    b.load_library()


def run_gpu(li, sm_count=None, out_fill=float("nan")):
    step = b.LayerStep.for_inputs(li, sm_count)
    out = torch.full_like(li.q, out_fill)
    step.run(li, out)
    flags = step.check()
    assert flags == 0
    return out, step


def run_oracle(li):
    return oracle.decode(synth.bits_u16(li.q), synth.bits_u16(li.k_pool),
                         None if li.v_pool is None else synth.bits_u16(li.v_pool),
                         li.block_tables.cpu().numpy(), li.seq_lens.cpu().numpy(), li.scale, li.window)


def compare(gpu_out, ref, li, tag=""):
    got = gpu_out.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all(), f"{tag}: non-finite output"
    err = np.abs(got - ref).max()
    empty = np.array([n == 0 for n in li.attended()])
    if empty.any():
        assert (got[empty] == 0).all(), f"{tag}: empty rows not zero"
    g, r = got[~empty].ravel(), ref[~empty].ravel()
    cos = float(g @ r / (np.linalg.norm(g) * np.linalg.norm(r))) if g.size else 1.0
    assert err <= MAX_ABS, f"{tag}: max abs {err:.3e}"
    assert cos > MIN_COS, f"{tag}: cosine {cos:.7f}"
    # per (request, head) row as well: at long contexts the outputs are small and
    # max |err| alone says little. Two bf16 roundings of at most 2^-9 relative
    # each (the probabilities entering PV, and the output) bound the relative
    # L2 error near 2^-8 = 3.9e-3 (allowed: 5e-3), and so 1 - cosine of any row
    # near (5e-3)^2 / 2 (allowed: 1e-4)
    gr, rr = got[~empty], ref[~empty]
    num = (gr * rr).sum(-1)
    den = np.linalg.norm(gr, axis=-1) * np.linalg.norm(rr, axis=-1)
    ok = den > 0
    row_cos = float((num[ok] / den[ok]).min()) if ok.any() else 1.0
    rel_l2 = float(np.linalg.norm(g - r) / np.linalg.norm(r)) if g.size and np.linalg.norm(r) > 0 else 0.0
    assert row_cos > 0.9999, f"{tag}: worst row cosine {row_cos:.6f}"
    assert rel_l2 < 5e-3, f"{tag}: relative L2 {rel_l2:.3e}"
    return err, cos, row_cos, rel_l2


# ---- the five named workloads at full size -------------------------------------

@pytest.mark.parametrize("cid,part", [(1, None), (2, None), (3, None), (4, "a"), (4, "b"), (4, "c"),
                                      (5, "global"), (5, "sliding")])
def test_workload_matches_oracle(cid, part):
    """Full size, in the launch configuration bench.py times: the plan's
    early_kv set, two steps queued back to back with no host sync (the second
    copying its first blocks while the first drains); both against the oracle."""
    for li in synth.workload(cid, device="cuda", part=part):
        step = b.LayerStep.for_inputs(li, early_kv=True)
        first = step.run(li, torch.full_like(li.q, float("nan")))
        out = step.run(li, torch.full_like(li.q, float("nan")))
        assert step.check() == 0
        ref = run_oracle(li)
        compare(first, ref, li, f"{li.name} first step")
        err, cos, row_cos, rel = compare(out, ref, li, f"{li.name} S={step.plan.num_splits}")
        print(f"{li.name}: splits {step.plan.num_splits} chunk {step.plan.chunk_tokens} max_abs {err:.2e} "
              f"cos {cos:.7f} worst row cos {row_cos:.6f} rel L2 {rel:.2e}")


# ---- every kernel instance on ragged batches ----------------------------------

VARIANTS = [(d, G, kvs) for d in (512, 256, 128) for G in (1, 2, 4, 8) for kvs in (False, True)]
FP8_VARIANTS = [v for v in VARIANTS if v[0] != 128]  # the FP8 instances are d = 512 and 256


@pytest.mark.parametrize("d,G,kvs", VARIANTS)
@pytest.mark.parametrize("window", [0, 37, 1000])
def test_variants_ragged(d, G, kvs, window):
    Hkv = 2
    lens = [1, 17, 300, 0, 1000, 33]
    li = synth.make_layer("v", lens, Hkv * G, Hkv, d, window=window, kv_shared=kvs,
                          pool_pages=sum((L + 15) // 16 for L in lens) + 5, seed=d + G + 100 * kvs + window,
                          device="cuda")
    ref = run_oracle(li)
    for sms in (3, 152):  # different split counts
        out, step = run_gpu(li, sm_count=sms)
        compare(out, ref, li, f"d{d} G{G} kvs{kvs} W{window} sms{sms} S{step.plan.num_splits}")


@pytest.mark.parametrize("d,G,kvs", [(512, 16, False), (512, 12, True), (256, 16, True), (256, 9, False)])
@pytest.mark.parametrize("window", [0, 37, 1000])
@pytest.mark.parametrize("long", [False, True])
def test_groups_above_8_ragged(d, G, kvs, window, long):
    """Groups of 9..16 query heads per KV head (two 8-column tiles: a CTA per
    tile over short contexts, one CTA for both over a span of 4096+ tokens):
    ragged lengths, windows, one piece / cluster merge / merge kernel."""
    Hkv = 2
    lens = [1, 17, 300, 0, 1000, 33] + ([5000] if long else [])
    li = synth.make_layer("g", lens, Hkv * G, Hkv, d, window=window, kv_shared=kvs,
                          pool_pages=sum((L + 15) // 16 for L in lens) + 5, seed=7 * d + G + 100 * kvs + window,
                          device="cuda")
    ref = run_oracle(li)
    modes = set()
    for sms in (1, 3, 40, 152):
        out, step = run_gpu(li, sm_count=sms)
        span = max(min(L, window) if window else L for L in lens)
        assert step.plan.grid_y == (Hkv if span >= 4096 else 2 * Hkv)
        modes.add(int(step.plan.merge_mode))
        compare(out, ref, li, f"d{d} G{G} kvs{kvs} W{window} sms{sms} S{step.plan.num_splits}")
    if window == 0:  # short windows always fit one piece
        assert 0 in modes and len(modes) >= 2, modes


@pytest.mark.parametrize("d,G,kvs", [(512, 3, False), (512, 6, True), (256, 5, False), (256, 7, True)])
@pytest.mark.parametrize("window", [0, 37, 1000])
def test_groups_between_the_decode_instances_ragged(d, G, kvs, window):
    """Groups of 3, 5, 6 and 7 query heads per KV head (no decode instance of
    their own: one 8-column tile per KV head): ragged lengths with an empty
    request, windows, one piece / cluster merge / merge kernel."""
    Hkv = 2
    lens = [1, 17, 300, 0, 1000, 33, 3000]
    li = synth.make_layer("gm", lens, Hkv * G, Hkv, d, window=window, kv_shared=kvs,
                          pool_pages=sum((L + 15) // 16 for L in lens) + 5, seed=11 * d + G + 100 * kvs + window,
                          device="cuda")
    ref = run_oracle(li)
    modes = set()
    for sms in (1, 3, 40, 152, 1000):
        out, step = run_gpu(li, sm_count=sms)
        assert step.plan.grid_y == Hkv
        modes.add(int(step.plan.merge_mode))
        compare(out, ref, li, f"d{d} G{G} kvs{kvs} W{window} sms{sms} S{step.plan.num_splits}")
    if window == 1000:
        assert modes == {0, 1, 2}, modes


@pytest.mark.parametrize("G", [3, 6])
def test_groups_between_the_decode_instances_over_fp8(G):
    li = synth.make_layer("gm8", [1, 17, 300, 1000, 33], 2 * G, 2, 512, window=37,
                          pool_pages=100, seed=90 + G, device="cuda")
    f = synth.quantize_kv_fp8(li)
    ref = run_oracle_fp8(f)
    for sms in (3, 152):
        out, step = run_gpu(f, sm_count=sms)
        compare(out, ref, f, f"fp8 G{G} sms{sms} S{step.plan.num_splits}")


def test_group_16_single_token_is_bit_exact():
    li = synth.make_layer("one16", [1, 1], 32, 2, 512, pool_pages=5, seed=13, device="cuda")
    out, _ = run_gpu(li)
    for bi in range(2):
        page = int(li.block_tables[bi, 0])
        assert torch.equal(out[bi], li.v_pool[page, :, 0, :].repeat_interleave(16, dim=0))


def test_page_size_32():
    lens = [100, 64, 5]
    li = synth.make_layer("p32", lens, 8, 2, 512, page_size=32, pool_pages=12, seed=5, device="cuda")
    compare(run_gpu(li)[0], run_oracle(li), li, "P32")


# ---- closed forms and invariants on the GPU ------------------------------------

@pytest.mark.parametrize("d,G,kvs", [(512, 4, False), (512, 4, True), (256, 2, False)])
def test_single_token_is_bit_exact(d, G, kvs):
    li = synth.make_layer("one", [1, 1, 1], 2 * G, 2, d, kv_shared=kvs, pool_pages=7, seed=3, device="cuda")
    for sms in (1, 152):
        out, _ = run_gpu(li, sm_count=sms)
        pool = li.k_pool if kvs else li.v_pool
        for bi in range(3):
            page = int(li.block_tables[bi, 0])
            want = pool[page, :, 0, :].repeat_interleave(G, dim=0)
            assert torch.equal(out[bi], want)


def test_empty_sequences_give_zero():
    li = synth.make_layer("empty", [0, 0, 40], 8, 2, 512, pool_pages=8, seed=4, device="cuda")
    out, _ = run_gpu(li)
    assert (out[:2] == 0).all()
    compare(out, run_oracle(li), li, "empty")


def test_deterministic_and_split_consistent():
    li = synth.workload(2, device="cuda")[0]
    a, _ = run_gpu(li)
    a2, _ = run_gpu(li)
    assert torch.equal(a, a2), "repeated runs differ"
    c, step_c = run_gpu(li, sm_count=1)
    assert step_c.plan.num_splits == 1
    diff = (a.float() - c.float()).abs().max().item()
    assert diff <= 2 * MAX_ABS


def test_page_permutation_is_bitwise_invariant():
    li = synth.make_layer("perm", [300, 1000, 77], 16, 4, 512, pool_pages=120, seed=6, device="cuda")
    a, step = run_gpu(li)
    g = torch.Generator().manual_seed(1)
    perm = torch.randperm(li.num_pages, generator=g)
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(li.num_pages)
    inv = inv.cuda()
    t2 = li.block_tables.clone()
    valid = t2 >= 0
    t2[valid] = perm.cuda()[t2[valid].long()].to(torch.int32)
    out2 = torch.empty_like(li.q)
    step(li.q, li.k_pool[inv].contiguous(), li.v_pool[inv].contiguous(), t2, li.seq_lens, li.scale, out2)
    assert step.check() == 0
    assert torch.equal(a, out2)


def test_window_ignores_rows_before_the_window():
    W = 100
    li = synth.make_layer("win", [1000, 517, 250], 16, 8, 256, window=W, pool_pages=120, seed=8, device="cuda")
    a, step = run_gpu(li)
    k2, v2 = li.k_pool.clone(), li.v_pool.clone()
    for bi, L in enumerate(li.seq_lens_list()):
        for t in range(0, L - W):
            page = int(li.block_tables[bi, t // 16])
            k2[page, :, t % 16] = 50.0
            v2[page, :, t % 16] = -50.0
    out2 = torch.empty_like(li.q)
    step(li.q, k2, v2, li.block_tables, li.seq_lens, li.scale, out2)
    assert torch.equal(a, out2)


# ---- device-side error reporting (the kernel's own checks; nothing faults) -------

@pytest.mark.parametrize("early_kv", [False, True])
def test_bad_page_id_sets_flag_and_skips_the_page(early_kv):
    # with early_kv the producer meets the bad page before its dependency wait;
    # the flag still reaches the error word (written only after that wait)
    li = synth.make_layer("bad", [64, 64], 8, 2, 512, pool_pages=10, seed=9, device="cuda")
    bt = li.block_tables.clone()
    bt[1, 2] = 10 ** 6  # far outside the pool
    step = b.LayerStep.for_inputs(li, early_kv=early_kv)
    out = torch.empty_like(li.q)
    step(li.q, li.k_pool, li.v_pool, bt, li.seq_lens, li.scale, out)
    with pytest.raises(b.PagedDecodeError) as e:
        step.check()
    assert e.value.status == b.PD_ERR_DEVICE_FAULT and e.value.flags & b.PD_DEVFLAG_BAD_PAGE
    assert step.check() == 0  # cleared
    ref = run_oracle(li)
    compare(out[:1], ref[:1], synth.make_layer("x", [64], 8, 2, 512, pool_pages=10, seed=9), "untouched row")
    assert torch.isfinite(out[1].float()).all()


def test_bad_seq_len_sets_flag():
    li = synth.make_layer("len", [64, 64], 8, 2, 512, pool_pages=10, seed=10, device="cuda")
    step = b.LayerStep.for_inputs(li)
    out = torch.empty_like(li.q)
    sl = li.seq_lens.clone()
    sl[0] = -5
    step(li.q, li.k_pool, li.v_pool, li.block_tables, sl, li.scale, out)
    with pytest.raises(b.PagedDecodeError) as e:
        step.check()
    assert e.value.flags & b.PD_DEVFLAG_BAD_SEQLEN
    assert (out[0] == 0).all()


def test_abi_rejects_bad_arguments_without_launching():
    li = synth.make_layer("args", [64], 8, 2, 512, pool_pages=5, seed=11, device="cuda")
    step = b.LayerStep.for_inputs(li)
    out = torch.zeros_like(li.q)
    cases = [
        dict(v_pool=None),                       # K != V layer without V
        dict(v_pool=li.k_pool),                  # V aliasing K on a K != V layer
        dict(scale=float("inf")),
        dict(q=li.q.view(-1)[1:]),               # misaligned q
    ]
    for kw in cases:
        args = dict(q=li.q, v_pool=li.v_pool, scale=li.scale)
        args.update(kw)
        with pytest.raises(b.PagedDecodeError) as e:
            b.paged_decode_global(step.plan, args["q"], li.k_pool, args["v_pool"], li.block_tables, li.seq_lens,
                                  args["scale"], step.workspace, out)
        assert e.value.status == b.PD_ERR_INVALID_ARG
    with pytest.raises(b.PagedDecodeError) as e:
        b.paged_decode_window(step.plan, li.q, li.k_pool, li.v_pool, li.block_tables, li.seq_lens, 16, li.scale,
                              step.workspace, out)
    assert e.value.status == b.PD_ERR_INVALID_ARG
    if step.plan.num_splits > 1:
        with pytest.raises(b.PagedDecodeError) as e:
            b.paged_decode_global(step.plan, li.q, li.k_pool, li.v_pool, li.block_tables, li.seq_lens, li.scale,
                                  step.workspace, out, workspace_bytes=16)
        assert e.value.status == b.PD_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert (out == 0).all()  # nothing ran
    assert step.check() == 0


@pytest.mark.parametrize("kvs,window,d", [(False, 0, 512), (True, 0, 512), (False, 45, 256)])
def test_nan_in_unattended_rows_does_not_leak(kvs, window, d):
    """Rows a page holds past the sequence end (and before a window) are never
    attended; whatever bits they hold must not reach the output."""
    lens = [37, 100, 250]
    li = synth.make_layer("nan", lens, 8, 2, d, window=window, kv_shared=kvs, pool_pages=30, seed=12,
                          device="cuda")
    ref = run_oracle(li)
    for bi, L in enumerate(lens):
        lo = max(0, L - window) if window else 0
        npages = (L + 15) // 16
        for t in list(range((lo // 16) * 16, lo)) + list(range(L, npages * 16)):
            page = int(li.block_tables[bi, t // 16])
            li.k_pool[page, :, t % 16] = float("nan")
            if li.v_pool is not None:
                li.v_pool[page, :, t % 16] = float("nan")
    out, _ = run_gpu(li)
    compare(out, ref, li, "nan rows")


MERGE_CASES = [  # (lengths, SM count given to the planner, merge mode it picks)
    ([1000, 977, 513, 64], 20, 2),      # 2 pieces merged in the cluster
    ([1000, 977, 513, 64], 4000, 2),    # 8 pieces merged in the cluster
    ([8000, 7000, 513, 64], 20, 1),     # 5 pieces, the merge launch
    ([8000, 7000, 513, 64], 1000, 1),   # 63 pieces
    ([9000], 1000, 1),                  # 141 pieces of one request
]


@pytest.mark.parametrize("lens,sms,mode", MERGE_CASES)
def test_many_pieces_merge(lens, sms, mode):
    """From a few pieces to one per 16-token page, in both merge modes: the
    merge matches the oracle, and a second call on the same workspace gives the
    same bits."""
    li = synth.make_layer("mm", lens, 16, 2, 512, pool_pages=sum((L + 15) // 16 for L in lens) + 8, seed=13,
                          device="cuda")
    ref = run_oracle(li)
    out, step = run_gpu(li, sm_count=sms)
    assert step.plan.num_splits > 1 and step.plan.merge_mode == mode
    compare(out, ref, li, f"S={step.plan.num_splits}")
    again = torch.empty_like(out)
    step.run(li, again)
    assert step.check() == 0
    assert torch.equal(out, again)


@pytest.mark.parametrize("lens,sms,mode", [([32], 152, 0), ([4000, 3000], 152, 1), ([1000, 900], 20, 2)])
def test_pipeline_wait_timeout_is_reported_and_context_survives(lens, sms, mode):
    """A stage that never completes (the copies deliver fewer bytes than the
    stage expects): every wait gives up after ~1 s, the kernel returns, the
    host reads PD_DEVFLAG_WAIT_TIMEOUT, and the next call on the same context
    is correct."""
    li = synth.make_layer("stall", lens, 4, 2, 256, pool_pages=sum((L + 15) // 16 for L in lens) + 2, seed=30,
                          device="cuda")
    step = b.LayerStep.for_inputs(li, sm_count=sms)
    assert step.plan.merge_mode == mode
    step.plan.test_stall_bytes = 16
    out = torch.zeros_like(li.q)
    step.run(li, out)
    with pytest.raises(b.PagedDecodeError) as e:
        step.check()
    assert e.value.status == b.PD_ERR_DEVICE_FAULT and e.value.flags & b.PD_DEVFLAG_WAIT_TIMEOUT
    step.plan.test_stall_bytes = 0
    out2, _ = run_gpu(li, sm_count=sms)
    compare(out2, run_oracle(li), li, "after a timed-out call")


# ---- FP8 (e4m3) KV cache -----------------------------------------------------------

def run_oracle_fp8(f):
    return oracle.decode_fp8(synth.bits_u16(f.q), f.k8.cpu().numpy(),
                             None if f.v8 is None else f.v8.cpu().numpy(), f.k_scale.cpu().numpy(),
                             None if f.v_scale is None else f.v_scale.cpu().numpy(), f.block_tables.cpu().numpy(),
                             f.seq_lens.cpu().numpy(), f.scale, f.window)


@pytest.mark.parametrize("d,G,kvs", FP8_VARIANTS + [(512, 16, True), (256, 12, False)])
@pytest.mark.parametrize("window", [0, 37])
@pytest.mark.parametrize("long", [False, True])
def test_fp8_variants_ragged(d, G, kvs, window, long):
    """Every FP8 instance on a ragged batch; K != V spans under 4096 tokens run
    on the six-warp instances, longer ones on the seven-warp ones."""
    Hkv = 2
    lens = [1, 17, 300, 0, 1000, 33] + ([5000] if long else [])
    li = synth.make_layer("f8", lens, Hkv * G, Hkv, d, window=window, kv_shared=kvs,
                          pool_pages=sum((L + 15) // 16 for L in lens) + 5, seed=500 + d + G + 100 * kvs + window,
                          device="cuda")
    f = synth.quantize_kv_fp8(li)
    ref = run_oracle_fp8(f)
    span = max(min(L, window) if window else L for L in lens)
    for sms in (3, 152):
        out, step = run_gpu(f, sm_count=sms)
        assert step.plan.threads_per_cta == (224 if not kvs and G <= 8 and span < 4096 else 256)
        compare(out, ref, f, f"fp8 d{d} G{G} kvs{kvs} W{window} sms{sms} S{step.plan.num_splits}")


@pytest.mark.parametrize("cid,part", [(2, None), (3, None), (4, "c"), (5, "global"), (5, "sliding")])
def test_fp8_workload_matches_oracle(cid, part):
    for li in synth.workload(cid, device="cuda", part=part):
        f = synth.quantize_kv_fp8(li)
        step = b.LayerStep.for_inputs(f, early_kv=True)
        first = step.run(f, torch.full_like(f.q, float("nan")))
        out = step.run(f, torch.full_like(f.q, float("nan")))
        assert step.check() == 0
        ref = run_oracle_fp8(f)
        compare(first, ref, f, f"{f.name} first step")
        err, cos, row_cos, rel = compare(out, ref, f, f"{f.name} S={step.plan.num_splits}")
        print(f"{f.name}: splits {step.plan.num_splits} max_abs {err:.2e} cos {cos:.7f} worst row cos {row_cos:.6f} "
              f"rel L2 {rel:.2e}")


def test_fp8_nan_bytes_in_unattended_rows_do_not_leak():
    lens = [37, 100, 250]
    li = synth.make_layer("f8nan", lens, 8, 2, 512, pool_pages=30, seed=31, device="cuda")
    f = synth.quantize_kv_fp8(li)
    ref = run_oracle_fp8(f)
    for bi, L in enumerate(lens):
        for t in range(L, (L + 15) // 16 * 16):
            page = int(f.block_tables[bi, t // 16])
            f.k8[page, :, t % 16] = 0x7F  # e4m3 NaN
            f.v8[page, :, t % 16] = 0xFF
    out, _ = run_gpu(f)
    compare(out, ref, f, "fp8 nan rows")


def test_fp8_scales_reach_the_result():
    """Doubling every V scale doubles the output; doubling every K scale equals
    doubling the softmax scale."""
    li = synth.make_layer("f8s", [500, 70], 8, 2, 512, pool_pages=40, seed=32, device="cuda")
    f = synth.quantize_kv_fp8(li)
    out, step = run_gpu(f)
    f.v_scale.mul_(2)
    out2 = torch.empty_like(out)
    step.run(f, out2)
    assert step.check() == 0
    assert torch.allclose(out2.float(), 2 * out.float(), rtol=1e-2, atol=1e-3)
    f.v_scale.div_(2)
    import dataclasses
    f.k_scale.mul_(2)
    out3 = torch.empty_like(out)
    step.run(f, out3)
    f.k_scale.div_(2)
    out4 = torch.empty_like(out)
    step.run(dataclasses.replace(f, scale=2 * f.scale), out4)
    assert step.check() == 0
    assert torch.equal(out3, out4)  # products with 2 are exact in fp32
    assert not torch.equal(out3, out)


def test_one_workspace_serves_changing_plans():
    """Serving replans every step: one workspace, zeroed once, runs plans of
    every merge mode and of different batches in turn, each call matching the
    oracle and leaving the error word clear."""
    shapes = [  # (lengths, SM count, merge mode)
        ([4097, 1500, 77, 0, 3000], 152, 1),
        ([9000], 1000, 1),
        ([2000] * 8, 152, 2),
        ([8000, 7000, 513, 64, 1, 4000, 300, 2500], 40, 1),
        ([300, 17], 1, 0),
        ([4097, 1500, 77, 0, 3000], 152, 1),
    ]
    layers, plans, need = [], [], 0
    for i, (lens, sms, mode) in enumerate(shapes):
        li = synth.make_layer(f"ws{i}", lens, 16, 4, 512, pool_pages=sum((L + 15) // 16 for L in lens) + 8,
                              seed=40 + i, device="cuda")
        step = b.LayerStep.for_inputs(li, sm_count=sms)
        assert step.plan.merge_mode == mode, (lens, sms, step.plan.merge_mode)
        layers.append(li)
        plans.append(step.plan)
        need = max(need, int(step.plan.workspace_bytes))
    ws = torch.zeros((need + 255) // 256 * 256, dtype=torch.uint8, device="cuda")
    for rep in range(2):
        for li, plan in zip(layers, plans):
            out = torch.full_like(li.q, float("nan"))
            b.paged_decode_global(plan, li.q, li.k_pool, li.v_pool, li.block_tables, li.seq_lens, li.scale, ws, out)
            b.paged_decode_merge(plan, ws, out)
            assert b.paged_decode_check_device_error(plan, ws) == 0
            compare(out, run_oracle(li), li, f"rep {rep} mode {plan.merge_mode} S={plan.num_splits}")


@pytest.mark.parametrize("d,G,kvs,window,T,fp8", [(512, 4, False, 0, 1, False), (512, 4, True, 0, 1, False),
                                                  (256, 2, False, 1024, 1, False), (512, 4, False, 0, 3, False),
                                                  (256, 8, False, 37, 2, False), (512, 4, False, 0, 1, True),
                                                  (256, 2, True, 1024, 1, True)])
@pytest.mark.parametrize("sms", [3, 40, 152, 1000])
def test_plan_made_for_longer_lengths_serves_shorter_ones(d, G, kvs, window, T, fp8, sms):
    """A plan stays valid for any later step whose lengths do not exceed the
    ones it was made for: planned with headroom (lengths + 2000), run on the
    actual lengths (a request one token long, an empty one when decoding one
    token), against the oracle at the actual lengths."""
    Hkv = 2
    lens = [max(T, L) for L in [4100, 1, 777, 0, 3000]] if T > 1 else [4100, 1, 777, 0, 3000]
    plan_lens = [L + 2000 for L in lens]
    li = synth.make_layer("hr", lens, Hkv * G, Hkv, d, window=window, kv_shared=kvs,
                          pool_pages=sum((L + 15) // 16 for L in lens) + 3, seed=d + G + window + T + 7 * fp8,
                          device="cuda")
    desc = b.layer_desc(Hkv * G, Hkv, d, 16, li.num_pages, (max(plan_lens) + 15) // 16, window, kvs,
                        b.PD_KV_FP8_E4M3 if fp8 else b.PD_KV_BF16)
    plan = b.paged_decode_plan_multi(desc, T, plan_lens, sms) if T > 1 else b.paged_decode_plan(desc, plan_lens, sms)
    # the block table is as wide as the plan's layer says: pad the rows
    table = torch.zeros(len(lens), desc.max_pages_per_seq, dtype=torch.int32, device="cuda")
    table[:, :li.block_tables.shape[1]] = li.block_tables
    g = torch.Generator(device="cuda").manual_seed(3 + sms)
    q = li.q if T == 1 else torch.randn(len(lens), T, Hkv * G, d, generator=g, device="cuda").to(torch.bfloat16)
    ws = torch.zeros(max(256, int(plan.workspace_bytes)), dtype=torch.uint8, device="cuda")
    out = torch.full_like(q, float("nan"))
    if fp8:
        f8 = synth.quantize_kv_fp8(li)
        args = (plan, q, f8.k8, f8.v8, f8.k_scale, f8.v_scale, table, li.seq_lens)
        if window > 0:
            b.paged_decode_window_fp8(*args, window, li.scale, ws, out)
        else:
            b.paged_decode_global_fp8(*args, li.scale, ws, out)
    else:
        args = (plan, q, li.k_pool, li.v_pool, table, li.seq_lens)
        if window > 0:
            b.paged_decode_window(*args, window, li.scale, ws, out)
        else:
            b.paged_decode_global(*args, li.scale, ws, out)
    b.paged_decode_merge(plan, ws, out)
    assert b.paged_decode_check_device_error(plan, ws) == 0
    tables, seq = li.block_tables.cpu().numpy(), li.seq_lens.cpu().numpy()
    if fp8:
        k8, v8 = f8.k8.cpu().numpy(), None if f8.v8 is None else f8.v8.cpu().numpy()
        ks, vs = f8.k_scale.cpu().numpy(), None if f8.v_scale is None else f8.v_scale.cpu().numpy()
        ref = oracle.decode_fp8(synth.bits_u16(q), k8, v8, ks, vs, tables, seq, li.scale, window)
        compare(out, ref, f8, f"fp8 S={plan.num_splits} mode={plan.merge_mode}")
    elif T == 1:
        compare(out, run_oracle(li), li, f"S={plan.num_splits} mode={plan.merge_mode}")
    else:
        ref = oracle.decode_multi(synth.bits_u16(q.cpu()), synth.bits_u16(li.k_pool),
                                  None if li.v_pool is None else synth.bits_u16(li.v_pool), tables, seq, li.scale,
                                  window)
        got = out.float().cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all() and np.abs(got - ref).max() <= MAX_ABS
