"""The allocation-free entry point (paged_decode_noalloc) against the fp64
oracle and against the workspace entry points.

paged_decode_noalloc serves callers that may not allocate device memory, such
as an engine plugin whose host owns all device memory or a serving loop that
must not call cudaMalloc mid-step; it runs the same decode step on a scratch
array inside the library. Each case makes two calls in a row with different
queries: the second call finds the first call's partials in the shared array
and must not be affected by them. The cases cover each merge mode: one piece
(nothing in the array but the error word), pieces merged inside a
thread-block cluster (likewise), and pieces merged by the merge kernel, whose
fp32 partials and log-sum-exps live in the array.

This file is named to be collected last.
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


def _close(a, ref, tag):
    x = a.float().cpu().numpy().astype(np.float64).ravel() if torch.is_tensor(a) else a.ravel()
    y = ref.float().cpu().numpy().astype(np.float64).ravel() if torch.is_tensor(ref) else ref.ravel()
    assert np.isfinite(x).all(), tag
    err = np.abs(x - y).max()
    cos = float(x @ y / (np.linalg.norm(x) * np.linalg.norm(y)))
    assert err <= MAX_ABS and cos > MIN_COS, f"{tag}: max abs {err:.3e} cos {cos:.7f}"


def _oracle(li, q):
    return oracle.decode(synth.bits_u16(q), synth.bits_u16(li.k_pool),
                         None if li.v_pool is None else synth.bits_u16(li.v_pool),
                         li.block_tables.cpu().numpy(), li.seq_lens.cpu().numpy(), li.scale, li.window)


LENS = [4097, 1500, 77, 0, 3000]

# (lengths, window, K=V, head_dim, group, merge mode the plan must have)
CASES = [
    (LENS, 0, False, 512, 4, 0),
    (LENS, 0, False, 512, 4, 1),
    (LENS, 0, True, 512, 4, 1),
    (LENS, 1024, False, 256, 2, 1),
    (LENS, 1024, False, 256, 2, 2),
    ([1024] * 8, 0, False, 512, 4, 2),
]


def _step_with_mode(li, mode):
    """A plan in the wanted merge mode: the first of these SM counts (given to
    the planner) that makes the planner choose it."""
    for sms in (152, 160, 132, 100, 64, 48, 40, 32, 24, 16, 8, 4, 1):
        step = b.LayerStep.for_inputs(li, sm_count=sms)
        if int(step.plan.merge_mode) == mode:
            return step
    raise AssertionError(f"no SM count gives merge mode {mode}")


@pytest.mark.parametrize("lens,window,kvs,d,G,mode", CASES)
def test_noalloc_matches_oracle_and_workspace_path_twice(lens, window, kvs, d, G, mode):
    li = synth.make_layer("na", lens, 4 * G, 4, d, window=window, kv_shared=kvs,
                          pool_pages=sum((L + 15) // 16 for L in lens) + 8, seed=21 + d + window + kvs + mode,
                          device="cuda")
    step = _step_with_mode(li, mode)
    sms = int(step.plan.sm_count)
    if mode == 1:
        # the merge kernel reads partials from the scratch array
        assert step.plan.workspace_bytes > 256 and step.plan.num_splits > 1
    gen = torch.Generator(device="cuda").manual_seed(77 + sms)
    queries = [li.q, torch.randn(li.q.shape, generator=gen, device="cuda").to(torch.bfloat16)]
    flags = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call, q in enumerate(queries):
        ref_ws = torch.full_like(q, float("nan"))
        step(q, li.k_pool, li.v_pool, li.block_tables, li.seq_lens, li.scale, ref_ws)
        assert step.check() == 0
        out = torch.full_like(q, float("nan"))
        b.paged_decode_noalloc(step.plan, q, li.k_pool, li.v_pool, li.block_tables, li.seq_lens, window,
                               li.scale, out, device_flags=flags)
        torch.cuda.synchronize()
        assert int(flags.item()) == 0, f"call {call}: device flags {int(flags.item()):#x}"
        tag = f"call {call}, merge mode {mode}, S={step.plan.num_splits}"
        _close(out, ref_ws, tag + " vs the workspace path")
        _close(out.float().cpu().numpy().astype(np.float64), _oracle(li, q), tag + " vs the oracle")


def test_noalloc_rejects_plans_beyond_its_scratch():
    # a plan for 4 requests x 16 heads x ~150 pieces (planned for 4000 SMs) needs
    # far more than 8 MiB of partials; the call must refuse it before touching
    # any buffer
    lens = [131072] * 4
    plan = b.paged_decode_plan(b.layer_desc(16, 4, 512, 16, 4 * 8192 + 1, 8192), lens, 4000)
    li = synth.make_layer("small", [16], 16, 4, 512, pool_pages=2, seed=3, device="cuda")
    assert plan.workspace_bytes > 8 << 20
    out = torch.zeros_like(li.q)
    with pytest.raises(b.PagedDecodeError) as e:
        b.paged_decode_noalloc(plan, li.q, li.k_pool, li.v_pool, li.block_tables, li.seq_lens, 0, li.scale, out)
    assert e.value.status == b.PD_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert (out == 0).all()


def _random_cases(n=20, seed=20261208):
    """Seeded random bf16 shapes (head_dim, group 1..16, K=V, 1..4 query
    tokens, windows, ragged requests, the SM count the plan is sized for)
    whose plans fit the 8 MiB scratch array."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        d = int(rng.choice([256, 512]))
        G = int(rng.choice([1, 2, 3, 4, 8, 12, 16]))
        Hkv = int(rng.choice([1, 2, 4]))
        kvs = bool(rng.random() < 0.4)
        T = 1 if rng.random() < 0.6 else int(rng.choice([2, 4]))
        window = int(rng.choice([0, 0, 37, 1024]))
        B = int(rng.integers(1, 7))
        lens = [max(T, int(x)) for x in np.exp(rng.uniform(0.0, np.log(6000), B))]
        sms = int(rng.choice([3, 40, 152, 1000]))
        if B * T * G * Hkv * max(lens) > 3_000_000:
            continue
        desc = b.layer_desc(G * Hkv, Hkv, d, 16, sum((L + 15) // 16 for L in lens) + 3,
                            max((L + 15) // 16 for L in lens), window, kvs)
        plan = b.paged_decode_plan_multi(desc, T, lens, sms) if T > 1 else b.paged_decode_plan(desc, lens, sms)
        if plan.workspace_bytes > 8 << 20:
            continue
        out.append((d, G, Hkv, kvs, T, window, lens, sms))
    return out


def _random_id(c):
    d, G, Hkv, kvs, T, window, lens, sms = c
    return f"d{d}-G{G}-Hkv{Hkv}-kvs{int(kvs)}-T{T}-W{window}-B{len(lens)}-sm{sms}"


@pytest.mark.parametrize("case", _random_cases(), ids=_random_id)
def test_noalloc_random_shapes_match_oracle_twice(case):
    d, G, Hkv, kvs, T, window, lens, sms = case
    li = synth.make_layer("nar", lens, G * Hkv, Hkv, d, window=window, kv_shared=kvs,
                          pool_pages=sum((L + 15) // 16 for L in lens) + 3, seed=d + G + T + len(lens),
                          device="cuda")
    desc = b.layer_desc(G * Hkv, Hkv, d, 16, li.num_pages, li.block_tables.shape[1], window, kvs)
    plan = b.paged_decode_plan_multi(desc, T, lens, sms) if T > 1 else b.paged_decode_plan(desc, lens, sms)
    gen = torch.Generator(device="cuda").manual_seed(5 + sms)
    flags = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    kp = synth.bits_u16(li.k_pool)
    vp = None if li.v_pool is None else synth.bits_u16(li.v_pool)
    tables, seq = li.block_tables.cpu().numpy(), li.seq_lens.cpu().numpy()
    for call in range(2):
        q = (torch.randn((len(lens), T, G * Hkv, d) if T > 1 else tuple(li.q.shape), generator=gen,
                         device="cuda")).to(torch.bfloat16)
        out = torch.full_like(q, float("nan"))
        b.paged_decode_noalloc(plan, q, li.k_pool, li.v_pool, li.block_tables, li.seq_lens, window, li.scale, out,
                               device_flags=flags)
        torch.cuda.synchronize()
        assert int(flags.item()) == 0, f"call {call}: device flags {int(flags.item()):#x}"
        if T == 1:
            ref = oracle.decode(synth.bits_u16(q), kp, vp, tables, seq, li.scale, window)
        else:
            ref = oracle.decode_multi(synth.bits_u16(q.cpu()), kp, vp, tables, seq, li.scale, window)
        _close(out.float().cpu().numpy().astype(np.float64), ref, f"call {call}, S={plan.num_splits} "
               f"mode={plan.merge_mode}")
