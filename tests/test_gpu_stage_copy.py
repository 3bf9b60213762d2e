"""paged_decode_stage_copy: copies between page-locked host memory and device
memory as one kernel in the stream's chain of programmatic dependent launches,
and the host-in/host-out decode loop built on it (after step i's kernels one
copy brings step i + 1's q in, the block table and lengths of the step one
on -- two on with pd_plan.early_kv, whose stage 1 reads them before its wait --
and takes step i - 1's result out; a last copy, waiting first, takes the final
result out).

The loop's steps each get their own q and lengths, so a copy that landed late
or a result taken before its step finished shows up as a wrong step; every
host result is compared bit for bit with the same decode run on its own
(itself held to the oracle by the parity tests). Eager calls and a CUDA graph
of the loop, with and without early_kv, merge in a cluster and through the
merge kernel, K=V and K!=V, a window layer, FP8.
"""
import numpy as np
import pytest
import torch

from paged_gqa_decode_global_gb300 import binding as b
from paged_gqa_decode_global_gb300 import host_loop
from paged_gqa_decode_global_gb300 import inputs as synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("nbytes", [16, 4096 + 16, 3 << 20])
@pytest.mark.parametrize("after_wait", [0, 1])
def test_round_trip_through_the_device(nbytes, after_wait):
    g = torch.Generator().manual_seed(nbytes + after_wait)
    src = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, generator=g).pin_memory()
    dev = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    back = torch.zeros(nbytes, dtype=torch.uint8).pin_memory()
    b.paged_decode_stage_copy([(dev, src)], after_wait)
    b.paged_decode_stage_copy([(back, dev)], 1)  # waits for the copy in front
    torch.cuda.synchronize()
    assert torch.equal(back, src)
    assert torch.equal(dev.cpu(), src)


def test_four_copies_of_one_launch():
    g = torch.Generator().manual_seed(7)
    a = torch.randint(0, 256, (1 << 16,), dtype=torch.uint8, generator=g).pin_memory()
    c = torch.randint(0, 256, (3 * 1024,), dtype=torch.uint8, generator=g).cuda()
    e = torch.randint(0, 256, (48,), dtype=torch.uint8, generator=g).pin_memory()
    f = torch.randint(0, 256, (5 << 20,), dtype=torch.uint8, generator=g).cuda()
    a_dev, e_dev = torch.empty_like(a, device="cuda"), torch.empty_like(e, device="cuda")
    c_host = torch.zeros(c.shape, dtype=torch.uint8).pin_memory()
    f_dev = torch.zeros_like(f)
    b.paged_decode_stage_copy([(a_dev, a), (c_host, c), (e_dev, e), (f_dev, f)], 0)
    torch.cuda.synchronize()
    assert torch.equal(a_dev.cpu(), a)
    assert torch.equal(c_host, c.cpu())
    assert torch.equal(e_dev.cpu(), e)
    assert torch.equal(f_dev, f)


def test_refused_without_launching():
    dev = torch.zeros(256, dtype=torch.uint8, device="cuda")
    pinned = torch.zeros(256, dtype=torch.uint8).pin_memory()
    pageable = torch.zeros(256, dtype=torch.uint8)
    cases = [
        (dev, pageable, 0),               # pageable host memory
        (dev[8:24], pinned[:16], 0),      # misaligned destination
        (dev[:8], pinned[:8], 0),         # not a multiple of 16 bytes
        (dev[16:48], dev[0:32], 0),       # source and destination overlap
        (dev[:16], pinned[:16], 2),       # after_wait neither 0 nor 1
    ]
    for dst, src, wait in cases:
        with pytest.raises(b.PagedDecodeError) as e:
            b.paged_decode_stage_copy([(dst, src)], wait)
        assert e.value.status == b.PD_ERR_INVALID_ARG
    with pytest.raises(b.PagedDecodeError) as e:  # more than PD_MAX_STAGE_COPIES
        b.paged_decode_stage_copy([(dev[16 * i:16 * i + 16], pinned[16 * i:16 * i + 16]) for i in range(5)])
    assert e.value.status == b.PD_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        b.paged_decode_stage_copy([(dev, None)])
    torch.cuda.synchronize()
    assert int(dev.count_nonzero()) == 0


LOOP_CASES = [
    # (head_dim, group, kv heads, K=V, window, lengths, SM count the plan is made for, fp8)
    (512, 4, 4, False, 0, [1024] * 8, 152, False),        # clusters of 4 (64 MiB layer's shape)
    (512, 4, 4, False, 0, [3000, 777, 4096, 1], 400, False),  # many pieces: the merge kernel
    (256, 2, 8, False, 1024, [1500, 4000, 300], 152, False),  # window layer
    (512, 4, 2, True, 0, [2048, 513], 152, False),            # K=V
    (512, 4, 4, False, 0, [2000, 1024, 64], 152, True),       # FP8 cache
]


def _layer(case, seed):
    d, G, Hkv, kvs, window, lens, sms, fp8 = case
    li = synth.make_layer("loop", lens, G * Hkv, Hkv, d, window=window, kv_shared=kvs,
                          pool_pages=sum((L + 15) // 16 for L in lens) + 4, seed=seed, device="cuda")
    return (synth.quantize_kv_fp8(li) if fp8 else li), sms


def _staged(tensors_per_step, parts):
    """One pinned host buffer per step holding its tensors (each 256-byte
    aligned) and the layout (offsets, total bytes) of `parts`."""
    offs, total = [], 0
    for t in parts:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    hosts = []
    for tensors in tensors_per_step:
        h = torch.zeros(total, dtype=torch.uint8).pin_memory()
        for t, o in zip(tensors, offs):
            n = t.numel() * t.element_size()
            h[o:o + n].view(t.dtype).view(t.shape).copy_(t.cpu())
        hosts.append(h)
    return hosts, offs, total


def _device_buffers(parts, offs, total, n):
    bufs = [torch.zeros(total, dtype=torch.uint8, device="cuda") for _ in range(n)]
    views = [[s[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for t, o in zip(parts, offs)]
             for s in bufs]
    return bufs, views


@pytest.mark.parametrize("graph", [False, True], ids=["eager", "graph"])
@pytest.mark.parametrize("early_kv", [0, 1], ids=["table-1-ahead", "early_kv-table-2-ahead"])
@pytest.mark.parametrize("case", LOOP_CASES, ids=[f"d{c[0]}-G{c[1]}-kvs{int(c[3])}-W{c[4]}-sm{c[6]}-fp8{int(c[7])}"
                                                  for c in LOOP_CASES])
def test_host_in_host_out_loop(case, early_kv, graph):
    li, sms = _layer(case, seed=11)
    step = b.LayerStep.for_inputs(li, sm_count=sms, early_kv=bool(early_kv))
    ahead = 2 if early_kv else 1  # steps the block table and lengths go ahead of their decode
    fp8 = hasattr(li, "k8")
    k, v = (li.k8, li.v8) if fp8 else (li.k_pool, li.v_pool)
    ks, vs = (li.k_scale, li.v_scale) if fp8 else (None, None)
    n_steps = 7
    gen = torch.Generator(device="cuda").manual_seed(3)
    lens0 = li.seq_lens.cpu()
    # each step its own q and lengths (a request shrinking by 5 tokens a step, never below 1 if it had any)
    qs = [(torch.randn(li.q.shape, generator=gen, device="cuda")).to(torch.bfloat16) for _ in range(n_steps)]
    lens = [torch.where(lens0 > 0, torch.clamp(lens0 - 5 * j, min=1), lens0).to(torch.int32) for j in range(n_steps)]

    # what each step gives run on its own
    expect = []
    for j in range(n_steps):
        out = torch.empty_like(li.q)
        step(qs[j], k, v, li.block_tables, lens[j].cuda(), li.scale, out, k_scale=ks, v_scale=vs)
        expect.append(out.cpu())
    torch.cuda.synchronize()
    assert step.check() == 0

    q_h, q_offs, q_total = _staged([[qs[j]] for j in range(n_steps)], [li.q])
    meta_parts = [li.block_tables, li.seq_lens]
    meta_h, m_offs, m_total = _staged([[li.block_tables, lens[j]] for j in range(n_steps)], meta_parts)
    q_dev, q_views = _device_buffers([li.q], q_offs, q_total, 2)
    m_dev, m_views = _device_buffers(meta_parts, m_offs, m_total, 3)
    dev_out = [torch.empty_like(li.q) for _ in range(2)]
    host_out = [torch.zeros(li.q.shape, dtype=torch.bfloat16).pin_memory() for _ in range(n_steps)]
    stream = torch.cuda.Stream()

    sch = host_loop.schedule(n_steps, early_kv=bool(early_kv))
    assert sch.ahead == ahead

    def dst(c):
        return q_dev[c.buffer] if c.kind == "q" else m_dev[c.buffer] if c.kind == "meta" else host_out[c.step]

    def src(c):
        return q_h[c.step] if c.kind == "q" else meta_h[c.step] if c.kind == "meta" else dev_out[c.buffer]

    def loop():
        for c in sch.before:  # ordinary copies before the loop
            dst(c).copy_(src(c), non_blocking=True)
        for j in range(n_steps):
            (q,), (bt, sl) = q_views[host_loop.q_buffer(j)], m_views[host_loop.meta_buffer(j)]
            step(q, k, v, bt, sl, li.scale, dev_out[host_loop.out_buffer(j)], stream, k_scale=ks, v_scale=vs)
            b.paged_decode_stage_copy([(dst(c), src(c)) for c in sch.after_step[j]], 0, stream)
        b.paged_decode_stage_copy([(dst(c), src(c)) for c in sch.final], 1, stream)

    if graph:
        with torch.cuda.stream(stream):
            loop()  # warm-up outside the capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            loop()
        for h in host_out:
            h.zero_()
        for _ in range(2):
            g.replay()
    else:
        with torch.cuda.stream(stream):
            loop()
    torch.cuda.synchronize()
    assert step.check() == 0
    for j in range(n_steps):
        assert torch.equal(host_out[j], expect[j]), f"step {j}"


@pytest.mark.parametrize("graph", [False, True], ids=["eager", "graph"])
def test_new_token_step_loop_copies_after_waiting(graph):
    """Behind paged_decode_qkv_norm_rope_write, which lets its dependents start
    before its own wait, the loop copies with after_wait 1: the next step's new
    rows in and that step's q out. Seven steps, each with its own rows; every
    host q equals the step run on its own."""
    lens = [1000, 17, 4096, 1]
    li = synth.make_layer("newtok", lens, 16, 4, 512, pool_pages=sum((L + 15) // 16 for L in lens) + 4, seed=5,
                          device="cuda")
    pi = synth.make_prepare(li, rot=128, theta=1e6, seed=5)
    desc = b.layer_desc(li.num_q_heads, li.num_kv_heads, li.head_dim, li.page_size, li.num_pages,
                        li.block_tables.shape[1], 0, False)
    cos_sin = torch.empty(pi.max_positions, pi.rot, dtype=torch.float32, device="cuda")
    b.paged_decode_rope_table(pi.theta, pi.rot, pi.max_positions, cos_sin)
    k_pool, v_pool = li.k_pool.clone(), li.v_pool.clone()
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    n_steps = 7
    gen = torch.Generator(device="cuda").manual_seed(9)
    rows = [[(3.0 * torch.randn(t.shape, generator=gen, device="cuda")).to(torch.bfloat16)
             for t in (pi.q_in, pi.k_in, pi.v_in)] for _ in range(n_steps)]

    def prep(q_in, k_in, v_in, seq, q_out, stream=None):
        b.paged_decode_qkv_norm_rope_write(desc, pi.rot, pi.max_positions, pi.eps, q_in, k_in, v_in, pi.q_w,
                                           pi.k_w, pi.v_w, cos_sin, li.block_tables, seq, q_out, k_pool, v_pool,
                                           flags, stream)

    expect = []
    for j in range(n_steps):
        q_out = torch.empty_like(pi.q_in)
        prep(*rows[j], li.seq_lens, q_out)
        expect.append(q_out.cpu())
    torch.cuda.synchronize()
    assert int(flags.item()) == 0

    parts = [pi.q_in, pi.k_in, pi.v_in, li.seq_lens]
    offs, total = [], 0
    for t in parts:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    stage_h = []
    for j in range(n_steps):
        h = torch.zeros(total, dtype=torch.uint8).pin_memory()
        for t, o in zip(rows[j] + [li.seq_lens], offs):
            n = t.numel() * t.element_size()
            h[o:o + n].view(t.dtype).view(t.shape).copy_(t.cpu())
        stage_h.append(h)
    dev_stage = [torch.zeros(total, dtype=torch.uint8, device="cuda") for _ in range(2)]
    views = [[s[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for t, o in zip(parts, offs)]
             for s in dev_stage]
    dev_q = [torch.empty_like(pi.q_in) for _ in range(2)]
    host_q = [torch.zeros(pi.q_in.shape, dtype=torch.bfloat16).pin_memory() for _ in range(n_steps)]
    stream = torch.cuda.Stream()

    def loop():
        b.paged_decode_stage_copy([(dev_stage[0], stage_h[0])], 0, stream)
        for j in range(n_steps):
            cur, other = j % 2, (j + 1) % 2
            q, k, v, sl = views[cur]
            prep(q, k, v, sl, dev_q[cur], stream)
            more = j + 1 < n_steps
            b.paged_decode_stage_copy([(dev_stage[other], stage_h[j + 1]) if more else (None, None),
                                       (host_q[j], dev_q[cur])], 1, stream)

    if graph:
        with torch.cuda.stream(stream):
            loop()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            loop()
        for h in host_q:
            h.zero_()
        g.replay()
    else:
        with torch.cuda.stream(stream):
            loop()
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    for j in range(n_steps):
        assert torch.equal(host_q[j], expect[j]), f"step {j}"
