"""Decode with pd_plan.early_kv, launched back to back on one stream, against
the fp64 oracle.

Each case queues three decodes of the same layer with no host sync between
them, so every decode after the first becomes resident while the one before
drains (programmatic dependent launch) and its producer copies the first
ring fill before its dependency wait. Every output must still equal the
oracle's at the decode bar (max |err| <= 2e-2, cosine > 0.9995), with no
device flag. The cases cover one piece, the in-cluster merge and the merge
kernel, K=V and K!=V, the window, the FP8 cache and several query tokens
(whose newest T rows the producer copies only after the wait). A case where
the kernel before writes the newest row (the new-token step) is in
test_gpu_prepare.py.
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


def _compare(out, ref, tag):
    got = out.float().cpu().double().numpy()
    assert np.isfinite(got).all(), f"{tag}: non-finite output"
    err = np.abs(got - ref).max()
    g, r = got.ravel(), ref.ravel()
    cos = float(g @ r / (np.linalg.norm(g) * np.linalg.norm(r)))
    assert err <= MAX_ABS, f"{tag}: max abs {err:.3e}"
    assert cos > MIN_COS, f"{tag}: cosine {cos:.7f}"


def _layer(lens, Hq, Hkv, d, window, kvs, seed):
    pool = sum((L + 15) // 16 for L in lens) + 4
    return synth.make_layer("early", lens, Hq, Hkv, d, window=window, kv_shared=kvs, pool_pages=pool, seed=seed,
                            device="cuda")


def _chain(step, calls, stream):
    """Queue calls() three times on `stream` without a host sync; returns the outputs."""
    outs = []
    with torch.cuda.stream(stream):
        for _ in range(3):
            outs.append(calls())
    stream.synchronize()
    assert step.check(stream) == 0
    return outs


CASES = [
    # name, lens, Hq, Hkv, d, window, kv_shared, sm_count (sets the merge mode)
    ("global d512 one piece", [300, 17, 1, 64], 16, 4, 512, 0, False, 4),
    ("global d512 cluster", [1000, 977, 513, 64], 16, 4, 512, 0, False, 152),
    ("global d512 K=V cluster of 8", [1000, 977, 513, 64], 16, 2, 512, 0, True, 4000),
    ("global d512 K=V merge kernel", [8000, 7000, 513, 64], 16, 2, 512, 0, True, 20),
    ("global d512 K=V merge kernel, 125 pieces", [20000, 64], 16, 2, 512, 0, True, 1000),
    ("sliding d256", [4100, 4000, 1, 15], 16, 8, 256, 1024, False, 152),
    ("sliding d256 K=V", [700, 33, 129], 8, 4, 256, 100, True, 152),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_early_kv_chain_matches_oracle(case):
    name, lens, Hq, Hkv, d, window, kvs, sms = case
    li = _layer(lens, Hq, Hkv, d, window, kvs, seed=len(name) + d)
    ref = oracle.decode(synth.bits_u16(li.q), synth.bits_u16(li.k_pool),
                        None if li.v_pool is None else synth.bits_u16(li.v_pool), li.block_tables.cpu().numpy(),
                        li.seq_lens.cpu().numpy(), li.scale, li.window)
    step = b.LayerStep.for_inputs(li, sm_count=sms, early_kv=True)
    assert step.plan.early_kv == 1
    s = torch.cuda.Stream()
    outs = _chain(step, lambda: step.run(li, stream=s), s)
    for i, out in enumerate(outs):
        _compare(out, ref, f"{name} call {i} (S={step.plan.num_splits}, mode {step.plan.merge_mode})")
    assert torch.equal(outs[1], outs[2])


@pytest.mark.parametrize("window,kvs", [(0, False), (0, True), (37, False)])
def test_early_kv_chain_fp8(window, kvs):
    li = _layer([1, 17, 300, 1000, 33], 8, 2, 512, window, kvs, seed=71 + window)
    f = synth.quantize_kv_fp8(li)
    ref = oracle.decode_fp8(synth.bits_u16(f.q), f.k8.cpu().numpy(), None if f.v8 is None else f.v8.cpu().numpy(),
                            f.k_scale.cpu().numpy(), None if f.v_scale is None else f.v_scale.cpu().numpy(),
                            f.block_tables.cpu().numpy(), f.seq_lens.cpu().numpy(), f.scale, f.window)
    step = b.LayerStep.for_inputs(f, early_kv=True)
    s = torch.cuda.Stream()
    outs = _chain(step, lambda: step.run(f, stream=s), s)
    for i, out in enumerate(outs):
        _compare(out, ref, f"fp8 W{window} kvs{kvs} call {i}")


@pytest.mark.parametrize("T,window,sms", [(2, 0, 152), (4, 0, 152), (4, 50, 152), (3, 0, 4000)])
def test_early_kv_chain_multi_token(T, window, sms):
    lens = [T, 17, 300, 1000]
    li = _layer(lens, 16, 4, 512, window, False, seed=90 + T + window)
    g = torch.Generator(device="cuda").manual_seed(5 + T)
    q = (0.5 * torch.randn(len(lens), T, 16, 512, generator=g, device="cuda")).to(torch.bfloat16)
    ref = oracle.decode_multi(synth.bits_u16(q.cpu()), synth.bits_u16(li.k_pool.cpu()),
                              synth.bits_u16(li.v_pool.cpu()), li.block_tables.cpu().numpy(),
                              li.seq_lens.cpu().numpy(), li.scale, li.window)
    step = b.LayerStep.for_inputs(li, sm_count=sms, query_tokens=T, early_kv=True)
    s = torch.cuda.Stream()

    def call():
        out = torch.empty_like(q)
        return step(q, li.k_pool, li.v_pool, li.block_tables, li.seq_lens, li.scale, out, s)

    outs = _chain(step, call, s)
    for i, out in enumerate(outs):
        _compare(out, ref, f"T={T} W{window} call {i} (S={step.plan.num_splits}, mode {step.plan.merge_mode})")
