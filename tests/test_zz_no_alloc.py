"""The allocation-free entry point (paged_decode_noalloc) against the
workspace entry points.

paged_decode_noalloc serves callers that may not allocate device memory, such
as an engine plugin whose host owns all device memory or a serving loop that
must not call cudaMalloc mid-step; it runs the same decode step on a scratch
array inside the library. Its output must match the workspace path's on two
calls in a row (the second call finds the first call's contents in the shared
array).

This file is named to be collected last.
"""
import numpy as np
import pytest
import torch

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
    x = a.float().cpu().numpy().astype(np.float64).ravel()
    y = ref.float().cpu().numpy().astype(np.float64).ravel()
    assert np.isfinite(x).all(), tag
    err = np.abs(x - y).max()
    cos = float(x @ y / (np.linalg.norm(x) * np.linalg.norm(y)))
    assert err <= MAX_ABS and cos > MIN_COS, f"{tag}: max abs {err:.3e} cos {cos:.7f}"


@pytest.mark.parametrize("window,kvs,d,G", [(0, False, 512, 4), (0, True, 512, 4), (1024, False, 256, 2)])
def test_noalloc_matches_workspace_path_twice(window, kvs, d, G):
    lens = [4097, 1500, 77, 0, 3000]
    li = synth.make_layer("na", lens, 4 * G, 4, d, window=window, kv_shared=kvs,
                          pool_pages=sum((L + 15) // 16 for L in lens) + 8, seed=21 + d + window + kvs,
                          device="cuda")
    step = b.LayerStep.for_inputs(li)
    assert step.plan.num_splits > 1  # the scratch array really carries partials
    ref = step.run(li)
    assert step.check() == 0
    flags = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = torch.full_like(li.q, float("nan"))
        b.paged_decode_noalloc(step.plan, li.q, li.k_pool, li.v_pool, li.block_tables, li.seq_lens, window,
                               li.scale, out, device_flags=flags)
        torch.cuda.synchronize()
        assert int(flags.item()) == 0, f"call {call}: device flags {int(flags.item()):#x}"
        _close(out, ref, f"call {call}")


def test_noalloc_rejects_plans_beyond_its_scratch():
    # a plan for 64 requests x 16 heads x 31 pieces needs far more than 8 MiB of
    # partials; the call must refuse it before touching any buffer
    lens = [8192] * 64
    plan = b.paged_decode_plan(b.layer_desc(16, 4, 512, 16, 64 * 512 + 1, 512), lens, 4000)
    li = synth.make_layer("small", [16], 16, 4, 512, pool_pages=2, seed=3, device="cuda")
    assert plan.workspace_bytes > 8 << 20
    out = torch.zeros_like(li.q)
    with pytest.raises(b.PagedDecodeError) as e:
        b.paged_decode_noalloc(plan, li.q, li.k_pool, li.v_pool, li.block_tables, li.seq_lens, 0, li.scale, out)
    assert e.value.status == b.PD_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert (out == 0).all()
