"""Host-side checks of the C ABI (no GPU): the library builds, loads and exports
every function declared in include/*.h; the planner validates its arguments
and its plans cover every attended token."""
import ctypes
import glob
import os
import re

import pytest
import torch

from paged_gqa_decode_global_gb300 import binding as b
from paged_gqa_decode_global_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return b.load_library()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M):
            if not m.group(1).startswith(("if", "sizeof")):
                names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in b.EXPORTED:
        assert n in names, n


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} declared but not exported"


def test_build_targets_sm103a_only():
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_status_strings_and_version(lib):
    assert b.status_string(b.PD_OK) == "ok"
    assert "workspace" in b.status_string(b.PD_ERR_WORKSPACE_TOO_SMALL)
    assert b.abi_version() == 5 == b.ABI_VERSION


def _plan(lens, Hq=16, Hkv=4, d=512, P=16, pages=4096, maxp=None, window=0, kv_shared=False, sms=152):
    if maxp is None:
        maxp = max(1, max([(L + P - 1) // P for L in lens] or [1]))
    return b.paged_decode_plan(b.layer_desc(Hq, Hkv, d, P, pages, maxp, window, kv_shared), lens, sms)


@pytest.mark.parametrize("kw,status", [
    (dict(Hq=15), b.PD_ERR_INVALID_ARG),          # Hq not a multiple of Hkv
    (dict(P=24), b.PD_ERR_INVALID_ARG),           # page size not a multiple of 16
    (dict(window=-1), b.PD_ERR_INVALID_ARG),
    (dict(sms=0), b.PD_ERR_INVALID_ARG),
    (dict(d=384), b.PD_ERR_UNSUPPORTED),
    (dict(d=192), b.PD_ERR_UNSUPPORTED),
    (dict(Hq=128, Hkv=4), b.PD_ERR_UNSUPPORTED),  # group of 32
    (dict(Hq=68, Hkv=4), b.PD_ERR_UNSUPPORTED),   # group of 17
    (dict(Hq=64, Hkv=4, d=128), b.PD_ERR_UNSUPPORTED),  # group of 16 at head_dim 128
])
def test_plan_rejects(lib, kw, status):
    with pytest.raises(b.PagedDecodeError) as e:
        _plan([100, 200], **kw)
    assert e.value.status == status


def test_plan_kv_dtypes(lib):
    for dt in (b.PD_KV_BF16, b.PD_KV_FP8_E4M3):
        pl = b.paged_decode_plan(b.layer_desc(16, 4, 512, 16, 4096, 64, kv_dtype=dt), [1024] * 8, 152)
        assert pl.layer.kv_dtype == dt
    with pytest.raises(b.PagedDecodeError) as e:
        b.paged_decode_plan(b.layer_desc(16, 4, 512, 16, 4096, 64, kv_dtype=7), [1024] * 8, 152)
    assert e.value.status == b.PD_ERR_INVALID_ARG
    # the bf16 and FP8 entry points refuse each other's plans before touching CUDA
    bf = b.paged_decode_plan(b.layer_desc(16, 4, 512, 16, 4096, 64), [64], 152)
    f8 = b.paged_decode_plan(b.layer_desc(16, 4, 512, 16, 4096, 64, kv_dtype=b.PD_KV_FP8_E4M3), [64], 152)
    assert lib.paged_decode_global_fp8(ctypes.byref(bf), 16, 16, 32, 48, 48, 64, 64, 1.0, 256, 1 << 20, 512,
                                       None) == b.PD_ERR_INVALID_ARG
    assert lib.paged_decode_global(ctypes.byref(f8), 16, 16, 32, 64, 64, 1.0, 256, 1 << 20, 512,
                                   None) == b.PD_ERR_INVALID_ARG


def test_plan_rejects_length_beyond_table(lib):
    with pytest.raises(b.PagedDecodeError) as e:
        _plan([100, 200], maxp=5)
    assert e.value.status == b.PD_ERR_INVALID_ARG


@pytest.mark.parametrize("lens,window,d,Hkv", [
    ([1024] * 8, 0, 512, 4),
    ([32768] * 4, 0, 512, 4),
    ([131072], 0, 512, 4),
    ([4000, 4100, 4200, 4033], 1024, 256, 8),
    ([1, 0, 17, 300000], 0, 512, 4),
    ([1024, 131072, 5000, 77777, 1500], 0, 512, 4),
    ([0, 0], 0, 256, 8),
])
def test_plan_covers_every_token(lib, lens, window, d, Hkv):
    for sms in (1, 8, 152, 1000):
        pl = _plan(lens, Hkv=Hkv, Hq=Hkv * 2, d=d, window=window, pages=10 ** 6, sms=sms)
        TB = pl.block_tokens
        assert pl.chunk_tokens % 16 == 0 and pl.num_splits >= 1
        for L in lens:
            lo = max(0, L - window) if window else 0
            span = L - (lo // TB) * TB if L else 0
            assert pl.num_splits * pl.chunk_tokens >= span
        if pl.num_splits > 1 and pl.merge_mode == 1:
            rows = len(lens) * Hkv * 2
            assert pl.workspace_bytes >= pl.opart_offset + rows * pl.num_splits * d * 4
            assert pl.opart_offset >= pl.lse_offset + rows * pl.num_splits * 4
            assert pl.lse_offset >= 4
        elif pl.num_splits > 1:
            assert pl.merge_mode == 2 and 2 <= pl.num_splits <= 8
        else:
            assert pl.merge_mode == 0
        assert pl.workspace_bytes >= 256
        assert (pl.grid_x, pl.grid_y, pl.grid_z) == (pl.num_splits, Hkv, len(lens))


def test_plan_fills_the_machine_on_long_contexts(lib):
    pl = _plan([131072], sms=152)
    assert pl.grid_x * pl.grid_y >= 152
    pl = _plan([1024] * 8, sms=152)
    assert pl.grid_x * pl.grid_y * pl.grid_z >= 100


def test_no_gpu_calls_fail_cleanly_without_a_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    pl = _plan([64])
    # a host-side argument error is reported before anything touches CUDA
    st = lib.paged_decode_global(ctypes.byref(pl), None, None, None, None, None, 1.0, None, 0, None, None)
    assert st == b.PD_ERR_INVALID_ARG


def test_prepare_rejects_bad_arguments_without_launching(lib):
    """Host checks of the fused norm / RoPE / cache-write entry point (nothing is launched)."""
    fake = 1 << 20  # an aligned address that is never touched: every call below is refused first
    desc = b.layer_desc(16, 4, 512, 16, 64, 8, 0, False)

    def call(desc=desc, rot=128, n_pos=128, eps=1e-6, batch=2, q_in=fake, flags=fake):
        ptrs = [q_in, fake, fake, fake, fake, None, fake, fake, fake, fake, fake, fake, flags, None]
        return lib.paged_decode_qkv_norm_rope_write(ctypes.byref(desc), batch, rot, n_pos, eps, *ptrs)

    fp8 = b.layer_desc(16, 4, 512, 16, 64, 8, 0, False, b.PD_KV_FP8_E4M3)
    assert call(desc=fp8) == b.PD_ERR_UNSUPPORTED
    assert call(desc=b.layer_desc(16, 4, 128, 16, 64, 8, 0, False)) == b.PD_ERR_UNSUPPORTED
    assert call(desc=b.layer_desc(16, 3, 512, 16, 64, 8, 0, False)) == b.PD_ERR_INVALID_ARG
    assert call(rot=3) == b.PD_ERR_INVALID_ARG
    assert call(rot=1024) == b.PD_ERR_INVALID_ARG
    assert call(eps=-1.0) == b.PD_ERR_INVALID_ARG
    assert call(eps=float("nan")) == b.PD_ERR_INVALID_ARG
    assert call(n_pos=0) == b.PD_ERR_INVALID_ARG
    assert call(batch=-1) == b.PD_ERR_INVALID_ARG
    assert call(q_in=None) == b.PD_ERR_INVALID_ARG
    assert call(q_in=fake + 2) == b.PD_ERR_INVALID_ARG
    assert call(flags=None) == b.PD_ERR_INVALID_ARG
    assert lib.paged_decode_rope_table(1e4, 63, 10, fake, None) == b.PD_ERR_INVALID_ARG
    assert lib.paged_decode_rope_table(-1.0, 64, 10, fake, None) == b.PD_ERR_INVALID_ARG
    assert lib.paged_decode_rope_table(1e4, 64, 0, fake, None) == b.PD_ERR_INVALID_ARG
    assert lib.paged_decode_rope_table(1e4, 64, 10, None, None) == b.PD_ERR_INVALID_ARG


def test_combine_and_partial_reject_bad_arguments_without_launching(lib):
    fake = 1 << 20
    assert lib.paged_decode_combine(0, 4, 512, fake, fake, fake, None) == b.PD_ERR_INVALID_ARG
    assert lib.paged_decode_combine(1025, 4, 512, fake, fake, fake, None) == b.PD_ERR_INVALID_ARG
    assert lib.paged_decode_combine(2, 4, 510, fake, fake, fake, None) == b.PD_ERR_INVALID_ARG
    assert lib.paged_decode_combine(2, -1, 512, fake, fake, fake, None) == b.PD_ERR_INVALID_ARG
    assert lib.paged_decode_combine(2, 4, 512, fake + 4, fake, fake, None) == b.PD_ERR_INVALID_ARG
    assert lib.paged_decode_combine(2, 4, 512, None, fake, fake, None) == b.PD_ERR_INVALID_ARG
    assert lib.paged_decode_combine(2, 0, 512, None, None, None, None) == b.PD_OK  # nothing to do
    win = b.layer_desc(16, 4, 512, 16, 64, 8, window=128)
    pl = b.Plan()
    arr = (ctypes.c_int32 * 1)(16)
    assert lib.paged_decode_plan_partial(ctypes.byref(win), 1, ctypes.cast(arr, ctypes.c_void_p), 152,
                                         ctypes.byref(pl)) == b.PD_ERR_UNSUPPORTED
    desc = b.layer_desc(16, 4, 512, 16, 64, 8)
    assert lib.paged_decode_plan_partial(ctypes.byref(desc), 1, ctypes.cast(arr, ctypes.c_void_p), 152,
                                         ctypes.byref(pl)) == b.PD_OK
    assert pl.partial == 1 and pl.merge_mode == 1
    # a decode plan is not a partial plan
    dec = b.paged_decode_plan(desc, [16], 152)
    st = lib.paged_decode_global_partial(ctypes.byref(dec), fake, fake, fake, fake, fake, 1.0, fake, 1 << 20, fake,
                                         fake, None)
    assert st == b.PD_ERR_INVALID_ARG


@pytest.mark.parametrize("G", [9, 12, 16])
@pytest.mark.parametrize("d,window,kvs", [(512, 0, False), (512, 0, True), (256, 1024, False)])
def test_groups_above_8_are_served_by_column_tiles(lib, G, d, window, kvs):
    lens = [5000, 100, 0, 30000]
    pl = _plan(lens, Hq=4 * G, Hkv=4, d=d, window=window, kv_shared=kvs, pages=10 ** 5)
    tiles = (G + 7) // 8
    # bf16 over a long context (a span of 4096 tokens or more): one CTA per KV
    # head serves both 8-column tiles (one copy of each block); a short one
    # (the 1024-token window) keeps a CTA per tile
    per_cta = 2 if window == 0 else 1
    assert pl.query_tokens == 1 and (pl.grid_y, pl.grid_z) == (4 * tiles // per_cta, len(lens))
    assert b.load_library().paged_decode_abi_version() == 5
    # the same group over several query tokens: T x G pairs, 16 per CTA
    desc = b.layer_desc(4 * G, 4, d, 16, 10 ** 5, 2000, window, kvs)
    pm = b.paged_decode_plan_multi(desc, 3, [3000, 40], 152)
    t3 = (3 * G + 7) // 8
    assert pm.grid_y == 4 * ((t3 + 1) // 2 if t3 >= 3 else t3)
    # and its FP8 form: 8 columns per CTA
    f8 = b.paged_decode_plan(b.layer_desc(4 * G, 4, d, 16, 10 ** 5, 2000, window, kvs, b.PD_KV_FP8_E4M3),
                             [3000, 40], 152)
    assert f8.grid_y == 4 * tiles


def test_stage_copy_rejects_bad_arguments_before_any_cuda_call(lib):
    """Refusals that need no pointer lookup come first, so they answer here,
    with no GPU: a copy count off 0..4, a missing list, a bad wait flag, a size
    off 16 bytes, a NULL or misaligned pointer, overlapping ends."""
    fake = 1 << 20

    def copies(*entries):
        arr = (b.Copy * max(1, len(entries)))(*[b.Copy(d, s_, n) for d, s_, n in entries])
        return ctypes.cast(arr, ctypes.c_void_p), len(entries)

    call = lib.paged_decode_stage_copy
    assert b.MAX_STAGE_COPIES == 4
    arr, _ = copies(*[(fake + 64 * i, 2 * fake + 64 * i, 16) for i in range(5)])
    assert call(arr, 5, 0, None) == b.PD_ERR_INVALID_ARG
    assert call(arr, -1, 0, None) == b.PD_ERR_INVALID_ARG
    assert call(None, 1, 0, None) == b.PD_ERR_INVALID_ARG
    assert call(*copies((fake, 2 * fake, 16)), 2, None) == b.PD_ERR_INVALID_ARG
    assert call(*copies((fake, 2 * fake, 24)), 0, None) == b.PD_ERR_INVALID_ARG
    assert call(*copies((None, 2 * fake, 16)), 0, None) == b.PD_ERR_INVALID_ARG
    assert call(*copies((fake + 8, 2 * fake, 16)), 1, None) == b.PD_ERR_INVALID_ARG
    assert call(*copies((fake, fake + 16, 32)), 0, None) == b.PD_ERR_INVALID_ARG
    # a refused copy anywhere in the list refuses the call
    assert call(*copies((None, None, 0), (fake, 2 * fake, 16), (fake, 2 * fake, 8)), 0, None) == b.PD_ERR_INVALID_ARG
    # the binding checks the pairs before calling
    with pytest.raises(ValueError):
        b.paged_decode_stage_copy([(torch.zeros(16, dtype=torch.uint8), None)])
    with pytest.raises(ValueError):
        b.paged_decode_stage_copy([(torch.zeros(16, dtype=torch.uint8), torch.zeros(32, dtype=torch.uint8))])


def test_noalloc_checks_every_argument_before_queueing_work(lib):
    """paged_decode_noalloc refuses bad calls with no CUDA call at all: on a
    machine without a GPU, a call that got past its checks would fail with
    PD_ERR_CUDA instead."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    fake = 1 << 20
    bf = b.paged_decode_plan(b.layer_desc(16, 4, 512, 16, 4096, 64), [1024] * 4, 152)
    win = b.paged_decode_plan(b.layer_desc(16, 8, 256, 16, 4096, 300, 1024), [4000] * 4, 152)
    f8 = b.paged_decode_plan(b.layer_desc(16, 4, 512, 16, 4096, 64, kv_dtype=b.PD_KV_FP8_E4M3), [1024] * 4, 152)
    part = b.paged_decode_plan_partial(b.layer_desc(16, 4, 512, 16, 4096, 64), [1024] * 4, 152)

    def call(plan, window=0, q=fake, k=fake, v=fake + 4096, scale=0.05):
        return lib.paged_decode_noalloc(ctypes.byref(plan), q, k, v, fake, fake, window, ctypes.c_float(scale),
                                        fake, None, None)

    assert call(f8) == b.PD_ERR_INVALID_ARG           # FP8: no scales to pass
    assert call(part) == b.PD_ERR_INVALID_ARG         # partial plans keep fp32 pieces for the caller
    assert call(win, window=512) == b.PD_ERR_INVALID_ARG   # window differs from the plan's
    assert call(bf, window=1024) == b.PD_ERR_INVALID_ARG   # a window on a global plan
    assert call(bf, q=None) == b.PD_ERR_INVALID_ARG
    assert call(bf, q=fake + 2) == b.PD_ERR_INVALID_ARG    # misaligned q
    assert call(bf, v=fake) == b.PD_ERR_INVALID_ARG        # V aliasing K on a K != V layer
    assert call(bf, scale=float("nan")) == b.PD_ERR_INVALID_ARG
    big = b.paged_decode_plan(b.layer_desc(16, 4, 512, 16, 4 * 8192 + 1, 8192), [131072] * 4, 4000)
    assert big.workspace_bytes > 8 << 20 and call(big) == b.PD_ERR_WORKSPACE_TOO_SMALL
    assert call(bf) == b.PD_ERR_CUDA                  # valid: gets as far as CUDA, which is absent here


def test_head_dim_128_is_planned_for_bf16_single_token(lib):
    pl = _plan([100, 2000], d=128)
    assert pl.layer.head_dim == 128 and pl.threads_per_cta == 128
    desc = b.layer_desc(16, 4, 128, 16, 4096, 64, kv_dtype=b.PD_KV_FP8_E4M3)
    with pytest.raises(b.PagedDecodeError) as e:
        b.paged_decode_plan(desc, [100], 152)
    assert e.value.status == b.PD_ERR_UNSUPPORTED
    with pytest.raises(b.PagedDecodeError) as e:
        b.paged_decode_plan_multi(b.layer_desc(16, 4, 128, 16, 4096, 64), 2, [100], 152)
    assert e.value.status == b.PD_ERR_UNSUPPORTED


def test_early_kv_is_a_flag_the_caller_sets(lib):
    """pd_plan.early_kv: 0 as planned; 1 accepted; anything else refused before any launch."""
    fake = 1 << 20
    desc = b.layer_desc(16, 4, 512, 16, 64, 8)
    pl = b.paged_decode_plan(desc, [100], 152)
    assert pl.early_kv == 0
    pl.early_kv = 2
    st = lib.paged_decode_global(ctypes.byref(pl), fake, fake, fake, fake, fake, 1.0, fake, 1 << 20, fake, None)
    assert st == b.PD_ERR_INVALID_ARG
    assert lib.paged_decode_merge(ctypes.byref(pl), fake, 1 << 20, fake, None) == b.PD_ERR_INVALID_ARG


def test_plans_edited_past_their_workspace_are_refused(lib):
    """A plan whose pieces, grid or workspace offsets were changed after
    planning, so that its launches would write past the workspace it asks for,
    is refused before any launch (here: no CUDA call, so INVALID_ARG rather
    than PD_ERR_CUDA)."""
    import copy
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    fake = 1 << 20
    pl = b.paged_decode_plan(b.layer_desc(16, 4, 512, 16, 8192, 4096), [65536, 65536], 152)
    assert pl.merge_mode == 1 and pl.num_splits > 1

    def launch(p, ws_bytes=None):
        wb = p.workspace_bytes if ws_bytes is None else ws_bytes
        return lib.paged_decode_global(ctypes.byref(p), fake, fake, fake + 4096, fake, fake, 0.05, fake, wb, fake,
                                       None)

    assert launch(pl) == b.PD_ERR_CUDA  # valid: reaches CUDA, absent here
    edits = [
        lambda p: (setattr(p, "num_splits", p.num_splits * 2), setattr(p, "grid_x", p.num_splits)),
        lambda p: setattr(p, "opart_offset", p.lse_offset),
        lambda p: setattr(p, "workspace_bytes", p.workspace_bytes - 4),
        lambda p: setattr(p, "lse_offset", 0),
        lambda p: setattr(p, "opart_offset", p.opart_offset + 4),
        lambda p: setattr(p, "grid_z", p.batch + 1),
        lambda p: setattr(p, "block_tokens", 32),
        lambda p: (setattr(p, "num_splits", 2000), setattr(p, "grid_x", 2000)),
    ]
    for i, edit in enumerate(edits):
        bad = copy.copy(pl)
        edit(bad)
        assert launch(bad, ws_bytes=1 << 40) == b.PD_ERR_INVALID_ARG, i
        assert lib.paged_decode_merge(ctypes.byref(bad), fake, 1 << 40, fake, None) == b.PD_ERR_INVALID_ARG, i
    # one-piece and cluster plans still need the error word
    one = b.paged_decode_plan(b.layer_desc(16, 4, 512, 16, 64, 8), [100], 152)
    assert one.merge_mode in (0, 2)
    one.workspace_bytes = 4
    assert launch(one, ws_bytes=1 << 20) == b.PD_ERR_INVALID_ARG


@pytest.mark.parametrize("lens,Hq,Hkv,d,window,want", [
    ([32768] * 4, 16, 4, 512, 0, (9, 3648, 1)),     # one wave of 144 CTAs, then the merge kernel
    ([65536] * 2, 16, 4, 512, 0, (19, 3456, 1)),    # one wave of 152
    ([131072], 16, 4, 512, 0, (38, 3456, 1)),
    ([1024] * 8, 16, 4, 512, 0, (4, 256, 2)),       # clusters of 4 (36 fit at once: all 32 run together)
    ([256], 8, 2, 512, 0, (4, 64, 2)),
    ([4100] * 8, 16, 8, 256, 1024, (2, 544, 2)),    # pieces of whole two-block stages
])
def test_planner_choices_on_the_measured_workloads(lib, lens, Hq, Hkv, d, window, want):
    """The plans the measured steps ran (152 SMs): pieces, piece size, merge mode."""
    pl = _plan(lens, Hq=Hq, Hkv=Hkv, d=d, window=window, pages=10 ** 6, sms=152)
    assert (pl.num_splits, pl.chunk_tokens, pl.merge_mode) == want


@pytest.mark.parametrize("G", [3, 5, 6, 7])
def test_groups_between_the_decode_instances_are_served(lib, G):
    """Groups without an instance of their own (3, 5, 6, 7) go to the column-
    tiled instances at one query token as well: one CTA of 8 columns per KV
    head; head_dim 128 has no such instance."""
    for d, window, kvs, fp8 in [(512, 0, False, False), (256, 1024, True, False), (512, 37, False, True)]:
        desc = b.layer_desc(4 * G, 4, d, 16, 10 ** 5, 2000, window, kvs, b.PD_KV_FP8_E4M3 if fp8 else b.PD_KV_BF16)
        pl = b.paged_decode_plan(desc, [3000, 40, 0], 152)
        assert pl.grid_y == 4 and pl.query_tokens == 1
    with pytest.raises(b.PagedDecodeError) as e:
        b.paged_decode_plan(b.layer_desc(4 * G, 4, 128, 16, 10 ** 5, 2000), [3000], 152)
    assert e.value.status == b.PD_ERR_UNSUPPORTED


def test_fp8_kneqv_decode_instance_follows_the_span(lib):
    """FP8 K != V decode: six consumer warps (224 threads) for spans under 4096
    tokens, seven (256) for longer ones; K = V and the column-tiled instances
    have one form."""
    for d in (256, 512):
        for G in (1, 2, 4, 8):
            fp8 = b.layer_desc(2 * G, 2, d, 16, 10 ** 5, 2000, 0, False, b.PD_KV_FP8_E4M3)
            assert b.paged_decode_plan(fp8, [4095, 12], 152).threads_per_cta == 224
            assert b.paged_decode_plan(fp8, [4096, 12], 152).threads_per_cta == 256
            win = b.layer_desc(2 * G, 2, d, 16, 10 ** 5, 2000, 1024, False, b.PD_KV_FP8_E4M3)
            assert b.paged_decode_plan(win, [30000], 152).threads_per_cta == 224  # the window bounds the span
            kvs = b.layer_desc(2 * G, 2, d, 16, 10 ** 5, 2000, 0, True, b.PD_KV_FP8_E4M3)
            assert b.paged_decode_plan(kvs, [100], 152).threads_per_cta == 256


def test_planner_invariants_on_random_shapes(lib):
    """300 seeded random layer shapes and batches, decode / multi-token / partial
    plans, bf16 and FP8: every plan covers every attended token, its grid and
    workspace match its merge mode, and stage 1 launches fit the hardware."""
    import numpy as np
    rng = np.random.default_rng(20261202)
    shapes = [(512, 0), (256, 0), (256, 1024), (512, 64), (128, 0)]
    made = {0: 0, 1: 0, 2: 0}
    for _ in range(300):
        d, window = shapes[rng.integers(len(shapes))]
        Hkv = int(rng.choice([1, 2, 4, 8]))
        G = int(rng.choice([1, 2, 3, 4, 6, 8, 12, 16] if d != 128 else [1, 2, 4, 8]))
        kvs = bool(rng.integers(2))
        fp8 = d != 128 and bool(rng.integers(2))
        T = 1 if d == 128 or rng.random() < 0.6 else int(rng.integers(2, 9))
        partial = T == 1 and window == 0 and not fp8 and rng.random() < 0.2
        B = int(rng.integers(1, 40))
        lens = [int(x) for x in np.exp(rng.uniform(np.log(T), np.log(200000), B)).astype(int)]
        lens = [max(L, T) for L in lens]
        maxp = max((L + 15) // 16 for L in lens)
        sms = int(rng.choice([1, 20, 148, 152, 1000]))
        desc = b.layer_desc(Hkv * G, Hkv, d, 16, 10 ** 6, maxp, window, kvs,
                            b.PD_KV_FP8_E4M3 if fp8 else b.PD_KV_BF16)
        if partial:
            pl = b.paged_decode_plan_partial(desc, lens, sms)
        elif T > 1:
            pl = b.paged_decode_plan_multi(desc, T, lens, sms)
        else:
            pl = b.paged_decode_plan(desc, lens, sms)
        S, chunk, TB = pl.num_splits, pl.chunk_tokens, pl.block_tokens
        assert chunk % 16 == 0 and 1 <= S <= 1024
        for L in lens:
            first_hi = L - T + 1
            lo = first_hi - window if window and first_hi > window else 0
            assert S * chunk >= L - (lo // TB) * TB  # every attended token is in some piece
        tiles = (T * G + 7) // 8 if T > 1 or G > 8 else 1
        spans = [L - ((L - T + 1 - window) if window and L - T + 1 > window else 0) for L in lens]
        # bf16 CTAs serve two 8-column tiles for 3+ tiles, or 2 over a span of 4096+ tokens
        per_cta = 2 if not fp8 and (tiles >= 3 or (tiles == 2 and max(spans) >= 4096)) else 1
        assert (pl.grid_x, pl.grid_y, pl.grid_z) == (S, Hkv * ((tiles + per_cta - 1) // per_cta), B)
        assert pl.threads_per_cta in (128, 224, 256) and 0 < pl.smem_bytes <= 227 * 1024
        assert pl.query_tokens == T and pl.partial == int(partial) and pl.early_kv == 0
        rows = B * T * Hkv * G
        if pl.merge_mode == 1:
            assert pl.opart_offset >= pl.lse_offset + rows * S * 4 >= 256
            assert pl.workspace_bytes >= pl.opart_offset + rows * S * d * 4
        else:
            assert not partial and pl.workspace_bytes >= 4
            assert (pl.merge_mode == 0) == (S == 1)
            if pl.merge_mode == 2:
                assert 2 <= S <= 8
        made[pl.merge_mode] += 1
    assert all(made.values()), made  # every merge mode was planned for some shape
