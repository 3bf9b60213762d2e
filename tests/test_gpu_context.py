"""The library in a CUDA context other than the device's primary one.

State the library keeps per context -- the raised shared-memory limit of each
kernel instance and the allocation-free entry point's scratch address -- is
keyed on the context's id, so a caller that makes its own context current (an
engine plugin) starts from nothing there. The decode (workspace path and
allocation-free path) runs in a context made with the driver API, on buffers
allocated in it, interleaved with runs in the primary context, and must give
the primary context's results bit for bit.
"""
import ctypes

import numpy as np
import pytest
import torch

from paged_gqa_decode_global_gb300 import binding as b
from paged_gqa_decode_global_gb300 import inputs as synth

pytestmark = pytest.mark.gpu


class Driver:
    """The few driver calls the test needs (libcuda through ctypes)."""

    def __init__(self):
        self.lib = ctypes.CDLL("libcuda.so.1")
        self.ptr = ctypes.c_uint64

    def check(self, r, what):
        assert r == 0, f"{what}: CUresult {r}"

    def call(self, name, *args):
        self.check(getattr(self.lib, name)(*args), name)

    def new_context(self, ordinal):
        self.call("cuInit", ctypes.c_uint(0))
        dev = ctypes.c_int()
        self.call("cuDeviceGet", ctypes.byref(dev), ctypes.c_int(ordinal))
        ctx = ctypes.c_void_p()
        self.call("cuCtxCreate_v2", ctypes.byref(ctx), ctypes.c_uint(0), dev)  # made current
        return ctx

    def alloc_copy(self, arr):
        p = self.ptr()
        n = max(arr.nbytes, 256)
        self.call("cuMemAlloc_v2", ctypes.byref(p), ctypes.c_size_t(n))
        if arr.nbytes:
            self.call("cuMemcpyHtoD_v2", p, arr.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(arr.nbytes))
        return p

    def zeros(self, nbytes):
        return self.alloc_copy(np.zeros(nbytes, dtype=np.uint8))

    def read(self, p, like):
        out = np.empty_like(like)
        self.call("cuCtxSynchronize")
        self.call("cuMemcpyDtoH_v2", out.ctypes.data_as(ctypes.c_void_p), p, ctypes.c_size_t(out.nbytes))
        return out


def _u16(t):
    return t.contiguous().view(torch.int16).cpu().numpy()


@pytest.mark.parametrize("sms", [152, 400], ids=["cluster-merge", "merge-kernel"])
def test_decode_in_a_context_of_its_own(sms):
    lens = [1500, 64, 3000, 700]
    li = synth.make_layer("ctx", lens, 16, 4, 512, pool_pages=sum((L + 15) // 16 for L in lens) + 4, seed=21,
                          device="cuda")
    step = b.LayerStep.for_inputs(li, sm_count=sms)
    plan = step.plan
    assert int(plan.workspace_bytes) <= 8 << 20
    ref = step.run(li)
    ref_noalloc = torch.empty_like(li.q)
    b.paged_decode_noalloc(plan, li.q, li.k_pool, li.v_pool, li.block_tables, li.seq_lens, 0, li.scale, ref_noalloc)
    torch.cuda.synchronize()
    host = [_u16(li.q), _u16(li.k_pool), _u16(li.v_pool), li.block_tables.cpu().numpy(), li.seq_lens.cpu().numpy()]
    want, want_noalloc = _u16(ref), _u16(ref_noalloc)

    drv = Driver()
    lib = b.load_library()
    ctx = drv.new_context(torch.cuda.current_device())
    try:
        bufs = [drv.alloc_copy(a) for a in host] + [drv.zeros(int(plan.workspace_bytes)), drv.zeros(want.nbytes),
                                                    drv.zeros(want.nbytes)]
        q, k, v, bt, sl, ws, out, out2 = (p.value for p in bufs)
        wsb = int(plan.workspace_bytes)
        stream = ctypes.c_void_p()
        drv.call("cuStreamCreate", ctypes.byref(stream), ctypes.c_uint(0))
        for _ in range(2):  # the second call finds this context's state in place
            st = lib.paged_decode_global(ctypes.byref(plan), q, k, v, bt, sl, li.scale, ws, wsb, out, stream)
            assert st == b.PD_OK, b.status_string(st)
            st = lib.paged_decode_merge(ctypes.byref(plan), ws, wsb, out, stream)
            assert st == b.PD_OK, b.status_string(st)
            assert np.array_equal(drv.read(bufs[6], want), want)
            st = lib.paged_decode_noalloc(ctypes.byref(plan), q, k, v, bt, sl, 0, li.scale, out2, None, stream)
            assert st == b.PD_OK, b.status_string(st)
            assert np.array_equal(drv.read(bufs[7], want_noalloc), want_noalloc)
        drv.call("cuStreamDestroy_v2", stream)
        for p in bufs:
            drv.call("cuMemFree_v2", p)
    finally:
        popped = ctypes.c_void_p()
        drv.call("cuCtxPopCurrent_v2", ctypes.byref(popped))
        drv.call("cuCtxDestroy_v2", ctx)
    # and the primary context still gives the same results afterwards
    again = step.run(li)
    again_noalloc = torch.empty_like(li.q)
    b.paged_decode_noalloc(plan, li.q, li.k_pool, li.v_pool, li.block_tables, li.seq_lens, 0, li.scale,
                          again_noalloc)
    torch.cuda.synchronize()
    assert np.array_equal(_u16(again), want)
    assert np.array_equal(_u16(again_noalloc), want_noalloc)
