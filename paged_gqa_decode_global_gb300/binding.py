"""ctypes binding of libpaged_decode.so (argument marshalling only).

The functions carry the names of the C entry points declared in
include/paged_decode.h and take torch tensors (device memory) or plain
integers; every step of the computation runs in the library's CUDA kernels.
There is no fallback: if the library is missing, loading raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional, Sequence

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libpaged_decode.so")

PD_OK = 0
PD_ERR_INVALID_ARG = 1
PD_ERR_UNSUPPORTED = 2
PD_ERR_WORKSPACE_TOO_SMALL = 3
PD_ERR_CUDA = 4
PD_ERR_DEVICE_FAULT = 5

# layout of pd_plan / pd_layer_desc this binding marshals (paged_decode_abi_version)
ABI_VERSION = 5

PD_KV_BF16 = 0
PD_KV_FP8_E4M3 = 1

PD_DEVFLAG_BAD_PAGE = 0x1
PD_DEVFLAG_BAD_SEQLEN = 0x2
PD_DEVFLAG_WAIT_TIMEOUT = 0x4

EXPORTED = (
    "paged_decode_plan",
    "paged_decode_global",
    "paged_decode_window",
    "paged_decode_merge",
    "paged_decode_check_device_error",
    "paged_decode_status_string",
    "paged_decode_abi_version",
    "paged_decode_noalloc",
    "paged_decode_global_fp8",
    "paged_decode_window_fp8",
    "paged_decode_plan_multi",
    "paged_decode_plan_partial",
    "paged_decode_global_partial",
    "paged_decode_combine",
    "paged_decode_rope_table",
    "paged_decode_qkv_norm_rope_write",
    "paged_decode_stage_copy",
)


class LayerDesc(ctypes.Structure):
    _fields_ = [
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("max_pages_per_seq", ctypes.c_int32),
        ("window", ctypes.c_int32),
        ("kv_shared", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32),
    ]


class Plan(ctypes.Structure):
    _fields_ = [
        ("layer", LayerDesc),
        ("batch", ctypes.c_int32),
        ("num_splits", ctypes.c_int32),
        ("chunk_tokens", ctypes.c_int32),
        ("block_tokens", ctypes.c_int32),
        ("variant", ctypes.c_int32),
        ("grid_x", ctypes.c_int32),
        ("grid_y", ctypes.c_int32),
        ("grid_z", ctypes.c_int32),
        ("threads_per_cta", ctypes.c_int32),
        ("smem_bytes", ctypes.c_int32),
        ("sm_count", ctypes.c_int32),
        ("max_seq_len", ctypes.c_int32),
        ("merge_mode", ctypes.c_int32),
        ("test_stall_bytes", ctypes.c_int32),
        ("query_tokens", ctypes.c_int32),
        ("partial", ctypes.c_int32),
        ("early_kv", ctypes.c_int32),
        ("workspace_bytes", ctypes.c_uint64),
        ("lse_offset", ctypes.c_uint64),
        ("opart_offset", ctypes.c_uint64),
        ("magic", ctypes.c_uint32),
        ("version", ctypes.c_uint32),
    ]


class PagedDecodeError(RuntimeError):
    def __init__(self, status: int, where: str, flags: int = 0):
        self.status = status
        self.flags = flags
        msg = f"{where}: {status_string(status)} (status {status})"
        if flags:
            msg += f", device flags 0x{flags:x}"
        super().__init__(msg)


_lock = threading.Lock()
_lib = None


def load_library(path: Optional[str] = None):
    """Load the CUDA library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"CUDA library not found at {p}; build it with "
                "`python -m paged_gqa_decode_global_gb300.build` (no CPU fallback exists)")
        lib = ctypes.CDLL(p)
        vp, i32, u64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
        lib.paged_decode_plan.argtypes = [ctypes.POINTER(LayerDesc), i32, vp, i32, ctypes.POINTER(Plan)]
        lib.paged_decode_plan.restype = ctypes.c_int
        lib.paged_decode_global.argtypes = [ctypes.POINTER(Plan), vp, vp, vp, vp, vp, f32, vp, u64, vp, vp]
        lib.paged_decode_global.restype = ctypes.c_int
        lib.paged_decode_window.argtypes = [ctypes.POINTER(Plan), vp, vp, vp, vp, vp, i32, f32, vp, u64, vp, vp]
        lib.paged_decode_window.restype = ctypes.c_int
        lib.paged_decode_merge.argtypes = [ctypes.POINTER(Plan), vp, u64, vp, vp]
        lib.paged_decode_merge.restype = ctypes.c_int
        lib.paged_decode_check_device_error.argtypes = [ctypes.POINTER(Plan), vp, u64, vp,
                                                        ctypes.POINTER(ctypes.c_uint32)]
        lib.paged_decode_check_device_error.restype = ctypes.c_int
        lib.paged_decode_status_string.argtypes = [ctypes.c_int]
        lib.paged_decode_status_string.restype = ctypes.c_char_p
        lib.paged_decode_abi_version.argtypes = []
        lib.paged_decode_abi_version.restype = i32
        lib.paged_decode_noalloc.argtypes = [ctypes.POINTER(Plan), vp, vp, vp, vp, vp, i32, f32, vp, vp, vp]
        lib.paged_decode_noalloc.restype = ctypes.c_int
        lib.paged_decode_global_fp8.argtypes = [ctypes.POINTER(Plan), vp, vp, vp, vp, vp, vp, vp, f32, vp, u64, vp,
                                                vp]
        lib.paged_decode_global_fp8.restype = ctypes.c_int
        lib.paged_decode_window_fp8.argtypes = [ctypes.POINTER(Plan), vp, vp, vp, vp, vp, vp, vp, i32, f32, vp, u64,
                                                vp, vp]
        lib.paged_decode_window_fp8.restype = ctypes.c_int
        lib.paged_decode_plan_multi.argtypes = [ctypes.POINTER(LayerDesc), i32, i32, vp, i32, ctypes.POINTER(Plan)]
        lib.paged_decode_plan_multi.restype = ctypes.c_int
        lib.paged_decode_plan_partial.argtypes = [ctypes.POINTER(LayerDesc), i32, vp, i32, ctypes.POINTER(Plan)]
        lib.paged_decode_plan_partial.restype = ctypes.c_int
        lib.paged_decode_global_partial.argtypes = [ctypes.POINTER(Plan), vp, vp, vp, vp, vp, f32, vp, u64, vp, vp, vp]
        lib.paged_decode_global_partial.restype = ctypes.c_int
        lib.paged_decode_combine.argtypes = [i32, i32, i32, vp, vp, vp, vp]
        lib.paged_decode_combine.restype = ctypes.c_int
        lib.paged_decode_stage_copy.argtypes = [ctypes.c_void_p, i32, i32, vp]
        lib.paged_decode_stage_copy.restype = ctypes.c_int
        lib.paged_decode_rope_table.argtypes = [ctypes.c_double, i32, i32, vp, vp]
        lib.paged_decode_rope_table.restype = ctypes.c_int
        lib.paged_decode_qkv_norm_rope_write.argtypes = [ctypes.POINTER(LayerDesc), i32, i32, i32, f32] + [vp] * 14
        lib.paged_decode_qkv_norm_rope_write.restype = ctypes.c_int
        found = int(lib.paged_decode_abi_version())
        if found != ABI_VERSION:
            raise RuntimeError(f"{p} has ABI version {found}, this binding marshals version {ABI_VERSION}: rebuild it "
                               "with `python -m paged_gqa_decode_global_gb300.build`")
        if path is None:
            _lib = lib
        return lib


def status_string(status: int) -> str:
    try:
        return load_library().paged_decode_status_string(status).decode()
    except Exception:  # noqa: BLE001 - message formatting must not fail
        return f"status {status}"


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str):
    if status != PD_OK:
        raise PagedDecodeError(status, where)


def layer_desc(num_q_heads: int, num_kv_heads: int, head_dim: int, page_size: int, num_pages: int,
               max_pages_per_seq: int, window: int = 0, kv_shared: bool = False,
               kv_dtype: int = PD_KV_BF16) -> LayerDesc:
    return LayerDesc(num_q_heads, num_kv_heads, head_dim, page_size, num_pages, max_pages_per_seq,
                     window, 1 if kv_shared else 0, int(kv_dtype))


def paged_decode_plan(desc: LayerDesc, seq_lens_host: Sequence[int], sm_count: int) -> Plan:
    lib = load_library()
    n = len(seq_lens_host)
    arr = (ctypes.c_int32 * max(1, n))(*[int(x) for x in seq_lens_host])
    plan = Plan()
    st = lib.paged_decode_plan(ctypes.byref(desc), n, ctypes.cast(arr, ctypes.c_void_p) if n else None,
                               int(sm_count), ctypes.byref(plan))
    _check(st, "paged_decode_plan")
    return plan


def paged_decode_plan_multi(desc: LayerDesc, query_tokens: int, seq_lens_host: Sequence[int],
                            sm_count: int) -> Plan:
    """Plan for `query_tokens` new tokens per request (q / out [B, T, Hq, d])."""
    lib = load_library()
    n = len(seq_lens_host)
    arr = (ctypes.c_int32 * max(1, n))(*[int(x) for x in seq_lens_host])
    plan = Plan()
    st = lib.paged_decode_plan_multi(ctypes.byref(desc), n, int(query_tokens),
                                     ctypes.cast(arr, ctypes.c_void_p) if n else None, int(sm_count),
                                     ctypes.byref(plan))
    _check(st, "paged_decode_plan_multi")
    return plan


def paged_decode_global(plan: Plan, q, k_pool, v_pool, block_tables, seq_lens, scale: float, workspace,
                        out, stream=None, workspace_bytes: Optional[int] = None) -> None:
    lib = load_library()
    wb = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    st = lib.paged_decode_global(ctypes.byref(plan), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables),
                                 _ptr(seq_lens), float(scale), _ptr(workspace), int(wb), _ptr(out),
                                 _stream_ptr(stream))
    _check(st, "paged_decode_global")


def paged_decode_window(plan: Plan, q, k_pool, v_pool, block_tables, seq_lens, window: int, scale: float,
                        workspace, out, stream=None, workspace_bytes: Optional[int] = None) -> None:
    lib = load_library()
    wb = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    st = lib.paged_decode_window(ctypes.byref(plan), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables),
                                 _ptr(seq_lens), int(window), float(scale), _ptr(workspace), int(wb), _ptr(out),
                                 _stream_ptr(stream))
    _check(st, "paged_decode_window")


def paged_decode_global_fp8(plan: Plan, q, k_pool, v_pool, k_scale, v_scale, block_tables, seq_lens,
                            scale: float, workspace, out, stream=None, workspace_bytes: Optional[int] = None) -> None:
    lib = load_library()
    wb = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    st = lib.paged_decode_global_fp8(ctypes.byref(plan), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale),
                                     _ptr(v_scale), _ptr(block_tables), _ptr(seq_lens), float(scale),
                                     _ptr(workspace), int(wb), _ptr(out), _stream_ptr(stream))
    _check(st, "paged_decode_global_fp8")


def paged_decode_window_fp8(plan: Plan, q, k_pool, v_pool, k_scale, v_scale, block_tables, seq_lens, window: int,
                            scale: float, workspace, out, stream=None, workspace_bytes: Optional[int] = None) -> None:
    lib = load_library()
    wb = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    st = lib.paged_decode_window_fp8(ctypes.byref(plan), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale),
                                     _ptr(v_scale), _ptr(block_tables), _ptr(seq_lens), int(window), float(scale),
                                     _ptr(workspace), int(wb), _ptr(out), _stream_ptr(stream))
    _check(st, "paged_decode_window_fp8")


def paged_decode_merge(plan: Plan, workspace, out, stream=None, workspace_bytes: Optional[int] = None) -> None:
    lib = load_library()
    wb = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    st = lib.paged_decode_merge(ctypes.byref(plan), _ptr(workspace), int(wb), _ptr(out), _stream_ptr(stream))
    _check(st, "paged_decode_merge")


def paged_decode_check_device_error(plan: Plan, workspace, stream=None) -> int:
    """Synchronise, read and clear the device error word; raises on a non-zero word."""
    lib = load_library()
    flags = ctypes.c_uint32(0)
    wb = workspace.numel() * workspace.element_size()
    st = lib.paged_decode_check_device_error(ctypes.byref(plan), _ptr(workspace), int(wb), _stream_ptr(stream),
                                             ctypes.byref(flags))
    if st != PD_OK:
        raise PagedDecodeError(st, "paged_decode_check_device_error", flags.value)
    return flags.value


def paged_decode_noalloc(plan: Plan, q, k_pool, v_pool, block_tables, seq_lens, window: int, scale: float, out,
                         device_flags=None, stream=None) -> None:
    """Stage 1 + merge using the library's own scratch array instead of a
    workspace, for callers that cannot allocate device memory (see the C
    header). `device_flags`: optional int32/uint32 device tensor receiving the
    call's device error word."""
    lib = load_library()
    st = lib.paged_decode_noalloc(ctypes.byref(plan), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables),
                                  _ptr(seq_lens), int(window), float(scale), _ptr(out), _ptr(device_flags),
                                  _stream_ptr(stream))
    _check(st, "paged_decode_noalloc")


def abi_version() -> int:
    return int(load_library().paged_decode_abi_version())


# ----------------------------------------------------------------------------
# Convenience: one layer-step (stage 1 + stage 2) on torch tensors
# ----------------------------------------------------------------------------

class LayerStep:
    """Plan + workspace for one layer, reusable across steps whose sequences
    are no longer than the planned ones."""

    def __init__(self, num_q_heads, num_kv_heads, head_dim, page_size, num_pages, max_pages_per_seq,
                 seq_lens_host, *, window=0, kv_shared=False, kv_dtype=PD_KV_BF16, sm_count=None, device=None,
                 query_tokens=1, early_kv=False):
        import torch
        device = torch.device("cuda") if device is None else torch.device(device)
        if sm_count is None:
            sm_count = torch.cuda.get_device_properties(device).multi_processor_count
        self.desc = layer_desc(num_q_heads, num_kv_heads, head_dim, page_size, num_pages, max_pages_per_seq,
                               window, kv_shared, kv_dtype)
        self.fp8 = kv_dtype == PD_KV_FP8_E4M3
        self.query_tokens = int(query_tokens)
        if self.query_tokens > 1:
            self.plan = paged_decode_plan_multi(self.desc, self.query_tokens, list(seq_lens_host), sm_count)
        else:
            self.plan = paged_decode_plan(self.desc, list(seq_lens_host), sm_count)
        # the caller's promise about the kernel launched just before stage 1 (pd_plan.early_kv)
        self.plan.early_kv = 1 if early_kv else 0
        nbytes = int(self.plan.workspace_bytes)
        # zeroed once: the first word is the device error flag
        self.workspace = torch.zeros((nbytes + 255) // 256 * 256, dtype=torch.uint8, device=device)
        self.window = window

    @classmethod
    def for_inputs(cls, li, sm_count=None, query_tokens=1, early_kv=False):
        """A step for a LayerInputs (bf16 cache) or Fp8LayerInputs (e4m3 cache);
        query_tokens > 1: q and out are [B, T, Hq, d]."""
        fp8 = hasattr(li, "k8")
        return cls(li.num_q_heads, li.num_kv_heads, li.head_dim, li.page_size, li.num_pages, li.max_pages,
                   li.seq_lens_list(), window=li.window, kv_shared=li.kv_shared,
                   kv_dtype=PD_KV_FP8_E4M3 if fp8 else PD_KV_BF16, sm_count=sm_count, device=li.q.device,
                   query_tokens=query_tokens, early_kv=early_kv)

    def __call__(self, q, k_pool, v_pool, block_tables, seq_lens, scale, out, stream=None, k_scale=None,
                 v_scale=None):
        if self.fp8:
            if self.window > 0:
                paged_decode_window_fp8(self.plan, q, k_pool, v_pool, k_scale, v_scale, block_tables, seq_lens,
                                        self.window, scale, self.workspace, out, stream)
            else:
                paged_decode_global_fp8(self.plan, q, k_pool, v_pool, k_scale, v_scale, block_tables, seq_lens,
                                        scale, self.workspace, out, stream)
        elif self.window > 0:
            paged_decode_window(self.plan, q, k_pool, v_pool, block_tables, seq_lens, self.window, scale,
                                self.workspace, out, stream)
        else:
            paged_decode_global(self.plan, q, k_pool, v_pool, block_tables, seq_lens, scale, self.workspace,
                                out, stream)
        paged_decode_merge(self.plan, self.workspace, out, stream)
        return out

    def run(self, li, out=None, stream=None):
        import torch
        if out is None:
            out = torch.empty_like(li.q)
        if self.fp8:
            return self(li.q, li.k8, li.v8, li.block_tables, li.seq_lens, li.scale, out, stream,
                        k_scale=li.k_scale, v_scale=li.v_scale)
        return self(li.q, li.k_pool, li.v_pool, li.block_tables, li.seq_lens, li.scale, out, stream)

    def check(self, stream=None) -> int:
        return paged_decode_check_device_error(self.plan, self.workspace, stream)


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)


def paged_decode_rope_table(theta: float, rotary_dim: int, num_positions: int, cos_sin, stream=None) -> None:
    """Fill cos_sin (fp32 [num_positions, rotary_dim], device) with the layer's RoPE table."""
    st = load_library().paged_decode_rope_table(float(theta), int(rotary_dim), int(num_positions), _ptr(cos_sin),
                                                _stream_ptr(stream))
    _check(st, "paged_decode_rope_table")


def paged_decode_qkv_norm_rope_write(desc: LayerDesc, rotary_dim: int, num_positions: int, eps: float, q_in, k_in,
                                     v_in, q_norm_weight, k_norm_weight, v_norm_weight, cos_sin, block_tables,
                                     seq_lens, q_out, k_pool, v_pool, device_flags, stream=None) -> None:
    """QKV norm + RoPE of the new tokens, k / v rows written into the pools, q into q_out."""
    batch = q_in.shape[0]
    st = load_library().paged_decode_qkv_norm_rope_write(
        ctypes.byref(desc), int(batch), int(rotary_dim), int(num_positions), float(eps), _ptr(q_in), _ptr(k_in),
        _ptr(v_in), _ptr(q_norm_weight), _ptr(k_norm_weight), _ptr(v_norm_weight), _ptr(cos_sin),
        _ptr(block_tables), _ptr(seq_lens), _ptr(q_out), _ptr(k_pool), _ptr(v_pool), _ptr(device_flags),
        _stream_ptr(stream))
    _check(st, "paged_decode_qkv_norm_rope_write")


def paged_decode_plan_partial(desc: LayerDesc, seq_lens_host: Sequence[int], sm_count: int) -> Plan:
    """Plan for paged_decode_global_partial (a global bf16 layer's local tokens)."""
    lib = load_library()
    n = len(seq_lens_host)
    arr = (ctypes.c_int32 * max(1, n))(*[int(x) for x in seq_lens_host])
    plan = Plan()
    st = lib.paged_decode_plan_partial(ctypes.byref(desc), n, ctypes.cast(arr, ctypes.c_void_p) if n else None,
                                       int(sm_count), ctypes.byref(plan))
    _check(st, "paged_decode_plan_partial")
    return plan


def paged_decode_global_partial(plan: Plan, q, k_pool, v_pool, block_tables, seq_lens, scale: float, workspace,
                                o_out, lse_out, stream=None, workspace_bytes: Optional[int] = None) -> None:
    """This rank's normalised fp32 partial output o_out [B, Hq, d] and its log-sum-exp lse_out [B, Hq]."""
    wb = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    st = load_library().paged_decode_global_partial(
        ctypes.byref(plan), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables), _ptr(seq_lens), float(scale),
        _ptr(workspace), int(wb), _ptr(o_out), _ptr(lse_out), _stream_ptr(stream))
    _check(st, "paged_decode_global_partial")


MAX_STAGE_COPIES = 4  # PD_MAX_STAGE_COPIES


class Copy(ctypes.Structure):
    _fields_ = [("dst", ctypes.c_void_p), ("src", ctypes.c_void_p), ("bytes", ctypes.c_size_t)]


def paged_decode_stage_copy(pairs, after_wait: int = 0, stream=None) -> None:
    """Copy each (dst, src) pair of tensors (equal byte sizes; device or
    page-locked host memory; a pair of Nones is skipped) as one kernel in the
    stream's chain of programmatic dependent launches; after_wait 1 waits for
    the launch in front first."""
    entries = []
    for dst, src in pairs:
        if dst is None and src is None:
            continue
        if dst is None or src is None:
            raise ValueError("a copy needs both its source and its destination")
        n = dst.numel() * dst.element_size()
        if src.numel() * src.element_size() != n:
            raise ValueError(f"copy of {src.numel() * src.element_size()} bytes into {n} bytes")
        entries.append(Copy(_ptr(dst), _ptr(src), n))
    arr = (Copy * max(1, len(entries)))(*entries)
    st = load_library().paged_decode_stage_copy(ctypes.cast(arr, ctypes.c_void_p), len(entries), int(after_wait),
                                                _stream_ptr(stream))
    _check(st, "paged_decode_stage_copy")


def paged_decode_combine(o_parts, lse_parts, out, stream=None) -> None:
    """Merge gathered partials o_parts [R, rows..., d] fp32, lse_parts [R, rows...] into bf16 out [rows..., d]."""
    R = o_parts.shape[0]
    d = o_parts.shape[-1]
    rows = o_parts[0].numel() // d
    st = load_library().paged_decode_combine(int(R), int(rows), int(d), _ptr(o_parts), _ptr(lse_parts), _ptr(out),
                                             _stream_ptr(stream))
    _check(st, "paged_decode_combine")
