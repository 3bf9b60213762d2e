"""fp64 CPU oracle for paged GQA decode attention.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline may import this package; the product package never does. It shares
no code with the CUDA path. The arithmetic lives in ``ref_decode.c`` (decode
attention; plain C, fp64, OpenMP over query rows) and ``ref_prepare.c`` (the
per-token norm / RoPE / cache-slot step before it); this module only compiles
them with gcc and marshals numpy arrays into them.

bf16 tensors are passed as their raw bit patterns (numpy ``uint16``); the C
code widens them exactly to fp64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCES = [os.path.join(_HERE, "ref_decode.c"), os.path.join(_HERE, "ref_prepare.c")]
_LIB_PATH = os.path.join(_HERE, "libref_decode.so")
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-shared", "-fPIC"]
_lock = threading.Lock()
_lib = None

_STATUS = {
    0: "ok",
    -1: "invalid argument",
    -2: "block table names a page outside the pool",
    -3: "sequence length outside [0, max_pages * page_size]",
    -4: "out of host memory",
}


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile the C sources into libref_decode.so next to them (gcc, -fopenmp)."""
    if not force and os.path.exists(_LIB_PATH) and all(
            os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src) for src in SOURCES):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, "-o", tmp, *SOURCES, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            p = ctypes.c_void_p
            i = ctypes.c_int
            d = ctypes.c_double
            lib.ref_decode_rows.argtypes = [i, i, i, i, i, i, i, p, p, p, p, p, i, d, p, i, p, p, i]
            lib.ref_decode_rows.restype = i
            lib.ref_decode_split.argtypes = [i, i, i, i, i, i, i, p, p, p, p, p, i, d, i, i, p, p, i]
            lib.ref_decode_split.restype = i
            lib.ref_merge.argtypes = [i, i, i, p, p, p]
            lib.ref_merge.restype = i
            lib.ref_max_threads.argtypes = []
            lib.ref_max_threads.restype = i
            lib.ref_decode_rows_fp8.argtypes = [i, i, i, i, i, i, i, p, p, p, p, p, p, p, i, d, p, i, p, p, i]
            lib.ref_decode_rows_fp8.restype = i
            lib.ref_e4m3_to_f64.argtypes = [i]
            lib.ref_e4m3_to_f64.restype = d
            lib.ref_decode_multi.argtypes = [i, i, i, i, i, i, i, i, p, p, p, p, p, i, d, p, p, i]
            lib.ref_decode_multi.restype = i
            set_prepare_signatures(lib)
            _lib = lib
    return _lib


def set_prepare_signatures(lib):
    p = ctypes.c_void_p
    i = ctypes.c_int
    d = ctypes.c_double
    lib.ref_prepare_qkv.argtypes = [i, i, i, i, i, i, i, i, i, d, d] + [p] * 12
    lib.ref_prepare_qkv.restype = i
    lib.ref_rope_table.argtypes = [i, d, i, p]
    lib.ref_rope_table.restype = i


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"bf16 operands must be passed as uint16 bit patterns, got {a.dtype}")
    return a


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(status: int):
    if status != 0:
        raise OracleError(_STATUS.get(status, f"status {status}"))


def _shapes(q, k_pool, block_tables):
    B, Hq, d = q.shape
    num_pages, Hkv, P, d2 = k_pool.shape
    if d2 != d:
        raise ValueError("q and pool head_dim differ")
    max_pages = block_tables.shape[1] if block_tables.ndim == 2 else 0
    return B, Hq, Hkv, d, P, num_pages, max_pages


def max_threads() -> int:
    return int(_load().ref_max_threads())


def decode(q, k_pool, v_pool, block_tables, seq_lens, scale: float, window: int = 0,
           rows=None, nthreads: int = 0, return_lse: bool = False):
    """Decode attention in fp64.

    q: uint16 [B, Hq, d]; k_pool / v_pool: uint16 [num_pages, Hkv, P, d]
    (v_pool None = K=V layer); block_tables: int32 [B, max_pages];
    seq_lens: int32 [B]; window 0 = global layer.
    rows: optional list of b * Hq + h to compute (others stay zero).
    Returns float64 [B, Hq, d] (and [B, Hq] log-sum-exp if return_lse).
    """
    lib = _load()
    q, k_pool = _u16(q), _u16(k_pool)
    v_pool = None if v_pool is None else _u16(v_pool)
    block_tables, seq_lens = _i32(block_tables), _i32(seq_lens)
    B, Hq, Hkv, d, P, num_pages, max_pages = _shapes(q, k_pool, block_tables)
    if v_pool is not None and v_pool.shape != k_pool.shape:
        raise ValueError("k_pool and v_pool shapes differ")
    out = np.zeros((B, Hq, d), dtype=np.float64)
    lse = np.full((B, Hq), -np.inf, dtype=np.float64)
    rows_arr = None if rows is None else _i32(rows)
    n_rows = 0 if rows_arr is None else int(rows_arr.size)
    st = lib.ref_decode_rows(B, Hq, Hkv, d, P, num_pages, max_pages, _ptr(q), _ptr(k_pool),
                             _ptr(v_pool), _ptr(block_tables), _ptr(seq_lens), int(window),
                             float(scale), _ptr(rows_arr), n_rows, _ptr(out), _ptr(lse), int(nthreads))
    _check(st)
    return (out, lse) if return_lse else out


def decode_fp8(q, k8, v8, k_scale, v_scale, block_tables, seq_lens, scale: float, window: int = 0,
               rows=None, nthreads: int = 0, return_lse: bool = False):
    """Decode over an FP8 KV cache in fp64.

    q: uint16 (bf16 bits) [B, Hq, d]; k8 / v8: uint8 e4m3 bytes
    [num_pages, Hkv, P, d] (v8 None = K=V layer, K's scales);
    k_scale / v_scale: float32 [num_pages, Hkv] (the cached value is the e4m3
    value times its (page, KV head) scale). Otherwise as `decode`.
    """
    lib = _load()
    q = _u16(q)
    k8 = np.ascontiguousarray(k8, dtype=np.uint8)
    v8 = None if v8 is None else np.ascontiguousarray(v8, dtype=np.uint8)
    k_scale = np.ascontiguousarray(k_scale, dtype=np.float32)
    v_scale = None if v_scale is None else np.ascontiguousarray(v_scale, dtype=np.float32)
    block_tables, seq_lens = _i32(block_tables), _i32(seq_lens)
    B, Hq, Hkv, d, P, num_pages, max_pages = _shapes(q, k8, block_tables)
    if k_scale.shape != (num_pages, Hkv) or (v8 is not None and (v8.shape != k8.shape or v_scale is None
                                                                  or v_scale.shape != k_scale.shape)):
        raise ValueError("fp8 pool / scale shapes disagree")
    out = np.zeros((B, Hq, d), dtype=np.float64)
    lse = np.full((B, Hq), -np.inf, dtype=np.float64)
    rows_arr = None if rows is None else _i32(rows)
    n_rows = 0 if rows_arr is None else int(rows_arr.size)
    st = lib.ref_decode_rows_fp8(B, Hq, Hkv, d, P, num_pages, max_pages, _ptr(q), _ptr(k8), _ptr(v8),
                                 _ptr(k_scale), _ptr(v_scale), _ptr(block_tables), _ptr(seq_lens), int(window),
                                 float(scale), _ptr(rows_arr), n_rows, _ptr(out), _ptr(lse), int(nthreads))
    _check(st)
    return (out, lse) if return_lse else out


def decode_multi(q, k_pool, v_pool, block_tables, seq_lens, scale: float, window: int = 0, nthreads: int = 0,
                 return_lse: bool = False):
    """T new tokens per request, causal over the paged cache, in fp64.

    q: uint16 [B, T, Hq, d], the last T positions of each request (seq_lens
    counts them); otherwise as `decode`. Returns float64 [B, T, Hq, d] (and the
    log-sum-exp [B, T, Hq] if return_lse).
    """
    lib = _load()
    q, k_pool = _u16(q), _u16(k_pool)
    v_pool = None if v_pool is None else _u16(v_pool)
    block_tables, seq_lens = _i32(block_tables), _i32(seq_lens)
    B, T, Hq, d = q.shape
    num_pages, Hkv, P, d2 = k_pool.shape
    if d2 != d or (v_pool is not None and v_pool.shape != k_pool.shape):
        raise ValueError("shapes disagree")
    max_pages = block_tables.shape[1] if block_tables.ndim == 2 else 0
    out = np.zeros((B, T, Hq, d), dtype=np.float64)
    lse = np.full((B, T, Hq), -np.inf, dtype=np.float64)
    st = lib.ref_decode_multi(B, T, Hq, Hkv, d, P, num_pages, max_pages, _ptr(q), _ptr(k_pool), _ptr(v_pool),
                              _ptr(block_tables), _ptr(seq_lens), int(window), float(scale), _ptr(out), _ptr(lse),
                              int(nthreads))
    _check(st)
    return (out, lse) if return_lse else out


def e4m3_to_f64(code: int) -> float:
    """The oracle's e4m3 decoder, for its pin."""
    return float(_load().ref_e4m3_to_f64(int(code)))


def decode_split(q, k_pool, v_pool, block_tables, seq_lens, scale: float, window: int,
                 num_splits: int, chunk: int, nthreads: int = 0):
    """Split-KV stage 1 in fp64: returns (o_part [B, Hq, S, d], lse_part [B, Hq, S])."""
    lib = _load()
    q, k_pool = _u16(q), _u16(k_pool)
    v_pool = None if v_pool is None else _u16(v_pool)
    block_tables, seq_lens = _i32(block_tables), _i32(seq_lens)
    B, Hq, Hkv, d, P, num_pages, max_pages = _shapes(q, k_pool, block_tables)
    o_part = np.zeros((B, Hq, num_splits, d), dtype=np.float64)
    lse_part = np.full((B, Hq, num_splits), -np.inf, dtype=np.float64)
    st = lib.ref_decode_split(B, Hq, Hkv, d, P, num_pages, max_pages, _ptr(q), _ptr(k_pool),
                              _ptr(v_pool), _ptr(block_tables), _ptr(seq_lens), int(window),
                              float(scale), int(num_splits), int(chunk), _ptr(o_part), _ptr(lse_part),
                              int(nthreads))
    _check(st)
    return o_part, lse_part


def merge(o_part, lse_part):
    """Split-KV stage 2 in fp64: o_part [..., S, d], lse_part [..., S] -> [..., d]."""
    lib = _load()
    o_part = np.ascontiguousarray(o_part, dtype=np.float64)
    lse_part = np.ascontiguousarray(lse_part, dtype=np.float64)
    lead = o_part.shape[:-2]
    S, d = o_part.shape[-2:]
    if lse_part.shape != lead + (S,):
        raise ValueError("lse_part shape does not match o_part")
    rows = int(np.prod(lead)) if lead else 1
    out = np.zeros(lead + (d,), dtype=np.float64)
    _check(lib.ref_merge(rows, S, d, _ptr(o_part), _ptr(lse_part), _ptr(out)))
    return out


def rope_table(rot: int, theta: float, n_pos: int):
    """float64 [n_pos, rot]: cos of the pair angles, then their sin."""
    out = np.zeros((n_pos, rot), dtype=np.float64)
    _check(_load().ref_rope_table(int(rot), float(theta), int(n_pos), _ptr(out)))
    return out


def prepare_qkv(q_in, k_in, v_in, q_w, k_w, v_w, block_tables, seq_lens, num_pages: int, page_size: int,
                rot: int, theta: float, eps: float):
    """The per-token step before decode, in fp64.

    q_in uint16 [B, Hq, d]; k_in / v_in uint16 [B, Hkv, d] (v_in None = K=V
    layer); weights uint16 [d] (v_w None = unit weight); block_tables int32
    [B, max_pages]; seq_lens int32 [B] (including the new token).
    Returns (q_out [B, Hq, d], k_out [B, Hkv, d], v_out [B, Hkv, d] or None,
    slot_page [B] (-1 outside the pool), slot_row [B]).
    """
    lib = _load()
    q_in, k_in, q_w, k_w = _u16(q_in), _u16(k_in), _u16(q_w), _u16(k_w)
    v_in = None if v_in is None else _u16(v_in)
    v_w = None if v_w is None else _u16(v_w)
    block_tables, seq_lens = _i32(block_tables), _i32(seq_lens)
    B, Hq, d = q_in.shape
    Hkv = k_in.shape[1]
    max_pages = block_tables.shape[1] if block_tables.ndim == 2 else 0
    kv_shared = v_in is None
    q_out = np.zeros((B, Hq, d), dtype=np.float64)
    k_out = np.zeros((B, Hkv, d), dtype=np.float64)
    v_out = None if kv_shared else np.zeros((B, Hkv, d), dtype=np.float64)
    slot_page = np.zeros(B, dtype=np.int32)
    slot_row = np.zeros(B, dtype=np.int32)
    st = lib.ref_prepare_qkv(B, Hq, Hkv, d, int(page_size), int(num_pages), max_pages, int(kv_shared), int(rot),
                             float(theta), float(eps), _ptr(q_in), _ptr(k_in), _ptr(v_in), _ptr(q_w), _ptr(k_w),
                             _ptr(v_w), _ptr(block_tables), _ptr(seq_lens), _ptr(q_out), _ptr(k_out), _ptr(v_out),
                             _ptr(slot_page), _ptr(slot_row))
    _check(st)
    return q_out, k_out, v_out, slot_page, slot_row
