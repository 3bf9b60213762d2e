"""Paged GQA decode attention for GB300 (sm_103a).

Single-token decode attention over a paged bf16 KV cache for the global
(head_dim 512, optional K=V storage) and sliding-window (head_dim 256) layers of
a Gemma-4-style model: a split-KV stage 1 in hand-written CUDA and a
log-sum-exp merge stage 2, behind the C ABI of include/paged_decode.h.

`binding` wraps that ABI (ctypes; torch only supplies device memory and
streams); `inputs` draws seeded synthetic workloads; `build` compiles the
library in-tree. Importing the package does not load the library; the first
call does, and raises if it has not been built.
"""
from . import binding, inputs  # noqa: F401
from .binding import (  # noqa: F401
    LayerStep,
    PagedDecodeError,
    layer_desc,
    paged_decode_check_device_error,
    paged_decode_global,
    paged_decode_merge,
    paged_decode_plan,
    paged_decode_window,
)
