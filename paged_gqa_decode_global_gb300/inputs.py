"""Seeded synthetic inputs for paged decode attention.

This module only draws random numbers and lays out pages: it holds none of
the attention arithmetic, so both the CUDA path and the CPU oracle can take
their inputs from it.

Recipe (the same for every workload):
  * structure (sequence lengths, the page permutation, block tables) is drawn
    from a seeded CPU ``torch.Generator`` so it is identical on every device;
  * values (q, K, V) are fp32 ``torch.randn`` from a seeded generator on the
    target device, multiplied by the stated standard deviation and rounded to
    bf16 (round to nearest even);
  * page ids come from one ``randperm`` of the pool and are handed to the
    requests in order; block-table entries past a request's last page are -1;
  * the layer's scale is 1/sqrt(head_dim) unless a case says otherwise.

The five named workloads follow the decode configurations of a Gemma-4-style
model (global layers: head_dim 512; sliding-window layers: head_dim 256, with
their own KV-head counts), 16-token pages.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np
import torch

PAGE = 16


@dataclass
class LayerInputs:
    """One attention layer's decode inputs (all tensors on one device)."""

    name: str
    q: torch.Tensor                 # bf16 [B, Hq, d]
    k_pool: torch.Tensor            # bf16 [num_pages, Hkv, P, d]
    v_pool: Optional[torch.Tensor]  # bf16 like k_pool, None for a K=V layer
    block_tables: torch.Tensor      # int32 [B, max_pages], -1 past the end
    seq_lens: torch.Tensor          # int32 [B]
    window: int                     # 0 = global layer
    scale: float
    extra: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_q_heads(self) -> int:
        return int(self.q.shape[1])

    @property
    def head_dim(self) -> int:
        return int(self.q.shape[2])

    @property
    def num_pages(self) -> int:
        return int(self.k_pool.shape[0])

    @property
    def num_kv_heads(self) -> int:
        return int(self.k_pool.shape[1])

    @property
    def page_size(self) -> int:
        return int(self.k_pool.shape[2])

    @property
    def max_pages(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def kv_shared(self) -> bool:
        return self.v_pool is None

    def seq_lens_list(self) -> List[int]:
        return [int(x) for x in self.seq_lens.cpu().tolist()]

    def attended(self) -> List[int]:
        """Number of attended positions per request."""
        out = []
        for L in self.seq_lens_list():
            out.append(min(L, self.window) if self.window > 0 else L)
        return out

    def kv_bytes(self) -> int:
        """Algorithmic KV bytes one decode step must read (each attended row once)."""
        per_token = self.num_kv_heads * self.head_dim * 2 * (1 if self.kv_shared else 2)
        return sum(self.attended()) * per_token

    def algorithmic_bytes(self) -> int:
        """KV bytes plus q read and out written (bf16)."""
        qo = 2 * self.batch * self.num_q_heads * self.head_dim * 2
        return self.kv_bytes() + qo

    def to(self, device) -> "LayerInputs":
        return LayerInputs(self.name, self.q.to(device), self.k_pool.to(device),
                           None if self.v_pool is None else self.v_pool.to(device),
                           self.block_tables.to(device), self.seq_lens.to(device),
                           self.window, self.scale, dict(self.extra))


def bits_u16(t: torch.Tensor) -> np.ndarray:
    """Raw bit patterns of a bf16 tensor as a host uint16 array."""
    if t.dtype != torch.bfloat16:
        raise TypeError("expected a bf16 tensor")
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _cpu_gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _dev_gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn_bf16(shape, std: float, gen: torch.Generator, device) -> torch.Tensor:
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def page_tables(seq_lens: Sequence[int], pool_pages: int, gen: torch.Generator,
                page_size: int = PAGE, max_pages: Optional[int] = None) -> torch.Tensor:
    """Hand out a shuffled pool's page ids to the requests, in order."""
    need = [(L + page_size - 1) // page_size for L in seq_lens]
    if sum(need) > pool_pages:
        raise ValueError(f"pool of {pool_pages} pages cannot hold {sum(need)} pages")
    width = max(1, max(need) if need else 1) if max_pages is None else max_pages
    perm = torch.randperm(pool_pages, generator=gen).to(torch.int32)
    table = torch.full((len(seq_lens), width), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[off:off + n]
        off += n
    return table


def make_layer(name: str, seq_lens: Sequence[int], num_q_heads: int, num_kv_heads: int,
               head_dim: int, *, window: int = 0, kv_shared: bool = False,
               pool_pages: Optional[int] = None, page_size: int = PAGE, q_std: float = 1.0,
               kv_std: float = 1.0, scale: Optional[float] = None, seed: int = 0,
               device="cpu", block_tables: Optional[torch.Tensor] = None) -> LayerInputs:
    """A single layer's inputs with a freshly shuffled pool (or a given table)."""
    sgen = _cpu_gen(seed)
    if pool_pages is None:
        pool_pages = max(1, sum((L + page_size - 1) // page_size for L in seq_lens))
    if block_tables is None:
        block_tables = page_tables(seq_lens, pool_pages, sgen, page_size)
    vgen = _dev_gen(seed + 7919, device)
    B = len(seq_lens)
    q = _randn_bf16((B, num_q_heads, head_dim), q_std, vgen, device)
    k_pool = _randn_bf16((pool_pages, num_kv_heads, page_size, head_dim), kv_std, vgen, device)
    v_pool = None if kv_shared else _randn_bf16((pool_pages, num_kv_heads, page_size, head_dim),
                                                kv_std, vgen, device)
    return LayerInputs(name, q, k_pool, v_pool, block_tables.to(device),
                       torch.tensor(list(seq_lens), dtype=torch.int32, device=device), window,
                       (1.0 / math.sqrt(head_dim)) if scale is None else scale)


# --------------------------------------------------------------------------
# The named workloads
# --------------------------------------------------------------------------

WORKLOADS = {
    1: "tiny global decode: B1, 8q/2kv, d512, L256, 16-page pool",
    2: "global-layer decode: B8, 16q/4kv, d512, L1024, 4096-page pool, K!=V",
    3: "sliding-window decode: B8, 16q/8kv, d256, W1024, L~U[4000,4200], K!=V",
    4: "long-context global decode: d512, 16q/4kv, {B4x32768, B2x65536, B1x131072}, q std 0.5",
    5: "mixed ragged decode step: 8 requests, L log-uniform [1K,128K]; global d512 16q/4kv K=V + "
       "sliding d256 16q/8kv W1024 K!=V over one page-id space",
}


def seed_of(cid: int) -> int:
    return 1000 + cid


def workload(cid: int, device="cpu", part: Optional[str] = None) -> List[LayerInputs]:
    """Layers of workload `cid` (1..5). Workload 4 has parts 'a', 'b', 'c'
    (B4x32768, B2x65536, B1x131072); workload 5 has 'global' and 'sliding'."""
    seed = seed_of(cid)
    if cid == 1:
        return [make_layer("w1", [256], 8, 2, 512, pool_pages=16, seed=seed, device=device)]
    if cid == 2:
        return [make_layer("w2", [1024] * 8, 16, 4, 512, pool_pages=4096, seed=seed, device=device)]
    if cid == 3:
        g = _cpu_gen(seed + 1)
        lens = torch.randint(4000, 4201, (8,), generator=g).tolist()
        return [make_layer("w3", lens, 16, 8, 256, window=1024, pool_pages=4096, seed=seed,
                           device=device)]
    if cid == 4:
        shapes = {"a": (4, 32768), "b": (2, 65536), "c": (1, 131072)}
        keys = [part] if part else ["a", "b", "c"]
        out = []
        for k in keys:
            B, L = shapes[k]
            out.append(make_layer(f"w4{k}", [L] * B, 16, 4, 512, pool_pages=8192, q_std=0.5,
                                  seed=seed + ord(k), device=device))
        return out
    if cid == 5:
        g = _cpu_gen(seed + 1)
        u = torch.rand(8, generator=g, dtype=torch.float64)
        lo, hi = math.log(1024.0), math.log(131072.0)
        lens = [int(min(131072, max(1024, round(math.exp(lo + float(x) * (hi - lo)))))) for x in u]
        pool = int(math.ceil(sum((L + PAGE - 1) // PAGE for L in lens) * 1.25))
        table = page_tables(lens, pool, g)
        layers = []
        if part in (None, "global"):
            layers.append(make_layer("w5-global", lens, 16, 4, 512, kv_shared=True, pool_pages=pool,
                                     seed=seed, device=device, block_tables=table))
        if part in (None, "sliding"):
            layers.append(make_layer("w5-sliding", lens, 16, 8, 256, window=1024, pool_pages=pool,
                                     seed=seed + 1, device=device, block_tables=table))
        return layers
    raise ValueError(f"unknown workload {cid}")


# --------------------------------------------------------------------------
# FP8 KV cache inputs
# --------------------------------------------------------------------------

E4M3_MAX = 448.0


@dataclass
class Fp8LayerInputs:
    """A layer whose KV cache holds e4m3 bytes with one fp32 scale per
    (page, KV head) for K and for V; the cached value is byte * scale."""

    name: str
    q: torch.Tensor                  # bf16 [B, Hq, d]
    k8: torch.Tensor                 # uint8 (e4m3 bits) [num_pages, Hkv, P, d]
    v8: Optional[torch.Tensor]       # like k8; None for a K=V layer
    k_scale: torch.Tensor            # float32 [num_pages, Hkv]
    v_scale: Optional[torch.Tensor]  # float32 [num_pages, Hkv]; None for a K=V layer
    block_tables: torch.Tensor
    seq_lens: torch.Tensor
    window: int
    scale: float

    batch = LayerInputs.batch
    num_q_heads = LayerInputs.num_q_heads
    head_dim = LayerInputs.head_dim
    max_pages = LayerInputs.max_pages
    seq_lens_list = LayerInputs.seq_lens_list
    attended = LayerInputs.attended

    @property
    def num_pages(self) -> int:
        return int(self.k8.shape[0])

    @property
    def num_kv_heads(self) -> int:
        return int(self.k8.shape[1])

    @property
    def page_size(self) -> int:
        return int(self.k8.shape[2])

    @property
    def kv_shared(self) -> bool:
        return self.v8 is None

    def kv_bytes(self) -> int:
        per_token = self.num_kv_heads * self.head_dim * (1 if self.kv_shared else 2)
        return sum(self.attended()) * per_token

    def algorithmic_bytes(self) -> int:
        """KV bytes, their scales (one per page and KV head touched), q read and out written."""
        qo = 2 * self.batch * self.num_q_heads * self.head_dim * 2
        pages = sum((n + self.page_size - 1) // self.page_size for n in self.attended())
        return self.kv_bytes() + pages * self.num_kv_heads * 4 * (1 if self.kv_shared else 2) + qo


def _quantize_pool(pool: torch.Tensor):
    """Per (page, KV head): scale = max |x| / 448, bytes = e4m3(x / scale)."""
    x = pool.float()
    amax = x.abs().amax(dim=(2, 3))
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    q8 = (x / scale[:, :, None, None]).clamp_(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return q8.view(torch.uint8), scale.contiguous()


def quantize_kv_fp8(li: LayerInputs) -> Fp8LayerInputs:
    """The same layer with its KV cache stored as e4m3 with per-(page, KV head) scales."""
    k8, ks = _quantize_pool(li.k_pool)
    v8, vs = (None, None) if li.v_pool is None else _quantize_pool(li.v_pool)
    return Fp8LayerInputs(li.name + "-fp8", li.q, k8, v8, ks, vs, li.block_tables, li.seq_lens, li.window,
                          li.scale)


# --------------------------------------------------------------------------
# The step before decode: the new token's raw q / k / v and the layer's norm
# weights and RoPE parameters
# --------------------------------------------------------------------------

# Per layer kind: RoPE base and the number of rotated dims (sliding layers
# rotate every dim with base 1e4; global layers rotate a quarter of d with
# base 1e6). The pages only say that the two kinds carry their own RoPE
# parameters; these values are inputs, not part of the method.
ROPE_PARAMS = {"global": (1.0e6, 0.25), "sliding": (1.0e4, 1.0)}
NORM_EPS = 1e-6


@dataclass
class PrepareInputs:
    """The new token of every request of one layer, before normalisation."""
    layer: LayerInputs        # pools, block tables, seq_lens (including the new token)
    q_in: torch.Tensor        # bf16 [B, Hq, d]
    k_in: torch.Tensor        # bf16 [B, Hkv, d]
    v_in: Optional[torch.Tensor]  # bf16 [B, Hkv, d]; None on a K=V layer
    q_w: torch.Tensor         # bf16 [d]
    k_w: torch.Tensor         # bf16 [d]
    v_w: Optional[torch.Tensor]   # bf16 [d] or None (unit weight)
    rot: int                  # rotated dims (even, <= d; 0 = none)
    theta: float              # RoPE base
    eps: float
    max_positions: int        # rows of the layer's RoPE table

    def rows_bytes(self) -> int:
        """Bytes of the head rows read and written per call (q in/out, k/v in, cache rows)."""
        li = self.layer
        d, B = li.head_dim, li.batch
        kv_rows = li.num_kv_heads * (1 if self.v_in is None else 2)
        return 2 * B * (li.num_q_heads + kv_rows) * d * 2


def make_prepare(li: LayerInputs, *, rot: Optional[int] = None, theta: Optional[float] = None,
                 eps: float = NORM_EPS, in_std: float = 3.0, seed: int = 0, with_v_weight: bool = True,
                 max_positions: Optional[int] = None) -> PrepareInputs:
    """Raw new-token rows (N(0, in_std), bf16) and norm weights (N(1, 0.25), bf16)
    for layer `li`; RoPE parameters from the layer kind unless given."""
    kind = "sliding" if li.window > 0 else "global"
    th, frac = ROPE_PARAMS[kind]
    theta = th if theta is None else theta
    rot = int(li.head_dim * frac) if rot is None else rot
    device = li.q.device
    gen = _dev_gen(seed + 104729, device)
    B, Hq, Hkv, d = li.batch, li.num_q_heads, li.num_kv_heads, li.head_dim
    q_in = _randn_bf16((B, Hq, d), in_std, gen, device)
    k_in = _randn_bf16((B, Hkv, d), in_std, gen, device)
    v_in = None if li.v_pool is None else _randn_bf16((B, Hkv, d), in_std, gen, device)

    def weight():
        return (1.0 + 0.25 * torch.randn(d, generator=gen, device=device)).to(torch.bfloat16)

    q_w, k_w = weight(), weight()
    v_w = weight() if (with_v_weight and v_in is not None) else None
    if max_positions is None:
        max_positions = li.block_tables.shape[1] * li.page_size
    return PrepareInputs(li, q_in, k_in, v_in, q_w, k_w, v_w, rot, theta, eps, max_positions)


# --------------------------------------------------------------------------
# Several query tokens per request (speculative-decode verification)
# --------------------------------------------------------------------------

def make_query_tokens(li: LayerInputs, T: int, seed: int = 0, q_std: float = 1.0) -> torch.Tensor:
    """q for the last T positions of each request: bf16 [B, T, Hq, d], N(0, q_std)."""
    gen = _dev_gen(seed + 15485863, li.q.device)
    return _randn_bf16((li.batch, T, li.num_q_heads, li.head_dim), q_std, gen, li.q.device)


def _multi_tokens(li, T: int) -> List[int]:
    """Positions T query tokens per request attend (the union of their causal
    ranges: the whole sequence, or the last W + T - 1 positions)."""
    return [min(L, li.window + T - 1) if li.window > 0 else L for L in li.seq_lens_list()]


def multi_kv_bytes(li, T: int) -> int:
    """KV bytes T query tokens per request must read (bf16 or e4m3 cache)."""
    elem = 1 if hasattr(li, "k8") else 2
    per_token = li.num_kv_heads * li.head_dim * elem * (1 if li.kv_shared else 2)
    return sum(_multi_tokens(li, T)) * per_token


def multi_algorithmic_bytes(li, T: int) -> int:
    """KV bytes (and, for an e4m3 cache, the scales of the pages touched) plus
    q read and out written (bf16) for T tokens per request."""
    scales = 0
    if hasattr(li, "k8"):
        pages = sum((n + li.page_size - 1) // li.page_size for n in _multi_tokens(li, T))
        scales = pages * li.num_kv_heads * 4 * (1 if li.kv_shared else 2)
    return multi_kv_bytes(li, T) + scales + 2 * li.batch * T * li.num_q_heads * li.head_dim * 2
