"""Sequence-sharded decode (decode context parallelism) over the C ABI.

The cached tokens of every request are spread over R ranks. Each rank attends
its own tokens with ``paged_decode_global_partial`` (a normalised fp32 partial
output and its log-sum-exp), the ranks all-gather those partials, and every
rank merges them with ``paged_decode_combine`` -- the same log-sum-exp merge
that joins the pieces of one request inside a rank (vLLM concepts page
"模型库与算子层 — 概念", MLA backend sections: DCP with an exchange of the
partial outputs and log-sum-exps).

This module holds only the layout of the shards and the collective: the
attention and the merge run in the library's kernels. ``shard_cache`` copies a
request's cached rows into the local pages of one rank (in a serving engine
each rank writes its own tokens when they are appended); ``exchange_partials``
is one all-gather of the fp32 partials (NCCL on GPUs, gloo on the host).
"""
from __future__ import annotations

from typing import List, Optional, Sequence, Tuple

import torch

from . import binding

MODES = ("interleaved", "contiguous")


def shard_positions(L: int, R: int, r: int, mode: str = "interleaved") -> List[int]:
    """Token positions of a length-L request held by rank r of R.

    interleaved: t with t % R == r (new tokens go round-robin);
    contiguous: the r-th of R consecutive runs of ceil(L / R) positions.
    """
    if mode == "interleaved":
        return list(range(r, L, R))
    if mode == "contiguous":
        chunk = (L + R - 1) // R if L > 0 else 0
        return list(range(min(L, r * chunk), min(L, (r + 1) * chunk)))
    raise ValueError(f"mode must be one of {MODES}")


def shard_cache(k_pool: torch.Tensor, v_pool: Optional[torch.Tensor], block_tables: torch.Tensor,
                seq_lens: Sequence[int], R: int, r: int, mode: str = "interleaved"
                ) -> Tuple[torch.Tensor, Optional[torch.Tensor], torch.Tensor, torch.Tensor]:
    """Rank r's local cache: its tokens of every request, in position order,
    packed into fresh pages [local_pages, Hkv, P, d] (v None on a K=V layer),
    with the local block table [B, max_local_pages] (-1 past the end) and the
    local lengths [B] (int32, on the pools' device)."""
    num_pages, Hkv, P, d = k_pool.shape
    dev = k_pool.device
    tables = block_tables.cpu()
    per_req = [shard_positions(int(L), R, r, mode) for L in seq_lens]
    n_pages = [(len(pos) + P - 1) // P for pos in per_req]
    total = max(1, sum(n_pages))
    width = max(1, max(n_pages) if n_pages else 1)
    k_loc = torch.zeros(total, Hkv, P, d, dtype=k_pool.dtype, device=dev)
    v_loc = None if v_pool is None else torch.zeros_like(k_loc)
    table = torch.full((len(per_req), width), -1, dtype=torch.int32)
    nxt = 0
    for b, pos in enumerate(per_req):
        if not pos:
            continue
        t = torch.tensor(pos, dtype=torch.long)
        src_page = tables[b, t // P].long().to(dev)
        src_row = (t % P).to(dev)
        dst = torch.arange(len(pos), device=dev)
        dst_page = nxt + dst // P
        dst_row = dst % P
        k_loc[dst_page, :, dst_row, :] = k_pool[src_page, :, src_row, :]
        if v_loc is not None:
            v_loc[dst_page, :, dst_row, :] = v_pool[src_page, :, src_row, :]
        table[b, :n_pages[b]] = torch.arange(nxt, nxt + n_pages[b], dtype=torch.int32)
        nxt += n_pages[b]
    lens = torch.tensor([len(pos) for pos in per_req], dtype=torch.int32, device=dev)
    return k_loc, v_loc, table.to(dev), lens


def exchange_partials(o: torch.Tensor, lse: torch.Tensor, group=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """All-gather this rank's partials: returns o [R, ...] and lse [R, ...] in rank order."""
    import torch.distributed as dist
    R = dist.get_world_size(group)
    o_all = [torch.empty_like(o) for _ in range(R)]
    lse_all = [torch.empty_like(lse) for _ in range(R)]
    dist.all_gather(o_all, o.contiguous(), group=group)
    dist.all_gather(lse_all, lse.contiguous(), group=group)
    return torch.stack(o_all), torch.stack(lse_all)


class PartialStep:
    """Plan + workspace for this rank's partial decode of one global layer."""

    def __init__(self, desc: binding.LayerDesc, local_lens: Sequence[int], sm_count: int, device,
                 early_kv: bool = False):
        self.plan = binding.paged_decode_plan_partial(desc, list(local_lens), sm_count)
        # the caller's promise about the kernels before each call (pd_plan.early_kv)
        self.plan.early_kv = 1 if early_kv else 0
        nbytes = int(self.plan.workspace_bytes)
        self.workspace = torch.zeros((nbytes + 255) // 256 * 256, dtype=torch.uint8, device=device)

    def __call__(self, q, k_pool, v_pool, block_tables, seq_lens, scale, stream=None):
        B, Hq, d = q.shape
        o = torch.empty(B, Hq, d, dtype=torch.float32, device=q.device)
        lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
        binding.paged_decode_global_partial(self.plan, q, k_pool, v_pool, block_tables, seq_lens, scale,
                                            self.workspace, o, lse, stream)
        return o, lse


def combine(o_all: torch.Tensor, lse_all: torch.Tensor, stream=None) -> torch.Tensor:
    """Merge gathered partials [R, B, Hq, d] / [R, B, Hq] into bf16 [B, Hq, d]."""
    out = torch.empty(o_all.shape[1:], dtype=torch.bfloat16, device=o_all.device)
    binding.paged_decode_combine(o_all.contiguous(), lse_all.contiguous(), out, stream)
    return out
