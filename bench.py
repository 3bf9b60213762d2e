#!/usr/bin/env python
"""Benchmark of one decode layer-step (stage 1 + stage 2) of paged GQA decode.

Default workload: long-context global-layer decode with split-K, batch 4 x
32768 cached tokens, 16 query / 4 KV heads, head_dim 512, 16-token pages
shuffled across an 8192-page pool, K and V in separate pools (bf16), q with
std 0.5: 1 GiB of KV per layer-step. --workload 1..5 (and --part) select the
other workloads.

A "step" is one layer-step: the stage-1 launch and the merge launch over one
batch. Timing: W warm-up steps, then regions of exactly K steps replayed from
CUDA graphs on one stream, each bracketed by CUDA events with a synchronize
(and, for N > 1, a barrier) on both sides; the region is timed several times
(at least 5, about 0.4 s in all) and the median is reported (max over ranks).
Each step reads a different replica of the K/V pools when one step's KV is
smaller than L2, and the replicas together are larger than 4x L2, so every
step streams its KV from HBM. The plan's early_kv flag is set (--no-early-kv clears it): a step's
stage 1 copies its first cached blocks while the step before it drains (each
step's rows are written by no kernel of the loop). Prints one JSON line
(rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 1..5] [--impl ours|reference]
                  [--op decode|prepare|layer] [--kv bf16|fp8] [--query-tokens T] [--dcp-ranks R]

Under torchrun (N > 1) every rank runs an independent replica of the step
(decode attention needs no exchange); the reported time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time
from typing import Optional

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_gqa_decode_global_gb300 import host_loop  # noqa: E402
from paged_gqa_decode_global_gb300 import binding as pdb  # noqa: E402
from paged_gqa_decode_global_gb300 import build as pd_build  # noqa: E402
from paged_gqa_decode_global_gb300 import inputs as synth  # noqa: E402

METRIC = "decode-attn µs/layer-step and KV HBM GB/s (% of GB300 peak), 1 GPU"
LAYER_METRIC = "new-token step + decode-attn µs/layer-step and KV HBM GB/s, 1 GPU"
MULTI_METRIC = "{T}-token-per-request (verification) attn µs/layer-step and KV HBM GB/s, 1 GPU"
UNIT = "us/layer-step"
L2_BYTES = 129 * 1000 * 1000
FALLBACK_HBM_GBS = 6800.0

# DRAM bytes (read + write) per stage-1 launch from an ncu capture, keyed by the
# hash of the kernel sources it was taken on, each with the plan that launch ran
# (pieces, tokens per piece, merge mode: they set the partials written); an
# entry whose sources or plan differ from the run's is not used (the captures
# and their commands are summarised under profiles/).
NCU_TRAFFIC = {
    "390644f8bf77bb67": {
        "w4a": (1073983488 + 2760704, (9, 3648, 1)),
        "w2": (67294976 + 501504, (4, 256, 2)),
        "w3": (68276992 + 407808, (2, 544, 2)),
        "w4a-fp8": (537289728 + 2464768, (9, 3648, 1)),
        "w5global": (1596576512 + 4325632, (19, 5456, 1)),
        "w5global-fp8": (798929920 + 4875776, (19, 5456, 1)),
        "w5sliding": (68173312 + 504320, (2, 544, 2)),
    },
}

# the same for the fused QKV norm + RoPE + cache-write kernel (--op prepare)
PREP_NCU_TRAFFIC = {
    "bddd86ff645abd50": {"w2": 221184},
}

STAGE1_SOURCES = ("stage1.cu", "pd_common.cuh", "pd_variants.h", "pd_kernels.h")


PREP_SOURCES = ("prepare.cu", "pd_common.cuh", "pd_variants.h")


def kernel_source_hash(sources=STAGE1_SOURCES) -> str:
    """Hash of a kernel's sources (what an ncu capture describes)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_gqa_decode_global_gb300", "csrc")
    for name in sources:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def hbm_peak_from(data) -> Optional[float]:
    """The measured HBM copy bandwidth (GB/s) in a peaks record: the number under
    a key naming HBM and GB/s ("hbm_gbs", "hbm_GBs", "hbm_copy_gbs", ...), at the
    top level or one level down, or such a key's {"value": ...}; None if absent."""
    def number(v):
        if isinstance(v, dict):
            v = v.get("value", v.get("gbs"))
        return float(v) if isinstance(v, (int, float)) and not isinstance(v, bool) and v > 0 else None

    def scan(d):
        for key, v in d.items():
            k = key.lower()
            if "hbm" in k and "gbs" in k.replace("/", "").replace("_", ""):
                x = number(v)
                if x is not None:
                    return x
        return None

    if not isinstance(data, dict):
        return None
    x = scan(data)
    if x is None:
        for key, v in data.items():
            if isinstance(v, dict):
                x = scan(v) if "hbm" not in key.lower() else (number(v) or scan(v))
                if x is not None:
                    break
    return x


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                x = hbm_peak_from(json.load(f))
        except (OSError, ValueError):
            x = None
        if x is not None:
            return x, "measured"
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.25)  # first sample lands before the region starts
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        return False

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), max=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hw_thermal=parts[6], sw_thermal=parts[7], sw_power=parts[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w": statistics.median(r["power"] for r in rows)}


def clocks_rejected(c) -> bool:
    """A timed region whose clock samples show a hardware or thermal slowdown, or
    SM clocks well below their maximum with no reason given (a leftover clock
    lock), does not count; sw_power_cap alone is kept (and reported)."""
    if not c or c.get("sm_mhz") is None:
        return False
    if set(c.get("reasons", ())) & {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}:
        return True
    return not c.get("reasons") and c["sm_mhz"] < 0.9 * c["sm_max_mhz"]


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload_layer(cid: int, part, device):
    layers = synth.workload(cid, device=device, part=part)
    if len(layers) != 1:
        raise SystemExit("pick one layer with --part (workload 4: a|b|c, workload 5: global|sliding)")
    return layers[0]


def config_of(li, cid, part, replicas, plan):
    return {
        "workload": synth.WORKLOADS[cid] + (f" [{li.name}]" if part or hasattr(li, "k8") else ""),
        "batch": li.batch, "num_q_heads": li.num_q_heads, "num_kv_heads": li.num_kv_heads,
        "head_dim": li.head_dim, "page_size": li.page_size, "pool_pages": li.num_pages,
        "seq_lens": li.seq_lens_list() if li.batch <= 8 else f"{li.batch} requests",
        "window": li.window, "kv_shared": li.kv_shared,
        "kv_bytes_per_step": li.kv_bytes(),
        "l2": f"{replicas} rotating K/V pool replicas, {replicas * li.kv_bytes() / 1e6:.0f} MB touched per cycle (> 4x L2)",
        "num_splits": int(plan.num_splits), "chunk_tokens": int(plan.chunk_tokens),
        "merge": {0: "none (one piece)", 1: "merge kernel", 2: "in-cluster (distributed shared memory)"}[
            int(plan.merge_mode)],
        "launch": "CUDA graph replay, one stream",
        "parallelism": "replicas (no exchange)",
    }


def timed_regions(graphs, stream, world, local, sample_clocks=False, stats=None, min_regions=5,
                  max_regions=400, budget_s=0.4):
    """Time the K-step region (one replay of every graph in `graphs`, on
    `stream`) several times and return the median region in ms, with the clock
    samples taken meanwhile. Each region is bracketed by a synchronize and a
    barrier on both sides and timed by CUDA events on `stream`. The number of
    regions (at least min_regions, about budget_s of timed work, at most
    max_regions) is agreed across ranks from the first region's time; the
    median is then taken per rank and the max over ranks reported."""
    # CUDAGraph.replay() launches on the current stream: make it `stream`,
    # the stream the events are recorded on
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)

    def region():
        torch.cuda.synchronize()
        barrier(world)
        with torch.cuda.stream(stream):
            start.record(stream)
            for g in graphs:
                g.replay()
            end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return start.elapsed_time(end)

    with torch.cuda.stream(stream):
        for g in graphs[:1]:  # warm the graph exec once
            g.replay()
    torch.cuda.synchronize()
    barrier(world)
    sampler = ClockSampler(local) if sample_clocks else None
    if sampler:
        sampler.__enter__()
    times = [region()]
    n = int(min(max_regions, max(min_regions, math.ceil(budget_s * 1e3 / max(times[0], 1e-3)))))
    n = int(max_over_ranks(float(n), world))
    while len(times) < n:
        times.append(region())
    if sampler:
        sampler.__exit__(None, None, None)
    med = statistics.median(times)
    if stats is not None:
        stats.clear()
        stats.update({"regions": len(times), "statistic": "median over regions of K steps (max over ranks)",
                      "region_ms_min": round(min(times), 4), "region_ms_median": round(med, 4),
                      "region_ms_max": round(max(times), 4)})
    return med, (sampler.summary() if sampler else None)


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------

def run_ours(args, world, rank, local):
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the library has no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pd_build.build()
    pdb.load_library()

    li = workload_layer(args.workload, args.part, dev)
    fp8 = args.kv == "fp8"
    T = args.query_tokens
    if fp8:
        li = synth.quantize_kv_fp8(li)
    step = pdb.LayerStep.for_inputs(li, query_tokens=T)
    stream = torch.cuda.Stream(device=dev)
    # the step's query rows: q [B, Hq, d], or [B, T, Hq, d] for T tokens per request
    q_rows = li.q if T == 1 else synth.make_query_tokens(li, T, seed=synth.seed_of(args.workload))
    plan = step.plan
    plan.early_kv = 1 if args.early_kv else 0
    S = int(plan.num_splits)
    launches_per_step = 1 + (1 if int(plan.merge_mode) == 1 else 0)  # mode 2 merges inside stage 1

    # --op layer: each step first runs the fused QKV norm + RoPE + cache write
    # of the new token (into the pool replica the step decodes), whose q_out is
    # the decode's q
    layer_op = args.op == "layer"
    prep = None
    if layer_op:
        if fp8 or T != 1:
            raise SystemExit("--op layer: bf16 cache, one query token per request")
        pi = synth.make_prepare(li, seed=synth.seed_of(args.workload))
        cos_sin = torch.empty(pi.max_positions, max(2, pi.rot), dtype=torch.float32, device=dev)
        pdb.paged_decode_rope_table(pi.theta, pi.rot, pi.max_positions, cos_sin)
        prep_desc = pdb.layer_desc(li.num_q_heads, li.num_kv_heads, li.head_dim, li.page_size, li.num_pages,
                                   li.block_tables.shape[1], li.window, li.kv_shared)
        prep_flags = torch.zeros(1, dtype=torch.int32, device=dev)
        q_rows = torch.empty_like(li.q)

        def prep(k, v, q_in=None, k_in=None, v_in=None, bt=None, sl=None, q_out=None):
            pdb.paged_decode_qkv_norm_rope_write(
                prep_desc, pi.rot, pi.max_positions, pi.eps, pi.q_in if q_in is None else q_in,
                pi.k_in if k_in is None else k_in, pi.v_in if v_in is None else v_in, pi.q_w, pi.k_w, pi.v_w,
                cos_sin, li.block_tables if bt is None else bt, li.seq_lens if sl is None else sl,
                q_rows if q_out is None else q_out, k, v, prep_flags, stream)

        launches_per_step += 1

    touched = max(1, li.kv_bytes() if T == 1 else synth.multi_kv_bytes(li, T))
    replicas = max(1, min(16, math.ceil(4 * L2_BYTES / touched)))
    kp, vp = (li.k8, li.v8) if fp8 else (li.k_pool, li.v_pool)
    pools = [(kp, vp)]
    for _ in range(replicas - 1):
        pools.append((kp.clone(), None if vp is None else vp.clone()))
    k_sc = li.k_scale if fp8 else None
    v_sc = li.v_scale if fp8 else None
    out = torch.empty_like(q_rows)

    def one_step(i, stage1_only=False):
        k, v = pools[i % replicas]
        if prep is not None and not stage1_only:
            prep(k, v)
        if fp8 and li.window > 0:
            pdb.paged_decode_window_fp8(plan, q_rows, k, v, k_sc, v_sc, li.block_tables, li.seq_lens, li.window,
                                        li.scale, step.workspace, out, stream)
        elif fp8:
            pdb.paged_decode_global_fp8(plan, q_rows, k, v, k_sc, v_sc, li.block_tables, li.seq_lens, li.scale,
                                        step.workspace, out, stream)
        elif li.window > 0:
            pdb.paged_decode_window(plan, q_rows, k, v, li.block_tables, li.seq_lens, li.window, li.scale,
                                    step.workspace, out, stream)
        else:
            pdb.paged_decode_global(plan, q_rows, k, v, li.block_tables, li.seq_lens, li.scale, step.workspace,
                                    out, stream)
        if not stage1_only:
            pdb.paged_decode_merge(plan, step.workspace, out, stream)

    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            one_step(i)
    torch.cuda.synchronize()
    step.check(stream)

    def capture(n, stage1_only=False):
        graphs = []
        per = min(n, 500)
        left = n
        i0 = 0
        while left > 0:
            m = min(per, left)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(m):
                    one_step(i0 + i, stage1_only)
            graphs.append(g)
            left -= m
            i0 += m
        return graphs

    def timed(graphs, sample_clocks=False):
        return timed_regions(graphs, stream, world, local, sample_clocks, region_stats)

    K = args.steps
    region_stats = {}
    step_graphs = capture(K)
    elapsed_ms, clocks = timed(step_graphs, sample_clocks=True)
    step_regions = dict(region_stats)
    # a region with rejected clocks on any rank is measured once more, by every rank
    if max_over_ranks(1.0 if clocks_rejected(clocks) else 0.0, world) > 0:
        first = clocks
        elapsed_ms, clocks = timed(step_graphs, sample_clocks=True)
        clocks = dict(clocks, remeasured_after=first)
        step_regions = dict(region_stats)
    elapsed_ms = max_over_ranks(elapsed_ms, world)
    del step_graphs
    s1_graphs = capture(K, stage1_only=True)
    s1_ms, _ = timed(s1_graphs)
    s1_ms = max_over_ranks(s1_ms, world)
    del s1_graphs
    step.check(stream)

    us_per_step = elapsed_ms * 1e3 / K
    s1_us = s1_ms * 1e3 / K
    alg_bytes = li.algorithmic_bytes() if T == 1 else synth.multi_algorithmic_bytes(li, T)
    peak, peak_kind = measured_peaks()
    achieved = alg_bytes / (s1_us * 1e-6) / 1e9
    kv_gbs = touched / (us_per_step * 1e-6) / 1e9
    src_hash = kernel_source_hash()
    captured = NCU_TRAFFIC.get(src_hash, {}).get(
        f"w{args.workload}{args.part or ''}{'-fp8' if fp8 else ''}{f'-t{T}' if T > 1 else ''}")
    run_plan = (int(plan.num_splits), int(plan.chunk_tokens), int(plan.merge_mode))
    traffic = captured[0] if captured is not None and tuple(captured[1]) == run_plan else None


    # end to end: every step copies its inputs (q, block table, seq_lens) from
    # pinned host memory, decodes, and copies out back to pinned host memory.
    # Timed as CUDA-graph replays of that whole host-in/host-out step (how a
    # decode loop runs), and, for reference, as eager calls.
    e2e = None
    if not args.no_e2e:
        # Every step copies its inputs (q -- or the new token's raw rows --,
        # block table, seq_lens) from pinned host memory and its result back to
        # pinned host memory. The decode loop a caller writes pipelines this and
        # keeps the chain of programmatic dependent launches unbroken: after
        # step i's kernels one paged_decode_stage_copy kernel copies step i + 1's
        # q (or rows) into the other q buffer, the block table and lengths of
        # the step `ahead` steps on, and step i - 1's result out, then waits
        # for step i; a last one (waiting first) copies the final result out.
        # With early_kv stage 1 reads its block table and lengths before its
        # wait, so those go two steps ahead (never written by the copy in front
        # of the stage 1 that reads them), else one. Two q / result buffers,
        # three for the table and lengths; before the loop, ordinary copies of
        # the first step's inputs (and, two steps ahead, the second's table).
        # The schedule of these copies is host_loop.schedule.
        q_parts = ([pi.q_in, pi.k_in] + ([] if pi.v_in is None else [pi.v_in])) if layer_op else [q_rows]
        meta_parts = [li.block_tables, li.seq_lens]

        def staged(parts, n_dev):
            offs, total = [], 0
            for t in parts:
                offs.append(total)
                total += (t.numel() * t.element_size() + 255) // 256 * 256
            host = torch.zeros(total, dtype=torch.uint8, pin_memory=True)
            for t, o in zip(parts, offs):
                n = t.numel() * t.element_size()
                host[o:o + n].view(t.dtype).view(t.shape).copy_(t.cpu())
            devs = []
            for _ in range(n_dev):
                sd = torch.empty(total, dtype=torch.uint8, device=dev)
                sd.copy_(host)
                devs.append({"stage": sd, "views": [sd[o:o + t.numel() * t.element_size()].view(t.dtype)
                                                    .view(t.shape) for t, o in zip(parts, offs)]})
            return host, devs

        q_h, qbufs = staged(q_parts, 2)
        meta_h, mbufs = staged(meta_parts, 3)
        for qb in qbufs:
            qb["q"] = torch.empty_like(q_rows) if layer_op else qb["views"][0]
            qb["out"] = torch.empty_like(q_rows)
            qb["out_h"] = torch.empty(q_rows.shape, dtype=q_rows.dtype, pin_memory=True)
        ahead = host_loop.schedule(1, early_kv=bool(plan.early_kv)).ahead

        def compute(i, qb, mb):
            k, v = pools[i % replicas]
            qv, (bt, sl) = qb["views"], mb["views"]
            if layer_op:
                prep(k, v, q_in=qv[0], k_in=qv[1], v_in=None if pi.v_in is None else qv[2], bt=bt, sl=sl,
                     q_out=qb["q"])
            step(qb["q"], k, v, bt, sl, li.scale, qb["out"], stream, k_scale=k_sc, v_scale=v_sc)

        def serial_steps(i0, m):
            qb, mb = qbufs[0], mbufs[0]
            for i in range(i0, i0 + m):
                qb["stage"].copy_(q_h, non_blocking=True)
                mb["stage"].copy_(meta_h, non_blocking=True)
                compute(i, qb, mb)
                qb["out_h"].copy_(qb["out"], non_blocking=True)

        def pipelined_steps(i0, m):
            # the copies of an m-step loop (buffers indexed from the loop's first step)
            sch = host_loop.schedule(m, early_kv=bool(plan.early_kv))

            def dst(c):
                return (qbufs[c.buffer]["stage"] if c.kind == "q" else mbufs[c.buffer]["stage"] if c.kind == "meta"
                        else qbufs[c.buffer]["out_h"])

            def src(c):
                return q_h if c.kind == "q" else meta_h if c.kind == "meta" else qbufs[c.buffer]["out"]

            for c in sch.before:
                dst(c).copy_(src(c), non_blocking=True)
            for j in range(m):
                compute(i0 + j, qbufs[host_loop.q_buffer(j)], mbufs[host_loop.meta_buffer(j)])
                pdb.paged_decode_stage_copy([(dst(c), src(c)) for c in sch.after_step[j]], 0, stream)
            pdb.paged_decode_stage_copy([(dst(c), src(c)) for c in sch.final], 1, stream)

        def e2e_graphs(fn):
            with torch.cuda.stream(stream):
                fn(0, 3)
            torch.cuda.synchronize()
            graphs = []
            left, i0 = K, 0
            while left > 0:
                m = min(500, left)
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    fn(i0, m)
                graphs.append(g)
                left -= m
                i0 += m
            return graphs

        graphs = e2e_graphs(pipelined_steps)
        e2e_ms, _ = timed(graphs)
        e2e_ms = max_over_ranks(e2e_ms, world)
        del graphs
        for qb in qbufs:  # the last two steps' results reached the host
            assert torch.equal(qb["out_h"], qb["out"].cpu())
        graphs = e2e_graphs(serial_steps)
        serial_ms, _ = timed(graphs)
        serial_ms = max_over_ranks(serial_ms, world)
        del graphs
        # the pipelined steps as eager C-ABI calls (host launch overhead included)
        n_eager = min(K, 2000)
        with torch.cuda.stream(stream):
            a = torch.cuda.Event(enable_timing=True)
            z = torch.cuda.Event(enable_timing=True)
            barrier(world)
            a.record(stream)
            pipelined_steps(0, n_eager)
            z.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        eager_ms = max_over_ranks(a.elapsed_time(z), world)
        e2e = {"value": round(e2e_ms * 1e3 / K, 3), "unit": UNIT,
               "h2d_bytes_per_step": int(q_h.numel() + meta_h.numel()),
               "d2h_bytes_per_step": qbufs[0]["out_h"].numel() * 2, "steps": K,
               "launch": "CUDA graph replay of, per step: the C-ABI " +
                         ("new-token step and " if layer_op else "") +
                         "decode calls, then one paged_decode_stage_copy kernel copying the next step's " +
                         ("new q/k/v rows" if layer_op else "q") +
                         f" in, the block table + seq_lens of the step {ahead} on, and the previous step's out "
                         "to pinned host memory (the last out by a final copy); one stream, one chain of "
                         "programmatic dependent launches" + (", early_kv set" if ahead == 2 else ""),
               "serial_value": round(serial_ms * 1e3 / K, 3),
               "eager_value": round(eager_ms * 1e3 / n_eager, 3), "eager_steps": n_eager}
        step.check(stream)

    cpu_baseline = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        if fp8:
            cpu_baseline = oracle_baseline_fp8(li, budget_s=args.cpu_seconds,
                                               q_multi=None if T == 1 else q_rows.cpu())
        else:
            cpu_baseline = oracle_baseline(li.to("cpu"), budget_s=args.cpu_seconds,
                                           q_multi=None if T == 1 else q_rows.cpu())
            if layer_op:
                prep_us = oracle_prepare_us(li.to("cpu"), synth.seed_of(args.workload))
                cpu_baseline = dict(cpu_baseline, value=round(cpu_baseline["value"] + prep_us, 1),
                                    sample=cpu_baseline["sample"] + f"; plus the new-token step, {prep_us:.0f} us "
                                                                    "(full layer-step, median of 5, one core)")

    if rank == 0:
        line = {
            "metric": LAYER_METRIC if layer_op else METRIC if T == 1 else MULTI_METRIC.format(T=T),
            "value": round(us_per_step, 3), "unit": UNIT,
            "n_gpus": world, "steps": K,
            "warmup": max(3, args.warmup), "ms_per_step": round(us_per_step / 1e3, 6),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "io_dtype": "bf16" if not fp8 else "bf16 q/out, e4m3 KV", "data": "synthetic",
            "config": dict(config_of(li, args.workload, args.part, replicas, plan), query_tokens=T,
                           kv_bytes_per_step=touched, early_kv=bool(args.early_kv),
                           **({"step": "fused QKV norm + RoPE + cache write of the new token, then decode"}
                              if layer_op else {})),
            "kv_gbs": round(kv_gbs, 1), "kv_hbm_frac": round(kv_gbs / peak, 4),
            "roofline": {"bound": "hbm", "kernel": "stage1", "achieved": round(achieved, 1), "peak": peak,
                         "peak_source": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "traffic": traffic, "algorithmic_bytes": alg_bytes, "kernel_us": round(s1_us, 3),
                         "kernel_source": src_hash},
            "cpu_baseline": cpu_baseline,
            "e2e": e2e,
            "gpu_launches": K * launches_per_step,
            "clocks": clocks,
            "timing": step_regions,
            "device": torch.cuda.get_device_name(dev),
        }
        print(json.dumps(line), flush=True)


def oracle_baseline(li_cpu, budget_s=10.0, q_multi=None):
    """The fp64 oracle, as it stands, on all host cores: full layer-steps
    repeated for about `budget_s` seconds (q_multi: [B, T, Hq, d] query tokens)."""
    import oracle
    q = synth.bits_u16(li_cpu.q if q_multi is None else q_multi)
    k = synth.bits_u16(li_cpu.k_pool)
    v = None if li_cpu.v_pool is None else synth.bits_u16(li_cpu.v_pool)
    bt = li_cpu.block_tables.numpy()
    sl = li_cpu.seq_lens.numpy()
    threads = oracle.max_threads()
    times = []
    t_end = time.perf_counter() + budget_s
    while True:
        t0 = time.perf_counter()
        if q_multi is None:
            oracle.decode(q, k, v, bt, sl, li_cpu.scale, li_cpu.window)
        else:
            oracle.decode_multi(q, k, v, bt, sl, li_cpu.scale, li_cpu.window)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() > t_end and len(times) >= 3:
            break
    t = statistics.median(times)
    # and once on one core
    t0 = time.perf_counter()
    if q_multi is None:
        oracle.decode(q, k, v, bt, sl, li_cpu.scale, li_cpu.window, nthreads=1)
    else:
        oracle.decode_multi(q, k, v, bt, sl, li_cpu.scale, li_cpu.window, nthreads=1)
    t1 = time.perf_counter() - t0
    return {"value": round(t * 1e6, 1), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"full layer-step ({li_cpu.batch}x{li_cpu.num_q_heads} rows, {sum(li_cpu.attended())} "
                      f"attended tokens), median of {len(times)} runs, fp64 C + OpenMP",
            "single_thread_value": round(t1 * 1e6, 1)}


def oracle_prepare_us(li_cpu, seed) -> float:
    """The oracle of the new-token step, one full layer-step on one core (median of 5), in us."""
    import oracle
    pc = synth.make_prepare(li_cpu, seed=seed)
    a = [synth.bits_u16(pc.q_in), synth.bits_u16(pc.k_in), None if pc.v_in is None else synth.bits_u16(pc.v_in),
         synth.bits_u16(pc.q_w), synth.bits_u16(pc.k_w), None if pc.v_w is None else synth.bits_u16(pc.v_w),
         li_cpu.block_tables.numpy(), li_cpu.seq_lens.numpy(), li_cpu.num_pages, li_cpu.page_size, pc.rot,
         pc.theta, pc.eps]
    times = []
    for _ in range(5):
        t0 = time.perf_counter()
        oracle.prepare_qkv(*a)
        times.append(time.perf_counter() - t0)
    return statistics.median(times) * 1e6


def oracle_baseline_fp8(li, budget_s=10.0, q_multi=None):
    """The fp64 oracle of the FP8 cache, as it stands, on all host cores: full
    layer-steps repeated for about `budget_s` seconds (q_multi [B, T, Hq, d]:
    token j of each request decoded at length L - T + 1 + j)."""
    import oracle
    q = synth.bits_u16(li.q.cpu())
    k8 = li.k8.cpu().numpy()
    v8 = None if li.v8 is None else li.v8.cpu().numpy()
    ks = li.k_scale.cpu().numpy()
    vs = None if li.v_scale is None else li.v_scale.cpu().numpy()
    bt = li.block_tables.cpu().numpy()
    sl = li.seq_lens.cpu().numpy()
    threads = oracle.max_threads()
    times = []
    t_end = time.perf_counter() + budget_s
    T = 1 if q_multi is None else q_multi.shape[1]
    qs = [q] if q_multi is None else [synth.bits_u16(q_multi[:, j].contiguous()) for j in range(T)]
    while True:
        t0 = time.perf_counter()
        for j in range(T):
            oracle.decode_fp8(qs[j], k8, v8, ks, vs, bt, sl - T + 1 + j, li.scale, li.window)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() > t_end and len(times) >= 3:
            break
    t = statistics.median(times)
    return {"value": round(t * 1e6, 1), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"full layer-step over the e4m3 cache ({li.batch}x{T}x{li.num_q_heads} rows, "
                      f"{sum(li.attended())} attended tokens per query token), median of {len(times)} runs, "
                      "fp64 C + OpenMP"}


# ----------------------------------------------------------------------------
# the step before decode: QKV norm + RoPE + paged-cache write (--op prepare)
# ----------------------------------------------------------------------------

PREP_METRIC = "qkv-norm-rope-cache-write µs/layer-step and HBM GB/s, 1 GPU"


def prepare_bytes(pi) -> int:
    """Algorithmic bytes of one fused call: head rows in and out, the three norm
    weights, one RoPE table row per request, one block-table entry and one length
    per request."""
    li = pi.layer
    d = li.head_dim
    weights = d * 2 * (2 + (1 if pi.v_w is not None else 0))
    return pi.rows_bytes() + weights + li.batch * (pi.rot * 4 + 4 + 4)


def run_prepare(args, world, rank, local):
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the library has no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pd_build.build()
    pdb.load_library()
    if args.kv != "bf16":
        raise SystemExit("--op prepare writes a bf16 cache")
    li = workload_layer(args.workload, args.part, dev)
    pi = synth.make_prepare(li, seed=synth.seed_of(args.workload))
    desc = pdb.layer_desc(li.num_q_heads, li.num_kv_heads, li.head_dim, li.page_size, li.num_pages,
                          li.block_tables.shape[1], li.window, li.kv_shared)
    cos_sin = torch.empty(pi.max_positions, max(2, pi.rot), dtype=torch.float32, device=dev)
    pdb.paged_decode_rope_table(pi.theta, pi.rot, pi.max_positions, cos_sin)
    # Each step reads its own copy of the new rows and writes its k / v rows to
    # a different page (its own block table), so the copies of all steps of a
    # cycle exceed 4x L2 and every step reaches HBM.
    per_step = prepare_bytes(pi)
    replicas = max(1, min(8192, math.ceil(4 * L2_BYTES / per_step)))
    q_in = pi.q_in.unsqueeze(0).repeat(replicas, 1, 1, 1)
    k_in = pi.k_in.unsqueeze(0).repeat(replicas, 1, 1, 1)
    v_in = None if pi.v_in is None else pi.v_in.unsqueeze(0).repeat(replicas, 1, 1, 1)
    q_out = torch.empty_like(q_in)
    g = torch.Generator(device="cpu")
    g.manual_seed(synth.seed_of(args.workload) + 31)
    perm = torch.randperm(li.num_pages, generator=g).to(torch.int32)
    tables = li.block_tables.cpu().unsqueeze(0).repeat(replicas, 1, 1)
    last = ((li.seq_lens.cpu() - 1) // li.page_size).long()
    for r in range(replicas):
        tables[r, torch.arange(li.batch), last] = perm[(r * li.batch + torch.arange(li.batch)) % li.num_pages]
    tables = tables.to(dev)
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    k_pool, v_pool = li.k_pool, li.v_pool
    stream = torch.cuda.Stream(device=dev)

    def one(i, qi=None, ki=None, vi=None, qo=None, seq=None):
        r = i % replicas
        pdb.paged_decode_qkv_norm_rope_write(
            desc, pi.rot, pi.max_positions, pi.eps, q_in[r] if qi is None else qi, k_in[r] if ki is None else ki,
            (None if v_in is None else v_in[r]) if vi is None else vi, pi.q_w, pi.k_w, pi.v_w, cos_sin, tables[r],
            li.seq_lens if seq is None else seq, q_out[r] if qo is None else qo, k_pool, v_pool, flags, stream)

    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            one(i)
    torch.cuda.synchronize()
    if int(flags.item()) != 0:
        raise SystemExit(f"device flags 0x{int(flags.item()):x}")

    def graphs_of(fn, n):
        out, left, i0 = [], n, 0
        while left > 0:
            m = min(1000, left)
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                for i in range(m):
                    fn(i0 + i)
            out.append(gr)
            left -= m
            i0 += m
        return out

    def timed(graphs, sample_clocks=False):
        return timed_regions(graphs, stream, world, local, sample_clocks)

    K = args.steps
    ms, clocks = timed(graphs_of(one, K), sample_clocks=True)
    ms = max_over_ranks(ms, world)
    us = ms * 1e3 / K
    peak, peak_kind = measured_peaks()
    achieved = per_step / (us * 1e-6) / 1e9

    e2e = None
    if not args.no_e2e:
        # host rows in (q, k, v, lengths) from a pinned staging buffer, q out back to the host: after
        # step i's kernel one paged_decode_stage_copy that waits for it first (this kernel lets its
        # dependents start before its own wait, so nothing behind it may assume step i - 1 done before
        # waiting) copies step i + 1's rows into the other device buffer and step i's q out
        parts = [pi.q_in, pi.k_in] + ([pi.v_in] if pi.v_in is not None else []) + [li.seq_lens]
        offs, total = [], 0
        for t in parts:
            offs.append(total)
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        stage_h = torch.zeros(total, dtype=torch.uint8, pin_memory=True)
        for t, o in zip(parts, offs):
            n = t.numel() * t.element_size()
            stage_h[o:o + n].view(t.dtype).view(t.shape).copy_(t.cpu())
        bufs = []
        for _ in range(2):
            sd = torch.empty(total, dtype=torch.uint8, device=dev)
            sd.copy_(stage_h)
            bufs.append({"stage": sd,
                         "views": [sd[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                                   for t, o in zip(parts, offs)],
                         "qo": torch.empty_like(pi.q_in),
                         "qo_h": torch.empty(pi.q_in.shape, dtype=torch.bfloat16, pin_memory=True)})

        def chain(i0, m):
            pdb.paged_decode_stage_copy([(bufs[i0 % 2]["stage"], stage_h)], 0, stream)
            for i in range(i0, i0 + m):
                bf, other = bufs[i % 2], bufs[(i + 1) % 2]
                vw = bf["views"]
                one(i, qi=vw[0], ki=vw[1], vi=vw[2] if pi.v_in is not None else None, qo=bf["qo"], seq=vw[-1])
                more = i + 1 < i0 + m
                pdb.paged_decode_stage_copy([(other["stage"], stage_h) if more else (None, None),
                                             (bf["qo_h"], bf["qo"])], 1, stream)

        with torch.cuda.stream(stream):
            chain(0, 3)
        torch.cuda.synchronize()
        graphs, left, i0 = [], K, 0
        while left > 0:
            m = min(1000, left)
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                chain(i0, m)
            graphs.append(gr)
            left -= m
            i0 += m
        e_ms, _ = timed(graphs)
        e_ms = max_over_ranks(e_ms, world)
        for bf in bufs:
            assert torch.equal(bf["qo_h"], bf["qo"].cpu())
        e2e = {"value": round(e_ms * 1e3 / K, 3), "unit": UNIT, "h2d_bytes_per_step": int(stage_h.numel()),
               "d2h_bytes_per_step": bufs[0]["qo_h"].numel() * 2, "steps": K,
               "launch": "CUDA graph replay of, per step: the C-ABI call, then one paged_decode_stage_copy kernel "
                         "(waiting for it first) copying the next step's new q / k / v rows + lengths in from a "
                         "pinned staging buffer and this step's q out to pinned host memory; one stream, two "
                         "device buffers each way"}
    if int(flags.item()) != 0:
        raise SystemExit(f"device flags 0x{int(flags.item()):x}")

    cpu_baseline = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        pc = synth.make_prepare(li.to("cpu"), seed=synth.seed_of(args.workload))
        a = [synth.bits_u16(pc.q_in), synth.bits_u16(pc.k_in), None if pc.v_in is None else synth.bits_u16(pc.v_in),
             synth.bits_u16(pc.q_w), synth.bits_u16(pc.k_w), None if pc.v_w is None else synth.bits_u16(pc.v_w),
             pc.layer.block_tables.numpy(), pc.layer.seq_lens.numpy(), li.num_pages, li.page_size, pc.rot, pc.theta,
             pc.eps]
        times, t_end = [], time.perf_counter() + args.cpu_seconds
        while True:
            t0 = time.perf_counter()
            oracle.prepare_qkv(*a)
            times.append(time.perf_counter() - t0)
            if time.perf_counter() > t_end and len(times) >= 3:
                break
        cpu_baseline = {"value": round(statistics.median(times) * 1e6, 1), "unit": UNIT, "cores": 1,
                        "kind": "oracle", "sample": f"full layer-step, median of {len(times)} runs, fp64 C"}

    if rank == 0:
        line = {
            "metric": PREP_METRIC, "value": round(us, 3), "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": max(3, args.warmup), "ms_per_step": round(us / 1e3, 6), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "io_dtype": "bf16", "data": "synthetic",
            "config": {"workload": synth.WORKLOADS[args.workload] + f" [{li.name}], new-token step",
                       "batch": li.batch, "num_q_heads": li.num_q_heads, "num_kv_heads": li.num_kv_heads,
                       "head_dim": li.head_dim, "kv_shared": li.kv_shared, "rotary_dim": pi.rot,
                       "rope_theta": pi.theta,
                       "l2": f"{replicas} input copies and block tables, {replicas * per_step / 1e6:.0f} MB per "
                             "cycle (> 4x L2)",
                       "launch": "CUDA graph replay, one stream"},
            "roofline": {"bound": "hbm", "kernel": "qkv_norm_rope_write", "achieved": round(achieved, 1),
                         "peak": peak, "peak_source": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "traffic": PREP_NCU_TRAFFIC.get(kernel_source_hash(PREP_SOURCES), {}).get(
                             f"w{args.workload}{args.part or ''}"),
                         "algorithmic_bytes": per_step, "kernel_us": round(us, 3),
                         "kernel_source": kernel_source_hash(PREP_SOURCES)},
            "cpu_baseline": cpu_baseline, "e2e": e2e, "gpu_launches": K, "clocks": clocks,
            "device": torch.cuda.get_device_name(dev),
        }
        print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# one rank of a sequence-sharded decode (--dcp-ranks R)
# ----------------------------------------------------------------------------

DCP_METRIC = "sequence-sharded decode, per-rank µs/layer-step (partial over 1/R of the tokens + combine of R), 1 GPU"


def run_dcp(args, world, rank, local):
    """What one of R ranks computes per layer-step: its partial over its
    interleaved shard of the cache, then the combine of the R gathered
    partials. The all-gather between them needs R GPUs and is not timed."""
    from paged_gqa_decode_global_gb300 import dcp
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the library has no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pd_build.build()
    pdb.load_library()
    R = args.dcp_ranks
    li = workload_layer(args.workload, args.part, dev)
    if li.window > 0 or args.kv != "bf16" or args.query_tokens != 1:
        raise SystemExit("--dcp-ranks: global bf16 layers, one query token")
    k, v, table, lens = dcp.shard_cache(li.k_pool, li.v_pool, li.block_tables, li.seq_lens_list(), R, 0)
    per_token = li.num_kv_heads * li.head_dim * 2 * (1 if li.kv_shared else 2)
    shard_bytes = int(lens.sum()) * per_token
    replicas = max(1, min(16, math.ceil(4 * L2_BYTES / max(1, shard_bytes))))
    pools = [(k, v)] + [(k.clone(), None if v is None else v.clone()) for _ in range(replicas - 1)]
    desc = pdb.layer_desc(li.num_q_heads, li.num_kv_heads, li.head_dim, li.page_size, k.shape[0], table.shape[1],
                          0, li.kv_shared)
    step = dcp.PartialStep(desc, lens.tolist(), torch.cuda.get_device_properties(dev).multi_processor_count, dev,
                           early_kv=args.early_kv)
    B, Hq, d = li.q.shape
    o_all = torch.zeros(R, B, Hq, d, dtype=torch.float32, device=dev)
    lse_all = torch.full((R, B, Hq), -float("inf"), dtype=torch.float32, device=dev)
    out = torch.empty(B, Hq, d, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def one(i):
        kk, vv = pools[i % replicas]
        # this rank's partial lands in its slot of the gathered buffers
        pdb.paged_decode_global_partial(step.plan, li.q, kk, vv, table, lens, li.scale, step.workspace, o_all[0],
                                        lse_all[0], stream)
        pdb.paged_decode_combine(o_all, lse_all, out, stream)

    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            one(i)
        for r in range(1, R):  # the other ranks' partials, as an all-gather would deliver them
            o_all[r].copy_(o_all[0])
            lse_all[r].copy_(lse_all[0])
    torch.cuda.synchronize()
    K = args.steps
    graphs, left, i0 = [], K, 0
    while left > 0:
        m = min(500, left)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(m):
                one(i0 + i)
        graphs.append(g)
        left -= m
        i0 += m
    with torch.cuda.stream(stream):
        graphs[0].replay()
    torch.cuda.synchronize()
    barrier(world)
    sampler = ClockSampler(local)
    sampler.__enter__()
    a = torch.cuda.Event(enable_timing=True)
    z = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for g in graphs:
            g.replay()
        z.record(stream)
    torch.cuda.synchronize()
    sampler.__exit__(None, None, None)
    barrier(world)
    us = max_over_ranks(a.elapsed_time(z), world) * 1e3 / K
    peak, peak_kind = measured_peaks()
    alg = shard_bytes + B * Hq * d * 2 + R * B * Hq * (d + 1) * 4 + B * Hq * d * 2
    if rank == 0:
        line = {
            "metric": DCP_METRIC, "value": round(us, 3), "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": max(3, args.warmup), "ms_per_step": round(us / 1e3, 6), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "io_dtype": "bf16", "data": "synthetic",
            "config": {"workload": synth.WORKLOADS[args.workload] + (f" [{li.name}]" if args.part else ""),
                       "dcp_ranks": R, "shard": "interleaved positions, rank 0", "early_kv": bool(args.early_kv),
                       "shard_kv_bytes": shard_bytes, "exchange": "all-gather of (o, lse) not timed (needs R GPUs)",
                       "l2": f"{replicas} rotating shard replicas", "launch": "CUDA graph replay, one stream"},
            "kv_gbs": round(shard_bytes / (us * 1e-6) / 1e9, 1),
            "roofline": {"bound": "hbm", "kernel": "partial + combine", "achieved": round(alg / (us * 1e-6) / 1e9, 1),
                         "peak": peak, "peak_source": peak_kind, "unit": "GB/s",
                         "frac": round(alg / (us * 1e-6) / 1e9 / peak, 4), "traffic": None, "algorithmic_bytes": alg},
            "cpu_baseline": None, "e2e": None, "gpu_launches": K * 3, "clocks": sampler.summary(),
            "device": torch.cuda.get_device_name(dev),
        }
        print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# reference arm: the oracle on the host cores
# ----------------------------------------------------------------------------

def run_reference_prepare(args, world):
    """The oracle of the fused new-token step, full layer-steps on the host."""
    import oracle
    li = workload_layer(args.workload, args.part, "cpu")
    pc = synth.make_prepare(li, seed=synth.seed_of(args.workload))
    a = [synth.bits_u16(pc.q_in), synth.bits_u16(pc.k_in), None if pc.v_in is None else synth.bits_u16(pc.v_in),
         synth.bits_u16(pc.q_w), synth.bits_u16(pc.k_w), None if pc.v_w is None else synth.bits_u16(pc.v_w),
         li.block_tables.numpy(), li.seq_lens.numpy(), li.num_pages, li.page_size, pc.rot, pc.theta, pc.eps]
    for _ in range(args.warmup):
        oracle.prepare_qkv(*a)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.prepare_qkv(*a)
    us = (time.perf_counter() - t0) / max(1, args.steps) * 1e6
    line = {
        "impl": "reference", "metric": PREP_METRIC, "value": round(us, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us / 1e3, 6), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": synth.WORKLOADS[args.workload] + f" [{li.name}], new-token step", "batch": li.batch,
                   "head_dim": li.head_dim},
        "cpu_baseline": {"value": round(us, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": "full layer-step per step, fp64 C"},
        "e2e": {"value": round(us, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_reference_multi(args, world):
    """The multi-token oracle on the host cores: each step is the full set of
    T x Hq query rows of one request (cycling through the batch), its time
    scaled by the (row, attended position) pairs to a full layer-step."""
    import numpy as np
    import oracle
    T = args.query_tokens
    li = workload_layer(args.workload, args.part, "cpu")
    q = synth.make_query_tokens(li, T, seed=synth.seed_of(args.workload))
    k = synth.bits_u16(li.k_pool)
    v = None if li.v_pool is None else synth.bits_u16(li.v_pool)
    lens = li.seq_lens_list()
    fp8 = args.kv == "fp8"
    if fp8:  # token j of a request is the FP8 decode at length L - T + 1 + j (what the multi-token pins show)
        f8 = synth.quantize_kv_fp8(li)
        k8, v8 = f8.k8.numpy(), None if f8.v8 is None else f8.v8.numpy()
        ks, vs = f8.k_scale.numpy(), None if f8.v_scale is None else f8.v_scale.numpy()

    def pairs(L):
        return sum(min(L - T + 1 + j, li.window) if li.window else L - T + 1 + j for j in range(T)) * li.num_q_heads

    full = sum(pairs(L) for L in lens)

    def sample(i):
        bi = i % li.batch
        t0 = time.perf_counter()
        if fp8:
            for j in range(T):
                oracle.decode_fp8(synth.bits_u16(q[bi:bi + 1, j]), k8, v8, ks, vs, li.block_tables[bi:bi + 1].numpy(),
                                  np.array([lens[bi] - T + 1 + j], np.int32), li.scale, li.window)
        else:
            oracle.decode_multi(synth.bits_u16(q[bi:bi + 1]), k, v, li.block_tables[bi:bi + 1].numpy(),
                                np.array([lens[bi]], np.int32), li.scale, li.window)
        return time.perf_counter() - t0, pairs(lens[bi])

    for i in range(args.warmup):
        sample(i)
    t_total, work = 0.0, 0
    for i in range(args.steps):
        dt, n = sample(i)
        t_total += dt
        work += n
    us = t_total / work * full * 1e6
    line = {
        "impl": "reference", "metric": MULTI_METRIC.format(T=T), "value": round(us, 3), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us / 1e3, 6),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": synth.WORKLOADS[args.workload], "batch": li.batch, "head_dim": li.head_dim,
                   "query_tokens": T, "kv": args.kv},
        "cpu_baseline": {"value": round(us, 3), "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
                         "sample": "one request's T x Hq rows per step, time scaled linearly to a full layer-step"},
        "e2e": {"value": round(us, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_reference(args, world, rank):
    if rank != 0:
        return
    if args.op == "prepare":
        run_reference_prepare(args, world)
        return
    if args.query_tokens > 1:
        run_reference_multi(args, world)
        return
    import numpy as np
    import oracle
    li = workload_layer(args.workload, args.part, "cpu")
    q = synth.bits_u16(li.q)
    fp8 = args.kv == "fp8"
    if fp8:  # the FP8 oracle over the e4m3 cache the GPU arm decodes
        f8 = synth.quantize_kv_fp8(li)
        k8, v8 = f8.k8.numpy(), None if f8.v8 is None else f8.v8.numpy()
        ks, vs = f8.k_scale.numpy(), None if f8.v_scale is None else f8.v_scale.numpy()
    else:
        k = synth.bits_u16(li.k_pool)
        v = None if li.v_pool is None else synth.bits_u16(li.v_pool)
    bt = li.block_tables.numpy()
    full_lens = li.seq_lens.numpy().astype(np.int32)
    threads = oracle.max_threads()
    rows_all = li.batch * li.num_q_heads
    rows = list(range(min(rows_all, threads)))
    full_tokens = sum(li.attended()) * li.num_q_heads  # (row, token) pairs of a layer-step

    def sample_step(frac):
        lens = np.maximum(1, (full_lens * frac).astype(np.int64)).astype(np.int32)
        if li.window > 0:
            lens = full_lens  # the window bounds the work already
        t0 = time.perf_counter()
        if fp8:
            oracle.decode_fp8(q, k8, v8, ks, vs, bt, lens, li.scale, li.window, rows=rows)
        else:
            oracle.decode(q, k, v, bt, lens, li.scale, li.window, rows=rows)
        dt = time.perf_counter() - t0
        att = [min(int(L), li.window) if li.window else int(L) for L in lens]
        done = sum(att[r // li.num_q_heads] for r in rows)
        return dt, done

    # size the sample so warmup + steps fit the time budget
    dt, done = sample_step(1.0)
    per_step_budget = args.ref_seconds / max(1, args.steps + args.warmup)
    frac = min(1.0, max(1e-4, per_step_budget / max(dt, 1e-9)))
    for _ in range(args.warmup):
        sample_step(frac)
    t_total, work = 0.0, 0
    for _ in range(args.steps):
        dt, done = sample_step(frac)
        t_total += dt
        work += done
    us_per_step = t_total / work * full_tokens * 1e6  # scaled to a full layer-step
    sample = (f"{len(rows)} query rows over {frac:.4f} of each attended range per step, "
              "time scaled linearly to a full layer-step")
    if args.op == "layer":  # plus the oracle's new-token step, timed whole
        prep_us = oracle_prepare_us(li, synth.seed_of(args.workload))
        us_per_step += prep_us
        sample += f"; plus the new-token step, {prep_us:.0f} us (full layer-step, median of 5, one core)"
    line = {
        "impl": "reference", "metric": LAYER_METRIC if args.op == "layer" else METRIC,
        "value": round(us_per_step, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us_per_step / 1e3, 6),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": synth.WORKLOADS[args.workload], "batch": li.batch, "head_dim": li.head_dim,
                   "kv": args.kv},
        "cpu_baseline": {"value": round(us_per_step, 3), "unit": UNIT, "cores": len(rows), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(us_per_step, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", type=int, default=4, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--part", default=None, help="workload 4: a|b|c; workload 5: global|sliding")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--kv", default="bf16", choices=["bf16", "fp8"],
                    help="KV-cache element type (fp8: e4m3 with per-(page, KV head) scales)")
    ap.add_argument("--op", default="decode", choices=["decode", "prepare", "layer"],
                    help="decode: the decode layer-step (default); prepare: the fused QKV norm + RoPE + "
                         "paged-cache write of the new tokens; layer: both, the new-token step then the decode")
    ap.add_argument("--query-tokens", type=int, default=1,
                    help="decode op: query tokens per request (> 1: speculative-decode verification, causal)")
    ap.add_argument("--dcp-ranks", type=int, default=1,
                    help="decode op: time one rank of an R-way sequence-sharded decode (partial + combine)")
    ap.add_argument("--early-kv", action=argparse.BooleanOptionalAction, default=True,
                    help="decode / layer: set pd_plan.early_kv (stage 1 copies older cache rows while the "
                         "previous kernel on the stream -- the last step's decode, or the new-token step -- "
                         "is still running; default on)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    args = ap.parse_args()
    if args.workload == 4 and args.part is None:
        args.part = "a"
    if args.workload == 5 and args.part is None:
        args.part = "global"
    world, rank, local = dist_setup()
    if args.gpus != world and world > 1 and rank == 0:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        elif args.op == "prepare":
            run_prepare(args, world, rank, local)
        elif args.dcp_ranks > 1:
            run_dcp(args, world, rank, local)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
