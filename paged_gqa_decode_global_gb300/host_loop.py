"""Buffer schedule of a host-in/host-out decode loop built on paged_decode_stage_copy.

Each step's q (or new rows) comes from page-locked host memory, its block
table and lengths too, and its result goes back. The loop keeps one chain of
programmatic dependent launches: after step i's kernels one stage copy brings
step i + 1's q into the other of two q buffers, the table and lengths of step
i + ahead into the third of three buffers, and takes step i - 1's result out of
the other of two result buffers (after_wait 0); a last copy, waiting first,
takes the final result out. `ahead` is 2 when the decode runs with
pd_plan.early_kv (its stage 1 reads the table and lengths before its
dependency wait, so the copy in front of it must not be the one writing them)
and 1 otherwise; before the loop, ordinary copies bring in step 0's q and the
first `ahead` steps' tables.

When a copy issued after step i starts, every kernel of steps before i has
completed (the decode and merge kernels signal their dependents only after
their own wait, and each copy completes only after the launch in front of it),
while step i's own kernels may still run: a copy may therefore touch any buffer
but those of step i, and, with early_kv, not the table buffer of step i + 1.

This module is host bookkeeping only: which buffer each copy uses. The copies
are issued with paged_decode_stage_copy.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List

Q_BUFFERS = 2
META_BUFFERS = 3
OUT_BUFFERS = 2


@dataclass(frozen=True)
class Copy:
    kind: str    # "q" (host -> device), "meta" (host -> device) or "out" (device -> host)
    step: int    # the step whose data it carries
    buffer: int  # index of the device buffer of that kind


@dataclass(frozen=True)
class Schedule:
    ahead: int                  # steps the table and lengths go ahead of their decode
    before: List[Copy]          # ordinary copies before the loop
    after_step: List[List[Copy]]  # the stage copy issued after each step's kernels (after_wait 0)
    final: List[Copy]           # the last stage copy (after_wait 1)


def q_buffer(step: int) -> int:
    return step % Q_BUFFERS


def meta_buffer(step: int) -> int:
    return step % META_BUFFERS


def out_buffer(step: int) -> int:
    return step % OUT_BUFFERS


def schedule(n_steps: int, early_kv: bool) -> Schedule:
    """The copies of an n_steps loop (n_steps >= 1)."""
    if n_steps < 1:
        raise ValueError("a loop of at least one step")
    ahead = 2 if early_kv else 1
    before = [Copy("q", 0, q_buffer(0))] + [Copy("meta", j, meta_buffer(j)) for j in range(min(ahead, n_steps))]
    after: List[List[Copy]] = []
    for i in range(n_steps):
        cps = []
        if i + 1 < n_steps:
            cps.append(Copy("q", i + 1, q_buffer(i + 1)))
        if i + ahead < n_steps:
            cps.append(Copy("meta", i + ahead, meta_buffer(i + ahead)))
        if i > 0:
            cps.append(Copy("out", i - 1, out_buffer(i - 1)))
        after.append(cps)
    final = [Copy("out", n_steps - 1, out_buffer(n_steps - 1))]
    return Schedule(ahead, before, after, final)
