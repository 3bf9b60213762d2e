"""The host-in/host-out loop's buffer schedule (no GPU).

Checks, for loops of 1..12 steps with and without early_kv, what the ordering
of the launch chain requires: every step's q, table/lengths and result cross
exactly once; inputs arrive before their step; a copy issued after step i
touches no buffer of step i (still running) and, with early_kv, not the table
buffer of step i + 1 (read before that stage 1's wait); a buffer is rewritten
only once no step in flight or before its new owner uses it. A schedule built
with the table one step ahead under early_kv is caught.
"""
import pytest

from paged_gqa_decode_global_gb300 import host_loop as hl

BUF = {"q": hl.q_buffer, "meta": hl.meta_buffer, "out": hl.out_buffer}


def violations(s: hl.Schedule, n: int, early_kv: bool):
    bad = []
    issued = {}  # (kind, step) -> position: -1 before the loop, i after step i, n for the final copy
    for pos, cps in [(-1, s.before)] + list(enumerate(s.after_step)) + [(n, s.final)]:
        for c in cps:
            if (c.kind, c.step) in issued:
                bad.append(f"{c.kind} of step {c.step} copied twice")
            issued[(c.kind, c.step)] = pos
            if c.buffer != BUF[c.kind](c.step):
                bad.append(f"{c.kind} of step {c.step} in buffer {c.buffer}")
            if pos < 0 or pos >= n:
                continue
            i = pos  # issued after step i: step i may still run, steps before it are done
            if c.kind in ("q", "meta"):
                if c.step <= i:
                    bad.append(f"{c.kind} of step {c.step} arrives after its step ({i})")
                # steps from i up to the new owner must not use the buffer being written
                for t in range(i, c.step):
                    if BUF[c.kind](t) == c.buffer:
                        bad.append(f"copy after step {i} overwrites the {c.kind} buffer of step {t}")
                if early_kv and c.kind == "meta" and c.step == i + 1:
                    bad.append(f"copy after step {i} writes the table step {i + 1} reads before its wait")
            else:
                if c.step >= i:
                    bad.append(f"result of step {c.step} taken while it may run (after step {i})")
                if hl.out_buffer(i) == c.buffer:
                    bad.append(f"copy after step {i} reads the result buffer step {i} writes")
    for j in range(n):
        for kind in ("q", "meta", "out"):
            if (kind, j) not in issued:
                bad.append(f"{kind} of step {j} never copied")
    for (kind, j), pos in issued.items():
        if kind == "out" and pos != (j + 1 if j + 1 < n else n):
            bad.append(f"result of step {j} copied at {pos}")
    return bad


@pytest.mark.parametrize("early_kv", [False, True])
@pytest.mark.parametrize("n", range(1, 13))
def test_schedule_keeps_the_chain_order(n, early_kv):
    s = hl.schedule(n, early_kv)
    assert s.ahead == (2 if early_kv else 1)
    assert violations(s, n, early_kv) == []
    assert all(len(cps) <= 4 for cps in s.after_step)  # one stage copy each (PD_MAX_STAGE_COPIES)


def test_table_one_step_ahead_under_early_kv_is_caught():
    s = hl.schedule(6, early_kv=False)
    assert any("before its wait" in v for v in violations(s, 6, early_kv=True))


def test_a_buffer_reused_too_soon_is_caught():
    s = hl.schedule(5, early_kv=False)
    wrong = hl.Schedule(s.ahead, s.before, [[hl.Copy(c.kind, c.step, 0) if c.kind == "q" else c for c in cps]
                                            for cps in s.after_step], s.final)
    assert any("overwrites the q buffer" in v or "in buffer" in v for v in violations(wrong, 5, False))


def test_rejects_an_empty_loop():
    with pytest.raises(ValueError):
        hl.schedule(0, early_kv=True)
