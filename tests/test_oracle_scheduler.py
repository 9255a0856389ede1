"""Pins for the scheduler oracle (CPU only): hand-worked runs (one child per
parent; several children forked in one step, sibling order by -m, nested
outputs, preemption and the N_max gate), mistakes planted in the oracle
that those runs catch, and pool accounting checked against an independent
count of live blocks."""
import os

import numpy as np
import pytest

from oracle import scheduler as osch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FORK, CHILD, EOS = 1, 2, 3


def _ids(x):
    return [] if x == "-" else [int(v) for v in x.split(",")]


GOLDEN_RUNS = ["sched_small.txt", "sched_multichild.txt"]


def replay(sched, name):
    """Drives a scheduler (the oracle, or the C++ port through an adapter
    with the same methods) through a hand-worked golden run and asserts
    every recorded decision, free-block count and output."""
    lines = [l.split() for l in open(os.path.join(GOLDEN, name)) if l.strip() and l[0] != "#"]
    cfg = dict(kv.split("=") for kv in lines[0][1:])
    s = sched(int(cfg["blocks"]), float(cfg["tau"]), int(cfg["n_max"]), int(cfg["window"]), int(cfg["max_len"]))
    for ln in lines[1:]:
        if ln[0] == "submit":
            s.submit(int(ln[1]), int(ln[2]))
        elif ln[0] == "step":
            step = int(ln[1])
            kv = dict(x.split("=") for x in ln[2:])
            adm, pre, batch = s.schedule(step)
            assert adm == _ids(kv["admitted"]) and pre == _ids(kv["preempted"]), (step, adm, pre)
            want = [(int(p), _ids(r)) for p, r in (x.split(":") for x in kv["batch"].split("|"))]
            assert batch == want, (step, batch)
            assert s.free() == int(kv["free_after_schedule"]), step
            s.update(step, [(int(r), _ids(t)) for r, t in (x.split(":") for x in kv["tokens"].split("|"))])
            if "free_after_update" in kv:
                assert s.free() == int(kv["free_after_update"]), step
        elif ln[0] == "output":
            assert s.output(int(ln[1])) == _ids(ln[2]), ln[1]
        elif ln[0] == "final_free":
            assert s.free() == int(ln[1])


class OracleSched:
    def __init__(self, blocks, tau, n_max, window, max_len):
        self.s = osch.Scheduler(blocks, tau, n_max, window, max_len, FORK, CHILD, EOS)

    def submit(self, prompt, at):
        return self.s.submit(prompt, at)

    def schedule(self, step):
        return self.s.schedule(step)

    def update(self, step, acc):
        self.s.update(step, acc)

    def output(self, rid):
        return self.s.output(rid)

    def free(self):
        return self.s.pool.free


@pytest.mark.parametrize("name", GOLDEN_RUNS)
def test_golden_run(name):
    replay(OracleSched, name)


def test_golden_catches_flipped_sibling_order(monkeypatch):
    """A planted mistake in the oracle: siblings ordered by +m instead of -m.
    The multi-child run admits child 4 instead of 6 at step 1 and fails."""
    def key_plus_m(self, rid):
        r = self.reqs[rid]
        if r.parent is None:
            return (1, r.arrival, 0, 0, rid)
        return (0, self.reqs[r.parent].arrival, r.m, r.arrival, rid)

    monkeypatch.setattr(osch.Scheduler, "key", key_plus_m)
    with pytest.raises(AssertionError):
        replay(OracleSched, "sched_multichild.txt")


def test_golden_catches_wrong_child_nesting(monkeypatch):
    """A planted mistake in the oracle: the children's outputs emitted in
    reverse order of their <FORK>s.  The multi-child run fails."""
    def output_reversed(self, rid):
        r = self.reqs[rid]
        out, kids = [], list(reversed(r.children))
        for t in r.out:
            out.append(t)
            if t == self.FORK:
                out.extend(output_reversed(self, kids.pop(0)))
        return out

    monkeypatch.setattr(osch.Scheduler, "output", output_reversed)
    with pytest.raises(AssertionError):
        replay(OracleSched, "sched_multichild.txt")


def test_golden_catches_parent_released_early(monkeypatch):
    """A planted mistake in the oracle: a parent's sequence released as soon
    as it ends, without waiting for its children.  At step 1 layout request
    A ends with two children still queued; its two blocks come back at once
    and the recorded free-block count no longer matches."""
    def release_now(self, rid):
        r = self.reqs[rid]
        if r.state == "ended" and r.seq >= 0:
            self.pool.release(r.seq)
            r.seq = -1
        if r.state == "ended" and all(self.reqs[c].state == "done" for c in r.children):
            r.state = "done"
            if r.parent is not None:
                release_now(self, r.parent)

    monkeypatch.setattr(osch.Scheduler, "_maybe_release", release_now)
    with pytest.raises(AssertionError):
        replay(OracleSched, "sched_multichild.txt")


def test_pool_accounting_against_live_blocks():
    """Blocks in use equal the distinct blocks referenced by live sequences,
    and every refcount equals the number of sequences holding the block."""
    from test_scheduler import tokens_for
    rng = np.random.default_rng(3)
    s = osch.Scheduler(40, 0.8, 3, 3, 40, FORK, CHILD, EOS)
    for _ in range(6):
        s.submit(int(rng.integers(1, 120)), int(rng.integers(0, 20)))
    for step in range(300):
        _, _, batch = s.schedule(step)
        held = {}
        for seq in s.pool.seqs.values():
            for b in seq["blocks"]:
                held[b] = held.get(b, 0) + 1
        assert s.pool.used() == len(held) and held == s.pool.ref
        act = [r for _, rids in batch for r in rids]
        s.update(step, [(r, tokens_for(9, r, len(s.reqs[r].out), s.reqs[r].parent is None, 3)) for r in act])
