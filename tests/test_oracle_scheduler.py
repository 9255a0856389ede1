"""Pins for the scheduler oracle (CPU only): a hand-worked run and pool
accounting checked against an independent count of live blocks."""
import os

import numpy as np

from oracle import scheduler as osch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FORK, CHILD, EOS = 1, 2, 3


def _ids(x):
    return [] if x == "-" else [int(v) for v in x.split(",")]


def test_golden_run():
    lines = [l.split() for l in open(os.path.join(GOLDEN, "sched_small.txt")) if l.strip() and l[0] != "#"]
    cfg = dict(kv.split("=") for kv in lines[0][1:])
    s = osch.Scheduler(int(cfg["blocks"]), float(cfg["tau"]), int(cfg["n_max"]), int(cfg["window"]),
                       int(cfg["max_len"]), FORK, CHILD, EOS)
    for ln in lines[1:]:
        if ln[0] == "submit":
            s.submit(int(ln[1]), int(ln[2]))
        elif ln[0] == "step":
            step = int(ln[1])
            kv = dict(x.split("=") for x in ln[2:])
            adm, pre, batch = s.schedule(step)
            assert adm == _ids(kv["admitted"]) and pre == _ids(kv["preempted"]), step
            want = [(int(p), _ids(r)) for p, r in (x.split(":") for x in kv["batch"].split("|"))]
            assert batch == want, (step, batch)
            assert s.pool.free == int(kv["free_after_schedule"]), step
            s.update(step, [(int(r), _ids(t)) for r, t in (x.split(":") for x in kv["tokens"].split("|"))])
        elif ln[0] == "output":
            assert s.output(int(ln[1])) == _ids(ln[2])
        elif ln[0] == "final_free":
            assert s.pool.free == int(ln[1])


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
