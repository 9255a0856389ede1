"""The C++ branch scheduler against the scheduler oracle (host code, CPU
only).  Both are driven by the same seeded token stream; every decision
(admissions, preemptions, the batch grouped by page), the pool's block
usage and the interleaved outputs must agree exactly."""
import os
import subprocess
import sys

import numpy as np
import pytest

from oracle import scheduler as osch
from tree_structured_shared_gb300 import padoc

FORK, CHILD, EOS = 1, 2, 3
FAKE = 1 << 20  # pool storage is never touched: the scheduler only keeps books


def tokens_for(seed, rid, n_out, is_main, window):
    """The 'model': verified tokens of one branch for one step, a pure
    function of (seed, request, output length)."""
    rng = np.random.default_rng([seed, rid, n_out])
    n = 1 + int(rng.integers(0, window + 1))
    out = []
    for i in range(n):
        L = n_out + i
        u = rng.random()
        if is_main and u < 0.15:
            out.append(FORK)
        elif u < (0.02 + L / 400.0 if is_main else 0.05 + L / 250.0):
            out.append(EOS)
        else:
            out.append(10 + int(rng.integers(0, 1000)))
    return out


def run_both(seed, n_blocks, tau, n_max, window, max_len, arrivals, n_steps):
    pool = padoc.KVPool(FAKE, FAKE, n_blocks, Hkv=2, d=128, max_seqs=512, max_blocks_per_seq=64)
    cs = padoc.Scheduler(pool, tau, n_max, window, max_len, FORK, CHILD, EOS)
    os_ = osch.Scheduler(n_blocks, tau, n_max, window, max_len, FORK, CHILD, EOS)
    parent = {}
    n_pre = 0
    for step in range(n_steps):
        for prompt, at in arrivals:
            if at == step:
                a, b = cs.submit(prompt, at), os_.submit(prompt, at)
                assert a == b
                parent[a] = -1
        adm_c, pre_c, pages_c = cs.schedule()
        adm_o, pre_o, pages_o = os_.schedule(step)
        assert adm_c == adm_o and pre_c == pre_o, (step, adm_c, adm_o, pre_c, pre_o)
        n_pre += len(pre_c)
        got = [([r for r, _ in br]) for _, br in pages_c]
        want = [rids for _, rids in pages_o]
        assert got == want, (step, got, want)
        for pseq, br in pages_c:  # the page's sequence is the parent's (or the main request's own)
            r0 = br[0][0]
            p = parent[r0] if parent[r0] >= 0 else r0
            assert pseq == cs.request(p)["seq"]
        assert pool.stats()["free_blocks"] == os_.pool.free, step
        batch = [r for _, rids in pages_o for r in rids]
        acc = []
        for r in batch:
            n_out = len(os_.reqs[r].out)
            assert cs.request(r)["n_out"] == n_out
            acc.append((r, tokens_for(seed, r, n_out, os_.reqs[r].parent is None, window)))
        cs.update(step, acc)
        os_.update(step, acc)
        for rid, rq in os_.reqs.items():
            parent.setdefault(rid, -1 if rq.parent is None else rq.parent)
        assert pool.stats()["free_blocks"] == os_.pool.free, step
    done = [rid for rid, r in os_.reqs.items() if r.parent is None and r.state == "done"]
    for rid in done:
        assert cs.request(rid)["state"] == "done"
        assert cs.output(rid) == os_.output(rid)
    return cs, os_, pool, done, n_pre


@pytest.mark.parametrize("seed", range(6))
def test_matches_oracle(padoc_lib, seed):
    rng = np.random.default_rng(seed)
    arrivals = [(int(rng.integers(1, 200)), int(rng.integers(0, 40))) for _ in range(10)]
    cs, os_, pool, done, n_pre = run_both(seed, n_blocks=48, tau=0.7, n_max=3, window=4, max_len=60,
                                          arrivals=arrivals, n_steps=400)
    assert len(done) >= 1


def test_preemption_and_full_release(padoc_lib):
    """A tight pool forces preemptions; once everything has ended every block
    is free again (children held their parents' blocks by reference)."""
    arrivals = [(60, 0), (90, 0), (40, 1), (120, 2), (30, 5)]
    cs, os_, pool, done, n_pre = run_both(11, n_blocks=26, tau=1.0, n_max=8, window=6, max_len=50,
                                          arrivals=arrivals, n_steps=2000)
    assert n_pre > 0
    assert len(done) == len(arrivals)
    assert pool.stats()["free_blocks"] == 26 and os_.pool.free == 26


def test_gate_and_child_bypass(padoc_lib):
    """With n_max = 1 only one main request runs at a time, yet its children
    are admitted next to it (they bypass the gate)."""
    arrivals = [(20, 0), (20, 0), (20, 0)]
    pool = padoc.KVPool(FAKE, FAKE, 400, Hkv=2, d=128, max_seqs=512, max_blocks_per_seq=64)
    cs = padoc.Scheduler(pool, 1.0, 1, 3, 40, FORK, CHILD, EOS)
    for p, a in arrivals:
        cs.submit(p, a)
    saw_children = False
    for step in range(600):
        adm, pre, pages = cs.schedule()
        act = [r for _, br in pages for r, _ in br]
        mains = [r for r in act if cs.request(r)["parent"] < 0]
        assert len(mains) <= 1
        saw_children |= len(act) > len(mains)
        cs.update(step, [(r, tokens_for(5, r, cs.request(r)["n_out"], cs.request(r)["parent"] < 0, 3))
                         for r in act])
    assert saw_children
    assert all(cs.request(r)["state"] == "done" for r in range(3))


def test_fault_injection(padoc_lib):
    """Block allocation failing after a fixed count (PADOC_FAULT_ALLOC_AFTER)
    looks like a full pool: the scheduler preempts and stalls instead of
    failing, and the pool's books stay consistent."""
    code = (
        "import sys; sys.path.insert(0, %r); sys.path.insert(0, %r)\n"
        "from tree_structured_shared_gb300 import padoc\n"
        "from test_scheduler import tokens_for, FORK, CHILD, EOS, FAKE\n"
        "pool = padoc.KVPool(FAKE, FAKE, 200, Hkv=2, d=128, max_seqs=64, max_blocks_per_seq=64)\n"
        "cs = padoc.Scheduler(pool, 1.0, 8, 4, 200, FORK, CHILD, EOS)\n"
        "for i in range(4): cs.submit(40, 0)\n"
        "npre = 0\n"
        "for step in range(300):\n"
        "    adm, pre, pages = cs.schedule(); npre += len(pre)\n"
        "    act = [r for _, br in pages for r, _ in br]\n"
        "    cs.update(step, [(r, [10 + step %% 7]) for r in act])\n"
        "print('OK', npre, pool.stats()['free_blocks'])\n"
    ) % (os.path.dirname(os.path.dirname(os.path.abspath(__file__))), os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, PADOC_FAULT_ALLOC_AFTER="12")
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    tag, npre, free = out.stdout.split()
    assert tag == "OK" and int(npre) > 0


def test_rejects_bad_arguments(padoc_lib):
    pool = padoc.KVPool(FAKE, FAKE, 10, Hkv=2, d=128)
    with pytest.raises(padoc.PadocError):
        padoc.Scheduler(pool, 1.5, 1, 3, 10, FORK, CHILD, EOS)
    with pytest.raises(padoc.PadocError):
        padoc.Scheduler(pool, 0.5, 0, 3, 10, FORK, CHILD, EOS)
    cs = padoc.Scheduler(pool, 0.5, 1, 3, 10, FORK, CHILD, EOS)
    with pytest.raises(padoc.PadocError):
        cs.submit(0, 0)
    with pytest.raises(padoc.PadocError):
        cs.update(0, [(0, [5])])  # not running
    with pytest.raises(padoc.PadocError):
        cs.output(0)


class PortSched:
    """The C++ scheduler behind the golden replay's interface: batches come
    back as (page request, branch ids), the page's pool sequence checked."""

    def __init__(self, blocks, tau, n_max, window, max_len):
        self.pool = padoc.KVPool(FAKE, FAKE, blocks, Hkv=2, d=128, max_seqs=64, max_blocks_per_seq=64)
        self.s = padoc.Scheduler(self.pool, tau, n_max, window, max_len, FORK, CHILD, EOS)

    def submit(self, prompt, at):
        return self.s.submit(prompt, at)

    def schedule(self, step):
        adm, pre, pages = self.s.schedule()
        out = []
        for pseq, br in pages:
            rids = [r for r, _ in br]
            par = self.s.request(rids[0])["parent"]
            page = par if par >= 0 else rids[0]
            assert pseq == self.s.request(page)["seq"]
            out.append((page, rids))
        return adm, pre, out

    def update(self, step, acc):
        self.s.update(step, acc)

    def output(self, rid):
        return self.s.output(rid)

    def free(self):
        return self.pool.stats()["free_blocks"]


@pytest.mark.parametrize("name", ["sched_small.txt", "sched_multichild.txt"])
def test_port_golden_run(padoc_lib, name):
    """The C++ port replays the hand-worked runs directly."""
    from test_oracle_scheduler import replay
    replay(PortSched, name)

