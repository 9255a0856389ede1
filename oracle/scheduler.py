"""Oracle for the branch scheduler of hierarchical parallel decoding.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain Python, one
decision at a time, with its own model of the paged KV pool (16-token
blocks, reference counts, zero-copy forks).

HPD-Parsing, inference workflow and its Algorithm 1 (the pages give the
steps in prose):
 * an active pool P and a waiting queue Q;
 * Q is ordered first-come-first-served by keys: a child branch has key
   (0, arrival(parent), -m, arrival(child)), a main (layout) request has key
   (1, arrival) -- children of earlier parents come before any new request;
 * a KV occupancy threshold tau and a concurrency cap N_max gate the
   admission of main requests; child branches bypass the gate;
 * KV is reserved ahead of each step for the draft window (K drafted tokens
   plus the anchor); when it runs out, the youngest request is preempted;
 * every step drafts and verifies all active branches in parallel;
 * a <FORK> among the accepted tokens of the layout branch spawns a child
   (content) branch that shares the parent's KV up to that point with zero
   copy;
 * a finished branch releases its KV by reference count, and a parent's
   result is emitted, interleaved with its children's, once all of them
   have finished.

Readings fixed here (also listed in the design notes):
 * m is the number of children the parent had spawned before this child
   (the child's ordinal), fixed when the child is created; keys sort
   ascending, ties by request id;
 * occupancy = blocks in use / pool blocks; the gate admits a main request
   only while occupancy <= tau and |P| < N_max;
 * a branch's token stream is its prefix (a main request's prompt, a
   child's fork_len parent tokens) followed by its output; every token but
   the newest is cached, the newest being the anchor of the next verify step
   (a main request's first anchor is its last prompt token, a child's is
   <CHILD>);
 * each step first reserves, for every active branch in key order, blocks
   for its cached tokens plus K + 1; on a shortage the youngest active
   request (latest arrival, then highest id) is preempted: its KV is
   released and it returns to Q to be rebuilt later, and the reservation is
   retried.  The youngest active request never has an active child (a child
   arrives after its parent), so no running branch loses its prefix;
 * then Q is scanned in key order: a main request passes the gate or is
   skipped; a child is ready once its parent is resident (it has cached the
   tokens before the <FORK>: everything but its newest token is cached); a request whose KV cannot be reserved keeps its place
   and the scan goes on (stopping there can deadlock: ended layout requests
   keep their prefixes for children that wait behind a larger request);
   requests preempted in this step wait for the next one;
 * admission reserves the cached tokens + K + 1 and rebuilds the cached
   tokens (a main request: prompt and output but the anchor; a child forks
   its parent at fork_len, the parent's tokens before the <FORK> -- the
   structural prefix of its region; it starts its own stream with <CHILD> --
   and rebuilds its own cached tokens in fresh blocks);
 * the accepted tokens of a step (n_acc drafted tokens plus the free token)
   extend the branch's output; the step's commit caches the old anchor and
   all new tokens but the newest; branches are updated in the order given;
 * a branch ends at <EOS> or after max_len generated tokens (tokens after
   the end are dropped); at its end the unused part of its reservation goes
   back to the pool, and its sequence is released once it and all its
   children have ended;
 * only main (layout) requests fork; a <FORK> in a content branch's output
   is an ordinary token;
 * a main request's output interleaves: after each <FORK> token comes the
   full output of the child spawned there.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Tuple

BS = 16


class Pool:
    """Block accounting of the paged KV pool: refcounted blocks, per-sequence
    block lists and token counts (cached tokens)."""

    def __init__(self, n_blocks: int):
        self.free = n_blocks
        self.total = n_blocks
        self.ref: Dict[int, int] = {}
        self.next_block = 0
        self.seqs: Dict[int, dict] = {}
        self.next_seq = 0

    def used(self) -> int:
        return self.total - self.free

    def _take(self, n: int) -> Optional[List[int]]:
        if n > self.free:
            return None
        out = []
        for _ in range(n):
            b = self.next_block
            self.next_block += 1
            self.ref[b] = 1
            out.append(b)
        self.free -= n
        return out

    def alloc(self, n_tokens: int) -> Optional[int]:
        blocks = self._take(-(-n_tokens // BS))
        if blocks is None:
            return None
        s = self.next_seq
        self.next_seq += 1
        self.seqs[s] = {"blocks": blocks, "n_shared": 0, "len": 0, "fork_len": 0}
        return s

    def fork(self, parent: int, fork_len: int) -> int:
        p = self.seqs[parent]
        nsh = -(-fork_len // BS)
        blocks = p["blocks"][:nsh]
        for b in blocks:
            self.ref[b] += 1
        s = self.next_seq
        self.next_seq += 1
        self.seqs[s] = {"blocks": list(blocks), "n_shared": nsh, "len": fork_len, "fork_len": fork_len}
        return s

    def reserve(self, seq: int, n_more: int) -> bool:
        """Blocks for len + n_more tokens; all or nothing."""
        s = self.seqs[seq]
        own = s["len"] - s["fork_len"]
        need = -(-(own + n_more) // BS)
        have = len(s["blocks"]) - s["n_shared"]
        if need > have:
            got = self._take(need - have)
            if got is None:
                return False
            s["blocks"].extend(got)
        return True

    def advance(self, seq: int, n: int):
        s = self.seqs[seq]
        s["len"] += n
        assert s["len"] - s["fork_len"] <= (len(s["blocks"]) - s["n_shared"]) * BS

    def trim(self, seq: int):
        """Drops the sequence's own blocks past its cached tokens."""
        s = self.seqs[seq]
        keep = s["n_shared"] + -(-(s["len"] - s["fork_len"]) // BS)
        for b in s["blocks"][keep:]:
            self.ref[b] -= 1
            if self.ref[b] == 0:
                del self.ref[b]
                self.free += 1
        del s["blocks"][keep:]

    def release(self, seq: int):
        s = self.seqs.pop(seq)
        for b in s["blocks"]:
            self.ref[b] -= 1
            if self.ref[b] == 0:
                del self.ref[b]
                self.free += 1


@dataclasses.dataclass
class Req:
    rid: int
    arrival: int
    parent: Optional[int]
    m: int = 0
    prompt_len: int = 0
    fork_len: int = 0
    out: List[int] = dataclasses.field(default_factory=list)
    children: List[int] = dataclasses.field(default_factory=list)
    n_spawned: int = 0
    state: str = "waiting"      # waiting | running | ended | done
    seq: int = -1


class Scheduler:
    def __init__(self, n_blocks: int, tau: float, n_max: int, window: int, max_len: int, fork: int, child: int,
                 eos: int):
        self.pool = Pool(n_blocks)
        self.tau, self.n_max, self.K, self.max_len = tau, n_max, window, max_len
        self.FORK, self.CHILD, self.EOS = fork, child, eos
        self.reqs: Dict[int, Req] = {}
        self.queue: List[int] = []
        self.active: List[int] = []
        self.next_id = 0

    # -- keys
    def key(self, rid: int) -> Tuple:
        r = self.reqs[rid]
        if r.parent is None:
            return (1, r.arrival, 0, 0, rid)
        return (0, self.reqs[r.parent].arrival, -r.m, r.arrival, rid)

    def submit(self, prompt_len: int, arrival: int) -> int:
        rid = self.next_id
        self.next_id += 1
        self.reqs[rid] = Req(rid, arrival, None, prompt_len=prompt_len)
        self.queue.append(rid)
        return rid

    def _stream_len(self, r: Req) -> int:
        return (r.prompt_len if r.parent is None else r.fork_len) + len(r.out)

    def _preempt(self, rid: int):
        r = self.reqs[rid]
        self.pool.release(r.seq)
        r.seq = -1
        r.state = "waiting"
        self.active.remove(rid)
        self.queue.append(rid)

    def _admit_kv(self, r: Req) -> bool:
        cached = self._stream_len(r) - 1  # all but the anchor
        if r.parent is None:
            s = self.pool.alloc(cached + self.K + 1)
            if s is None:
                return False
            self.pool.advance(s, cached)
        else:
            p = self.reqs[r.parent]
            s = self.pool.fork(p.seq, r.fork_len)
            if not self.pool.reserve(s, cached - r.fork_len + self.K + 1):
                self.pool.release(s)
                return False
            self.pool.advance(s, cached - r.fork_len)
        r.seq = s
        return True

    def schedule(self, now: int):
        """One step's decisions: returns (admitted ids, preempted ids, active
        ids in key order)."""
        preempted = []
        # 1. reserve the step's window for every active branch
        for rid in sorted(self.active, key=self.key):
            if rid not in self.active:
                continue
            while not self.pool.reserve(self.reqs[rid].seq, self.K + 1):
                victim = max(self.active, key=lambda a: (self.reqs[a].arrival, a))
                self._preempt(victim)
                preempted.append(victim)
                if victim == rid:
                    break
        # 2. admission in key order
        admitted = []
        for rid in sorted(self.queue, key=self.key):
            if rid in preempted:
                continue
            r = self.reqs[rid]
            if r.parent is None:
                occ = self.pool.used() / self.pool.total
                if occ > self.tau or len(self.active) >= self.n_max:
                    continue
            else:
                p = self.reqs[r.parent]
                if p.seq < 0 or self.pool.seqs[p.seq]["len"] < r.fork_len:
                    continue  # parent not resident, or its <FORK> not cached yet
            if not self._admit_kv(r):
                continue  # no room this step: it keeps its place
            r.state = "running"
            self.queue.remove(rid)
            self.active.append(rid)
            admitted.append(rid)
        return admitted, preempted, self.batch()

    def batch(self) -> List[Tuple[int, List[int]]]:
        """Active branches grouped by page (the request whose sequence holds
        the shared prefix: the parent of a child, a main request itself),
        pages in order of their first branch in key order."""
        pages: Dict[int, List[int]] = {}
        for rid in sorted(self.active, key=self.key):
            r = self.reqs[rid]
            pg = rid if r.parent is None else r.parent
            pages.setdefault(pg, []).append(rid)
        return list(pages.items())

    def update(self, now: int, accepted: List[Tuple[int, List[int]]]):
        """The verified tokens of each active branch (n_acc drafts plus the
        free token, at least one), in the given order."""
        for rid, toks in accepted:
            r = self.reqs[rid]
            assert len(toks) >= 1 and r.state == "running"
            ended = False
            taken = 0
            for t in toks:
                r.out.append(t)
                taken += 1
                if t == self.FORK and r.parent is None:
                    c = self.next_id
                    self.next_id += 1
                    base = r.prompt_len if r.parent is None else r.fork_len
                    self.reqs[c] = Req(c, now, rid, m=r.n_spawned, fork_len=base + len(r.out) - 1, out=[self.CHILD])
                    r.n_spawned += 1
                    r.children.append(c)
                    self.queue.append(c)
                if t == self.EOS or len(r.out) >= self.max_len:
                    ended = True
                    break
            # the old anchor and the new tokens but the newest are now cached
            self.pool.advance(r.seq, taken)
            if ended:
                r.state = "ended"
                self.active.remove(rid)
                self.pool.trim(r.seq)  # the unused part of its reservation
                self._maybe_release(rid)

    def _maybe_release(self, rid: int):
        r = self.reqs[rid]
        if r.state != "ended" or any(self.reqs[c].state != "done" for c in r.children):
            return
        self.pool.release(r.seq)
        r.seq = -1
        r.state = "done"
        if r.parent is not None:
            self._maybe_release(r.parent)

    def output(self, rid: int) -> List[int]:
        r = self.reqs[rid]
        assert r.state == "done"
        out, k = [], 0
        for t in r.out:
            out.append(t)
            if t == self.FORK:
                out.extend(self.output(r.children[k]))
                k += 1
        return out
