"""Pins for the accept-step oracle (CPU only)."""
import math
import os

import numpy as np
import pytest

from oracle import accept as acc
from tree_structured_shared_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_golden_small_tree():
    rows, expects = [], []
    with open(os.path.join(GOLDEN, "accept_small.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            p = line.split()
            if p[0] == "parents":
                parents = [int(x) for x in p[1:]]
            elif p[0] == "tokens":
                tokens = [int(x) for x in p[1:]]
            elif p[0] == "row":
                rows.append([float(x) for x in p[1:]])
            elif p[0] == "expect":
                path = [] if p[3] == "-" else [int(x) for x in p[3].split(",")]
                expects.append((float(p[1]), path, int(p[5])))
    logits = np.array(rows, np.float32)
    for tau, path, free in expects:
        assert acc.accept_tree(logits, tokens, parents, tau) == (path, free)


def test_chain_tau_one_is_greedy_prefix_match():
    """HPD-Parsing: n_acc = max{k : y*_{n+i} = t_hat_i for all i <= k}.
    (Tie-free logits: under an exact tie the log-ratio rule with tau = 1
    accepts any maximiser, while 'equals the argmax' names one of them.)"""
    rng = np.random.default_rng(0)
    for _ in range(200):
        n = int(rng.integers(1, 9))
        V = 6
        logits = rng.standard_normal((n, V)).astype(np.float32)
        tokens = rng.integers(0, V, size=n).tolist()
        for i in range(n - 1):  # make some drafts agree with the greedy choice
            if rng.random() < 0.6:
                tokens[i + 1] = int(np.argmax(logits[i]))
        parents = [-1] + list(range(n - 1))
        # greedy predictions y* written directly: row i predicts node i+1
        ystar = [int(np.argmax(logits[i])) for i in range(n)]
        k = 0
        while k + 1 < n and tokens[k + 1] == ystar[k]:
            k += 1
        path, free = acc.accept_tree(logits, tokens, parents, 1.0)
        assert path == list(range(1, k + 1))
        assert free == ystar[k]


def test_tau_limits():
    rng = np.random.default_rng(1)
    for _ in range(100):
        par = wl.draft_tree(rng)
        n, V = len(par), 7
        logits = rng.standard_normal((n, V)).astype(np.float32)
        tokens = rng.integers(0, V, size=n).tolist()
        # tau > 1: log tau > 0 and logit(u*) - logit(u_hat) <= 0, nothing accepted
        path, free = acc.accept_tree(logits, tokens, par, 2.0)
        assert path == [] and free == int(np.argmax(logits[0]))
        # tau tiny: every step accepts; the walk ends at a leaf
        path, _ = acc.accept_tree(logits, tokens, par, 1e-30)
        last = path[-1] if path else 0
        assert last not in par[1:]  # no children


def test_accepted_steps_satisfy_the_rule():
    rng = np.random.default_rng(2)
    log_tau = np.float32(math.log(0.75))
    for _ in range(200):
        par = wl.draft_tree(rng)
        n, V = len(par), 9
        logits = rng.integers(-4, 5, size=(n, V)).astype(np.float32)
        tokens = rng.integers(0, V, size=n).tolist()
        path, free = acc.accept_tree(logits, tokens, par, 0.75)
        s = 0
        for node in path + [None]:
            kids = [c for c in range(1, n) if par[c] == s]
            row = logits[s]
            top = row.max()
            if node is None:
                # stopped: no children, or the best child fails the rule
                assert free == int(np.argmax(row))
                if kids:
                    assert max(row[tokens[c]] for c in kids) - top < log_tau
                break
            assert par[node] == s
            assert row[tokens[node]] == max(row[tokens[c]] for c in kids)
            assert row[tokens[node]] - top >= log_tau
            s = node
