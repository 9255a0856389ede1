"""Pins for the draft-trie oracle (CPU only)."""
import os

import numpy as np
import pytest

from oracle import draft_trie as dt

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden():
    drafts, accepted, cases = [], None, []
    with open(os.path.join(GOLDEN, "draft_trie_small.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            p = line.split()
            if p[0] == "draft":
                drafts.append([int(x) for x in p[1:]])
            elif p[0] == "accepted":
                accepted = [int(x) for x in p[1:]]
            elif p[0] == "expect":
                kv = dict(x.split("=") for x in p[1:])
                cases.append((int(kv["n"]), int(kv["max_nodes"]), int(kv["max_depth"]),
                              [int(x) for x in kv["tokens"].split(",")], [int(x) for x in kv["parents"].split(",")]))
    return drafts, accepted, cases


def test_golden_trie():
    drafts, accepted, cases = _golden()
    for n, mn, md, tokens, parents in cases:
        assert dt.draft_tree(drafts, accepted, n, mn, md) == (tokens, parents), (n, mn, md)


def _random_case(rng, vocab=4):
    drafts = [rng.integers(0, vocab, int(rng.integers(0, 30))).tolist() for _ in range(int(rng.integers(1, 6)))]
    accepted = rng.integers(0, vocab, int(rng.integers(1, 8))).tolist()
    return drafts, accepted


def _paths(tokens, parents):
    out = []
    for i in range(1, len(tokens)):
        p, j = [], i
        while j > 0:
            p.append(tokens[j])
            j = parents[j]
        out.append(tuple(reversed(p)))
    return out


@pytest.mark.parametrize("n", [1, 2, 3])
def test_unbounded_trie_is_the_set_of_candidate_prefixes(n):
    """With no budget the non-root nodes are exactly the distinct non-empty
    prefixes of the candidates, each once (brute-force set)."""
    rng = np.random.default_rng(n)
    for _ in range(300):
        drafts, accepted = _random_case(rng)
        tokens, parents = dt.draft_tree(drafts, accepted, n, max_nodes=10**6, max_depth=10**6)
        # candidates by brute force over every (draft, position) pair
        w = accepted[-n:] if len(accepted) >= n else None
        prefixes = set()
        for d in drafts:
            for j in range(len(d)):
                if w is not None and d[j:j + n] == w and len(d[j:j + n]) == n:
                    rest = d[j + n:]
                    for k in range(1, len(rest) + 1):
                        prefixes.add(tuple(rest[:k]))
        paths = _paths(tokens, parents)
        assert len(paths) == len(set(paths)) == len(prefixes)
        assert set(paths) == prefixes
        assert tokens[0] == accepted[-1] and parents[0] == -1
        assert all(0 <= parents[i] < i for i in range(1, len(tokens)))


def test_budget_and_depth():
    rng = np.random.default_rng(9)
    for _ in range(300):
        drafts, accepted = _random_case(rng, vocab=3)
        full_t, full_p = dt.draft_tree(drafts, accepted, 2, max_nodes=10**6, max_depth=10**6)
        for mn, md in ((16, 7), (5, 3), (1, 7), (16, 1), (3, 10)):
            t, p = dt.draft_tree(drafts, accepted, 2, mn, md)
            assert len(t) <= mn
            depth = [1]
            for i in range(1, len(t)):
                depth.append(depth[p[i]] + 1)
            assert max(depth) <= md
            # every path is a path of the unbounded trie, cut to the depth
            assert set(_paths(t, p)) <= set(_paths(full_t, full_p))
            # siblings carry distinct tokens (a prefix tree)
            sib = {}
            for i in range(1, len(t)):
                assert (p[i], t[i]) not in sib
                sib[(p[i], t[i])] = i
            # under budget, nothing of depth <= md is missing
            if len(t) < mn:
                want = {q for q in _paths(full_t, full_p) if len(q) <= md - 1}
                assert set(_paths(t, p)) == want


def test_short_accepted_sequence_gives_the_anchor_alone():
    assert dt.draft_tree([[1, 2, 3, 4]], [3], n=3) == ([3], [-1])
    assert dt.draft_tree([[1, 2, 3, 4]], [2, 3], n=3) == ([3], [-1])
    assert dt.draft_tree([[1, 2, 3, 4]], [2, 3], n=2) == ([3, 4], [-1, 0])
