"""The C++ draft-trie builder against the oracle (host code, CPU only).
Node order and token values are integers, so the match is exact."""
import os
import time

import numpy as np
import pytest

from oracle import draft_trie as dt
from oracle import tree_attention as ta
from tree_structured_shared_gb300 import padoc
from tree_structured_shared_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_golden_trie(padoc_lib):
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
                cases.append(kv)
    for kv in cases:
        ix = padoc.DraftIndex(drafts, int(kv["n"]))
        got = ix.trie(accepted, int(kv["max_nodes"]), int(kv["max_depth"]))
        assert got == ([int(x) for x in kv["tokens"].split(",")], [int(x) for x in kv["parents"].split(",")])


@pytest.mark.parametrize("n", [1, 2, 3, 4])
def test_random_drafts_match_oracle(padoc_lib, n):
    """Small vocabularies give many window occurrences, shared prefixes and
    budget cut-offs."""
    rng = np.random.default_rng(100 + n)
    for _ in range(400):
        vocab = int(rng.integers(2, 6))
        drafts = [rng.integers(0, vocab, int(rng.integers(0, 40))).tolist() for _ in range(int(rng.integers(0, 6)))]
        ix = padoc.DraftIndex(drafts, n)
        for _ in range(4):
            accepted = rng.integers(0, vocab, int(rng.integers(1, 9))).tolist()
            mn, md = int(rng.integers(1, 20)), int(rng.integers(1, 10))
            assert ix.trie(accepted, mn, md) == dt.draft_tree(drafts, accepted, n, mn, md), (drafts, accepted, mn, md)
        # no budget at all
        accepted = rng.integers(0, vocab, 5).tolist()
        assert ix.trie(accepted, 4096, 4096) == dt.draft_tree(drafts, accepted, n, 4096, 4096)


def test_decoding_a_noisy_page(padoc_lib):
    """Walk a target sequence with pipeline-like drafts: every step's block
    equals the oracle's, and the batch call equals the single calls with
    tree bits equal to the oracle's ancestor masks."""
    target, drafts = wl.hsd_drafts(5, n_regions=6, vocab=50)
    ix = padoc.DraftIndex(drafts, 3)
    steps = list(range(1, len(target), 7))
    blocks = []
    for t in steps:
        acc = target[:t]
        got = ix.trie(acc)
        assert got == dt.draft_tree(drafts, acc), t
        blocks.append(got)
    assert max(len(b[0]) for b in blocks) > 4  # the window finds drafts most of the time
    tok, par, qoff, bits = padoc.draft_trie_batch([ix] * len(steps), [target[:t] for t in steps])
    for b, (tk, pr) in enumerate(blocks):
        a, e = qoff[b], qoff[b + 1]
        assert tok[a:e].tolist() == tk and par[a:e].tolist() == pr
        assert bits[a:e].tolist() == [int(x) for x in ta.tree_mask_bits(pr)]


def test_rejects_bad_arguments(padoc_lib):
    with pytest.raises(padoc.PadocError):
        padoc.DraftIndex([[1, 2]], 0)
    ix = padoc.DraftIndex([[1, 2, 3]], 2)
    with pytest.raises(padoc.PadocError):
        ix.trie([], 16, 7)
    with pytest.raises(padoc.PadocError):
        ix.trie([1, 2], 0, 7)
    with pytest.raises(padoc.PadocError):
        padoc.draft_trie_batch([ix], [[1, 2]], max_nodes=17)
    with pytest.raises(padoc.PadocError):
        padoc.draft_trie_batch([ix], [[]])
    assert ix.trie([1, 2]) == ([2, 3], [-1, 0])
    empty = padoc.DraftIndex([], 3)
    assert empty.trie([1, 2, 3]) == ([3], [-1])


def test_host_cost_per_block(padoc_lib):
    """Host time of one verify block on a pipeline-like page (reported, and
    bounded loosely so a pathological slowdown shows)."""
    target, drafts = wl.hsd_drafts(9, n_regions=12)
    ix = padoc.DraftIndex(drafts, 3)
    accs = [target[t - 3:t] for t in range(3, len(target), 3)]  # only the window is read
    t0 = time.perf_counter()
    tok, par, qoff, bits = padoc.draft_trie_batch([ix] * len(accs), accs)
    dt_us = (time.perf_counter() - t0) / len(accs) * 1e6
    print(f"draft trie: {dt_us:.2f} us per block over {len(accs)} blocks (mean {len(tok) / len(accs):.1f} nodes)")
    assert dt_us < 200
