"""C-ABI checks that need no GPU: exported symbols, the tree-descriptor
builder (bit-exact against the oracle's ancestor sets), the draft-tree mask
and depth helpers, and the KV pool's host bookkeeping."""
import os
import re
import subprocess
import sys

import numpy as np
import pytest

from oracle import tree_attention as ta
from tree_structured_shared_gb300 import padoc
from tree_structured_shared_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_exports_every_declared_symbol(padoc_lib):
    hdr = open(os.path.join(ROOT, "include", "padoc.h")).read()
    declared = set(re.findall(r"PADOC_API\s+[\w\s\*]+?\b(padoc_\w+)\s*\(", hdr))
    assert len(declared) >= 20
    out = subprocess.run(["nm", "-D", "--defined-only", padoc.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT\s+(padoc_\w+)", out))
    assert declared <= exported, declared - exported
    assert set(padoc.EXPORTED) == declared
    assert padoc_lib.padoc_version() == 100


def _expand(qs, kv, T):
    """Per-token visible key runs from the descriptor's segment lists."""
    runs = [None] * T
    for q_start, q_len, kv_first, kv_count in qs:
        for t in range(q_start, q_start + q_len):
            r = []
            for s in range(kv_first, kv_first + kv_count):
                a, n, causal = kv[s]
                b = min(a + n, t + 1) if causal else a + n
                if b > a:
                    if r and r[-1][1] == a:
                        r[-1] = (r[-1][0], b)
                    else:
                        r.append((a, b))
            assert runs[t] is None, "token covered twice"
            runs[t] = r
    return runs


@pytest.mark.parametrize("seed", range(10))
@pytest.mark.parametrize("order", [padoc.PACK_CANONICAL, padoc.PACK_DOCUMENT])
def test_descriptor_matches_oracle_ancestors(padoc_lib, seed, order):
    w = wl.random_pages(seed, n_pages=4, max_prefix=30, max_regions=6, max_layout=5, max_content=25)
    desc = padoc.TreeDesc(w.pages, order)
    inf = desc.info()
    assert inf["n_tokens"] == w.n_tokens
    qs, kv = desc.segments()
    got = _expand(qs, kv, w.n_tokens)
    want = ta.segment_intervals(w.pages, order)
    assert got == [list(x) for x in want]
    assert inf["ancestor_pairs"] == sum(len(a) for a in ta.ancestor_positions(w.pages, order))


def test_descriptor_config_shapes(padoc_lib):
    for w in (wl.tiny_fp32_page(0), wl.qwen_page(0)):
        desc = padoc.TreeDesc(w.pages)
        qs, kv = desc.segments()
        # canonical packing: one causal layout stream plus one segment per content branch
        assert len(qs) == 1 + sum(1 for c in w.pages[0].content_len if c > 0)
        assert max(qs[:, 3]) <= 2
        got = _expand(qs, kv, w.n_tokens)
        want = ta.segment_intervals(w.pages)
        assert got == [list(x) for x in want]


def test_descriptor_rejects_bad_input(padoc_lib):
    with pytest.raises(padoc.PadocError) as e:
        padoc.TreeDesc([wl.Page(-1, [], [])])
    assert e.value.code == padoc.ERR_INVALID
    with pytest.raises(padoc.PadocError):
        padoc.TreeDesc([wl.Page(3, [2], [-4])])
    with pytest.raises(padoc.PadocError):
        padoc.TreeDesc([wl.Page(3, [], [])], order=7)
    d = padoc.TreeDesc([])
    assert d.info()["n_tokens"] == 0


def test_tree_mask_build_matches_oracle(padoc_lib):
    rng = np.random.default_rng(0)
    for _ in range(200):
        par = wl.draft_tree(rng)
        if len(par) > 2 and rng.random() < 0.3:
            par[int(rng.integers(1, len(par)))] = -1
        assert list(padoc.tree_mask_build(par)) == ta.tree_mask_bits(par)
    with pytest.raises(padoc.PadocError):
        padoc.tree_mask_build([0])       # a node cannot be its own parent
    with pytest.raises(padoc.PadocError):
        padoc.tree_mask_build([-1] * 17)  # more than 16 nodes


def test_depths_match_oracle(padoc_lib):
    rng = np.random.default_rng(1)
    for _ in range(100):
        n = int(rng.integers(0, 30))
        lay = rng.integers(0, 20, n).tolist()
        con = rng.integers(0, 200, n).tolist()
        assert padoc.depths(lay, con) == ta.depths(lay, con)


# ---------------------------------------------------------------- KV pool (host bookkeeping)


def _pool(nb=64, max_seqs=16, max_bps=16):
    return padoc.KVPool(None, None, nb, Hkv=2, d=128, max_seqs=max_seqs, max_blocks_per_seq=max_bps)


def test_pool_alloc_fork_release_refcounts(padoc_lib):
    pool = _pool()
    a = pool.alloc(40)  # 3 blocks reserved, length 0
    assert pool.seq_info(a) == {"length": 0, "fork_len": 0, "n_blocks": 3}
    assert pool.stats() == {"free_blocks": 61, "live_seqs": 1}
    blocks = pool.seq_blocks(a)
    assert all(pool.refcount(b) == 1 for b in blocks)
    with pytest.raises(padoc.PadocError):
        pool.fork(a, 1)  # fork beyond the parent's length
    c = pool.fork(a, 0)
    assert pool.seq_info(c)["n_blocks"] == 0
    pool.release(c)
    assert pool.stats()["live_seqs"] == 1
    pool.release(a)
    assert pool.stats() == {"free_blocks": 64, "live_seqs": 0}
    assert all(pool.refcount(b) == 0 for b in blocks)
    with pytest.raises(padoc.PadocError):
        pool.release(a)


def test_pool_oom_changes_nothing(padoc_lib):
    pool = _pool(nb=8, max_seqs=4)
    a = pool.alloc(100)  # 7 blocks
    before = pool.stats()
    with pytest.raises(padoc.PadocError) as e:
        pool.alloc(33)   # 3 blocks, only 1 left
    assert e.value.code == padoc.ERR_OOM
    assert pool.stats() == before
    pool.alloc(16)
    pool.alloc(0)
    pool.alloc(0)
    with pytest.raises(padoc.PadocError) as e:
        pool.alloc(0)    # no sequence slot left
    assert e.value.code == padoc.ERR_OOM
    pool.release(a)


def test_pool_fault_injection_after_n_blocks(padoc_lib):
    code = (
        "import os, sys; sys.path.insert(0, %r)\n"
        "from tree_structured_shared_gb300 import padoc\n"
        "pool = padoc.KVPool(None, None, 64, Hkv=2, d=128, max_seqs=8, max_blocks_per_seq=16)\n"
        "a = pool.alloc(48)\n"
        "s0 = pool.stats()\n"
        "try:\n"
        "    pool.alloc(32)\n"
        "    print('NOFAULT')\n"
        "except padoc.PadocError as e:\n"
        "    print('FAULT', e.code, pool.stats() == s0, pool.seq_info(a)['n_blocks'])\n"
    ) % ROOT
    env = dict(os.environ, PADOC_FAULT_ALLOC_AFTER="4")
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=120)
    assert out.stdout.strip() == "FAULT -2 True 3", out.stdout + out.stderr


def test_pool_rejects_bad_arguments(padoc_lib):
    with pytest.raises(padoc.PadocError) as e:
        padoc.KVPool(None, None, 8, Hkv=2, d=64)
    assert e.value.code == padoc.ERR_UNSUPPORTED
    with pytest.raises(padoc.PadocError):
        padoc.KVPool(None, None, 0, Hkv=2, d=128)
    pool = _pool(max_bps=2)
    with pytest.raises(padoc.PadocError):
        pool.alloc(33)  # 3 blocks > max_blocks_per_seq
    with pytest.raises(padoc.PadocError):
        pool.seq_info(5)


FAKE = 1 << 20  # a pointer value nothing dereferences: every call below fails host checks first


def test_pool_device_before_sync(padoc_lib):
    """Before its first sync a pool has no device table: its device reads
    -1 and the testing relabel is refused (host only; decode calls compare
    this device with the current one before any launch)."""
    pool = padoc.KVPool(1 << 20, 1 << 20, 8, Hkv=2, d=128)
    assert pool.device() == -1
    with pytest.raises(padoc.PadocError) as e:
        pool.debug_rehome(1)
    assert e.value.code == padoc.ERR_INVALID


def test_commit_rejects_bad_lists_and_oom_changes_nothing(padoc_lib):
    pool = padoc.KVPool(FAKE, FAKE, 4, Hkv=2, d=128, max_seqs=4, max_blocks_per_seq=8)
    a, b = pool.alloc(0), pool.alloc(0)
    s0 = (pool.stats(), pool.seq_info(a), pool.seq_info(b))
    dev = dict(n_src_rows=40, k_new=FAKE, v_new=FAKE, ws=FAKE, ws_bytes=1 << 20)
    for seqs, offs, rows in [([a, a], [0, 1, 2], [0, 1]),    # listed twice
                             ([a, 3], [0, 1, 2], [0, 1]),    # not live
                             ([a], [0, 2], [0, 40]),         # row out of range
                             ([a], [1, 2], [0]),             # row_offsets[0] != 0
                             ([a, b], [0, 2, 1], [0, 1])]:   # decreasing offsets
        with pytest.raises(padoc.PadocError) as e:
            pool.commit(seqs, offs, rows, **dev)
        assert e.value.code == padoc.ERR_INVALID
    with pytest.raises(padoc.PadocError) as e:  # 3 + 2 blocks wanted, 4 free
        pool.commit([a, b], [0, 40, 60], list(range(40)) + list(range(20)), **dev)
    assert e.value.code == padoc.ERR_OOM
    with pytest.raises(padoc.PadocError) as e:  # workspace below 16 bytes per row
        pool.commit([a], [0, 2], [0, 1], n_src_rows=40, k_new=FAKE, v_new=FAKE, ws=FAKE, ws_bytes=16)
    assert e.value.code == padoc.ERR_INVALID
    with pytest.raises(padoc.PadocError):  # beyond max_blocks_per_seq
        pool.commit([a], [0, 140], list(range(140)), n_src_rows=140, k_new=FAKE, v_new=FAKE, ws=FAKE,
                    ws_bytes=1 << 20)
    assert (pool.stats(), pool.seq_info(a), pool.seq_info(b)) == s0
    pool.commit([a, b], [0, 0, 0], [], **dev)  # nothing to commit: no device work


def test_verify_accept_host_checks(padoc_lib):
    base = dict(logits=FAKE, nq=4, vocab=10, tokens=FAKE, parents=FAKE, q_offsets=FAKE, n_branches=1,
                n_acc=FAKE, path=FAKE, free_token=FAKE)
    for bad in (dict(max_nodes=0, tau=0.75), dict(max_nodes=17, tau=0.75), dict(max_nodes=4, tau=0.0),
                dict(max_nodes=4, tau=-1.0), dict(max_nodes=4, tau=float("nan")), dict(max_nodes=4, tau=float("inf")),
                dict(max_nodes=4, tau=0.75, vocab=0), dict(max_nodes=4, tau=0.75, q_offsets=None),
                dict(max_nodes=4, tau=0.75, path=None), dict(max_nodes=4, tau=0.75, n_branches=-1)):
        with pytest.raises(padoc.PadocError) as e:
            padoc.verify_accept(**{**base, **bad})
        assert e.value.code == padoc.ERR_INVALID
    padoc.verify_accept(**{**base, "n_branches": 0}, max_nodes=4, tau=0.75)  # nothing to do


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("order", [padoc.PACK_CANONICAL, padoc.PACK_DOCUMENT])
def test_backward_plan_covers_every_pair_once(padoc_lib, seed, order):
    """The key-stationary backward entries enumerate exactly the oracle's
    (query, ancestor) pairs, each once, inside 128-key tiles."""
    w = wl.random_pages(seed, n_pages=3, max_prefix=300, max_regions=5, max_layout=40, max_content=150)
    desc = padoc.TreeDesc(w.pages, order)
    items, entries = desc.bwd_plan()
    anc = ta.ancestor_positions(w.pages, order)
    want = np.zeros((w.n_tokens, w.n_tokens), np.int32)
    for t, a in enumerate(anc):
        want[t, a] = 1
    got = np.zeros_like(want)
    for k_start, k_len, e0, ne in items:
        assert k_start % 128 == 0 and 0 < k_len <= 128
        for k_lo, k_hi, causal, q_lo, q_hi in entries[e0:e0 + ne]:
            assert k_start <= k_lo < k_hi <= k_start + k_len
            for t in range(q_lo, q_hi):
                hi = min(k_hi, t + 1) if causal else k_hi
                if hi > k_lo:
                    got[t, k_lo:hi] += 1
    assert np.array_equal(got, want)


def test_backward_plan_key_tiles_in_position_order(padoc_lib):
    """The key-stationary units stay in position order (the kernel draws them
    in order, so CTAs at work together hold key tiles of one page and share
    its queries' Q and dO in L2); every key tile with a query appears once."""
    w = wl.random_pages(7, n_pages=4, max_prefix=400, max_regions=5, max_layout=40, max_content=200)
    items, _ = padoc.TreeDesc(w.pages, padoc.PACK_CANONICAL).bwd_plan()
    starts = [int(it[0]) for it in items]
    assert starts == sorted(starts) and len(set(starts)) == len(starts)


def _verify_plan(Hq, prefix, q_len, n_branches=3, own=40):
    """A host-only plan of one page: `prefix` tokens shared by n_branches
    forks with `own` tokens each and `q_len` query rows per branch."""
    pool = padoc.KVPool(None, None, 2048, Hkv=2, d=128, max_seqs=16, max_blocks_per_seq=512)
    page = pool.alloc(prefix)
    pool.advance(page, prefix)
    branches = []
    for _ in range(n_branches):
        c = pool.fork(page, prefix)
        pool.reserve(c, own)
        pool.advance(c, own)
        branches.append(c)
    batch = padoc.Batch([page], [0, n_branches], branches, [q_len * i for i in range(n_branches + 1)])
    return padoc.DecodePlan(pool, batch, Hq), (pool, batch)


def test_decode_plan_fusion_decision(padoc_lib):
    """A verify step runs as one kernel when Hq / Hkv >= 2, each branch
    stacks enough query rows for the tensor cores, and every page prefix
    fits one 40-tile chunk (5120 tokens); otherwise as the two passes."""
    plan, keep = _verify_plan(Hq=4, prefix=700, q_len=8)
    assert plan.fused()
    plan, keep = _verify_plan(Hq=4, prefix=5120, q_len=8)
    assert plan.fused()
    plan, keep = _verify_plan(Hq=4, prefix=5121, q_len=8)  # 41 key tiles: several chunks
    assert not plan.fused()
    plan, keep = _verify_plan(Hq=2, prefix=700, q_len=8)  # one head per kv head
    assert not plan.fused()
    plan, keep = _verify_plan(Hq=4, prefix=700, q_len=1)  # decode: one row per branch and head pair
    assert not plan.fused()
