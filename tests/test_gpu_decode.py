"""Branch decode / speculative verify on the GPU against the float64 oracle."""
import numpy as np
import pytest

from oracle import tree_attention as ta
from tree_structured_shared_gb300 import padoc
from tree_structured_shared_gb300 import workloads as wl

from parity import check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def harness(padoc_lib):
    from tree_structured_shared_gb300 import harness as h
    return h


def _decode(harness, w, seed=0, tree=True):
    import torch
    vals = wl.decode_values(w, seed)
    d = harness.Decode(w, vals, tree=tree)
    o, lse = d.run()
    torch.cuda.synchronize()
    padoc.device_status()
    O, L = ta.branch_decode(w, vals, tree=tree)
    return o.float().cpu().numpy()[: w.n_queries], lse.cpu().numpy()[: w.n_queries], O, L


@pytest.mark.parametrize("seed", range(4))
def test_small_verify_ragged(harness, seed):
    """Draft trees and forests, empty own suffixes, per-branch prefix lengths
    below the page prefix, G = 2."""
    w = wl.small_decode(seed, n_pages=4, max_prefix=700, max_branches=6, max_own=300, Hq=4, Hkv=2)
    og, lg, O, L = _decode(harness, w, seed)
    check(og, lg, O, L, "bf16", f"small verify seed {seed}")


@pytest.mark.parametrize("G", [1, 4, 8])
def test_small_decode_groups(harness, G):
    w = wl.small_decode(20 + G, n_pages=3, max_prefix=400, max_branches=5, max_own=100, verify=False,
                        Hq=2 * G, Hkv=2)
    og, lg, O, L = _decode(harness, w, G, tree=False)
    check(og, lg, O, L, "bf16", f"decode G={G}")


@pytest.mark.parametrize("G", [1, 4, 8])
def test_small_verify_groups(harness, G):
    """Draft trees with G = 1 (two passes, keys-on-M own pass) and G = 4 and
    8 (the fused pass; at G = 8 a row tile holds 16 query tokens)."""
    w = wl.small_decode(40 + G, n_pages=3, max_prefix=500, max_branches=5, max_own=300, Hq=2 * G, Hkv=2)
    og, lg, O, L = _decode(harness, w, 40 + G)
    check(og, lg, O, L, "bf16", f"verify G={G}")


def test_verify_long_prefix_one_chunk(harness):
    """Page prefixes up to 4500 tokens (at most 36 key tiles) with draft
    trees and ragged per-branch prefixes: the fused verify pass walks each
    page's whole prefix as one chunk, then the own suffixes and the query
    block."""
    w = wl.small_decode(60, n_pages=2, max_prefix=4500, max_branches=4, max_own=300, Hq=4, Hkv=2)
    og, lg, O, L = _decode(harness, w, 60)
    check(og, lg, O, L, "bf16", "verify, long prefixes in one chunk")


def test_verify_prefix_above_one_chunk(harness):
    """A page prefix of 6000 tokens (47 key tiles, above the 40 of one
    chunk): the step runs as two passes, the prefix split into several
    chunks whose partial results the own pass merges."""
    rng = np.random.default_rng(61)
    pages = []
    for P in (6000, 1300):
        N = 5
        bpl = rng.integers(0, P, N).tolist()
        bpl[0] = P
        parents = [wl.draft_tree(rng, max_nodes=16) for _ in range(N)]
        pages.append(wl.DecodePage(P, bpl, rng.integers(0, 300, N).tolist(), [len(t) for t in parents], parents))
    w = wl.DecodeWorkload("long_prefix", pages, 4, 2, 128, 1.0)
    og, lg, O, L = _decode(harness, w, 61)
    check(og, lg, O, L, "bf16", "verify, several prefix chunks per page")


@pytest.mark.parametrize("verify", [True, False])
def test_fragmented_pool(harness, verify):
    """Pages and branches whose blocks are scattered over the pool in a
    shuffled order: every key tile is loaded block by block (no tile of
    eight consecutive blocks), for the fused verify pass and for the prefix
    pass of branch decode."""
    import torch
    w = wl.small_decode(70 + verify, n_pages=3, max_prefix=1500, max_branches=5, max_own=400, verify=verify,
                        Hq=4, Hkv=2)
    vals = wl.decode_values(w, 70)
    d = harness.Decode(w, vals, tree=verify, fragment=True)
    def longest_run(b):
        best = cur = 1
        for i in range(1, len(b)):
            cur = cur + 1 if b[i] == b[i - 1] + 1 else 1
            best = max(best, cur)
        return best
    assert max(longest_run(d.pool.seq_blocks(s)) for s in d.page_seq + d.branch_seq) < 8
    o, lse = d.run()
    torch.cuda.synchronize()
    padoc.device_status()
    O, L = ta.branch_decode(w, vals, tree=verify)
    check(o.float().cpu().numpy()[: w.n_queries], lse.cpu().numpy()[: w.n_queries], O, L, "bf16",
          "fragmented pool")


def test_verify_output_16_byte_aligned(harness):
    """The fused verify pass writing O into a tensor that is 16- but not
    32-byte aligned (16-byte stores per row)."""
    import torch
    w = wl.small_decode(80, n_pages=3, max_prefix=700, max_branches=6, max_own=300, Hq=4, Hkv=2)
    vals = wl.decode_values(w, 80)
    d = harness.Decode(w, vals, tree=True)
    buf = torch.empty(d.o.numel() + 8, dtype=d.o.dtype, device=d.o.device)
    d.o = buf[8:].view(d.o.shape)
    assert d.o.data_ptr() % 32 == 16
    o, lse = d.run()
    torch.cuda.synchronize()
    padoc.device_status()
    O, L = ta.branch_decode(w, vals, tree=True)
    check(o.float().cpu().numpy()[: w.n_queries], lse.cpu().numpy()[: w.n_queries], O, L, "bf16",
          "verify, 16-byte aligned output")


def _child_verify(tmp_path, env_over, seed=3):
    """One small draft-tree verify batch run in a child process under the
    given environment (the kernel choices are read once per process)."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = tmp_path / "o.npz"
    code = (
        "import sys, numpy as np, torch; sys.path.insert(0, %r)\n"
        "from tree_structured_shared_gb300 import harness, padoc, workloads as wl\n"
        "w = wl.small_decode(%d, n_pages=4, max_prefix=700, max_branches=6, max_own=300, Hq=4, Hkv=2)\n"
        "d = harness.Decode(w, wl.decode_values(w, %d), tree=True); o, l = d.run(); torch.cuda.synchronize()\n"
        "padoc.device_status()\n"
        "np.savez(%r, o=o.float().cpu().numpy()[:w.n_queries], l=l.cpu().numpy()[:w.n_queries])\n"
    ) % (root, seed, seed, str(out))
    env = dict(os.environ, **env_over)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    got = np.load(out)
    w = wl.small_decode(seed, n_pages=4, max_prefix=700, max_branches=6, max_own=300, Hq=4, Hkv=2)
    O, L = ta.branch_decode(w, wl.decode_values(w, seed), tree=True)
    return got["o"], got["l"], O, L


def test_verify_two_pass_keys_on_m(padoc_lib, tmp_path):
    """The same verify batch as two passes (PADOC_VERIFY_FUSED=0): the
    prefix pass, then the keys-on-M own pass that merges its partials."""
    og, lg, O, L = _child_verify(tmp_path, {"PADOC_VERIFY_FUSED": "0"})
    check(og, lg, O, L, "bf16", "two-pass verify, keys-on-M own pass")


def test_verify_rows_major_own_pass(padoc_lib, tmp_path):
    """The rows-on-M tensor-core own pass (two passes, PADOC_OWN_KERNEL=rows)
    on the same draft-tree pages."""
    og, lg, O, L = _child_verify(tmp_path, {"PADOC_VERIFY_FUSED": "0", "PADOC_OWN_KERNEL": "rows"})
    check(og, lg, O, L, "bf16", "rows-major own pass")


def test_verify_repeat_runs_bit_identical(harness):
    """The full 64-page verify batch run repeatedly: any ordering race in
    the pipelines shows up as a difference between runs."""
    import torch
    w = wl.spec_verify(1)
    d = harness.Decode(w, seed=1, tree=True)
    o0, l0 = [x.clone() for x in d.run()]
    for _ in range(3):
        o, l = d.run()
        torch.cuda.synchronize()
        assert torch.equal(o, o0) and torch.equal(l, l0)
    padoc.device_status()


def test_chain_block_without_tree(harness):
    w = wl.small_decode(9, n_pages=2, max_prefix=300, max_branches=4, max_own=60, verify=True, Hq=4, Hkv=2)
    og, lg, O, L = _decode(harness, w, 9, tree=False)
    check(og, lg, O, L, "bf16", "chain block")


def test_many_rows_per_page(harness):
    """More than 128 stacked query rows on one page (several row tiles)."""
    rng = np.random.default_rng(4)
    pages = [wl.DecodePage(900, [900] * 12, rng.integers(0, 80, 12).tolist(), [16] * 12,
                           [wl.draft_tree(rng, max_nodes=16) for _ in range(12)])]
    for pg in pages:
        pg.q_len = [len(t) for t in pg.parents]
    w = wl.DecodeWorkload("rows", pages, 16, 8, 128, 0.5)
    og, lg, O, L = _decode(harness, w, 4)
    check(og, lg, O, L, "bf16", "many rows")


def test_branch_decode_full(harness):
    """16 pages, prefix 4809, 8-40 branches, own suffix 0-512: every query."""
    w = wl.branch_decode(0)
    og, lg, O, L = _decode(harness, w, 0, tree=False)
    check(og, lg, O, L, "bf16", "branch decode")


def test_page_decode_matches_forward_rows(harness):
    """Cross-regime: one decode step per content branch of the qwen-shaped
    page, the cache holding exactly each branch's ancestors, reproduces the
    forward's rows for the last token of every Y_k."""
    import torch
    tree = wl.qwen_page(1)
    pg = tree.pages[0]
    q, k, v = wl.tree_qkv(tree, 1)
    fwd = harness.Forward(tree, q, k, v)
    o_f, l_f = fwd.run()
    ident, pos = ta.packed_layout(tree.pages)
    N = pg.n_regions
    lay_pos = list(range(pg.prefix_len + sum(pg.layout_len)))
    own, qpos = [], []
    for kk in range(N):
        ys = [pos[(0, ta.Y_KIND, kk, i)] for i in range(pg.content_len[kk])]
        own.append(ys[:-1])
        qpos.append(ys[-1])
    dp = wl.DecodePage(len(lay_pos), [pg.prefix_len + sum(pg.layout_len[: kk + 1]) for kk in range(N)],
                       [len(o) for o in own], [1] * N, [[-1]] * N)
    dw = wl.DecodeWorkload("cross", [dp], tree.Hq, tree.Hkv, tree.d, 0.5)
    vals = wl.DecodeValues([k[lay_pos]], [v[lay_pos]], [k[o] for o in own], [v[o] for o in own],
                           q[qpos], k[qpos], v[qpos])
    d = harness.Decode(dw, vals, tree=False)
    o_d, l_d = d.run()
    torch.cuda.synchronize()
    O, L = ta.tree_forward(q, k, v, tree.pages, positions=qpos)
    check(o_d.float().cpu().numpy(), l_d.cpu().numpy(), O[qpos], L[:, qpos].T, "bf16", "decode vs oracle")
    check(o_d.float().cpu().numpy(), l_d.cpu().numpy(), o_f.float().cpu().numpy()[qpos],
          l_f.cpu().numpy()[:, qpos].T, "bf16", "decode vs forward")


def test_decode_rejects_bad_batches(harness):
    import torch
    w = wl.small_decode(1, n_pages=2, max_prefix=50, max_branches=3, max_own=20, verify=False)
    d = harness.Decode(w, wl.decode_values(w, 1), tree=False)
    bad = padoc.Batch(d.page_seq[::-1], [0, 1, len(d.branch_seq)], d.branch_seq,
                      list(range(len(d.branch_seq) + 1)))
    with pytest.raises(padoc.PadocError):
        # branch 0 is not a fork of the sequence now listed first
        padoc.branch_decode(d.pool, bad, w.Hq, d.q, d.k_new, d.v_new, None, d.o, d.lse, d.ws, d.ws_bytes)
    with pytest.raises(padoc.PadocError):
        padoc.branch_decode(d.pool, d.batch, w.Hq, d.q, d.k_new, d.v_new, None, d.o, d.lse, d.ws, 16)
    torch.cuda.synchronize()


def test_plan_and_passes_equal_all_in_one(harness):
    """The planned two-pass path writes the same bits as padoc_branch_decode."""
    import torch
    w = wl.small_decode(31, n_pages=3, max_prefix=500, max_branches=5, max_own=200, Hq=4, Hkv=2)
    d = harness.Decode(w, wl.decode_values(w, 31), tree=True)
    o1, l1 = [x.clone() for x in d.run()]
    d.o.zero_()
    d.lse.zero_()
    d.plan()
    d.prefix_pass()
    d.own_pass()
    torch.cuda.synchronize()
    assert torch.equal(o1, d.o) and torch.equal(l1, d.lse)


def test_repeat_decode_bit_identical(harness):
    import torch
    w = wl.spec_verify(1)
    w.pages = w.pages[:12]
    d = harness.Decode(w, seed=1, tree=True)
    d.plan()
    d.prefix_pass()
    d.own_pass()
    o0, l0 = d.o.clone(), d.lse.clone()
    for _ in range(4):
        d.prefix_pass()
        d.own_pass()
        torch.cuda.synchronize()
        assert torch.equal(d.o, o0) and torch.equal(d.lse, l0)
    padoc.device_status()


def test_cuda_core_own_pass_short_blocks(harness):
    """G = 1 with 1-3 query tokens per branch stays on the CUDA-core own pass
    (fewer than 4 rows per branch and kv head on average)."""
    rng = np.random.default_rng(12)
    pages = []
    for _ in range(3):
        N = int(rng.integers(2, 6))
        par = [[-1] + list(range(int(rng.integers(0, 2)))) for _ in range(N)]
        pages.append(wl.DecodePage(300, [300] * N, rng.integers(0, 90, N).tolist(), [len(t) for t in par], par))
    w = wl.DecodeWorkload("short", pages, 2, 2, 128, 1.0)
    og, lg, O, L = _decode(harness, w, 12)
    check(og, lg, O, L, "bf16", "short blocks")
