"""Pins for the float64 oracle (CPU only).

Each check compares the oracle with something that does not come from it:
hand-worked fixtures, a brute-force dense mask built from region comparisons,
plain causal attention, closed forms, invariants and a DAG longest path.
"""
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle
from oracle import tree_attention as ta
from tree_structured_shared_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- fixtures


def _small_page():
    return [wl.Page(2, [1, 2], [2, 1])]


def test_golden_ancestor_sets():
    pages = _small_page()
    want = {"canonical": {}, "document": {}}
    with open(os.path.join(GOLDEN, "ancestors_small_page.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            parts = line.split()
            want[parts[0]][int(parts[2])] = [int(x) for x in parts[3:]]
    for name, order in (("canonical", ta.PACK_CANONICAL), ("document", ta.PACK_DOCUMENT)):
        got = ta.ancestor_positions(pages, order)
        assert len(got) == 8
        for t, anc in enumerate(got):
            assert list(anc) == want[name][t], (name, t)


def test_golden_tree_mask():
    with open(os.path.join(GOLDEN, "tree_mask_small.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            lhs, rhs = line.split(";")
            parents = [int(x) for x in lhs.split(",")]
            bits = [int(x) for x in rhs.split()]
            assert ta.tree_mask_bits(parents) == bits


def test_golden_closed_form_two_keys():
    rows = {"q": {}, "k": {}, "v": {}, "O": {}, "LSE": {}}
    with open(os.path.join(GOLDEN, "closed_form_two_keys.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            p = line.split()
            rows[p[0]][int(p[1])] = [float(x) for x in p[2:]]
    pages = [wl.Page(1, [1], [0])]
    q = np.array([rows["q"][0], rows["q"][1]])[:, None, :]
    k = np.array([rows["k"][0], rows["k"][1]])[:, None, :]
    v = np.array([rows["v"][0], rows["v"][1]])[:, None, :]
    O, L = ta.tree_forward(q, k, v, pages)
    np.testing.assert_allclose(O[:, 0, :], np.array([rows["O"][0], rows["O"][1]]), atol=1e-14)
    np.testing.assert_allclose(L[0], [rows["LSE"][0][0], rows["LSE"][1][0]], atol=1e-14)


# ---------------------------------------------------------------- brute force


def _dense_mask(pages, order):
    """Visibility matrix written as comparisons of (page, region kind, region
    index, index inside the region): a formulation separate from the
    oracle's per-token ancestor enumeration."""
    attrs = []  # (page, kind, region, idx)
    for p, pg in enumerate(pages):
        xs = [(p, 0, 0, i) for i in range(pg.prefix_len)]
        bs = [[(p, 1, k, i) for i in range(pg.layout_len[k])] for k in range(len(pg.layout_len))]
        ys = [[(p, 2, k, i) for i in range(pg.content_len[k])] for k in range(len(pg.layout_len))]
        attrs += xs
        if order == ta.PACK_CANONICAL:
            for b in bs:
                attrs += b
            for y in ys:
                attrs += y
        else:
            for b, y in zip(bs, ys):
                attrs += b + y
    a = np.array(attrs, dtype=np.int64).reshape(-1, 4)
    pq, kq, rq, iq = (a[:, None, c] for c in range(4))
    pk, kk, rk, ik = (a[None, :, c] for c in range(4))
    same = pq == pk
    key_x = kk == 0
    key_b = kk == 1
    key_y = kk == 2
    q_x, q_b, q_y = kq == 0, kq == 1, kq == 2
    vis = np.zeros(same.shape, dtype=bool)
    vis |= q_x & key_x & (ik <= iq)
    vis |= (q_b | q_y) & key_x
    vis |= q_b & key_b & ((rk < rq) | ((rk == rq) & (ik <= iq)))
    vis |= q_y & key_b & (rk <= rq)
    vis |= q_y & key_y & (rk == rq) & (ik <= iq)
    return vis & same


def _dense_attention(q, k, v, mask, scale):
    G = q.shape[1] // k.shape[1]
    kr = np.repeat(k, G, axis=1)  # head h -> kv head h // G
    vr = np.repeat(v, G, axis=1)
    s = np.einsum("qhd,khd->hqk", q, kr) * scale
    s = np.where(mask[None], s, -np.inf)
    lse = scipy.special.logsumexp(s, axis=2)
    p = np.exp(s - lse[:, :, None])
    o = np.einsum("hqk,khd->qhd", p, vr)
    return o, lse


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("order", [ta.PACK_CANONICAL, ta.PACK_DOCUMENT])
def test_bruteforce_dense_mask(seed, order):
    w = wl.random_pages(seed, n_pages=3, max_prefix=12, max_regions=4, max_layout=4,
                        max_content=7, Hq=4, Hkv=2, d=8)
    T = w.n_tokens
    if T == 0:
        pytest.skip("empty draw")
    q, k, v = (wl.normal_f32(100 + seed * 3 + i, s) for i, s in
               enumerate([(T, 4, 8), (T, 2, 8), (T, 2, 8)]))
    O, L = ta.tree_forward(q, k, v, w.pages, order)
    mask = _dense_mask(w.pages, order)
    Od, Ld = _dense_attention(q.astype(np.float64), k.astype(np.float64), v.astype(np.float64),
                              mask, 1 / math.sqrt(8))
    np.testing.assert_allclose(O, Od, atol=1e-12, rtol=0)
    np.testing.assert_allclose(L, Ld, atol=1e-12, rtol=0)


def test_one_region_is_causal_attention():
    """N = 1: the page X, B_1, Y_1 in canonical order is one causal sequence."""
    pages = [wl.Page(9, [3], [6])]
    T = 18
    q = wl.normal_f32(1, (T, 6, 16))
    k = wl.normal_f32(2, (T, 3, 16))
    v = wl.normal_f32(3, (T, 3, 16))
    O, L = ta.tree_forward(q, k, v, pages)
    # textbook causal attention, head h uses kv head h // 2
    scale = 0.25
    for h in range(6):
        s = q[:, h, :].astype(np.float64) @ k[:, h // 2, :].astype(np.float64).T * scale
        s[np.triu_indices(T, 1)] = -np.inf
        p = scipy.special.softmax(s, axis=1)
        np.testing.assert_allclose(O[:, h, :], p @ v[:, h // 2, :].astype(np.float64), atol=1e-12)
        np.testing.assert_allclose(L[h], scipy.special.logsumexp(s, axis=1), atol=1e-12)


def test_isolation_under_perturbation():
    """Changing Y_j leaves every token outside Y_j bit-identical."""
    pages = [wl.Page(7, [2, 3, 1], [4, 5, 3])]
    T = pages[0].n_tokens
    q = wl.normal_f32(5, (T, 2, 8))
    k = wl.normal_f32(6, (T, 2, 8))
    v = wl.normal_f32(7, (T, 2, 8))
    O, L = ta.tree_forward(q, k, v, pages)
    ident, pos = ta.packed_layout(pages)
    yj = [pos[(0, ta.Y_KIND, 1, i)] for i in range(5)]
    k2, v2, q2 = k.copy(), v.copy(), q.copy()
    k2[yj] += 3.0
    v2[yj] -= 2.0
    q2[yj] *= -1.5
    O2, L2 = ta.tree_forward(q2, k2, v2, pages)
    others = [t for t in range(T) if t not in yj]
    assert np.array_equal(O[others], O2[others])
    assert np.array_equal(L[:, others], L2[:, others])
    assert not np.allclose(O[yj], O2[yj])


def test_packing_invariance():
    """The two packings give the same output per logical token."""
    w = wl.random_pages(11, n_pages=2, max_prefix=10, max_regions=4, max_layout=4, max_content=6,
                        allow_empty=False, Hq=2, Hkv=1, d=8)
    T = w.n_tokens
    ic, pc = ta.packed_layout(w.pages, ta.PACK_CANONICAL)
    idoc, pdoc = ta.packed_layout(w.pages, ta.PACK_DOCUMENT)
    q = wl.normal_f32(1, (T, 2, 8))
    k = wl.normal_f32(2, (T, 1, 8))
    v = wl.normal_f32(3, (T, 1, 8))
    perm = np.array([pc[t] for t in idoc])  # document position -> canonical position
    Oc, Lc = ta.tree_forward(q, k, v, w.pages, ta.PACK_CANONICAL)
    Od, Ld = ta.tree_forward(q[perm], k[perm], v[perm], w.pages, ta.PACK_DOCUMENT)
    np.testing.assert_allclose(Od, Oc[perm], atol=1e-13)
    np.testing.assert_allclose(Ld, Lc[:, perm], atol=1e-13)


# ---------------------------------------------------------------- closed forms


def test_zero_query_is_mean_of_ancestors():
    pages = [wl.Page(5, [2, 2], [3, 4])]
    T = pages[0].n_tokens
    q = np.zeros((T, 2, 8))
    k = wl.normal_f32(1, (T, 1, 8))
    v = wl.normal_f32(2, (T, 1, 8))
    O, L = ta.tree_forward(q, k, v, pages)
    # ancestor counts written out by hand from the rules for this page:
    # X: 1..5; B1: 6,7; B2: 8,9; Y1: 8..10 (X + B1 + own); Y2: 10..13
    counts = [1, 2, 3, 4, 5, 6, 7, 8, 9, 8, 9, 10, 10, 11, 12, 13]
    assert T == len(counts)
    np.testing.assert_allclose(L[0], np.log(counts), atol=1e-13)
    anc = ta.ancestor_positions(pages)
    for t in range(T):
        assert len(anc[t]) == counts[t]
        np.testing.assert_allclose(O[t, 0], v[anc[t], 0].astype(np.float64).mean(axis=0), atol=1e-13)


def test_constant_values_and_one_hot():
    pages = [wl.Page(4, [2], [3])]
    T = 9
    q = wl.normal_f32(1, (T, 1, 4))
    k = wl.normal_f32(2, (T, 1, 4))
    v = np.tile(np.array([1.5, -2.0, 0.25, 7.0]), (T, 1, 1))
    O, _ = ta.tree_forward(q, k, v, pages)
    np.testing.assert_allclose(O[:, 0, :], v[:, 0, :], atol=1e-13)
    # one-hot: the last content token's query aligned with X2's key, huge gain
    k1 = np.zeros((T, 1, 4))
    for t in range(T):
        k1[t, 0, t % 4] = 1.0
    q1 = np.zeros((T, 1, 4))
    q1[8, 0, 2] = 2000.0          # token 8 (Y1.2) sees X, B1, Y1; X2 has key e_2
    v1 = wl.normal_f32(3, (T, 1, 4)).astype(np.float64)
    k1[6, 0, :] = 0               # Y1.0 (position 6 = 2 mod 4) would tie; zero it
    O1, _ = ta.tree_forward(q1, k1, v1, pages)
    np.testing.assert_allclose(O1[8, 0], v1[2, 0], atol=1e-12)


def test_split_merge_equals_direct():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((4, 16))
    K = rng.standard_normal((50, 2, 16))
    V = rng.standard_normal((50, 2, 16))
    o, l = ta._attend(q, K, V, 0.25)
    cut = sorted(rng.choice(np.arange(1, 50), size=4, replace=False))
    idx = np.split(rng.permutation(50), cut)
    parts = [ta._attend(q, K[i], V[i], 0.25) for i in idx]
    parts.append(ta._attend(q, K[:0], V[:0], 0.25))  # an empty part
    om, lm = ta.lse_merge(parts)
    np.testing.assert_allclose(om, o, atol=1e-12)
    np.testing.assert_allclose(lm, l, atol=1e-12)


# ---------------------------------------------------------------- decode


def test_decode_matches_forward_row():
    """A decode query equal to a teacher-forced token, with the cache holding
    exactly its ancestors, reproduces that token's forward row."""
    tree = wl.random_pages(3, n_pages=1, max_prefix=20, max_regions=4, max_layout=4, max_content=9,
                           allow_empty=False, Hq=4, Hkv=2, d=16)
    pg = tree.pages[0]
    T = pg.n_tokens
    q, k, v = (wl.normal_f32(40 + i, s) for i, s in enumerate([(T, 4, 16), (T, 2, 16), (T, 2, 16)]))
    O, L = ta.tree_forward(q, k, v, tree.pages)
    ident, pos = ta.packed_layout(tree.pages)
    N = pg.n_regions
    # branch k decodes the last token of Y_k: prefix = X + B1..Bk of the layout
    # stream, own = Y_k without its last token, query block = that last token
    P = pg.prefix_len + sum(pg.layout_len)
    layout_pos = [pos[(0, ta.X_KIND, -1, i)] for i in range(pg.prefix_len)]
    for kk in range(N):
        layout_pos += [pos[(0, ta.B_KIND, kk, i)] for i in range(pg.layout_len[kk])]
    own, qpos = [], []
    for kk in range(N):
        ys = [pos[(0, ta.Y_KIND, kk, i)] for i in range(pg.content_len[kk])]
        own.append(ys[:-1])
        qpos.append(ys[-1])
    dp = wl.DecodePage(P, [pg.prefix_len + sum(pg.layout_len[: kk + 1]) for kk in range(N)],
                       [len(o) for o in own], [1] * N, [[-1]] * N)
    dw = wl.DecodeWorkload("x", [dp], 4, 2, 16, 1.0)
    vals = wl.DecodeValues([k[layout_pos]], [v[layout_pos]], [k[o] for o in own], [v[o] for o in own],
                           q[qpos], k[qpos], v[qpos])
    Od, Ld = ta.branch_decode(dw, vals)
    np.testing.assert_allclose(Od, O[qpos], atol=1e-12)
    np.testing.assert_allclose(Ld, L[:, qpos].T, atol=1e-12)


def test_decode_bruteforce_block_mask():
    """Verify rows: dense attention over [prefix | own | block] with a mask
    from networkx ancestor queries on the draft tree."""
    nx = pytest.importorskip("networkx")
    w = wl.small_decode(7, n_pages=2, max_prefix=12, max_branches=3, max_own=6, d=8)
    vals = wl.decode_values(w, 1, bf16=False)
    O, L = ta.branch_decode(w, vals)
    row, b = 0, 0
    scale = 1 / math.sqrt(8)
    for p, pg in enumerate(w.pages):
        for j in range(len(pg.own_len)):
            par = pg.parents[j]
            g = nx.DiGraph()
            g.add_nodes_from(range(len(par)))
            g.add_edges_from((pp, c) for c, pp in enumerate(par) if pp >= 0)
            plen = pg.branch_prefix_len[j]
            nb = len(par)
            Kc = np.concatenate([vals.prefix_k[p][:plen], vals.own_k[b], vals.k_new[row:row + nb]])
            Vc = np.concatenate([vals.prefix_v[p][:plen], vals.own_v[b], vals.v_new[row:row + nb]])
            ctx = plen + pg.own_len[j]
            mask = np.zeros((nb, ctx + nb), bool)
            mask[:, :ctx] = True
            for i in range(nb):
                for a in nx.ancestors(g, i) | {i}:
                    mask[i, ctx + a] = True
            Od, Ld = _dense_attention(vals.q[row:row + nb].astype(np.float64), Kc.astype(np.float64),
                                      Vc.astype(np.float64), mask, scale)
            np.testing.assert_allclose(O[row:row + nb], Od, atol=1e-12)
            np.testing.assert_allclose(L[row:row + nb], Ld.T, atol=1e-12)
            row += nb
            b += 1


def test_tree_mask_matches_networkx():
    nx = pytest.importorskip("networkx")
    rng = np.random.default_rng(3)
    for _ in range(50):
        par = wl.draft_tree(rng)
        g = nx.DiGraph()
        g.add_nodes_from(range(len(par)))
        g.add_edges_from((p, c) for c, p in enumerate(par) if p >= 0)
        bits = ta.tree_mask_bits(par)
        for i in range(len(par)):
            want = sum(1 << a for a in nx.ancestors(g, i) | {i})
            assert bits[i] == want
        # the generator's limits: at most 16 nodes, 3 children, depth 7
        assert 1 <= len(par) <= 16
        assert max(np.bincount([p for p in par if p >= 0], minlength=1)) <= 3
        assert max(len(nx.ancestors(g, i)) + 1 for i in range(len(par))) <= 7


# ---------------------------------------------------------------- depths


def _dag_longest_path(pg):
    """Longest chain of decoded tokens in the dependency DAG, with edges
    ancestor -> token taken from the dense region-comparison mask (X is
    prefilled, so its tokens are not decode steps)."""
    nx = pytest.importorskip("networkx")
    mask = _dense_mask([pg], ta.PACK_CANONICAL)
    P = pg.prefix_len
    g = nx.DiGraph()
    n = mask.shape[0]
    g.add_nodes_from(range(P, n))
    for i in range(P, n):
        for j in range(P, n):
            if i != j and mask[i, j]:
                g.add_edge(j, i)
    if g.number_of_nodes() == 0:
        return 0
    return nx.dag_longest_path_length(g) + 1


@pytest.mark.parametrize("seed", range(8))
def test_depths_against_dag(seed):
    w = wl.random_pages(seed, n_pages=1, max_prefix=3, max_regions=6, max_layout=4, max_content=9,
                        allow_empty=False, Hq=1, Hkv=1, d=1)
    pg = w.pages[0]
    dd = ta.depths(pg.layout_len, pg.content_len)
    assert dd["D_seq"] == sum(pg.layout_len) + sum(pg.content_len)
    assert dd["D_tree"] == _dag_longest_path(pg)
    assert dd["D_tree"] <= dd["D_seq"]


def test_segment_intervals_are_runs():
    pages = _small_page()
    runs = ta.segment_intervals(pages)
    assert runs[7] == [(0, 5), (7, 8)]
    assert runs[5] == [(0, 3), (5, 6)]
    assert runs[4] == [(0, 5)]


def test_workload_shapes():
    a = wl.tiny_fp32_page(0)
    assert a.pages[0].prefix_len == 256 and len(a.pages[0].layout_len) == 4
    assert all(16 <= c <= 64 for c in a.pages[0].content_len)
    b = wl.qwen_page(0)
    assert b.pages[0].layout_len == [12] * 24
    assert all(1 <= c <= 1024 for c in b.pages[0].content_len)
    c = wl.packed_sequences(0)
    per_seq = np.bincount(c.seq_of_page, weights=[p.n_tokens for p in c.pages])
    assert len(per_seq) == 8
    assert all(16384 - 13 < s <= 16384 for s in per_seq)
    d3 = wl.branch_decode(0)
    assert len(d3.pages) == 16 and all(p.prefix_len == 4809 for p in d3.pages)
    assert all(8 <= len(p.own_len) <= 40 for p in d3.pages)
    d4 = wl.spec_verify(0)
    assert all(1 <= q <= 16 for p in d4.pages for q in p.q_len)
    x = wl.round_bf16(np.array([1.0, 1.00390625, 1.01171875, -3.0000001], np.float32))
    assert list(x) == [1.0, 1.0, 1.015625, -3.0]
