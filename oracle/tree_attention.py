"""Plain float64 reference for ancestor-masked tree attention.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Slow on purpose: every
query's softmax is taken over its explicitly enumerated ancestor set, with no
tiling, fusion or reordering.

Readings of the pages that this file fixes (each one also listed in the design
notes of the repository):

1. The prefix X is the front of the one causal layout stream, so a token of X
   sees X up to and including itself (PaDoc, "Training paradigm": the whole
   layout stream is a single causal sequence).
2. Every query sees itself (standard next-token attention; PaDoc, "Training
   paradigm", teacher-forced next-token objective).
3. A layout token of B_k sees X, B_1..B_{k-1} and the tokens of B_k up to
   itself (Anc(B_k) = {X, B<k} plus causal order inside B_k).
4. A content token of Y_k sees X, B_1..B_k and the tokens of Y_k up to itself
   (Anc(Y_k) = {X, B<=k}; a query of Y_k reads the keys and values of X,
   B<=k and Y_k as if they were one sequence).  The branch-start token is
   simply the first token of Y_k.
5. Pages never see each other, whatever their packing.
6. scale = 1/sqrt(d); LSE is the natural log of sum(exp(scale * q.k)).
7. GQA: query head h reads kv head floor(h / (Hq / Hkv)).
8. A decode/verify query of a branch sees the first prefix_len tokens of its
   page's shared prefix, all cached tokens of its own suffix, and the query
   block tokens of the same branch that are its draft-tree ancestors or itself
   (HSD page, "prefix-tree batching": each token attends to the accepted
   sequence plus its own ancestor path).  With no tree given, the block is a
   chain (token j visible to token i iff j <= i).
"""
from __future__ import annotations

import math
from typing import Dict, List, Sequence, Tuple

import numpy as np

X_KIND, B_KIND, Y_KIND = 0, 1, 2
PACK_CANONICAL, PACK_DOCUMENT = 0, 1


# ---------------------------------------------------------------------------
# Token identities and packing
# ---------------------------------------------------------------------------


def packed_layout(pages, order: int = PACK_CANONICAL):
    """Lay pages back to back and, inside each page, place X, the layout
    segments and the content branches in the given order.

    Returns (ident, pos) where ident[t] = (page, kind, region, index) for
    packed position t, and pos maps that tuple back to t.  Canonical order is
    [X | B_1..B_N | Y_1..Y_N]; document order is [X | B_1 Y_1 | B_2 Y_2 | ...].
    The pages fix no packing: the oracle's answers per identity do not depend
    on it (a test checks that)."""
    ident: List[Tuple[int, int, int, int]] = []
    for p, pg in enumerate(pages):
        ident.extend((p, X_KIND, -1, i) for i in range(pg.prefix_len))
        N = len(pg.layout_len)
        if order == PACK_CANONICAL:
            for k in range(N):
                ident.extend((p, B_KIND, k, i) for i in range(pg.layout_len[k]))
            for k in range(N):
                ident.extend((p, Y_KIND, k, i) for i in range(pg.content_len[k]))
        elif order == PACK_DOCUMENT:
            for k in range(N):
                ident.extend((p, B_KIND, k, i) for i in range(pg.layout_len[k]))
                ident.extend((p, Y_KIND, k, i) for i in range(pg.content_len[k]))
        else:
            raise ValueError(f"unknown packing order {order}")
    pos = {t: i for i, t in enumerate(ident)}
    return ident, pos


def _ancestor_identities(pg, page: int, kind: int, k: int, t: int):
    """Ancestor set of one token, by logical identity (readings 1-4)."""
    out = []
    if kind == X_KIND:
        out.extend((page, X_KIND, -1, i) for i in range(t + 1))
        return out
    out.extend((page, X_KIND, -1, i) for i in range(pg.prefix_len))
    if kind == B_KIND:
        for kk in range(k):
            out.extend((page, B_KIND, kk, i) for i in range(pg.layout_len[kk]))
        out.extend((page, B_KIND, k, i) for i in range(t + 1))
        return out
    for kk in range(k + 1):
        out.extend((page, B_KIND, kk, i) for i in range(pg.layout_len[kk]))
    out.extend((page, Y_KIND, k, i) for i in range(t + 1))
    return out


def ancestor_positions(pages, order: int = PACK_CANONICAL) -> List[np.ndarray]:
    """For every packed position, the sorted packed positions of its ancestors
    (itself included)."""
    ident, pos = packed_layout(pages, order)
    res = []
    for (p, kind, k, t) in ident:
        anc = _ancestor_identities(pages[p], p, kind, k, t)
        res.append(np.sort(np.fromiter((pos[a] for a in anc), dtype=np.int64, count=len(anc))))
    return res


def segment_intervals(pages, order: int = PACK_CANONICAL) -> List[List[Tuple[int, int]]]:
    """Each token's ancestor positions compressed into maximal [start, end)
    runs of consecutive positions (for bit-exact index checks)."""
    out = []
    for a in ancestor_positions(pages, order):
        runs: List[Tuple[int, int]] = []
        if len(a):
            start = prev = int(a[0])
            for x in a[1:]:
                x = int(x)
                if x != prev + 1:
                    runs.append((start, prev + 1))
                    start = x
                prev = x
            runs.append((start, prev + 1))
        out.append(runs)
    return out


# ---------------------------------------------------------------------------
# Attention over an explicit key set
# ---------------------------------------------------------------------------


def _attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """softmax(scale * q K^T) V for one query token.

    q [Hq, d]; K, V [n, Hkv, d] (the visible keys only).  Query head h reads
    kv head h // (Hq // Hkv) (reading 7).  Returns O [Hq, d] and the natural
    log-sum-exp [Hq] (reading 6)."""
    Hq, d = q.shape
    n, Hkv, _ = K.shape
    if n == 0:
        return np.zeros((Hq, d)), np.full(Hq, -np.inf)
    g = Hq // Hkv
    kv_head = np.arange(Hq) // g
    Kh = K[:, kv_head, :]                      # [n, Hq, d]
    Vh = V[:, kv_head, :]
    s = np.einsum("hd,nhd->hn", q, Kh) * scale  # [Hq, n]
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=1)
    o = np.einsum("hn,nhd->hd", e, Vh) / l[:, None]
    lse = m[:, 0] + np.log(l)
    return o, lse


def tree_forward(q, k, v, pages, order: int = PACK_CANONICAL, scale=None, positions=None):
    """Tree-varlen forward (PaDoc, "Training paradigm"): for every packed token,
    softmax over its ancestor set only.

    q [T, Hq, d], k/v [T, Hkv, d] (any float dtype; computed in float64).
    Returns O [T, Hq, d] and LSE [Hq, T], both float64.  `positions` limits
    the work to a subset of query positions (rows not listed stay NaN)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    T, Hq, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    anc = ancestor_positions(pages, order)
    assert len(anc) == T, (len(anc), T)
    O = np.full((T, Hq, d), np.nan)
    L = np.full((Hq, T), np.nan)
    rows = range(T) if positions is None else positions
    for t in rows:
        a = anc[t]
        o, lse = _attend(q[t], k[a], v[a], scale)
        O[t] = o
        L[:, t] = lse
    return O, L


def tree_mask_bits(parent: Sequence[int]) -> List[int]:
    """Visibility inside a draft token tree (HSD page, "prefix-tree batching"):
    bit j of row i is set iff node j is node i or one of its ancestors.
    `parent` lists each node's parent index (-1 for a root)."""
    n = len(parent)
    out = []
    for i in range(n):
        bits = 0
        j = i
        seen = 0
        while j >= 0:
            bits |= 1 << j
            j = parent[j]
            seen += 1
            if seen > n:
                raise ValueError("parent array has a cycle")
        out.append(bits)
    return out


def branch_decode(w, vals, tree: bool = True, scale=None):
    """Branch-parallel decode / speculative verify.

    For branch b of page p and its query row i: visible keys are the first
    branch_prefix_len[b] tokens of page p's shared prefix, all own_len[b]
    cached tokens of the branch's own suffix, and the query-block tokens j of
    the same branch with bit j set in row i's draft-tree mask (reading 8).
    With tree=False the block is a chain.  Returns O [nq, Hq, d], LSE [nq, Hq]
    in float64."""
    Hq, d = w.Hq, w.d
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    q = np.asarray(vals.q, np.float64)
    kn = np.asarray(vals.k_new, np.float64)
    vn = np.asarray(vals.v_new, np.float64)
    nq = q.shape[0]
    O = np.zeros((nq, Hq, d))
    L = np.zeros((nq, Hq))
    b = 0
    row = 0
    for p, pg in enumerate(w.pages):
        PK = np.asarray(vals.prefix_k[p], np.float64)
        PV = np.asarray(vals.prefix_v[p], np.float64)
        for j in range(len(pg.own_len)):
            plen = pg.branch_prefix_len[j]
            OK = np.asarray(vals.own_k[b], np.float64)
            OV = np.asarray(vals.own_v[b], np.float64)
            nb = pg.q_len[j]
            if tree:
                bits = tree_mask_bits(pg.parents[j])
            else:
                bits = [(1 << (i + 1)) - 1 for i in range(nb)]
            for i in range(nb):
                vis = [r for r in range(nb) if (bits[i] >> r) & 1]
                K = np.concatenate([PK[:plen], OK, kn[row + np.asarray(vis, dtype=np.int64)]], axis=0)
                V = np.concatenate([PV[:plen], OV, vn[row + np.asarray(vis, dtype=np.int64)]], axis=0)
                O[row + i], L[row + i] = _attend(q[row + i], K, V, scale)
            row += nb
            b += 1
    return O, L


def lse_merge(parts):
    """Merge partial softmax results computed over disjoint key sets.

    Each part is (O_i, lse_i) with O_i normalised over its own keys.  The
    merged result weights each part by exp(lse_i - LSE) with
    LSE = log(sum_i exp(lse_i)); empty parts carry lse = -inf."""
    lses = np.stack([np.asarray(p[1], np.float64) for p in parts])
    m = np.max(lses, axis=0)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    w = np.exp(lses - m_safe)
    tot = w.sum(axis=0)
    LSE = m_safe + np.log(tot)
    O = sum(np.asarray(p[0], np.float64) * (wi / tot)[..., None] for p, wi in zip(parts, w))
    return O, LSE


def depths(layout_len: Sequence[int], content_len: Sequence[int]) -> Dict[str, int]:
    """Critical-path decoding depths of one page (PaDoc, theoretical speedup):
    D_seq = l(B_1:N) + sum_k l(Y_k) for one serialised stream, and
    D_PaDoc = max_k [l(B<=k) + l(Y_k)] when every content branch starts as
    soon as its layout prefix exists.  The prefix X is prefilled, not decoded,
    so it is in neither depth."""
    d_seq = int(sum(layout_len) + sum(content_len))
    d_tree = 0
    acc = 0
    for lk, ck in zip(layout_len, content_len):
        acc += lk
        d_tree = max(d_tree, acc + ck)
    d_tree = max(d_tree, int(sum(layout_len)))
    return {"D_seq": d_seq, "D_tree": d_tree}
