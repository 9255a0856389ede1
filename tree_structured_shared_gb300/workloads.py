"""Seeded synthetic inputs for ancestor-masked tree attention.

This module draws lengths, draft trees and Q/K/V values.  It holds none of the
attention arithmetic: the oracle (test infrastructure) and the CUDA path both
take what it returns as plain inputs, so it is the only code the two share.

Shapes follow the workloads the PaDoc and HPD-Parsing pages describe:

* one page = a shared prefix X (visual + layout-start tokens), N layout
  segments B1..BN and N content branches Y1..YN (PaDoc, "Training paradigm");
* HPD-Parsing (Table 2) reports about 4,809 input tokens per page, which
  sets the decode prefix length;
* draft token trees for the speculative-verify step hold up to 16 nodes,
  branching factor at most 3, depth at most 7.

Conventions (one reading each, used by every caller):

* "uniform int in [a, b]" is inclusive of both ends;
* lognormal content lengths use mu = ln(median), the given sigma, rounding to
  the nearest integer and clamping to [1, cap];
* random values are drawn as float32 and, for bf16 workloads, rounded to
  bf16 with round-to-nearest-even before either side sees them.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np

# ----------------------------------------------------------------------------
# Page (tree) descriptions for the tree-varlen forward
# ----------------------------------------------------------------------------


@dataclasses.dataclass
class Page:
    """Lengths of one page: prefix X, layout segments B_k, content branches Y_k."""

    prefix_len: int
    layout_len: List[int]
    content_len: List[int]

    @property
    def n_regions(self) -> int:
        return len(self.layout_len)

    @property
    def n_tokens(self) -> int:
        return self.prefix_len + sum(self.layout_len) + sum(self.content_len)


PACK_CANONICAL = 0  # [X | B1..BN | Y1..YN]
PACK_DOCUMENT = 1   # [X | B1 Y1 | B2 Y2 | ... ]


@dataclasses.dataclass
class TreeWorkload:
    name: str
    pages: List[Page]
    Hq: int
    Hkv: int
    d: int
    dtype: str  # "f32" or "bf16"
    value_scale: float
    seq_of_page: List[int]

    @property
    def n_tokens(self) -> int:
        return sum(p.n_tokens for p in self.pages)


def _uniform_int(rng: np.random.Generator, lo: int, hi: int, size=None):
    return rng.integers(lo, hi + 1, size=size)


def _lognormal_len(rng, median: float, sigma: float, cap: int, size: int):
    x = rng.lognormal(mean=math.log(median), sigma=sigma, size=size)
    return np.clip(np.rint(x), 1, cap).astype(np.int64)


def tiny_fp32_page(seed: int = 0) -> TreeWorkload:
    """Single-layer fp32 forward: Hq=4, Hkv=2, d=64, one page, X=256, N=4,
    8 layout tokens per region, content lengths uniform in [16, 64]."""
    rng = np.random.default_rng(seed)
    content = [int(c) for c in _uniform_int(rng, 16, 64, size=4)]
    page = Page(prefix_len=256, layout_len=[8] * 4, content_len=content)
    return TreeWorkload("tiny_fp32_page", [page], 4, 2, 64, "f32", 1.0, [0])


def qwen_page(seed: int = 0) -> TreeWorkload:
    """One page at a Qwen3-1.7B-like attention shape, bf16: Hq=16, Hkv=8,
    d=128, X=2048, N=24, 12 layout tokens/region, content lognormal
    (median 120, sigma 0.8, cap 1024), values N(0,1)*0.5."""
    rng = np.random.default_rng(seed)
    content = [int(c) for c in _lognormal_len(rng, 120.0, 0.8, 1024, 24)]
    page = Page(prefix_len=2048, layout_len=[12] * 24, content_len=content)
    return TreeWorkload("qwen_page", [page], 16, 8, 128, "bf16", 0.5, [0])


def packed_sequences(seed: int = 0, n_seq: int = 8, seq_tokens: int = 16384,
                     Hq: int = 16, Hkv: int = 8, d: int = 128) -> TreeWorkload:
    """Serving-scale forward: pages drawn as X ~ U[4000, 6144], N ~ U[8, 60],
    12 layout tokens/region, lognormal content, appended until each packed
    sequence holds seq_tokens tokens.  The page that overflows is cut
    region-wise: whole regions that fit are kept, the first one that does not
    fit keeps its layout and as much content as fits (at least one token),
    and if X alone overflows, X is cut and the page has no regions."""
    rng = np.random.default_rng(seed)
    pages: List[Page] = []
    seq_of_page: List[int] = []
    for s in range(n_seq):
        left = seq_tokens
        while left > 0:
            X = int(_uniform_int(rng, 4000, 6144))
            N = int(_uniform_int(rng, 8, 60))
            content = [int(c) for c in _lognormal_len(rng, 120.0, 0.8, 1024, N)]
            if X >= left:
                pages.append(Page(left, [], []))
                seq_of_page.append(s)
                left = 0
                break
            used = X
            lay: List[int] = []
            con: List[int] = []
            for k in range(N):
                if used + 12 + content[k] <= left:
                    lay.append(12)
                    con.append(content[k])
                    used += 12 + content[k]
                    continue
                if used + 12 + 1 <= left:
                    lay.append(12)
                    con.append(left - used - 12)
                    used = left
                break
            pages.append(Page(X, lay, con))
            seq_of_page.append(s)
            left -= used
            if used < X + sum(lay) + sum(con):  # pragma: no cover - guard
                raise AssertionError("page accounting")
            if left > 0 and len(lay) < N:
                # the page was cut but a few tokens (< 13) remain: the
                # sequence ends short rather than holding a sliver of a page
                left = 0
    return TreeWorkload("packed_sequences", pages, Hq, Hkv, d, "bf16", 0.5, seq_of_page)


def random_pages(seed: int, n_pages: int, max_prefix: int = 40, max_regions: int = 5,
                 max_layout: int = 6, max_content: int = 20, allow_empty: bool = True,
                 Hq: int = 4, Hkv: int = 2, d: int = 64, dtype: str = "f32") -> TreeWorkload:
    """Small random trees for edge-case tests (ragged, empty regions allowed)."""
    rng = np.random.default_rng(seed)
    lo = 0 if allow_empty else 1
    pages = []
    for _ in range(n_pages):
        X = int(_uniform_int(rng, lo, max_prefix))
        N = int(_uniform_int(rng, 0, max_regions))
        lay = [int(v) for v in _uniform_int(rng, lo, max_layout, size=N)]
        con = [int(v) for v in _uniform_int(rng, lo, max_content, size=N)]
        pages.append(Page(X, lay, con))
    return TreeWorkload("random_pages", pages, Hq, Hkv, d, dtype, 1.0, list(range(n_pages)))


# ----------------------------------------------------------------------------
# Decode / verify batches
# ----------------------------------------------------------------------------


@dataclasses.dataclass
class DecodePage:
    prefix_len: int            # tokens of the shared page prefix held in the cache
    branch_prefix_len: List[int]  # per branch: how much of the prefix it sees
    own_len: List[int]         # per branch: cached own-suffix tokens
    q_len: List[int]           # per branch: query tokens this step (1..16)
    parents: List[List[int]]   # per branch: draft-tree parent array (-1 = root)


@dataclasses.dataclass
class DecodeWorkload:
    name: str
    pages: List[DecodePage]
    Hq: int
    Hkv: int
    d: int
    value_scale: float

    @property
    def n_branches(self) -> int:
        return sum(len(p.own_len) for p in self.pages)

    @property
    def n_queries(self) -> int:
        return sum(sum(p.q_len) for p in self.pages)


def draft_tree(rng: np.random.Generator, max_nodes: int = 16, max_children: int = 3,
               max_depth: int = 7) -> List[int]:
    """A draft token tree in topological order (parent index < child index).

    Node count ~ U[1, max_nodes]; node 0 is the root at depth 1; each later node
    attaches to a uniformly chosen earlier node that still has fewer than
    max_children children and depth below max_depth."""
    n = int(_uniform_int(rng, 1, max_nodes))
    parent = [-1]
    depth = [1]
    children = [0]
    for _ in range(1, n):
        cands = [i for i in range(len(parent)) if children[i] < max_children and depth[i] < max_depth]
        if not cands:
            break
        p = cands[int(rng.integers(0, len(cands)))]
        parent.append(p)
        depth.append(depth[p] + 1)
        children.append(0)
        children[p] += 1
    return parent


def _decode_pages(rng, n_pages, prefix_lo, prefix_hi, n_lo, n_hi, suf_hi, verify):
    pages = []
    for _ in range(n_pages):
        P = int(_uniform_int(rng, prefix_lo, prefix_hi))
        N = int(_uniform_int(rng, n_lo, n_hi))
        own = [int(v) for v in _uniform_int(rng, 0, suf_hi, size=N)]
        if verify:
            parents = [draft_tree(rng) for _ in range(N)]
        else:
            parents = [[-1] for _ in range(N)]
        pages.append(DecodePage(P, [P] * N, own, [len(t) for t in parents], parents))
    return pages


def branch_decode(seed: int = 0) -> DecodeWorkload:
    """16 pages, prefix 4809, N ~ U[8, 40] branches, own suffix ~ U[0, 512],
    one query token per live branch, bf16 16/8/128."""
    rng = np.random.default_rng(seed)
    return DecodeWorkload("branch_decode", _decode_pages(rng, 16, 4809, 4809, 8, 40, 512, False),
                          16, 8, 128, 0.5)


def spec_verify(seed: int = 0) -> DecodeWorkload:
    """64 pages, prefix 4809, N ~ U[8, 40], own suffix ~ U[0, 512], each branch
    verifies a draft tree of up to 16 nodes (branching <= 3, depth <= 7)."""
    rng = np.random.default_rng(seed)
    return DecodeWorkload("spec_verify", _decode_pages(rng, 64, 4809, 4809, 8, 40, 512, True),
                          16, 8, 128, 0.5)


def serving_decode(seed: int = 0, n_pages: int = 512) -> DecodeWorkload:
    """512 pages, prefix ~ U[4000, 6144], N ~ U[8, 60], own suffix ~ U[0, 1024],
    one query token per branch, bf16 16/8/128."""
    rng = np.random.default_rng(seed)
    return DecodeWorkload("serving_decode", _decode_pages(rng, n_pages, 4000, 6144, 8, 60, 1024, False),
                          16, 8, 128, 0.5)


def page_branch_decode(tree: TreeWorkload) -> DecodeWorkload:
    """One decode step per content branch of a single forward page: branch k
    sees prefix X + B1..Bk of the layout stream (so prefix lengths differ per
    branch) and its own content tokens Y_k."""
    assert len(tree.pages) == 1
    pg = tree.pages[0]
    P = pg.prefix_len + sum(pg.layout_len)
    bpl = [pg.prefix_len + sum(pg.layout_len[: k + 1]) for k in range(pg.n_regions)]
    N = pg.n_regions
    dp = DecodePage(P, bpl, list(pg.content_len), [1] * N, [[-1]] * N)
    return DecodeWorkload("page_branch_decode", [dp], tree.Hq, tree.Hkv, tree.d, tree.value_scale)


def small_decode(seed: int, n_pages: int = 3, max_prefix: int = 70, max_branches: int = 5,
                 max_own: int = 40, verify: bool = True, Hq: int = 4, Hkv: int = 2,
                 d: int = 128, ragged_prefix: bool = True) -> DecodeWorkload:
    """Small ragged decode/verify batches for parity tests (empty own
    suffixes, per-branch prefix lengths below the page prefix, forests)."""
    rng = np.random.default_rng(seed)
    pages = []
    for _ in range(n_pages):
        P = int(_uniform_int(rng, 0, max_prefix))
        N = int(_uniform_int(rng, 1, max_branches))
        own = [int(v) for v in _uniform_int(rng, 0, max_own, size=N)]
        if ragged_prefix:
            bpl = [int(v) for v in _uniform_int(rng, 0, P, size=N)]
            bpl[int(rng.integers(0, N))] = P
        else:
            bpl = [P] * N
        parents = []
        for _ in range(N):
            if verify:
                t = draft_tree(rng)
                # occasionally split into a forest: a later node becomes a root
                if len(t) > 2 and rng.random() < 0.3:
                    t[int(rng.integers(1, len(t)))] = -1
                parents.append(t)
            else:
                parents.append([-1])
        pages.append(DecodePage(P, bpl, own, [len(t) for t in parents], parents))
    return DecodeWorkload("small_decode", pages, Hq, Hkv, d, 1.0)


# ----------------------------------------------------------------------------
# Values
# ----------------------------------------------------------------------------


def normal_f32(seed: int, shape: Sequence[int], scale: float = 1.0) -> np.ndarray:
    """i.i.d. N(0,1)*scale as float32 from numpy's PCG64 stream for `seed`."""
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(size=tuple(shape), dtype=np.float32) * np.float32(scale)).astype(np.float32)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32
    holding exactly representable bf16 values."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    nan = np.isnan(x)
    out = r.astype(np.uint32).view(np.float32)
    out = np.where(nan, np.float32(np.nan), out)
    return out.astype(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """The upper 16 bits of float32 values that are already bf16-exact."""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def tree_qkv(w: TreeWorkload, seed: int):
    """Q [T,Hq,d], K [T,Hkv,d], V [T,Hkv,d] float32 (bf16-exact for bf16)."""
    T = w.n_tokens
    q = normal_f32(seed * 3 + 0, (T, w.Hq, w.d), w.value_scale)
    k = normal_f32(seed * 3 + 1, (T, w.Hkv, w.d), w.value_scale)
    v = normal_f32(seed * 3 + 2, (T, w.Hkv, w.d), w.value_scale)
    if w.dtype == "bf16":
        q, k, v = round_bf16(q), round_bf16(k), round_bf16(v)
    return q, k, v


@dataclasses.dataclass
class DecodeValues:
    prefix_k: List[np.ndarray]  # per page [P, Hkv, d]
    prefix_v: List[np.ndarray]
    own_k: List[np.ndarray]     # per branch (global order) [own_len, Hkv, d]
    own_v: List[np.ndarray]
    q: np.ndarray               # [nq, Hq, d]
    k_new: np.ndarray           # [nq, Hkv, d]
    v_new: np.ndarray


def decode_values(w: DecodeWorkload, seed: int, bf16: bool = True) -> DecodeValues:
    s = float(w.value_scale)
    rd = round_bf16 if bf16 else (lambda a: a)
    pk, pv, ok, ov = [], [], [], []
    base = seed * 1000003
    for pi, pg in enumerate(w.pages):
        pk.append(rd(normal_f32(base + 4 * pi, (pg.prefix_len, w.Hkv, w.d), s)))
        pv.append(rd(normal_f32(base + 4 * pi + 1, (pg.prefix_len, w.Hkv, w.d), s)))
    b = 0
    for pg in w.pages:
        for L in pg.own_len:
            ok.append(rd(normal_f32(base + 500000 + 2 * b, (L, w.Hkv, w.d), s)))
            ov.append(rd(normal_f32(base + 500001 + 2 * b, (L, w.Hkv, w.d), s)))
            b += 1
    nq = w.n_queries
    q = rd(normal_f32(base + 900001, (nq, w.Hq, w.d), s))
    kn = rd(normal_f32(base + 900002, (nq, w.Hkv, w.d), s))
    vn = rd(normal_f32(base + 900003, (nq, w.Hkv, w.d), s))
    return DecodeValues(pk, pv, ok, ov, q, kn, vn)


def flatten_branches(w: DecodeWorkload):
    """Per-branch arrays in global branch order: page index, prefix length,
    own length, query offsets (CSR), and the concatenated parent arrays."""
    page, bpl, own, qoff, parents = [], [], [], [0], []
    for pi, pg in enumerate(w.pages):
        for j in range(len(pg.own_len)):
            page.append(pi)
            bpl.append(pg.branch_prefix_len[j])
            own.append(pg.own_len[j])
            qoff.append(qoff[-1] + pg.q_len[j])
            parents.extend(pg.parents[j])
    return (np.asarray(page, np.int32), np.asarray(bpl, np.int32), np.asarray(own, np.int32),
            np.asarray(qoff, np.int32), np.asarray(parents, np.int32))


# ----------------------------------------------------------------------------
# Accept step: draft tokens and next-token logits
# ----------------------------------------------------------------------------

# The pages name the decoder (HPD-Parsing's InternVL3.5-1B builds on
# Qwen3-0.6B) but not its vocabulary; this is the size of that model's
# published embedding table.
VOCAB = 151936


@dataclasses.dataclass
class AcceptInputs:
    logits: np.ndarray     # [nq, V] float32 holding bf16 values
    tokens: np.ndarray     # [nq] int32, the drafted token of each node
    parents: np.ndarray    # [nq] int32, parent node index within the branch (-1 for node 0)
    q_offsets: np.ndarray  # [B + 1] int32


def _agree_plan(rng: np.random.Generator, parents: np.ndarray, q_offsets: np.ndarray, p_agree: float):
    """Rows and boost flags for the drafter's agreement with the target: node
    c of branch b (c >= 1) is 'agreeing' with probability p_agree, and then
    its parent's row is raised at c's token."""
    nq = int(q_offsets[-1])
    base = np.repeat(q_offsets[:-1], np.diff(q_offsets)).astype(np.int64)
    has_parent = parents >= 0
    agree = has_parent & (rng.random(nq) < p_agree)
    parent_row = base + np.where(has_parent, parents, 0)
    return agree, parent_row


def accept_inputs(seed: int, parents_per_branch: Sequence[Sequence[int]], vocab: int, p_agree: float = 0.8,
                  boost: tuple = (4.0, 6.0), ties: bool = False) -> AcceptInputs:
    """Host inputs for the accept step.

    Logits are i.i.d. N(0, 1) rounded to bf16 (ties=True: small integers in
    [-3, 3], so equal scores are common).  Draft tokens are uniform over the
    vocabulary; each draft node then agrees with the target with probability
    p_agree, which sets its token's logit in its parent's row to U[boost]
    (ties=True: to 3 or 4).  That mimics a drafter that is often right, so
    accepted paths of every length occur."""
    rng = np.random.default_rng(seed)
    q_offsets = np.zeros(len(parents_per_branch) + 1, np.int32)
    q_offsets[1:] = np.cumsum([len(p) for p in parents_per_branch])
    parents = np.asarray([x for p in parents_per_branch for x in p], np.int32)
    nq = int(q_offsets[-1])
    if ties:
        logits = rng.integers(-3, 4, size=(nq, vocab)).astype(np.float32)
    else:
        logits = round_bf16(rng.standard_normal(size=(nq, vocab), dtype=np.float32))
    tokens = rng.integers(0, vocab, size=nq).astype(np.int32)
    agree, parent_row = _agree_plan(rng, parents, q_offsets, p_agree)
    if ties:
        val = rng.integers(3, 5, size=nq).astype(np.float32)
    else:
        val = round_bf16(rng.uniform(boost[0], boost[1], size=nq).astype(np.float32))
    idx = np.nonzero(agree)[0]
    logits[parent_row[idx], tokens[idx]] = val[idx]
    return AcceptInputs(logits, tokens, parents, q_offsets)


class DeviceAcceptInputs:
    """The same recipe drawn on the GPU (torch's seeded CUDA generator) for
    sizes the host would take long to fill: logits [nq, V] bf16 in HBM."""

    def __init__(self, seed: int, parents_per_branch: Sequence[Sequence[int]], vocab: int, device,
                 p_agree: float = 0.8, boost: tuple = (4.0, 6.0)):
        import torch
        rng = np.random.default_rng(seed)
        q_offsets = np.zeros(len(parents_per_branch) + 1, np.int32)
        q_offsets[1:] = np.cumsum([len(p) for p in parents_per_branch])
        parents = np.asarray([x for p in parents_per_branch for x in p], np.int32)
        nq = int(q_offsets[-1])
        tokens = rng.integers(0, vocab, size=nq).astype(np.int32)
        agree, parent_row = _agree_plan(rng, parents, q_offsets, p_agree)
        val = round_bf16(rng.uniform(boost[0], boost[1], size=nq).astype(np.float32))
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        self.logits = torch.randn((nq, vocab), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
        idx = np.nonzero(agree)[0]
        if len(idx):
            r = torch.from_numpy(parent_row[idx]).to(device)
            c = torch.from_numpy(tokens[idx].astype(np.int64)).to(device)
            self.logits[r, c] = torch.from_numpy(val[idx]).to(device).to(torch.bfloat16)
        self.tokens, self.parents, self.q_offsets, self.nq, self.vocab = tokens, parents, q_offsets, nq, vocab

    def host_rows(self, rows) -> np.ndarray:
        """float32 copy of the given logit rows (bf16-exact)."""
        import torch
        idx = torch.as_tensor(np.asarray(rows, np.int64), device=self.logits.device)
        return self.logits.index_select(0, idx).float().cpu().numpy()


def hsd_drafts(seed: int, n_regions: int = 6, region_len: tuple = (20, 120), vocab: int = 151936,
               p_sub: float = 0.03, p_del: float = 0.02, p_ins: float = 0.02):
    """A target token sequence and one fixed draft per region, as a parsing
    pipeline would give (HSD page: region-level drafts with local OCR
    errors).  Each region of the target is copied into its draft with
    independent substitutions, deletions and insertions at the given rates.
    Returns (target, drafts)."""
    rng = np.random.default_rng(seed)
    target, drafts = [], []
    for _ in range(n_regions):
        region = rng.integers(0, vocab, int(_uniform_int(rng, *region_len))).tolist()
        target.extend(region)
        d = []
        for t in region:
            u = rng.random()
            if u < p_del:
                continue
            if u < p_del + p_sub:
                d.append(int(rng.integers(0, vocab)))
            else:
                d.append(t)
            if rng.random() < p_ins:
                d.append(int(rng.integers(0, vocab)))
        drafts.append(d)
    return target, drafts
