"""Puts seeded workloads on the GPU and runs them through libpadoc.

Used by the GPU tests and by bench.py.  Holds no attention arithmetic: it
allocates device tensors, fills the KV pool through padoc_kv_append, builds the
decode batch arrays, and calls the C ABI.
"""
from __future__ import annotations

import dataclasses
import zlib
from typing import List, Optional

import numpy as np
import torch

from . import padoc
from . import workloads as wl


def _bf16(x: np.ndarray, device) -> torch.Tensor:
    """Exactly representable float32 values -> device bf16 (lossless)."""
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(device).to(torch.bfloat16)


# ------------------------------------------------------------------ forward


class Forward:
    """A tree-varlen forward over packed pages with inputs resident on the GPU."""

    def __init__(self, w: wl.TreeWorkload, q=None, k=None, v=None, order: int = padoc.PACK_CANONICAL,
                 device="cuda", seed: int = 0):
        self.w = w
        self.desc = padoc.TreeDesc(w.pages, order)
        T = w.n_tokens
        self.T = T
        self.dtype = padoc.BF16 if w.dtype == "bf16" else padoc.F32
        tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        if q is None:
            g = torch.Generator(device=device)
            g.manual_seed(seed)
            self.q = (torch.randn(T, w.Hq, w.d, device=device, generator=g) * w.value_scale).to(tdt)
            self.k = (torch.randn(T, w.Hkv, w.d, device=device, generator=g) * w.value_scale).to(tdt)
            self.v = (torch.randn(T, w.Hkv, w.d, device=device, generator=g) * w.value_scale).to(tdt)
        else:
            conv = (lambda a: _bf16(a, device)) if w.dtype == "bf16" else (
                lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device))
            self.q, self.k, self.v = conv(q), conv(k), conv(v)
        self.o = torch.empty(max(T, 1), w.Hq, w.d, dtype=tdt, device=device)
        self.lse = torch.empty(w.Hq, max(T, 1), dtype=torch.float32, device=device)
        self.desc.upload(w.Hq // w.Hkv)

    def run(self, stream=None):
        padoc.tree_attn_varlen(self.desc, self.q, self.k, self.v, self.o, self.lse, self.dtype, self.w.Hq,
                               self.w.Hkv, self.w.d, 0.0, stream)
        return self.o, self.lse

    @property
    def flops(self) -> float:
        """Algorithmic flops: 4 d Hq per (query, ancestor) pair."""
        return 4.0 * self.w.d * self.w.Hq * self.desc.info()["ancestor_pairs"]

    @property
    def executed_flops(self) -> float:
        """Flops the tensor cores execute on the bf16 path: per (query tile,
        kv head) unit, S and P V over every 128-key tile the unit walks (the
        key tiles of each of its key segments, a causal one cut at the tile's
        last token), 128 x 128 x d x 2 x 2 each -- masked and padded elements
        included."""
        w = self.w
        tt = 128 // (w.Hq // w.Hkv)
        qs, kv = self.desc.segments()
        tiles = 0
        for q_start, q_len, kv_first, kv_count in qs.tolist():
            for t0 in range(q_start, q_start + q_len, tt):
                last = min(t0 + tt, q_start + q_len) - 1
                for ks, kl, causal in kv[kv_first:kv_first + kv_count].tolist():
                    end = min(ks + kl, last + 1) if causal else ks + kl
                    if end > ks:
                        tiles += (end - ks + 127) // 128
        return float(tiles) * w.Hkv * 128 * 128 * w.d * 2 * 2


class Backward:
    """The backward of a Forward: upstream gradient dO resident on the GPU,
    gradients and workspace allocated once."""

    def __init__(self, fwd: Forward, d_o=None, seed: int = 0, device="cuda"):
        self.f = fwd
        w = fwd.w
        tdt = fwd.q.dtype
        if d_o is None:
            g = torch.Generator(device=device)
            g.manual_seed(seed + 77)
            self.d_o = (torch.randn(fwd.T, w.Hq, w.d, device=device, generator=g) * w.value_scale).to(tdt)
        elif w.dtype == "bf16":
            self.d_o = _bf16(d_o, device)
        else:
            self.d_o = torch.from_numpy(np.ascontiguousarray(d_o, np.float32)).to(device)
        self.dq = torch.empty_like(fwd.q)
        self.dk = torch.empty_like(fwd.k)
        self.dv = torch.empty_like(fwd.v)
        self.ws_bytes = padoc.tree_attn_varlen_bwd_ws_size(fwd.desc, w.Hq)
        self.ws = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=device)

    def run(self, stream=None):
        f, w = self.f, self.f.w
        padoc.tree_attn_varlen_bwd(f.desc, f.q, f.k, f.v, f.o, f.lse, self.d_o, self.dq, self.dk, self.dv, f.dtype,
                                   w.Hq, w.Hkv, w.d, self.ws, self.ws_bytes, 0.0, stream)
        return self.dq, self.dk, self.dv

    @property
    def flops(self) -> float:
        """Algorithmic flops: five products of 2 d flops per (query,
        ancestor) pair and query head -- q.k (the scores, recomputed),
        dO.v, dS k, dS q and P dO -- so 10 d, 2.5 times the forward."""
        return 10.0 * self.f.w.d * self.f.w.Hq * self.f.desc.info()["ancestor_pairs"]


# ------------------------------------------------------------------ decode


def _seed(*parts) -> int:
    return zlib.crc32(repr(parts).encode()) & 0x7FFFFFFF


@dataclasses.dataclass
class DeviceDecodeValues:
    """Per-item seeded device values; any item can be regenerated alone."""

    w: wl.DecodeWorkload
    seed: int
    device: str

    def _randn(self, tag, idx, shape):
        g = torch.Generator(device=self.device)
        g.manual_seed(_seed(self.seed, tag, idx))
        x = torch.randn(*shape, device=self.device, generator=g) * self.w.value_scale
        return x.to(torch.bfloat16)

    def prefix(self, p):
        P = self.w.pages[p].prefix_len
        return (self._randn("pk", p, (P, self.w.Hkv, self.w.d)), self._randn("pv", p, (P, self.w.Hkv, self.w.d)))

    def own(self, b, L):
        return (self._randn("ok", b, (L, self.w.Hkv, self.w.d)), self._randn("ov", b, (L, self.w.Hkv, self.w.d)))

    def block(self, nq):
        return (self._randn("q", 0, (nq, self.w.Hq, self.w.d)), self._randn("kn", 0, (nq, self.w.Hkv, self.w.d)),
                self._randn("vn", 0, (nq, self.w.Hkv, self.w.d)))


class Decode:
    """A branch-decode / verify step: pool filled with each page's prefix and
    each branch's own suffix (a zero-copy fork of its page), plus the query
    block, all resident on the GPU."""

    def __init__(self, w: wl.DecodeWorkload, vals: Optional[wl.DecodeValues] = None, seed: int = 0,
                 device="cuda", tree: bool = True, slack_blocks: int = 8, fragment: bool = False):
        """fragment: the pool has twice the blocks, every other one held by a
        spacer sequence and the rest handed out in a shuffled order, so no
        two blocks of a sequence are physically consecutive by design."""
        self.w = w
        Hkv, d = w.Hkv, w.d
        nb = sum((p.prefix_len + 15) // 16 for p in w.pages)
        nb += sum((L + 15) // 16 for p in w.pages for L in p.own_len) + slack_blocks
        n_spacers = nb if fragment else 0
        nb += n_spacers
        max_bps = max([(p.prefix_len + 15) // 16 + (max(p.own_len or [0]) + 15) // 16 + 2 for p in w.pages] + [4])
        self.k_pool = torch.empty(nb, Hkv, 16, d, dtype=torch.bfloat16, device=device)
        self.v_pool = torch.empty(nb, Hkv, 16, d, dtype=torch.bfloat16, device=device)
        self.pool = padoc.KVPool(self.k_pool, self.v_pool, nb, Hkv, d,
                                 max_seqs=len(w.pages) + w.n_branches + 8 + (nb if fragment else 0),
                                 max_blocks_per_seq=max_bps)
        self.pool.sync()
        if fragment:
            spacers = [self.pool.alloc(16) for _ in range(nb)]
            for i in np.random.default_rng(seed + 7919).permutation(nb)[:n_spacers]:
                self.pool.release(spacers[i])
        self.gen = DeviceDecodeValues(w, seed, device) if vals is None else None
        page_seq, branch_seq, boff, qoff = [], [], [0], [0]
        b = 0
        for p, pg in enumerate(w.pages):
            s = self.pool.alloc(pg.prefix_len)
            if pg.prefix_len:
                if vals is not None:
                    k, v = _bf16(vals.prefix_k[p], device), _bf16(vals.prefix_v[p], device)
                else:
                    k, v = self.gen.prefix(p)
                self.pool.append(s, k, v, pg.prefix_len)
            page_seq.append(s)
            for j in range(len(pg.own_len)):
                c = self.pool.fork(s, pg.branch_prefix_len[j])
                L = pg.own_len[j]
                if L:
                    if vals is not None:
                        k, v = _bf16(vals.own_k[b], device), _bf16(vals.own_v[b], device)
                    else:
                        k, v = self.gen.own(b, L)
                    self.pool.append(c, k, v, L)
                branch_seq.append(c)
                qoff.append(qoff[-1] + pg.q_len[j])
                b += 1
            boff.append(len(branch_seq))
        self.page_seq, self.branch_seq = page_seq, branch_seq
        self.batch = padoc.Batch(page_seq, boff, branch_seq, qoff)
        nq = qoff[-1]
        self.nq = nq
        if vals is not None:
            self.q, self.k_new, self.v_new = (_bf16(vals.q, device), _bf16(vals.k_new, device),
                                              _bf16(vals.v_new, device))
        else:
            self.q, self.k_new, self.v_new = self.gen.block(nq)
        if tree:
            bits = np.concatenate([padoc.tree_mask_build(par) for pg in w.pages for par in pg.parents])
            self.tree_bits = torch.from_numpy(bits.astype(np.int16)).to(device)
        else:
            self.tree_bits = None
        self.ws_bytes = padoc.branch_decode_ws_size(self.pool, self.batch, w.Hq)
        self.ws = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=device)
        self.o = torch.empty(max(nq, 1), w.Hq, d, dtype=torch.bfloat16, device=device)
        self.lse = torch.empty(max(nq, 1), w.Hq, dtype=torch.float32, device=device)
        torch.cuda.synchronize()

    def run(self, stream=None):
        padoc.branch_decode(self.pool, self.batch, self.w.Hq, self.q, self.k_new, self.v_new, self.tree_bits,
                            self.o, self.lse, self.ws, self.ws_bytes, 0.0, stream)
        return self.o, self.lse

    def plan(self):
        """Plans the step and uploads the plan into ws (before a timed region)."""
        self._plan = padoc.DecodePlan(self.pool, self.batch, self.w.Hq)
        self._plan.upload(self.ws, self.ws_bytes)
        return self._plan

    def prefix_pass(self, stream=None):
        self._plan.prefix_pass(self.q, self.ws, 0.0, stream)

    def own_pass(self, stream=None):
        self._plan.own_pass(self.q, self.k_new, self.v_new, self.tree_bits, self.o, self.lse, self.ws, 0.0, stream)

    def prefix_bytes(self) -> int:
        """Algorithmic bytes of the prefix pass: each page's shared prefix
        tokens once (K and V, all kv heads) and the query rows."""
        w = self.w
        row = w.Hkv * w.d * 2 * 2
        return sum(max(p.branch_prefix_len or [0]) for p in w.pages) * row + self.nq * w.Hq * w.d * 2

    def own_bytes(self) -> int:
        """Algorithmic bytes of the own pass: each own cached token once, the
        query block's Q, K and V, O and LSE out."""
        w = self.w
        row = w.Hkv * w.d * 2 * 2
        return (sum(sum(p.own_len) for p in w.pages) * row + self.nq * row + self.nq * w.Hq * w.d * 2 * 2
                + self.nq * w.Hq * 4)

    def unique_kv_bytes(self) -> int:
        """Algorithmic bytes of one step: each shared prefix token once per
        page (the longest prefix any of its branches sees), each own token
        once, the query block's K/V, Q in, O and LSE out."""
        w = self.w
        row = w.Hkv * w.d * 2 * 2
        toks = sum(max(p.branch_prefix_len or [0]) + sum(p.own_len) for p in w.pages)
        nq = self.nq
        return toks * row + nq * row + nq * w.Hq * w.d * 2 * 2 + nq * w.Hq * 4

    def flops(self) -> float:
        w = self.w
        pairs = 0
        for pg in w.pages:
            for j in range(len(pg.own_len)):
                nb = pg.q_len[j]
                bits = padoc.tree_mask_build(pg.parents[j]) if self.tree_bits is not None else None
                inblock = sum(bin(int(x)).count("1") for x in bits) if bits is not None else nb * (nb + 1) // 2
                pairs += nb * (pg.branch_prefix_len[j] + pg.own_len[j]) + inblock
        return 4.0 * w.d * w.Hq * pairs

    def host_values(self, p: int) -> dict:
        """Host copies of page p's inputs (from the seeded generator, not the
        pool), for checking sampled rows against the oracle."""
        assert self.gen is not None
        pk, pv = self.gen.prefix(p)
        b0 = sum(len(pg.own_len) for pg in self.w.pages[:p])
        own = [self.gen.own(b0 + j, L) for j, L in enumerate(self.w.pages[p].own_len)]
        return {"prefix_k": pk.float().cpu().numpy(), "prefix_v": pv.float().cpu().numpy(),
                "own_k": [o[0].float().cpu().numpy() for o in own],
                "own_v": [o[1].float().cpu().numpy() for o in own]}


class Accept:
    """The accept step of a verify batch: next-token logits of every draft
    node resident in HBM (bf16 [nq, vocab]), draft tokens and parents, and
    the outputs."""

    def __init__(self, trees, vocab: int, seed: int = 0, tau: float = 0.75, device="cuda"):
        self.inp = wl.DeviceAcceptInputs(seed, trees, vocab, device)
        self.nq, self.vocab, self.tau = self.inp.nq, vocab, tau
        self.B = len(trees)
        self.max_nodes = max(len(t) for t in trees)
        self.tokens = torch.from_numpy(self.inp.tokens).to(device)
        self.parents = torch.from_numpy(self.inp.parents).to(device)
        self.q_offsets = torch.from_numpy(self.inp.q_offsets).to(device)
        self.n_acc = torch.empty(self.B, dtype=torch.int32, device=device)
        self.path = torch.empty(self.B, 16, dtype=torch.int32, device=device)
        self.free = torch.empty(self.B, dtype=torch.int32, device=device)
        # algorithmic bytes: every logit once, plus the small per-node and per-branch arrays
        self.bytes = self.nq * vocab * 2 + self.nq * 8 + (self.B + 1) * 4 + self.B * (16 + 2) * 4

    def run(self, stream=None):
        padoc.verify_accept(self.inp.logits, self.nq, self.vocab, self.tokens, self.parents, self.q_offsets,
                            self.B, self.max_nodes, self.tau, self.n_acc, self.path, self.free, stream)
        return self.n_acc, self.path, self.free

    def mean_accepted(self) -> float:
        return float(self.n_acc.float().mean().item())
