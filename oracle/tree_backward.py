"""Float64 oracle for the backward pass of the tree-varlen forward.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The forward (PaDoc, "Training paradigm") gives every packed token t the
output O_t = softmax(s_t) V_A(t) over its ancestor set A(t), with scores
s_tj = scale * q_t . k_j.  Training back-propagates a loss through it; for an
upstream gradient dO the gradients of L = sum(dO * O) are the plain chain
rule through that softmax, taken here one query token at a time over the
same explicit ancestor set:

    P_tj  = exp(s_tj - LSE_t)                  (the forward's probabilities)
    dV_j += P_tj dO_t                          (O is linear in V)
    dP_tj = dO_t . v_j
    dS_tj = P_tj (dP_tj - dO_t . O_t)          (softmax Jacobian: the second term
                                                is sum_i P_ti dP_ti)
    dq_t  = scale * sum_j dS_tj k_j
    dk_j += scale * dS_tj q_t

With grouped heads, query head h reads kv head h // (Hq / Hkv) (reading 7 of
the forward), so dK and dV of a kv head sum over the query heads of its
group.  The pages train with a standard next-token objective and fix no
gradient formula beyond this; nothing here is reordered for speed.
"""
from __future__ import annotations

import math

import numpy as np

from .tree_attention import PACK_CANONICAL, _ancestor_identities, ancestor_positions, packed_layout


def _attend_grad(q, K, V, dO, scale):
    """One query token.  q, dO [Hq, d]; K, V [n, Hkv, d] (its ancestors).
    Returns dq [Hq, d], dK [n, Hkv, d], dV [n, Hkv, d]."""
    Hq, d = q.shape
    n, Hkv, _ = K.shape
    g = Hq // Hkv
    kv_head = np.arange(Hq) // g
    Kh = K[:, kv_head, :]                        # [n, Hq, d]
    Vh = V[:, kv_head, :]
    s = np.einsum("hd,nhd->hn", q, Kh) * scale   # [Hq, n]
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    P = e / e.sum(axis=1, keepdims=True)         # [Hq, n]
    O = np.einsum("hn,nhd->hd", P, Vh)
    dP = np.einsum("hd,nhd->hn", dO, Vh)
    Dt = np.einsum("hd,hd->h", dO, O)
    dS = P * (dP - Dt[:, None])
    dq = scale * np.einsum("hn,nhd->hd", dS, Kh)
    dKh = scale * np.einsum("hn,hd->nhd", dS, q)  # per query head
    dVh = np.einsum("hn,hd->nhd", P, dO)
    dK = dKh.reshape(n, Hkv, g, d).sum(axis=2)
    dV = dVh.reshape(n, Hkv, g, d).sum(axis=2)
    return dq, dK, dV


def tree_backward(q, k, v, dO, pages, order: int = PACK_CANONICAL, scale=None, positions=None):
    """Gradients of sum(dO * O) for the tree-varlen forward.

    q, dO [T, Hq, d]; k, v [T, Hkv, d] (any float dtype; float64 inside).
    Returns dQ [T, Hq, d], dK [T, Hkv, d], dV [T, Hkv, d] in float64.
    `positions` limits the work to those query positions: their dQ rows are
    exact (the rest stay NaN) and dK / dV hold only their contributions,
    which is the whole gradient for any key that no other query sees."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    dO = np.asarray(dO, np.float64)
    T, Hq, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if positions is None:
        anc = ancestor_positions(pages, order)
        assert len(anc) == T
        rows = range(T)
        dQ = np.zeros_like(q)
    else:
        ident, pos = packed_layout(pages, order)
        assert len(ident) == T
        rows = list(positions)
        anc = {}
        for t in rows:
            p, kind, r, i = ident[t]
            a = _ancestor_identities(pages[p], p, kind, r, i)
            anc[t] = np.sort(np.fromiter((pos[x] for x in a), dtype=np.int64, count=len(a)))
        dQ = np.full_like(q, np.nan)
    dK = np.zeros_like(k)
    dV = np.zeros_like(v)
    for t in rows:
        a = anc[t]
        dq, dk, dv = _attend_grad(q[t], k[a], v[a], dO[t], scale)
        dQ[t] = dq
        np.add.at(dK, a, dk)
        np.add.at(dV, a, dv)
    return dQ, dK, dV
