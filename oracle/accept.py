"""Float oracle for the accept step of speculative verify.

TEST INFRASTRUCTURE ONLY (see the package docstring).

HSD page (papernotes.org), "greedy tree traversal": starting at the root, among
the children of the current node pick the token u* with the highest model
probability; accept it when log p(u*) - log p(u_hat) >= log tau, where u_hat is
the most probable token over the whole vocabulary (tau = 0.75 by default), and
move to it; otherwise stop.  The accepted path is appended to the output,
followed by one free token: u_hat at the last accepted node.

HPD-Parsing notes, inference workflow: the accepted length of a drafted chain
is n_acc = max{k : y*_{n+i} = t_hat_i for all i <= k}, i.e. a draft token is
kept while it equals the target's greedy prediction.  This is the traversal
above on a chain with tau = 1 (accept exactly when the drafted token is an
argmax).

Readings fixed here (also listed in the design notes):
 * node 0 of a branch's draft tree is the anchor: the token emitted as free
   token by the previous step, whose logits are computed in this step; the
   traversal starts there and the anchor is always kept;
 * log p(a) - log p(b) under one softmax equals logit(a) - logit(b), so the
   rule compares logits; both sides take the decision in float32 (the logits
   are bf16 values, exactly representable) against float32(log tau);
 * ties (equal logits) go to the lowest vocabulary index for u_hat and to the
   lowest node index among children.
"""
from __future__ import annotations

import math
from typing import List, Sequence, Tuple

import numpy as np


def accept_tree(logits: np.ndarray, tokens: Sequence[int], parents: Sequence[int], tau: float):
    """One branch.  logits [n_nodes, V] (row i: the model's next-token scores
    after node i), tokens[i] the token of node i, parents[i] its parent
    (-1 for the root, node 0).  Returns (path, free_token) where path lists
    the accepted node indices after the root, in order."""
    logits = np.asarray(logits, dtype=np.float32)
    n = len(tokens)
    children: List[List[int]] = [[] for _ in range(n)]
    for i in range(1, n):
        children[parents[i]].append(i)
    log_tau = np.float32(math.log(tau))
    path = []
    s = 0
    while True:
        row = logits[s]
        u_hat = int(np.argmax(row))  # first maximum
        if not children[s]:
            return path, u_hat
        best = None
        for c in children[s]:  # children in index order; strict > keeps the lowest index on ties
            if best is None or row[tokens[c]] > row[tokens[best]]:
                best = c
        diff = np.float32(row[tokens[best]]) - np.float32(row[u_hat])
        if diff >= log_tau:
            path.append(best)
            s = best
        else:
            return path, u_hat


def accept_batch(logits: np.ndarray, tokens: Sequence[int], parents: Sequence[int], q_offsets: Sequence[int],
                 tau: float) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """All branches: rows [q_offsets[b], q_offsets[b+1]) belong to branch b.
    Returns n_acc [B], path [B, 16] (node indices within the branch, -1
    padded) and free_token [B]."""
    B = len(q_offsets) - 1
    n_acc = np.zeros(B, np.int32)
    path = np.full((B, 16), -1, np.int32)
    free = np.zeros(B, np.int32)
    for b in range(B):
        a, e = q_offsets[b], q_offsets[b + 1]
        p, f = accept_tree(logits[a:e], tokens[a:e], parents[a:e], tau)
        n_acc[b] = len(p)
        path[b, : len(p)] = p
        free[b] = f
    return n_acc, path, free
