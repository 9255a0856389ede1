"""Oracle for the draft trie of decoupled speculative verification.

TEST INFRASTRUCTURE ONLY (see the package docstring).

HSD page (papernotes.org), "decoupled speculative verification":
 (a) draft-target matching: at each step the last n accepted tokens form the
     reference window w (n = 3 by default); every position j of every fixed
     draft where the n tokens starting at j equal w is a match, and the draft's
     tokens after the match (from j + n to its end) are a candidate
     continuation;
 (b) prefix-tree batching: the candidates are merged into a prefix tree in
     which each node stands for one distinct prefix and its children are the
     distinct next tokens after it; the tree is linearised into one packed
     block that is verified in a single pass under the ancestor mask.

Readings fixed here (also listed in the design notes):
 * the tree's root (node 0) is the last accepted token, the anchor of the
   verify step; the window is the anchor and the n - 1 tokens before it;
 * fewer than n accepted tokens, or no match, give the anchor alone;
 * empty continuations (a match at the very end of a draft) add nothing;
 * candidates are taken draft by draft, and within a draft by match position;
 * the verify block holds at most max_nodes nodes (16) and paths of at most
   max_depth nodes counting the anchor (7): each candidate is cut to its first
   max_depth - 1 tokens, and nodes are created in candidate order until the
   budget is spent;
 * linearisation order = creation order, which puts every parent before its
   children.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple


def match_candidates(drafts: Sequence[Sequence[int]], accepted: Sequence[int], n: int) -> List[List[int]]:
    """Step (a): every continuation after an occurrence of the window."""
    if len(accepted) < n:
        return []
    w = list(accepted[len(accepted) - n:])
    cands = []
    for d in drafts:
        d = list(d)
        for j in range(len(d) - n + 1):
            if d[j:j + n] == w and j + n < len(d):
                cands.append(d[j + n:])
    return cands


def build_trie(anchor: int, candidates: Sequence[Sequence[int]], max_nodes: int = 16,
               max_depth: int = 7) -> Tuple[List[int], List[int]]:
    """Step (b): merge the candidates into a prefix tree rooted at the anchor.
    Returns (tokens, parents) in creation order; parents[0] = -1."""
    tokens, parents = [anchor], [-1]
    kids = [dict()]  # per node: next token -> child node
    for cand in candidates:
        node = 0
        for tok in list(cand)[: max_depth - 1]:
            if tok in kids[node]:
                node = kids[node][tok]
                continue
            if len(tokens) == max_nodes:
                return tokens, parents  # no room for another node, for this or any later candidate
            tokens.append(tok)
            parents.append(node)
            kids.append(dict())
            kids[node][tok] = len(tokens) - 1
            node = len(tokens) - 1
    return tokens, parents


def draft_tree(drafts: Sequence[Sequence[int]], accepted: Sequence[int], n: int = 3, max_nodes: int = 16,
               max_depth: int = 7) -> Tuple[List[int], List[int]]:
    """The verify block of one step: anchor = last accepted token."""
    cands = match_candidates(drafts, accepted, n)
    return build_trie(int(accepted[-1]), cands, max_nodes, max_depth)
