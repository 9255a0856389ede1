"""Float64 CPU oracle for ancestor-masked tree attention.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
CPU-baseline leg may import this package.  It shares no code with the CUDA
path (no kernels, headers, tables or helpers); the two meet only at the seeded
input generators, which hold none of the attention arithmetic.

What it computes, each function citing the passage it follows:

* ancestor sets of every token of a page tree (PaDoc, "Training paradigm":
  Anc(Bk) = {X, B<k}, Anc(Yk) = {X, B<=k}; the layout stream is one causal
  sequence and content tokens of Yk also see the earlier tokens of Yk);
* the tree-varlen forward: per query, softmax over its explicit ancestor set;
* branch decode / speculative verify: per query, softmax over the shared
  prefix it sees, its branch's own cached suffix and the draft-tree
  ancestors-or-self inside the step's query block (HSD page, "prefix-tree
  batching": each draft token sees the accepted sequence and its own
  ancestor path);
* the log-sum-exp merge of partial softmaxes;
* the critical-path depths D_seq and D_PaDoc (PaDoc, theoretical speedup);
* the backward pass of the tree-varlen forward (tree_backward.py: the chain
  rule through each token's softmax over its ancestor set);
* the accept step of speculative verify (accept.py: HSD page, greedy tree
  traversal; HPD-Parsing, accepted length of a drafted chain);
* the draft trie of decoupled speculative verification (draft_trie.py: HSD
  page, draft-target matching and prefix-tree batching).

Pins: every function here is checked in tests/test_oracle*.py against facts
that do not come from this code (brute-force dense masks built from region
comparisons, plain causal attention for one region, closed forms, isolation
under perturbation, hand-worked fixtures under tests/golden/).  No function is
left "parity unpinned".
"""
from .tree_attention import (  # noqa: F401
    ancestor_positions,
    branch_decode,
    depths,
    lse_merge,
    packed_layout,
    segment_intervals,
    tree_forward,
    tree_mask_bits,
)
