// Draft trie of decoupled speculative verification (HSD page, "decoupled
// speculative verification": (a) draft-target matching, (b) prefix-tree
// batching).
//
// The drafts of a request are fixed once they are produced, so the index is
// built once: a hash table from every window of n consecutive draft tokens to
// the positions where it starts, kept in (draft, position) order.  A step then
// costs one table lookup plus the insertion of the matched continuations into
// a small first-child / next-sibling tree.
#include <cstdint>
#include <algorithm>
#include <cstring>
#include <memory>
#include <new>
#include <string>
#include <unordered_map>
#include <vector>

#include "../../include/padoc.h"
#include "padoc_internal.h"

namespace {

uint64_t window_hash(const int32_t* t, int32_t n) {
  uint64_t h = 1469598103934665603ull;  // FNV-1a over the 32-bit tokens
  for (int32_t i = 0; i < n; ++i) {
    h ^= static_cast<uint32_t>(t[i]);
    h *= 1099511628211ull;
  }
  return h;
}

struct Match {
  int64_t start;  // first token of the window occurrence
  int64_t end;    // end of its draft (exclusive)
};

}  // namespace

struct padoc_draft_index {
  int32_t n = 0;
  std::vector<int32_t> tok;
  std::unordered_map<uint64_t, std::vector<Match>> table;
};

namespace {

// One verify block.  Returns the node count; tokens/parents hold max_nodes.
int32_t build_block(const padoc_draft_index* ix, const int32_t* accepted, int32_t n_accepted, int32_t max_nodes,
                    int32_t max_depth, int32_t* tokens, int32_t* parents) {
  int32_t count = 1;
  tokens[0] = accepted[n_accepted - 1];
  parents[0] = -1;
  const int32_t n = ix->n;
  if (n_accepted < n || max_nodes == 1 || max_depth == 1) return count;
  const int32_t* w = accepted + (n_accepted - n);
  auto it = ix->table.find(window_hash(w, n));
  if (it == ix->table.end()) return count;
  // first-child / next-sibling links of the nodes created so far
  int32_t small[2 * 64];
  std::vector<int32_t> big;
  int32_t* first = small;
  if (max_nodes > 64) {
    big.resize(2 * static_cast<size_t>(max_nodes));
    first = big.data();
  }
  int32_t* next = first + std::max(max_nodes, 64);
  std::fill(first, first + max_nodes, -1);
  std::fill(next, next + max_nodes, -1);
  const int32_t* t = ix->tok.data();
  for (const Match& m : it->second) {
    if (std::memcmp(t + m.start, w, sizeof(int32_t) * n) != 0) continue;  // hash collision
    const int64_t a = m.start + n;
    const int64_t b = std::min<int64_t>(m.end, a + (max_depth - 1));
    int32_t node = 0;
    for (int64_t p = a; p < b; ++p) {
      int32_t c = first[node];
      while (c >= 0 && tokens[c] != t[p]) c = next[c];
      if (c < 0) {
        if (count == max_nodes) return count;  // budget spent: nothing later can add a node
        c = count++;
        tokens[c] = t[p];
        parents[c] = node;
        // append as the last child, so siblings stay in creation order
        if (first[node] < 0) {
          first[node] = c;
        } else {
          int32_t s = first[node];
          while (next[s] >= 0) s = next[s];
          next[s] = c;
        }
      }
      node = c;
    }
  }
  return count;
}

}  // namespace

extern "C" int padoc_draft_index_create(const int32_t* tokens, const int64_t* draft_offsets, int32_t n_drafts,
                                        int32_t window, padoc_draft_index** out) {
  if (!out) return padoc::set_error(PADOC_ERR_INVALID, "draft_index_create: null out");
  *out = nullptr;
  if (window < 1) return padoc::set_error(PADOC_ERR_INVALID, "draft_index_create: window must be >= 1");
  if (n_drafts < 0 || (n_drafts > 0 && !draft_offsets))
    return padoc::set_error(PADOC_ERR_INVALID, "draft_index_create: bad draft count or null offsets");
  if (n_drafts > 0) {
    if (draft_offsets[0] != 0) return padoc::set_error(PADOC_ERR_INVALID, "draft_index_create: draft_offsets[0] must be 0");
    for (int32_t d = 0; d < n_drafts; ++d)
      if (draft_offsets[d + 1] < draft_offsets[d])
        return padoc::set_error(PADOC_ERR_INVALID, "draft_index_create: draft_offsets decrease");
    if (draft_offsets[n_drafts] > 0 && !tokens) return padoc::set_error(PADOC_ERR_INVALID, "draft_index_create: null tokens");
  }
  try {
    std::unique_ptr<padoc_draft_index> ix(new padoc_draft_index());
    ix->n = window;
    const int64_t total = n_drafts > 0 ? draft_offsets[n_drafts] : 0;
    ix->tok.assign(tokens, tokens + total);
    for (int32_t d = 0; d < n_drafts; ++d) {
      const int64_t a = draft_offsets[d], e = draft_offsets[d + 1];
      for (int64_t j = a; j + window <= e; ++j)
        ix->table[window_hash(ix->tok.data() + j, window)].push_back(Match{j, e});
    }
    *out = ix.release();
  } catch (const std::bad_alloc&) {
    return padoc::set_error(PADOC_ERR_OOM, "draft_index_create: out of host memory");
  }
  return PADOC_OK;
}

extern "C" int padoc_draft_index_free(padoc_draft_index* index) {
  delete index;
  return PADOC_OK;
}

extern "C" int padoc_draft_trie(const padoc_draft_index* index, const int32_t* accepted, int32_t n_accepted,
                                int32_t max_nodes, int32_t max_depth, int32_t* tokens, int32_t* parents,
                                int32_t* n_nodes) {
  if (!index || !accepted || !tokens || !parents || !n_nodes)
    return padoc::set_error(PADOC_ERR_INVALID, "draft_trie: null argument");
  if (n_accepted < 1) return padoc::set_error(PADOC_ERR_INVALID, "draft_trie: no accepted token");
  if (max_nodes < 1 || max_depth < 1) return padoc::set_error(PADOC_ERR_INVALID, "draft_trie: max_nodes and max_depth must be >= 1");
  try {
    *n_nodes = build_block(index, accepted, n_accepted, max_nodes, max_depth, tokens, parents);
  } catch (const std::bad_alloc&) {
    return padoc::set_error(PADOC_ERR_OOM, "draft_trie: out of host memory");
  }
  return PADOC_OK;
}

extern "C" int padoc_draft_trie_batch(const padoc_draft_index* const* index, int32_t n_branches,
                                      const int32_t* accepted, const int32_t* acc_offsets, int32_t max_nodes,
                                      int32_t max_depth, int32_t* tokens, int32_t* parents, int32_t* q_offsets,
                                      uint16_t* bits) {
  if (n_branches < 0) return padoc::set_error(PADOC_ERR_INVALID, "draft_trie_batch: n_branches < 0");
  if (!q_offsets) return padoc::set_error(PADOC_ERR_INVALID, "draft_trie_batch: null q_offsets");
  q_offsets[0] = 0;
  if (n_branches == 0) return PADOC_OK;
  if (!index || !accepted || !acc_offsets || !tokens || !parents)
    return padoc::set_error(PADOC_ERR_INVALID, "draft_trie_batch: null argument");
  if (max_nodes < 1 || max_nodes > 16 || max_depth < 1)
    return padoc::set_error(PADOC_ERR_INVALID, "draft_trie_batch: max_nodes must be in [1, 16] and max_depth >= 1");
  for (int32_t b = 0; b < n_branches; ++b) {
    if (!index[b]) return padoc::set_error(PADOC_ERR_INVALID, "draft_trie_batch: null index for branch %d", b);
    if (acc_offsets[b + 1] - acc_offsets[b] < 1 || acc_offsets[b] < 0)
      return padoc::set_error(PADOC_ERR_INVALID, "draft_trie_batch: branch %d has no accepted token", b);
  }
  try {
    int32_t row = 0;
    for (int32_t b = 0; b < n_branches; ++b) {
      const int32_t n = build_block(index[b], accepted + acc_offsets[b], acc_offsets[b + 1] - acc_offsets[b],
                                    max_nodes, max_depth, tokens + row, parents + row);
      if (bits) {
        for (int32_t i = 0; i < n; ++i)
          bits[row + i] = static_cast<uint16_t>((i ? bits[row + parents[row + i]] : 0u) | (1u << i));
      }
      row += n;
      q_offsets[b + 1] = row;
    }
  } catch (const std::bad_alloc&) {
    return padoc::set_error(PADOC_ERR_OOM, "draft_trie_batch: out of host memory");
  }
  return PADOC_OK;
}
