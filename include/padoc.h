/*
 * libpadoc: ancestor-masked tree attention over a shared page-prefix KV cache.
 *
 * A page is a shared prefix X followed by a layout stream B_1..B_N and N
 * content branches Y_1..Y_N.  Layout tokens attend causally to [X, B<=current];
 * content tokens of Y_k attend to [X, B<=k] and to the earlier tokens of Y_k,
 * and never to another branch (PaDoc, "Training paradigm": Anc(B_k) = {X, B<k},
 * Anc(Y_k) = {X, B<=k}, realised as a packed tree-varlen attention).
 *
 * Conventions for every call:
 *  - Return value: PADOC_OK (0) or a negative PADOC_ERR_* code.  On error,
 *    padoc_last_error() returns a message (thread-local, valid until the next
 *    call on the same thread).  No C++ exception crosses this boundary.
 *  - Ownership: the caller owns every device buffer (Q, K, V, O, LSE, KV pool
 *    storage, workspace) and the stream.  The library owns only the opaque
 *    host handles it returns and a little device metadata that it allocates
 *    outside the compute calls (descriptor upload, pool tables) and frees in
 *    the matching *_free / *_destroy call.
 *  - Compute calls enqueue work on `stream` and return without waiting.
 *    Host calls are synchronous.  A handle may be used from one thread at a
 *    time.
 *  - "device pointer" means memory of the current CUDA device; "host pointer"
 *    means ordinary CPU memory read during the call only.
 *  - Kernel waits are bounded: a kernel that gives up on a wait records an
 *    error that the next call on the same handle (or padoc_device_status)
 *    reports as PADOC_ERR_DEVICE_TIMEOUT.
 */
#ifndef PADOC_H_
#define PADOC_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PADOC_API __attribute__((visibility("default")))
#else
#define PADOC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; NULL means the legacy default stream. */
typedef struct CUstream_st* padoc_stream_t;

enum {
  PADOC_OK = 0,
  PADOC_ERR_INVALID = -1,        /* bad argument or malformed structure; nothing changed */
  PADOC_ERR_OOM = -2,            /* KV pool out of blocks or sequence slots; nothing changed */
  PADOC_ERR_CUDA = -3,           /* a CUDA runtime call failed (message names it) */
  PADOC_ERR_UNSUPPORTED = -4,    /* valid request this build does not implement */
  PADOC_ERR_DEVICE_TIMEOUT = -5  /* a kernel gave up a bounded wait */
};

enum { PADOC_F32 = 0, PADOC_BF16 = 1 };

/* Packing of one page's tokens in the packed (THD) token stream.  The pages
 * fix no order; attention results per logical token do not depend on it. */
enum {
  PADOC_PACK_CANONICAL = 0, /* [X | B_1 .. B_N | Y_1 .. Y_N] */
  PADOC_PACK_DOCUMENT = 1   /* [X | B_1 Y_1 | B_2 Y_2 | ...] */
};

PADOC_API const char* padoc_last_error(void);
PADOC_API int padoc_version(void); /* major*10000 + minor*100 + patch */

/* ------------------------------------------------------------------------
 * Tree descriptor (host).  Turns region lengths into query segments, each
 * with an ordered list of key/value segments, and a tile work list.
 * Basis: PaDoc, "Training paradigm" (the layout stream is one causal
 * sequence; Y_k queries attend to the virtual KV sequence [X, B<=k, Y_k]).
 * ---------------------------------------------------------------------- */
typedef struct {
  int32_t n_pages;             /* >= 0 */
  const int32_t* prefix_len;   /* host [n_pages], >= 0: tokens of X */
  const int32_t* n_regions;    /* host [n_pages], >= 0: N */
  const int32_t* layout_len;   /* host [sum n_regions], page-major, >= 0: l(B_k) */
  const int32_t* content_len;  /* host [sum n_regions], page-major, >= 0: l(Y_k) (the
                                  branch-start token counts as the first token of Y_k) */
  int32_t order;               /* PADOC_PACK_* */
} padoc_tree_spec;

typedef struct padoc_tree_desc padoc_tree_desc;

/* Builds the descriptor.  Pages are packed back to back in the given order;
 * no page sees another.  Total tokens must stay below 2^31.
 * Errors: PADOC_ERR_INVALID (negative length, bad order, overflow). */
PADOC_API int padoc_tree_desc_build(const padoc_tree_spec* spec, padoc_tree_desc** out);
PADOC_API int padoc_tree_desc_free(padoc_tree_desc* desc);

/* Sizes: packed tokens, query segments, key/value segments, and the number
 * of (query token, ancestor token) pairs (sum of ancestor-set sizes). */
PADOC_API int padoc_tree_desc_info(const padoc_tree_desc* desc, int64_t* n_tokens, int64_t* n_qsegs,
                         int64_t* n_kvsegs, int64_t* ancestor_pairs);

/* Copies the segment lists out (for bit-exact checks).
 *   qseg  host [n_qsegs][4]:  q_start, q_len, kv_first, kv_count
 *   kvseg host [n_kvsegs][3]: kv_start, kv_len, causal
 * A query at packed position t of segment s sees, for each of its key
 * segments, positions [kv_start, kv_start + kv_len) when causal == 0 and
 * [kv_start, min(kv_start + kv_len, t + 1)) when causal == 1. */
PADOC_API int padoc_tree_desc_segments(const padoc_tree_desc* desc, int32_t* qseg, int32_t* kvseg);

/* Allocates and fills the device copy of the descriptor for query-group size
 * `group` = Hq / Hkv on the current device (synchronous).  The forward does
 * this itself on first use; calling it first keeps allocation out of the
 * first forward. */
PADOC_API int padoc_tree_desc_upload(padoc_tree_desc* desc, int32_t group);

/* ------------------------------------------------------------------------
 * Packed tree-varlen forward (PaDoc, "Training paradigm"; tree-varlen).
 *   q   device [T, Hq, d]   (THD, row-major, contiguous)
 *   k,v device [T, Hkv, d]
 *   o   device [T, Hq, d]   same dtype as q
 *   lse device [Hq, T] f32  natural log of sum_j exp(scale * q.k_j) over the
 *                           query's ancestor set
 * dtype PADOC_BF16 (tensor-core path, f32 accumulation) or PADOC_F32 (f32
 * CUDA-core path).  d must be 128 for bf16 and 64 or 128 for f32; Hq must
 * be a multiple of Hkv with Hq / Hkv in {1, 2, 4, 8, 16}.  scale <= 0 means
 * 1/sqrt(d).  Query head h reads kv head h / (Hq / Hkv).  Pointers must be
 * 16-byte aligned.  T = 0 is a no-op. */
PADOC_API int padoc_tree_attn_varlen(padoc_tree_desc* desc, const void* q, const void* k, const void* v,
                           void* o, float* lse, int32_t dtype, int32_t Hq, int32_t Hkv,
                           int32_t d, float scale, padoc_stream_t stream);

/* ------------------------------------------------------------------------
 * Refcounted paged KV pool.  Storage is caller-owned device memory laid out
 * [num_blocks, Hkv, block_size, d] for K and for V (one layer).  A sequence
 * is a list of blocks; a fork shares the parent's blocks with zero copy and
 * bumps their reference counts; release drops them and frees blocks that
 * reach zero (HPD-Parsing: fork with zero-copy KV sharing and
 * reference-counted release).
 * ---------------------------------------------------------------------- */
typedef struct padoc_kv_pool padoc_kv_pool;

/* block_size must be 16; d must be 128; dtype PADOC_BF16.  max_seqs and
 * max_blocks_per_seq size the device block table (allocated on first device
 * use, see padoc_kv_pool_sync).  The environment variable
 * PADOC_FAULT_ALLOC_AFTER=n makes the n-th later block allocation fail with
 * PADOC_ERR_OOM (host fault injection for tests). */
PADOC_API int padoc_kv_pool_create(padoc_kv_pool** out, void* k_pool, void* v_pool, int32_t num_blocks,
                         int32_t block_size, int32_t Hkv, int32_t d, int32_t dtype,
                         int32_t max_seqs, int32_t max_blocks_per_seq);
PADOC_API int padoc_kv_pool_destroy(padoc_kv_pool* pool);

/* New empty sequence with room reserved for n_tokens (>= 0) tokens.
 * On PADOC_ERR_OOM nothing changes. */
PADOC_API int padoc_kv_alloc(padoc_kv_pool* pool, int32_t n_tokens, int32_t* seq);

/* Appends n tokens (device [n, Hkv, d] each for k and v, pool dtype) to the
 * end of seq, growing it by fresh blocks if needed.  A forked sequence never
 * writes into a shared block: its own tokens start in a fresh block.
 * On PADOC_ERR_OOM nothing changes.  The copy runs on `stream`. */
PADOC_API int padoc_kv_append(padoc_kv_pool* pool, int32_t seq, const void* k, const void* v, int32_t n,
                    padoc_stream_t stream);

/* New sequence whose first fork_len tokens are the parent's first fork_len
 * tokens, shared with zero copy (the blocks covering them get refcount + 1,
 * a partly used last block included).  0 <= fork_len <= length(parent). */
PADOC_API int padoc_kv_fork(padoc_kv_pool* pool, int32_t parent, int32_t fork_len, int32_t* child);

/* Grows seq's own blocks so that n_tokens more tokens fit after its current
 * length (all or nothing: PADOC_ERR_OOM changes nothing).  Host bookkeeping
 * only; a later append or commit of up to n_tokens then needs no block. */
PADOC_API int padoc_kv_reserve(padoc_kv_pool* pool, int32_t seq, int32_t n_tokens);
/* Marks n tokens after seq's current length as written, for callers that
 * write K/V into the reserved slots themselves (a prefill into the pool's
 * blocks through the block table).  The slots must already be reserved;
 * otherwise PADOC_ERR_INVALID.  Host bookkeeping only. */
PADOC_API int padoc_kv_advance(padoc_kv_pool* pool, int32_t seq, int32_t n);

/* Gives back seq's own blocks past the ones its current length uses (the
 * unused tail of a reservation); refcounts drop as in padoc_kv_release. */
PADOC_API int padoc_kv_trim(padoc_kv_pool* pool, int32_t seq);

/* Drops the sequence: refcount - 1 on each of its blocks, blocks at 0 return
 * to the free list, the sequence id becomes reusable. */
PADOC_API int padoc_kv_release(padoc_kv_pool* pool, int32_t seq);

/* Sequence facts: length, tokens shared from its fork parent, blocks held. */
PADOC_API int padoc_kv_seq_info(const padoc_kv_pool* pool, int32_t seq, int32_t* length, int32_t* fork_len,
                      int32_t* n_blocks);
/* Copies the block ids of seq into out (host, capacity cap). */
PADOC_API int padoc_kv_seq_blocks(const padoc_kv_pool* pool, int32_t seq, int32_t* out, int32_t cap);
/* Reference count of one block (0 = free). */
PADOC_API int padoc_kv_block_refcount(const padoc_kv_pool* pool, int32_t block, int32_t* refcount);
/* Free blocks and live sequences. */
PADOC_API int padoc_kv_pool_stats(const padoc_kv_pool* pool, int32_t* free_blocks, int32_t* live_seqs);
/* Allocates the device block table if needed and uploads changed rows
 * (synchronous with respect to the host tables; copies enqueue on stream). */
PADOC_API int padoc_kv_pool_sync(padoc_kv_pool* pool, padoc_stream_t stream);
/* The device that holds the pool's block table (the device current at the
 * first padoc_kv_pool_sync), or -1 before that.  Decode calls require it to
 * be the current device and return PADOC_ERR_INVALID otherwise. */
PADOC_API int padoc_kv_pool_device(const padoc_kv_pool* pool, int32_t* device);
/* Testing aid, not for normal use: records `device` as the pool's device
 * without moving anything, so that a machine with one GPU can exercise the
 * device-mismatch rejection.  Restore the true device before any decode
 * call is meant to run.  PADOC_ERR_INVALID before the first sync. */
PADOC_API int padoc_debug_kv_pool_rehome(padoc_kv_pool* pool, int32_t device);

/* ------------------------------------------------------------------------
 * Backward of the packed tree-varlen forward (training; PaDoc, "Training
 * paradigm" trains through the same ancestor-masked attention).  For an
 * upstream gradient dO it returns the gradients of sum(dO * O):
 *   P = exp(scale q.k - LSE), dP = dO . v, dS = P (dP - rowsum(dO * O)),
 *   dq = scale sum_j dS k_j,  dk_j = scale sum dS q,  dv_j = sum P dO,
 * over exactly the (query, ancestor key) pairs of the forward; dk and dv of
 * a kv head sum over the query heads of its group.
 *   q, k, v, o, lse  the forward's inputs and outputs (same layouts)
 *   d_o              device [T, Hq, d], dtype of q
 *   dq / dk / dv     device, shapes and dtype of q / k / v (overwritten)
 *   ws               device workspace of padoc_tree_attn_varlen_bwd_ws_size
 *                    bytes, 256-byte aligned, not in use by a running call
 * dtype PADOC_BF16 or PADOC_F32; d 64 or 128; Hq / Hkv in {1, 2, 4, 8, 16};
 * scale as in the forward.  Results are deterministic: every output row
 * belongs to one work unit (an atomic counter in ws only hands units out). */
PADOC_API int padoc_tree_attn_varlen_bwd_ws_size(const padoc_tree_desc* desc, int32_t Hq, size_t* bytes);
PADOC_API int padoc_tree_attn_varlen_bwd(padoc_tree_desc* desc, const void* q, const void* k, const void* v,
                                         const void* o, const float* lse, const void* d_o, void* dq, void* dk,
                                         void* dv, int32_t dtype, int32_t Hq, int32_t Hkv, int32_t d, float scale,
                                         void* ws, size_t ws_bytes, padoc_stream_t stream);
/* The key-stationary half of the backward plan, for checks: items [n][4] =
 * key tile start, keys in the tile, first entry, entries; entries [m][5] =
 * keys [k_lo, k_hi), causal, queries [q_lo, q_hi).  Keys of the tile that a
 * query of an entry sees are those in [k_lo, k_hi), and only j <= t when
 * causal.  Either output may be NULL. */
PADOC_API int padoc_tree_desc_bwd_plan(const padoc_tree_desc* desc, int32_t* items, int32_t* entries,
                                       int64_t* n_items, int64_t* n_entries);

/* ------------------------------------------------------------------------
 * Branch-parallel decode and speculative verify over the pool.
 * Every live branch queries 1..16 tokens against the shared prefix of its
 * page plus its own cached suffix; inside the query block each token sees
 * its draft-tree ancestors and itself (HSD page, "prefix-tree batching";
 * HPD-Parsing: parallel verify of drafted tokens on forked branches).
 * The shared prefix of a page is streamed from HBM once for all branches of
 * the page (cascade); partial softmaxes are merged by log-sum-exp.  A verify
 * step whose pages each fit one prefix chunk (see padoc_decode_plan_fused)
 * runs as one kernel that walks, per row tile, the prefix, the own suffixes
 * and the query block in a single running softmax.
 * ---------------------------------------------------------------------- */
typedef struct {
  int32_t n_pages;
  int32_t n_branches;
  const int32_t* page_seq;       /* host [n_pages]: sequence holding the page's shared prefix */
  const int32_t* branch_offsets; /* host [n_pages + 1]: page p owns branches
                                    [branch_offsets[p], branch_offsets[p+1]) */
  const int32_t* branch_seq;     /* host [n_branches]: the branch's sequence, a fork of its
                                    page's sequence; it sees the fork_len shared tokens as its
                                    prefix and the rest of its tokens as its own suffix */
  const int32_t* q_offsets;      /* host [n_branches + 1]: query rows of branch b are
                                    [q_offsets[b], q_offsets[b+1]), between 1 and 16 */
} padoc_decode_batch;

/* Workspace bytes padoc_branch_decode needs for this batch and head count. */
PADOC_API int padoc_branch_decode_ws_size(const padoc_kv_pool* pool, const padoc_decode_batch* batch,
                                int32_t Hq, size_t* bytes);

/*   q         device [nq, Hq, d] pool dtype; nq = q_offsets[n_branches]
 *   k_new     device [nq, Hkv, d]: keys of the step's own query tokens (not yet in the
 *   v_new               cache; commit accepted ones later with padoc_kv_append)
 *   tree_bits device [nq] uint16 or NULL: bit j of row i (within its branch) set iff
 *             query token j of the same branch is visible to token i; NULL means a chain
 *             (j <= i).  Bit i must be set for every row.  padoc_tree_mask_build fills it
 *             from a parent array.
 *   o         device [nq, Hq, d] pool dtype
 *   lse       device [nq, Hq] f32, natural log
 *   ws        device workspace of at least padoc_branch_decode_ws_size bytes, 256-byte
 *             aligned, not shared with a call still running
 * Hq must be a multiple of the pool's Hkv with Hq / Hkv <= 8.  scale <= 0 means
 * 1/sqrt(d).  Validation happens on the host before any launch. */
PADOC_API int padoc_branch_decode(padoc_kv_pool* pool, const padoc_decode_batch* batch, int32_t Hq,
                        const void* q, const void* k_new, const void* v_new,
                        const uint16_t* tree_bits, void* o, float* lse, float scale, void* ws,
                        size_t ws_bytes, padoc_stream_t stream);

/* ---- The same step split into a plan and its two device passes. ----
 * A plan is host state built from the pool and the batch.  It stays valid
 * until the pool changes (alloc/append/fork/release); build the next step's
 * plan while the current one runs.
 *   padoc_decode_plan_create  validates and plans (host only)
 *   padoc_decode_plan_ws_size workspace bytes the plan needs
 *   padoc_decode_plan_upload  uploads changed block-table rows and copies the
 *                             plan into ws (enqueued on stream)
 *   padoc_decode_prefix_pass  kernel 1: per page, kv head and prefix chunk,
 *                             the partial softmax of every query row of the
 *                             page over the chunk's shared blocks (tensor
 *                             cores; each prefix block read once per page)
 *   padoc_decode_own_pass     kernel 2: per branch and kv head, the own
 *                             suffix and the query block under the tree mask,
 *                             then the log-sum-exp merge with kernel 1's
 *                             partials into o and lse
 *   padoc_decode_plan_fused   *fused = 1 when the plan runs as one kernel: a
 *                             verify step (Hq / Hkv >= 2, several query rows
 *                             per branch) whose every page prefix fits one
 *                             40-tile chunk.  Its prefix pass then launches
 *                             nothing and its own pass walks, per page, row
 *                             tile and kv head, the prefix, the own suffixes
 *                             of the tile's branches and their query block,
 *                             and writes o and lse directly.  The
 *                             environment variable PADOC_VERIFY_FUSED=0
 *                             (read once per process) keeps two kernels.
 * Arguments mean what they mean for padoc_branch_decode; ws must hold the
 * uploaded plan.  The own pass reads what the prefix pass wrote to ws, so
 * run them in this order on one stream. */
typedef struct padoc_decode_plan padoc_decode_plan;
PADOC_API int padoc_decode_plan_create(padoc_kv_pool* pool, const padoc_decode_batch* batch, int32_t Hq,
                                       padoc_decode_plan** out);
PADOC_API int padoc_decode_plan_ws_size(const padoc_decode_plan* plan, size_t* bytes);
PADOC_API int padoc_decode_plan_fused(const padoc_decode_plan* plan, int32_t* fused);
PADOC_API int padoc_decode_plan_upload(padoc_decode_plan* plan, void* ws, size_t ws_bytes, padoc_stream_t stream);
PADOC_API int padoc_decode_prefix_pass(const padoc_decode_plan* plan, const void* q, float scale, void* ws,
                                       padoc_stream_t stream);
PADOC_API int padoc_decode_own_pass(const padoc_decode_plan* plan, const void* q, const void* k_new,
                                    const void* v_new, const uint16_t* tree_bits, void* o, float* lse,
                                    float scale, void* ws, padoc_stream_t stream);
PADOC_API int padoc_decode_plan_free(padoc_decode_plan* plan);

/* Draft-tree visibility (HSD page, "prefix-tree batching"): for n <= 16 nodes
 * in topological order (parent[i] < i, -1 for a root), bits[i] gets bit j set
 * iff node j is node i or one of its ancestors.  Host arrays. */
PADOC_API int padoc_tree_mask_build(const int32_t* parent, int32_t n, uint16_t* bits);

/* ------------------------------------------------------------------------
 * Accept step of speculative verify (HSD page, "greedy tree traversal";
 * HPD-Parsing, inference workflow: accepted length n_acc of a drafted chain).
 *
 * The query rows [q_offsets[b], q_offsets[b+1]) of branch b are the nodes of
 * its draft tree; node 0 is the anchor (the token fixed by the previous
 * step) and row r of logits holds the model's next-token scores after node r.
 * From the anchor the walk takes, among the current node's children, the one
 * whose token scores highest (lowest node index on ties) and accepts it when
 *     logit(child) - max(row) >= log(tau)            (float32 arithmetic)
 * -- the log-probability difference of the HSD rule, whose softmax
 * normaliser cancels -- and stops otherwise or at a leaf.  The free token is
 * the argmax of the last accepted node's row (lowest token index on ties).
 * tau = 1 is the greedy rule: a draft is kept while it is the argmax.
 *
 *   logits     device [nq, vocab] bf16, row-major, finite (NaN: unspecified)
 *   tokens     device [nq] int32: token of each node (node 0's is not read)
 *   parents    device [nq] int32: parent node index within the branch, -1
 *              for node 0 and in [0, i) for node i >= 1
 *   q_offsets  device [n_branches + 1] int32
 *   max_nodes  host bound on nodes per branch, 1..16; each branch gets this
 *              many argmax CTAs, so keep it tight (1 for plain decode)
 *   tau        acceptance threshold, > 0 (0.75 in the HSD page)
 *   n_acc      device [n_branches] int32 out: nodes accepted after the anchor
 *   path       device [n_branches, 16] int32 out: accepted node indices in
 *              order, -1 padded
 *   free_token device [n_branches] int32 out
 * A branch with no node or more than max_nodes nodes, rows outside [0, nq),
 * a parent on node 0, a parent that is not an earlier node, or a token
 * outside [0, vocab) gets n_acc = -1, free_token = -1 and a path of -1; the
 * other branches are unaffected.  Host checks (null pointers, sizes, tau)
 * return PADOC_ERR_INVALID before any launch.  Two launches on stream, no
 * workspace: the row argmaxes are parked in path between them. */
PADOC_API int padoc_verify_accept(const void* logits, int32_t nq, int32_t vocab, const int32_t* tokens,
                                  const int32_t* parents, const int32_t* q_offsets, int32_t n_branches,
                                  int32_t max_nodes, float tau, int32_t* n_acc, int32_t* path,
                                  int32_t* free_token, padoc_stream_t stream);

/* Commit of accepted draft tokens (HPD-Parsing, inference workflow: accepted
 * tokens join the branch's own KV, rejected drafts never reach the cache).
 * Appends to each listed sequence, in order, the rows of k_new / v_new that
 * it names.  For a verified branch b the rows are usually its anchor
 * q_offsets[b] followed by q_offsets[b] + path[b][0 .. n_acc[b]).
 *   seqs        host [n_seqs]: distinct live sequences
 *   row_offsets host [n_seqs + 1], row_offsets[0] = 0, non-decreasing:
 *               sequence i takes rows[row_offsets[i] .. row_offsets[i+1])
 *   rows        host: row indices into k_new / v_new, each in [0, n_src_rows)
 *   k_new/v_new device [n_src_rows, Hkv, d] pool dtype, 16-byte aligned
 *   ws          device, at least 16 * row_offsets[n_seqs] bytes, 16-byte
 *               aligned, not in use by a call still running
 * Blocks for every sequence are reserved before anything changes, so on
 * PADOC_ERR_OOM (or any validation error) the pool is as it was.  A forked
 * sequence's own tokens never go into a block it shares with its parent.
 * The row list is copied into ws and one scatter kernel runs on stream. */
PADOC_API int padoc_kv_commit(padoc_kv_pool* pool, int32_t n_seqs, const int32_t* seqs,
                              const int32_t* row_offsets, const int32_t* rows, int32_t n_src_rows,
                              const void* k_new, const void* v_new, void* ws, size_t ws_bytes,
                              padoc_stream_t stream);

/* ------------------------------------------------------------------------
 * Draft trie of decoupled speculative verification (HSD page, "decoupled
 * speculative verification": draft-target matching and prefix-tree batching).
 *
 * A draft index holds one request's fixed drafts (they do not change while
 * the request decodes) and a table of every window of `window` consecutive
 * draft tokens (n = 3 in the HSD page).  One step's verify block is then:
 *   node 0 = the last accepted token (the anchor);
 *   the last `window` accepted tokens are looked up; each occurrence in a
 *   draft, taken draft by draft and by position, contributes the draft's
 *   tokens after it, cut to max_depth - 1 tokens;
 *   the continuations are merged into a prefix tree (one node per distinct
 *   prefix, siblings with distinct tokens), nodes numbered in creation order
 *   (every parent before its children); creation stops once max_nodes nodes
 *   exist.
 * Fewer accepted tokens than `window`, or no occurrence, give the anchor
 * alone.  Everything here is host memory and host work. */
typedef struct padoc_draft_index padoc_draft_index;
/* tokens: the drafts concatenated; draft d is tokens[draft_offsets[d] ..
 * draft_offsets[d+1]) (draft_offsets[0] = 0, non-decreasing); window >= 1.
 * The index copies what it needs. */
PADOC_API int padoc_draft_index_create(const int32_t* tokens, const int64_t* draft_offsets, int32_t n_drafts,
                                       int32_t window, padoc_draft_index** out);
PADOC_API int padoc_draft_index_free(padoc_draft_index* index);
/* accepted: the accepted tokens so far (n_accepted >= 1; only the last
 * `window` are read).  tokens / parents: capacity max_nodes (>= 1);
 * parents[0] = -1.  max_depth >= 1 counts the anchor. */
PADOC_API int padoc_draft_trie(const padoc_draft_index* index, const int32_t* accepted, int32_t n_accepted,
                               int32_t max_nodes, int32_t max_depth, int32_t* tokens, int32_t* parents,
                               int32_t* n_nodes);
/* A whole verify batch: branch b uses index[b] and
 * accepted[acc_offsets[b] .. acc_offsets[b+1]) (at least one token).  Writes
 * the concatenated blocks: tokens and parents (capacity n_branches *
 * max_nodes, parents relative to the branch), q_offsets [n_branches + 1] and,
 * when bits is not NULL, the ancestor-or-self rows [nq] that
 * padoc_branch_decode takes as tree_bits.  max_nodes in [1, 16]. */
PADOC_API int padoc_draft_trie_batch(const padoc_draft_index* const* index, int32_t n_branches,
                                     const int32_t* accepted, const int32_t* acc_offsets, int32_t max_nodes,
                                     int32_t max_depth, int32_t* tokens, int32_t* parents, int32_t* q_offsets,
                                     uint16_t* bits);

/* ------------------------------------------------------------------------
 * Branch scheduler (HPD-Parsing, inference workflow, Algorithm 1).  Host
 * code over the KV pool; the model step (draft, verify, accept, commit) is
 * the caller's, between padoc_sched_schedule and padoc_sched_update.
 *   - Waiting requests are ordered first-come-first-served by keys: a child
 *     (content) branch (0, arrival(parent), -m, arrival(child)) with m the
 *     number of children its parent had spawned before it; a main (layout)
 *     request (1, arrival); ties by request id.
 *   - A main request is admitted only while pool occupancy (blocks in use /
 *     pool blocks) <= tau and fewer than n_max requests are active; child
 *     branches bypass that gate.  A child is ready once its parent is
 *     resident with the tokens before the <FORK> that spawned it cached.  A request the
 *     pool cannot hold now keeps its place; the scan goes on.
 *   - Each step first reserves, for every active branch, room for its
 *     cached tokens plus window + 1 (the anchor and the drafted tokens); when
 *     the pool runs short the youngest active request (latest arrival, then
 *     highest id) is preempted: its KV is released and it waits to be
 *     rebuilt.  Requests preempted in a step are not readmitted in it.
 *   - A branch's token stream is its prefix (the prompt; for a child, the
 *     parent's tokens before the <FORK>) and its output.  Every token but
 *     the newest is cached; the newest is the next step's anchor.  A child's
 *     output starts with child_token.  Only main requests fork.
 *   - A branch ends at eos_token or after max_len output tokens.  Its
 *     sequence is released when it and all its children have ended; a main
 *     request's output then interleaves each child's output after the <FORK>
 *     that spawned it.
 * The scheduler owns the pool sequences of its requests.  After admission
 * the caller rebuilds the cached tokens of each admitted request (the
 * request's sequence already counts them); after each step the caller
 * commits the old anchor and the accepted tokens but the newest
 * (padoc_kv_commit, or its own writes) before padoc_sched_update. */
typedef struct {
  float tau;            /* KV occupancy threshold in [0, 1] for admitting main requests */
  int32_t n_max;        /* cap on active requests for admitting main requests */
  int32_t window;       /* draft window K in [0, 15]: K + 1 query rows per branch and step */
  int32_t max_len;      /* output tokens after which a branch ends (8000 in HPD-Parsing) */
  int32_t fork_token;   /* <FORK> */
  int32_t child_token;  /* <CHILD>: first token of a child branch */
  int32_t eos_token;
} padoc_sched_config;
typedef struct padoc_sched padoc_sched;
/* One step's decisions.  The caller provides arrays of capacity cap
 * (branch_offsets cap + 1); the batch fields form a padoc_decode_batch
 * (page_seq, branch_offsets, branch_seq = active_seq). */
typedef struct {
  int32_t cap;
  int32_t n_admitted, n_preempted, n_active, n_pages;
  int32_t* admitted;        /* request ids admitted this step (their cached tokens need rebuilding) */
  int32_t* preempted;       /* request ids preempted this step */
  int32_t* active;          /* active request ids, grouped by page, key order inside a page */
  int32_t* active_seq;      /* their pool sequences */
  int32_t* page_seq;        /* per page: the sequence holding the shared prefix */
  int32_t* branch_offsets;  /* [n_pages + 1] */
} padoc_sched_step;
PADOC_API int padoc_sched_create(padoc_kv_pool* pool, const padoc_sched_config* cfg, padoc_sched** out);
/* Releases the pool sequences the scheduler still holds. */
PADOC_API int padoc_sched_destroy(padoc_sched* sched);
/* A main request with prompt_len >= 1 tokens (its last token is the first anchor). */
PADOC_API int padoc_sched_submit(padoc_sched* sched, int32_t prompt_len, int64_t arrival, int32_t* request);
PADOC_API int padoc_sched_schedule(padoc_sched* sched, padoc_sched_step* step);
/* The verified tokens of each listed running request (n_acc drafted tokens
 * plus the free token, at least one): request [n], token_offsets [n + 1],
 * tokens.  Processed in the given order; now is the arrival time of the
 * children spawned. */
PADOC_API int padoc_sched_update(padoc_sched* sched, int64_t now, int32_t n, const int32_t* request,
                                 const int32_t* token_offsets, const int32_t* tokens);
/* state: 0 waiting, 1 running, 2 ended (children pending), 3 done. */
PADOC_API int padoc_sched_request(const padoc_sched* sched, int32_t request, int32_t* state, int32_t* seq,
                                  int32_t* parent, int64_t* n_out);
/* The interleaved output of a done main request; tokens may be NULL to
 * query the length. */
PADOC_API int padoc_sched_output(const padoc_sched* sched, int32_t request, int32_t* tokens, int64_t cap,
                                 int64_t* n);

/* Critical-path depths of one page (PaDoc, theoretical speedup):
 * d_seq = l(B_1:N) + sum_k l(Y_k);  d_tree = max_k [l(B<=k) + l(Y_k)]. */
PADOC_API int padoc_depths(const int32_t* layout_len, const int32_t* content_len, int32_t n_regions,
                 int64_t* d_seq, int64_t* d_tree);

/* ------------------------------------------------------------------------
 * Branch decode without any device allocation.  (The papers have no
 * counterpart: this serves embedding, not the method.)
 *
 * Some callers may not call cudaMalloc at all: a host runtime that hands the
 * whole GPU to its own memory arena and owns every byte, a plug-in that lives
 * inside such a runtime, or a latency-critical loop that cannot afford the
 * device-wide synchronisation an allocation can cause.  They cannot provide
 * the workspace padoc_branch_decode needs.  This entry point computes the
 * same step with the workspace taken from one fixed array that the library
 * places in device memory when it is loaded (PADOC_NOALLOC_SCRATCH_BYTES on
 * every GPU that loads the library, held until the process exits).
 *
 * Arguments are those of padoc_branch_decode without ws / ws_bytes.
 *  - A step whose workspace (padoc_branch_decode_ws_size) exceeds
 *    PADOC_NOALLOC_SCRATCH_BYTES is rejected with PADOC_ERR_INVALID before
 *    any device work.  As a guide, a 16-page step with one query per branch
 *    needs about 10 MiB.
 *  - The pool's device block table must already exist (call
 *    padoc_kv_pool_sync once at set-up); otherwise PADOC_ERR_INVALID.
 *  - The pool's device (padoc_kv_pool_device) must be the current device;
 *    otherwise PADOC_ERR_INVALID before any device work.
 *  - The call allocates and frees no device memory itself; the host plan
 *    lives on the host heap.
 *  - The first call on a device looks up the array's device address (once
 *    per device, with that device current) and caches it.  With lazy module
 *    loading (CUDA_MODULE_LOADING=LAZY, the default) that lookup is also
 *    the moment the driver loads the library's module on the device and
 *    reserves the array, so the first call is the one that takes device
 *    memory.  Make that first call at set-up, before any stream capture and
 *    before the arena takes the rest of the GPU.  After cudaDeviceReset the
 *    cached address is stale: do not use the library on that device again
 *    in the same process (its pools' tables are gone as well).
 *  - All calls share the one array and it keeps the last call's contents.
 *    Nothing in it needs to start at zero: each call writes every byte it
 *    later reads.  Calls whose work overlaps on the GPU (other streams, other
 *    host threads) race on the array; order them on one stream. */
#define PADOC_NOALLOC_SCRATCH_BYTES (32u << 20)
PADOC_API int padoc_branch_decode_noalloc(padoc_kv_pool* pool, const padoc_decode_batch* batch, int32_t Hq,
                                          const void* q, const void* k_new, const void* v_new,
                                          const uint16_t* tree_bits, void* o, float* lse, float scale,
                                          padoc_stream_t stream);

/* Testing aid, not for normal use: sets, on the current device, the longest
 * time (nanoseconds) one wait of the verify own pass with keys on the MMA's
 * M side may take before the kernel gives up and reports
 * PADOC_ERR_DEVICE_TIMEOUT through padoc_device_status; 0 restores the
 * default of 2 s.  It applies to that kernel only: when one of its roles
 * gives up, the others leave their loops, its TMA producers wait for the
 * copies they issued and its MMA thread for its products before the CTA
 * releases tensor memory and exits, so a wait that runs out leaves the GPU
 * usable for the next call (HPD-Parsing's failure detection has no GPU-side
 * counterpart; this serves tests of the abort path). */
PADOC_API int padoc_debug_set_wait_limit(uint64_t ns);

/* Reports and clears the device error word of the current device: 0 when no
 * kernel has given up a wait since the last call, else PADOC_ERR_DEVICE_TIMEOUT
 * with the failing site in the message. */
PADOC_API int padoc_device_status(padoc_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* PADOC_H_ */
