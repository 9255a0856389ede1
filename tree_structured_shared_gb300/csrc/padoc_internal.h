// Structures shared by the host library and the kernel launchers.
#pragma once
#include <cstdint>
#include <string>
#include <cuda.h>
#include <cuda_runtime.h>

namespace padoc {

// ---------------------------------------------------------------- forward
// A query segment: packed positions [q_start, q_start + q_len) that share one
// ordered list of key/value segments kvsegs[kv_first .. kv_first + kv_count).
struct QSeg {
  int32_t q_start, q_len, kv_first, kv_count;
};
// Keys [start, start + len); when causal, a query at packed position t sees
// only keys <= t (all keys of the segment before the query are visible).
struct KVSeg {
  int32_t start, len, causal, pad;
};
// One query tile: tile_tokens consecutive tokens of one query segment.
struct FwdItem {
  int32_t qseg, tile_start;
  int32_t n_tiles;  // key tiles the tile's walk visits (every kernel role counts on it)
  // the query segment's fields and its first key segment, copied so a
  // kernel reads one record per unit
  int32_t q_end, kv_first, kv_count, tile_last, pad;
  KVSeg kv0;
};

constexpr int kTileKeys = 128;  // keys per K/V tile
constexpr int kTileRows = 128;  // MMA M: query rows (tokens x heads of a GQA group)
constexpr int kMaxChunkTiles = 40;  // prefix pass: key tiles in one chunk of a page's prefix, at most
constexpr int kHeadDim = 128;   // d of the tensor-core path

struct FwdPlan {
  const QSeg* qsegs;
  const KVSeg* kvsegs;
  const FwdItem* items;
  int32_t n_items;
  int32_t group;        // Hq / Hkv
  int32_t tile_tokens;  // kTileRows / group
};

struct FwdArgs {
  FwdPlan plan;
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int64_t T;
  int32_t Hq, Hkv, d;
  float scale;
};

// ---------------------------------------------------------------- backward
// Key-stationary work of the backward: keys are cut into tiles on a global
// kTileKeys grid; an entry lists queries [q_lo, q_hi) of one query segment
// that see keys [k_lo, k_hi) of the tile through one key segment (when
// causal, a query at t sees only keys <= t).  Entries of one tile cover
// disjoint (query, key) pairs, so their contributions simply add.
struct BwdEntry {
  int32_t k_lo, k_hi, causal, q_lo, q_hi, pad[3];
};
struct BwdItem {
  int32_t k_start, k_len, e_first, e_count;
};
struct BwdPlan {
  const BwdItem* items;
  const BwdEntry* entries;
  int32_t n_items;
};

struct BwdArgs {
  FwdPlan fwd;  // query-stationary work (dQ), as in the forward
  BwdPlan bwd;  // key-stationary work (dK, dV)
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const float* lse;   // [Hq, T]
  const void* dout;   // [T, Hq, d]
  void* dq;
  void* dk;
  void* dv;
  float* delta;       // workspace [Hq, T]: rowsum(dO * O)
  int32_t* work;      // workspace: unit counter of the dK/dV pass (zeroed by its launcher)
  int64_t T;
  int32_t Hq, Hkv, d;
  float scale;
};

// ---------------------------------------------------------------- decode
struct DecPage {
  int32_t seq;           // block-table row holding the shared prefix
  int32_t P;             // prefix tokens any branch of the page sees
  int32_t q_first;       // first query row of the page
  int32_t nq;            // query rows of the page
  int32_t item_base;     // first prefix item of the page
  int32_t n_chunks;      // prefix chunks
  int32_t chunk_tokens;  // tokens per chunk (multiple of kTileKeys)
  int32_t row_tiles;     // ceil(nq * group / kTileRows)
};
struct DecItem {
  int32_t page, tile, chunk;
  int32_t rows;      // valid rows of this row tile
  int32_t row_base;  // partial row index of head 0; head g adds g * rows
  // fused verify: the branches whose query rows the tile holds, and the
  // first query token of the first of them
  int32_t b_first, b_count, tok_lo;
  int32_t n_tiles;  // key tiles of the unit (prefix chunk; fused verify: + own suffixes + query block)
  int32_t pad[3];
};
struct DecBranch {
  int32_t page, seq;
  int32_t prefix_len;  // shared prefix tokens this branch sees
  int32_t own_len;     // own cached tokens
  int32_t n_shared;    // leading blocks of seq that belong to the prefix
  int32_t q_first, q_len;
  int32_t q_in_page;   // index of its first query among its page's queries
};

struct DecodeArgs {
  const DecPage* pages;
  const DecItem* items;
  const DecBranch* branches;
  const int32_t* q_plen;  // [nq] prefix tokens visible to each query row
  const int32_t* q_branch;  // [nq] branch of each query row
  const int32_t* table;   // device block table [max_seqs][max_bps]
  int32_t max_bps;
  int32_t n_pages, n_items, n_branches, nq;
  int32_t Hq, Hkv, group, d;
  float scale;
  const void* q;
  const void* k_new;
  const void* v_new;
  const uint16_t* tree_bits;
  void* o;
  float* lse;
  float* part_o;    // [rows][d] f32 normalised partial outputs of the prefix pass
  float* part_lse;  // [rows] f32
  int32_t* work;    // unit counter of the tensor-core passes (zeroed by their launchers)
  const void* k_pool;
  const void* v_pool;
  int64_t num_blocks;
};

// Launchers (return 0 or a PADOC_ERR_* code, message in *err).
int launch_fwd_bf16(const FwdArgs& a, cudaStream_t s, std::string* err);
int launch_fwd_f32(const FwdArgs& a, cudaStream_t s, std::string* err);
int launch_decode_prefix(const DecodeArgs& a, cudaStream_t s, std::string* err);
int launch_decode_own(const DecodeArgs& a, cudaStream_t s, std::string* err);
int launch_decode_own_tc(const DecodeArgs& a, cudaStream_t s, std::string* err);
// Verify own pass with keys on the MMA's M side (Hq / Hkv of 1 or 2).
int launch_decode_own_kmajor(const DecodeArgs& a, cudaStream_t s, std::string* err);
// Verify step in one pass (plans marked fused): each (page, row tile, kv
// head) walks the prefix, the own suffixes of the branches it holds and
// their query block, and writes the final O and LSE.
int launch_decode_verify_fused(const DecodeArgs& a, cudaStream_t s, std::string* err);
int launch_kv_append(void* k_pool, void* v_pool, const int32_t* table_row, int32_t first_own,
                     int32_t n, int32_t Hkv, int32_t d, const void* k, const void* v,
                     cudaStream_t s, std::string* err);

int launch_accept(const void* logits, int64_t V, int32_t nq, const int32_t* tokens, const int32_t* parents,
                  const int32_t* q_offsets, int32_t n_branches, int32_t max_nodes, float log_tau,
                  int32_t* n_acc, int32_t* path, int32_t* free_token, cudaStream_t s, std::string* err);
// plan: device int4 per row {source row, block, slot, 0}
int launch_commit(void* k_pool, void* v_pool, const void* plan, int64_t n_rows, int32_t Hkv, const void* k,
                  const void* v, cudaStream_t s, std::string* err);

int launch_bwd_core(const BwdArgs& a, int32_t dtype, cudaStream_t s, std::string* err);
int launch_bwd_delta(const BwdArgs& a, int32_t dtype, cudaStream_t s, std::string* err);
int launch_bwd_tc(const BwdArgs& a, cudaStream_t s, std::string* err);
int read_and_clear_bwd_error(cudaStream_t s, unsigned* word);

// Device error words (set by kernels that give up a bounded wait).
int read_and_clear_tc_error(cudaStream_t s, unsigned* word);
int read_and_clear_own_error(cudaStream_t s, unsigned* word);

// Driver entry point for tensor-map encoding (resolved through the runtime).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn get_encode_fn(std::string* err);
int num_sms();

// Records an error message for padoc_last_error() and returns code.
int set_error(int code, const char* fmt, ...);
int32_t pool_num_blocks(const padoc_kv_pool* pool);
// True once the pool's device block table exists (padoc_kv_pool_sync ran).
bool pool_has_device_table(const padoc_kv_pool* pool);
// PADOC_OK when the pool has no device table yet or its device is current;
// else PADOC_ERR_INVALID (message names the call).
int pool_check_device(const padoc_kv_pool* pool, const char* what);

}  // namespace padoc
