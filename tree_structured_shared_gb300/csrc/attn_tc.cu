// Tensor-core attention engine for sm_103a (tcgen05 + TMEM + TMA).
//
// One persistent, warp-specialised CTA per SM walks a list of work units.  A
// unit is 128 query rows (the tokens of one query tile times the query heads
// of one GQA group, so each K/V tile is read once for the whole group) and the
// ordered list of 128-key tiles those rows may see:
//
//   MODE_FWD     packed tree-varlen forward.  Rows are a tile of one query
//                segment; key tiles walk that segment's key segments (the
//                ancestors X, B<=k and the causal own segment).  Tiles of
//                non-ancestor keys are never listed, so they cost nothing.
//                (PaDoc, "Training paradigm": a query of Y_k reads the keys
//                of X, B<=k and Y_k as if they were one sequence.)
//   MODE_PREFIX  cascade prefix pass of branch decode.  Rows are the query
//                rows of every branch of one page; key tiles are one chunk of
//                the page's shared prefix blocks, read from HBM once for all
//                branches (HPD-Parsing: forked branches share the prefix KV
//                with zero copy).  Writes normalised partial O and LSE.
//   MODE_OWN     own pass of a verify step: rows are the query rows of one
//                branch; key tiles are its own cached suffix and its query
//                block; merges with the prefix partials into O and LSE.
//   MODE_VERIFY  a verify step in one pass: rows as in MODE_PREFIX; key
//                tiles are the page's prefix (one chunk), then the own
//                suffix of each branch the rows belong to (visible to that
//                branch's rows only), then one tile of the query-block keys
//                (visible by branch and draft-tree mask).  Writes O and LSE.
//
// Roles (224 threads):
//   warps 0-3  softmax: thread r owns TMEM lane r = query row r.  Reads S
//              from TMEM, masks, keeps the running max / sum, writes P (bf16
//              pairs) back over the S tile in TMEM, rescales O in TMEM when
//              the max grows by more than 2^8, and runs the epilogue.
//   warp 4     producer of Q and K tiles (TMA); decode: also stages the
//              chunk's block ids in shared memory.  Q and a unit's first K
//              tile share a barrier, the second K tile has its own, and later
//              K tiles complete the P_FULL barrier of the tile two before.
//   warp 6     producer of V tiles (TMA); a V tile's bytes complete the
//              P_FULL barrier of its key tile, next to the softmax's P.
//   warp 5     MMA issuer (one thread): S = Q K^T into one of three TMEM
//              tiles, two key tiles ahead of P V, and O += P V (P read from
//              TMEM) into a TMEM accumulator.
//
// TMEM: columns [0,128), [128,256) and [256,384) hold S (then P), [384,512)
// hold O (f32).  With three S tiles the S of tile j+2 needs only the P V of
// tile j-1 to have been issued, so the softmax never waits for its next S.
// K and V have rings of their own: a K stage is free once its S has run, a V
// stage once its P V has, so each ring prefetches as far as its lifetime
// allows.  tcgen05.mma issue stalls while the pipe is full, so the MMA
// thread does little else: one wait and two commits per key tile.
// Shared memory (1024-byte aligned, 128-byte swizzle, two 64-column halves):
//   Q 32 KB | K 3 x 32 KB | V 3 x 32 KB | barriers | block ids.
// Every wait is bounded; a unit that times out raises the CTA abort flag, the
// device error word, and all roles leave their loops.
#include <cuda_bf16.h>

#include "../../include/padoc.h"
#include "padoc_internal.h"
#include "ptx_sm103.cuh"

namespace padoc {

__device__ unsigned int g_tc_err;

namespace {

using namespace ptx;

enum { MODE_FWD = 0, MODE_PREFIX = 1, MODE_OWN = 2, MODE_VERIFY = 3 };

constexpr int kStages = 3;  // K and V tile rings
constexpr int kSBufs = 3;   // S / P tiles in tensor memory
constexpr int kThreads = 224;
constexpr int kHalf = 16384;  // bytes of one 64-column half of a 128-row tile
constexpr int SM_Q = 0;
constexpr int SM_K = SM_Q + 2 * kHalf;
constexpr int SM_V = SM_K + kStages * 2 * kHalf;
constexpr int SM_P = SM_V + kStages * 2 * kHalf;
constexpr int SM_BAR = SM_P;  // P lives in tensor memory, over the S tile it came from
constexpr int SM_IDS = SM_BAR + 256;  // prefix pass: block ids of the unit's chunk
constexpr int kMaxChunkBlocks = kMaxChunkTiles * kTileKeys / 16;
constexpr int SM_TOTAL = SM_IDS + kMaxChunkBlocks * 4;
constexpr int kSmemBytes = SM_TOTAL + 1024;

// barrier slots
enum {
  B_QK0_FULL = 0,    // count 2: Q and the K tile of the unit's first key tile have landed
  B_Q_EMPTY = 1,     // the unit's last S has run
  B_K1_FULL = 2,     // the K tile of the unit's second key tile has landed
  B_S_FULL = 3,      // +buffer (3): S of tile k (buffer and K stage k % 3) has run
  B_P_FULL = 6,      // +buffer (3), count 6: see below
  B_O_DONE = 9,      // +buffer (3): P V of tile k (V stage k % 3) has run
  B_IDS_READY = 12,  // prefix pass: the chunk's block ids are staged
  B_IDS_FREE = 13,   // prefix pass: the V producer is done with them
  B_UNIT_FULL = 14,  // +slot (4), decode: the unit ring's slot holds the next unit
  B_UNIT_EMPTY = 18, // +slot (4), count 6: the MMA thread, the V producer and the softmax warps read it
  N_BARS = 22
};
// Tiles are numbered k across all units of the CTA.  Tile k uses K stage, S
// buffer and V stage k % 3 alike, so the S_FULL commit also frees its K stage
// and the O_DONE commit its V stage: the producers wait on those.  P_FULL of
// tile k completes with six arrivals: the four softmax warps (P written), the
// V producer (V of tile k landed) and the K producer (K of the unit's tile
// two further on landed, or a plain arrival near the unit's end).  So the MMA
// thread waits once per key tile, issues S of tile k+2 and P V of tile k, and
// commits twice.
static_assert(kStages == kSBufs, "K / V stages must match the S buffers");
static_assert(N_BARS * 8 + 8 <= SM_IDS - SM_BAR, "barrier area");
// Decode kernels take their units from a counter in the workspace, in order
// (so the CTAs at work at one time still share pages), as they free up: the
// K producer draws two units ahead and publishes them in a ring of kURing
// slots after the barriers; the other roles read them there.
constexpr int kURing = 4;
constexpr int SM_URING = SM_BAR + 192;
static_assert(N_BARS * 8 + 8 <= 192 && SM_URING + kURing * 4 <= SM_IDS, "unit ring");

constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr uint32_t kTmemO = 384;           // TMEM columns [384, 512): O (f32)
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

struct Params {
  int mode;
  int n_units;
  int32_t Hq, Hkv, group;
  float sl2;  // scale * log2(e)
  // forward
  FwdPlan plan;
  int64_t T;
  __nv_bfloat16* o;
  int o_v8;  // o is 32-byte aligned (rows then take 32-byte stores)
  float* lse;
  // prefix pass
  const DecPage* pages;
  const DecItem* items;
  const int32_t* q_plen;
  const int32_t* table;
  int32_t max_bps;
  const __nv_bfloat16* q;
  float* part_o;
  float* part_lse;
  int32_t* work;  // decode: unit counter, zero at launch
  // own pass
  const DecBranch* branches;
  const uint16_t* tree_bits;
  const int32_t* q_branch;
};

// The work unit as seen by every role (computed identically by each).
struct Unit {
  int32_t g;         // kv head
  // forward
  int32_t tile_start, q_end, kv_first, kv_count, tile_last;
  // prefix / own
  int32_t page, tile, rows, row_base, k_begin, k_end, seq, q_first;
  // own
  int32_t own_len, n_shared, q_len, q_in_page;
  int32_t n_tiles;  // key tiles of the unit
  KVSeg kv0;        // forward: the first key segment
  // fused verify
  int32_t b_first, b_count, tok_lo;
};

__device__ __forceinline__ Unit load_unit(const Params& p, int u) {
  Unit w;
  // forward and prefix pass: head-major, so the CTAs at work at one time
  // share one kv head's K/V (forward: a working set that stays in L2; prefix
  // pass: a page's row tiles, adjacent items, read its prefix together);
  // own pass: the heads of one branch together
  const int n_it = p.mode == MODE_FWD ? p.plan.n_items : (p.mode == MODE_OWN ? 0 : p.n_units / p.Hkv);
  w.g = p.mode == MODE_OWN ? u % p.Hkv : u / n_it;
  const int item = p.mode == MODE_OWN ? u / p.Hkv : u % n_it;
  if (p.mode == MODE_FWD) {
    const FwdItem it = p.plan.items[item];
    w.tile_start = it.tile_start;
    w.q_end = it.q_end;
    w.kv_first = it.kv_first;
    w.kv_count = it.kv_count;
    w.tile_last = it.tile_last;
    w.n_tiles = it.n_tiles;
    w.kv0 = it.kv0;
  } else if (p.mode == MODE_OWN) {
    const DecBranch br = p.branches[item];
    w.page = br.page;
    w.seq = br.seq;
    w.q_first = br.q_first;
    w.own_len = br.own_len;
    w.n_shared = br.n_shared;
    w.q_len = br.q_len;
    w.q_in_page = br.q_in_page;
    w.rows = br.q_len * p.group;
    w.n_tiles = (br.own_len + kTileKeys - 1) / kTileKeys + 1;  // own suffix, then the query block
  } else {
    const DecItem it = p.items[item];
    const DecPage pg = p.pages[it.page];
    w.page = it.page;
    w.tile = it.tile;
    w.rows = it.rows;
    w.row_base = it.row_base;
    w.k_begin = it.chunk * pg.chunk_tokens;
    w.k_end = min(pg.P, w.k_begin + pg.chunk_tokens);
    w.seq = pg.seq;
    w.q_first = pg.q_first;
    w.b_first = it.b_first;
    w.b_count = it.b_count;
    w.tok_lo = it.tok_lo;
    w.n_tiles = it.n_tiles;
  }
  return w;
}

// Key tiles of a unit are enumerated in one fixed order by every role.
// Walk over a unit's key tiles.  The descriptor of the segment after the
// current one (forward: its KV segment; fused verify: the next own suffix's
// length) is loaded on entering a segment, so the switch does not wait on
// global memory.
struct TileIter {
  int32_t s, s_end, ks, end, causal;
  KVSeg nx;
};

__device__ __forceinline__ bool seg_setup(const Params& p, const Unit& w, TileIter& t) {
  while (t.s < t.s_end) {
    const KVSeg kv = t.nx;
    if (t.s + 1 < t.s_end) t.nx = p.plan.kvsegs[t.s + 1];
    int32_t end = kv.start + kv.len;
    if (kv.causal) end = min(end, w.tile_last + 1);
    if (end > kv.start) {
      t.ks = kv.start;
      t.end = end;
      t.causal = kv.causal;
      return true;
    }
    ++t.s;
  }
  return false;
}

// Fused verify: segment 0 is the prefix chunk, segments 1 .. b_count the own
// suffixes of the unit's branches (t.nx.len: the length of segment s + 1 when
// it is one), segment b_count + 1 the query-block tile.
__device__ __forceinline__ bool verify_setup(const Params& p, const Unit& w, TileIter& t) {
  while (t.s < t.s_end) {
    t.ks = 0;
    if (t.s == 0) {
      t.ks = w.k_begin;
      t.end = w.k_end;
    } else if (t.s <= w.b_count) {
      t.end = t.nx.len;
    } else {
      t.end = 1;
    }
    if (t.s + 1 <= w.b_count) t.nx.len = p.branches[w.b_first + t.s].own_len;
    if (t.ks < t.end) return true;
    ++t.s;
  }
  return false;
}

__device__ __forceinline__ bool tiles_begin(const Params& p, const Unit& w, TileIter& t) {
  t.causal = 0;
  if (p.mode == MODE_VERIFY) {
    t.s = 0;
    t.s_end = w.b_count + 2;
    return verify_setup(p, w, t);
  }
  if (p.mode == MODE_FWD) {
    t.s = w.kv_first;
    t.s_end = w.kv_first + w.kv_count;
    t.nx = w.kv0;
    return seg_setup(p, w, t);
  }
  if (p.mode == MODE_OWN) {
    // the branch's own cached tokens (t.s == 0), then one tile of the query
    // block's own keys (t.s == 1)
    t.s = w.own_len > 0 ? 0 : 1;
    t.s_end = 2;
    t.ks = 0;
    t.end = w.own_len > 0 ? w.own_len : w.q_len;
    t.causal = 0;
    return true;
  }
  t.s = 0;
  t.s_end = 1;
  t.ks = w.k_begin;
  t.end = w.k_end;
  t.causal = 0;
  return t.ks < t.end;
}

__device__ __forceinline__ bool tiles_next(const Params& p, const Unit& w, TileIter& t) {
  t.ks += kTileKeys;
  if (t.ks < t.end) return true;
  if (p.mode == MODE_FWD) {
    ++t.s;
    return seg_setup(p, w, t);
  }
  if (p.mode == MODE_VERIFY) {
    ++t.s;
    return verify_setup(p, w, t);
  }
  if (p.mode == MODE_OWN && t.s == 0) {
    t.s = 1;
    t.ks = 0;
    t.end = w.q_len;
    return true;
  }
  return false;
}

// Key tiles of the unit, counted by the host plan (the walk itself reads a
// segment list from global memory, a chain of loads every role would wait on).
__device__ __forceinline__ int count_tiles(const Params&, const Unit& w) { return w.n_tiles; }

// The next unit of a role that reads the unit ring (decode), or of the
// static round robin (forward).  `k` counts the units the role has taken;
// `single` when one thread runs the role.  False when a wait gave up.
template <int MODE>
__device__ __forceinline__ bool take_unit(const Params& p, uint32_t& k, int& u, volatile int32_t* uring,
                                          uint64_t* bars, volatile int* abort, bool single) {
  if (MODE == MODE_FWD) {
    u = blockIdx.x + static_cast<int>(k++) * gridDim.x;
    // the record of the unit after this one, into L1 while this one runs
    const int un = u + gridDim.x;
    if (un < p.n_units) asm volatile("prefetch.global.L1 [%0];" ::"l"(&p.plan.items[un % p.plan.n_items]));
    return true;
  }
  const int slot = k % kURing;
  const bool ok = mbar_wait(smem_u32(&bars[B_UNIT_FULL + slot]), (k / kURing) & 1, abort);
  if (single ? !ok : !__all_sync(0xffffffffu, ok)) return false;
  u = uring[slot];
  if (!single) __syncwarp();
  if (single || (threadIdx.x & 31) == 0) mbar_arrive(smem_u32(&bars[B_UNIT_EMPTY + slot]));
  ++k;
  return true;
}

__device__ __forceinline__ void raise_abort(volatile int* abort, unsigned site) {
  *abort = 1;
  atomicOr(&g_tc_err, site);
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_kn,
                   const __grid_constant__ CUtensorMap tm_vn, const __grid_constant__ CUtensorMap tm_k8,
                   const __grid_constant__ CUtensorMap tm_v8, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base; offsetting the shared array itself keeps the
  // compiler aware that every pointer below is a shared-memory pointer
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM_BAR + N_BARS * 8);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + SM_BAR + N_BARS * 8 + 4);
  volatile int32_t* uring = reinterpret_cast<volatile int32_t*>(smem + SM_URING);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < N_BARS; ++i) {
      uint32_t cnt = 1;
      if (i >= B_P_FULL && i < B_P_FULL + kSBufs) cnt = 6;
      if (i >= B_UNIT_EMPTY && i < B_UNIT_EMPTY + kURing) cnt = 6;
      if (i == B_QK0_FULL) cnt = 2;
      mbar_init(bar(i), cnt);
    }
    *abort = 0;
    fence_mbar_init();
  }
  if (MODE != MODE_FWD) {
    // stale bytes in a partly filled K/V tile are masked, but must be finite
    uint4 z = make_uint4(0, 0, 0, 0);
    for (int i = threadIdx.x; i < (SM_BAR - SM_K) / 16; i += kThreads)
      reinterpret_cast<uint4*>(smem + SM_K)[i] = z;
    fence_proxy_async_smem();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int G = p.group;

  if (warp == 4 || warp == 6) {
    // ------------------------------------------------------------ producers
    // warp 4: Q and K (and, for the prefix pass, the chunk's block ids);
    // warp 6: V.  Separate warps keep K loads from queueing behind V waits.
    const bool is_k = warp == 4;
    const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
    const int stages = kStages;
    const int b_empty = is_k ? B_S_FULL : B_O_DONE;  // the S / P V of the stage's last tile has run
    const uint32_t sm_base = sbase + (is_k ? SM_K : SM_V);
    if (lane == 0) {
      if (is_k) tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(tm);
    }
    int32_t* ids = reinterpret_cast<int32_t*>(smem + SM_IDS);
    uint32_t it = 0, item_it = 0;
    bool failed = false;
    // decode, K producer: draw a unit from the counter and publish it in
    // the ring (-1 when a wait gave up).  The next unit is drawn once the
    // current one's K tiles are issued: late enough that no CTA takes work
    // early, early enough that the draw overlaps the wait for Q.
    uint32_t n_pub = 0;
    auto publish = [&]() -> int {
      const int slot = n_pub % kURing;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_UNIT_EMPTY + slot), ((n_pub / kURing) & 1) ^ 1, abort)))
        return -1;
      int v = 0;
      if (lane == 0) {
        v = atomicAdd(p.work, 1);
        uring[slot] = v;
        mbar_arrive(bar(B_UNIT_FULL + slot));
      }
      ++n_pub;
      return __shfl_sync(0xffffffffu, v, 0);
    };
    int q_next = 0;  // K producer: the unit published, not yet loaded
    if (MODE != MODE_FWD && is_k) {
      q_next = publish();
      if (q_next < 0) failed = true;
    }
    auto publish_next = [&]() -> bool {
      if (MODE == MODE_FWD || !is_k) return true;
      q_next = publish();
      return q_next >= 0;
    };
    uint32_t n_taken = 0;
    while (!failed) {
      int u;
      if (MODE == MODE_FWD || !is_k) {
        if (!take_unit<MODE>(p, n_taken, u, uring, bars, abort, false)) {
          failed = true;
          break;
        }
      } else {
        u = q_next;
      }
      if (u >= p.n_units) break;
      const Unit w = load_unit(p, u);
      if (count_tiles(p, w) == 0) {
        if (!publish_next()) {
          failed = true;
          break;
        }
        continue;
      }
      if (is_k) {
        if (!__all_sync(0xffffffffu, mbar_wait(bar(B_Q_EMPTY), (item_it & 1) ^ 1, abort))) { failed = true; break; }
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(B_QK0_FULL), 2 * kHalf);
          if (MODE == MODE_FWD) {
            const int tt = p.plan.tile_tokens;
            for (int hh = 0; hh < G; ++hh)
              for (int h = 0; h < 2; ++h)
                tma_load_3d(sbase + SM_Q + h * kHalf + hh * tt * 128, &tm_q, bar(B_QK0_FULL), h * 64, w.g * G + hh,
                            w.tile_start);
          } else {
            // Query rows of the page, row R = (query R / G, head g*G + R % G):
            // a 4-D box {d/2, G, 1, 128/G} of q viewed as [nq][Hkv][G][d]
            // lands in exactly that row order.
            const int q0 = MODE == MODE_OWN ? w.q_first : w.q_first + w.tile * (kTileRows / G);
            for (int h = 0; h < 2; ++h) tma_load_4d(sbase + SM_Q + h * kHalf, &tm_q, bar(B_QK0_FULL), h * 64, 0, w.g, q0);
          }
        }
        if (MODE == MODE_PREFIX || MODE == MODE_VERIFY) {
          // block ids of the whole chunk, read once per unit and shared with warp 6
          if (!__all_sync(0xffffffffu, mbar_wait(bar(B_IDS_FREE), (item_it & 1) ^ 1, abort))) { failed = true; break; }
          const int n_ids = (w.k_end - w.k_begin + 15) >> 4;
          const int32_t* row = p.table + static_cast<int64_t>(w.seq) * p.max_bps + (w.k_begin >> 4);
          for (int i = lane; i < n_ids; i += 32) ids[i] = row[i];
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_IDS_READY));
        }
      } else if (MODE == MODE_PREFIX || MODE == MODE_VERIFY) {
        if (!__all_sync(0xffffffffu, mbar_wait(bar(B_IDS_READY), item_it & 1, abort))) { failed = true; break; }
      }
      const uint32_t it0 = it;  // number of the unit's first tile
      TileIter t;
      for (bool ok = tiles_begin(p, w, t); ok; ok = tiles_next(p, w, t), ++it) {
        const int st = it % stages;
        const uint32_t ph = ((it / stages) & 1) ^ 1;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(b_empty + st), ph, abort))) { failed = true; break; }
        const uint32_t dst = sm_base + st * 2 * kHalf;
        // where the tile's bytes land: V on P_FULL of its own tile; K of the
        // unit's first two tiles on QK0 / K1, later K on P_FULL of the tile
        // two before it (S of that K tile is issued after that wait)
        const int b_full = !is_k ? B_P_FULL + st
                                 : (it == it0 ? B_QK0_FULL
                                              : (it == it0 + 1 ? B_K1_FULL : B_P_FULL + (it - 2) % kSBufs));
        if (MODE == MODE_FWD) {
          if (lane == 0) {
            mbar_arrive_expect_tx(bar(b_full), 2 * kHalf);
            for (int h = 0; h < 2; ++h) tma_load_3d(dst + h * kHalf, tm, bar(b_full), h * 64, w.g, t.ks);
          }
        } else if (MODE == MODE_OWN && t.s == 1) {
          // the query block's own keys: 16 rows of k_new / v_new for kv head g
          if (lane == 0) {
            mbar_arrive_expect_tx(bar(b_full), 2 * 2048);
            for (int h = 0; h < 2; ++h)
              tma_load_3d(dst + h * kHalf, is_k ? &tm_kn : &tm_vn, bar(b_full), h * 64, w.g, w.q_first);
          }
        } else if (MODE == MODE_VERIFY && t.s == w.b_count + 1) {
          // the query-block keys of the unit's branches: 128 rows of k_new /
          // v_new for kv head g from the first branch's first query token
          if (lane == 0) {
            mbar_arrive_expect_tx(bar(b_full), 2 * kHalf);
            for (int h = 0; h < 2; ++h)
              tma_load_3d(dst + h * kHalf, is_k ? &tm_kn : &tm_vn, bar(b_full), h * 64, w.g, w.tok_lo);
          }
        } else {
          const int nblk = (min(kTileKeys, t.end - t.ks) + 15) >> 4;
          int32_t blk = 0;
          if (MODE == MODE_OWN) {
            if (lane < nblk)
              blk = p.table[static_cast<int64_t>(w.seq) * p.max_bps + w.n_shared + (t.ks >> 4) + lane];
          } else if (MODE == MODE_VERIFY && t.s > 0) {
            // an own tile of branch b_first + s - 1: its blocks after the shared ones
            const DecBranch br = p.branches[w.b_first + t.s - 1];
            if (lane < nblk) blk = p.table[static_cast<int64_t>(br.seq) * p.max_bps + br.n_shared + (t.ks >> 4) + lane];
          } else if (lane < nblk) {
            blk = ids[((t.ks - w.k_begin) >> 4) + lane];
          }
          // A tile of eight physically consecutive blocks comes in one box
          // per half (the TMA unit takes some 75 cycles per 2 KB box, so
          // sixteen boxes a tile for K and for V would bound the pass).
          const int32_t b0 = __shfl_sync(0xffffffffu, blk, 0);
          const bool run8 = nblk == 8 && __all_sync(0xffffffffu, lane >= 8 || blk == b0 + lane);
          if (lane == 0) mbar_arrive_expect_tx(bar(b_full), nblk * 2 * 2048);
          __syncwarp();
          if (run8) {
            if (lane == 0)
              for (int h = 0; h < 2; ++h) tma_load_4d(dst + h * kHalf, is_k ? &tm_k8 : &tm_v8, bar(b_full), h * 64, 0, w.g, b0);
          } else if (lane < nblk) {
            const int32_t row = (blk * p.Hkv + w.g) * 16;
            for (int h = 0; h < 2; ++h) tma_load_2d(dst + h * kHalf + lane * 2048, tm, bar(b_full), h * 64, row);
          }
        }
      }
      if (failed) break;
      if (!publish_next()) {
        failed = true;
        break;
      }
      if (is_k) {
        // tiles whose K tile two further on does not exist (the unit's last
        // two) still get the K producer's arrival on P_FULL.  Arriving for
        // tile k needs P_FULL of tile k-3 complete: S of tile k-1 is issued
        // only after that, so wait for S of tile k-1.
        const uint32_t n_t = it - it0;
        for (uint32_t k = it0 + (n_t > 2 ? n_t - 2 : 0); k < it && !failed; ++k) {
          if (k > 0 &&
              !__all_sync(0xffffffffu, mbar_wait(bar(B_S_FULL + (k - 1) % kSBufs), ((k - 1) / kSBufs) & 1, abort)))
            failed = true;
          if (!failed && lane == 0) mbar_arrive(bar(B_P_FULL + k % kSBufs));
        }
        if (failed) break;
      }
      if (!is_k && (MODE == MODE_PREFIX || MODE == MODE_VERIFY)) {
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_IDS_FREE));
      }
      ++item_it;
    }
    if (failed && lane == 0) raise_abort(abort, is_k ? 0x1 : 0x2);
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    // tcgen05.mma issue stalls while the pipe is full, so every instruction
    // between two MMA groups is pipe idle time: ring positions are kept as
    // (index, phase) pairs, and each key tile costs one wait and two commits.
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t id_pv = idesc_bf16_f32(128, 128, false, true);
      const uint32_t t_o = tmem + kTmemO;
      const uint64_t d_q = sdesc_sw128(sbase + SM_Q, 16, 1024);
      uint32_t sb = 0, s_ph = 0;  // ring position of the next S (K stage = S buffer)
      uint32_t pb = 0, p_ph = 0;  // ring position of the next P V (V stage = S buffer)
      uint32_t item_it = 0, k1_it = 0;
      bool failed = false;
      // S of the next key tile, its K tile already waited for.  Its S buffer
      // last held P of the tile three back, read by a P V issued earlier by
      // this thread (tcgen05.mma runs in issue order).  TMA-written operands
      // need no tcgen05 fence: the barrier's transaction count orders them
      // before the MMA reads.
      auto issue_s = [&]() {
        const uint64_t d_k = sdesc_sw128(sbase + SM_K + sb * 2 * kHalf, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t off = static_cast<uint64_t>(((kk >> 2) * kHalf + (kk & 3) * 32) >> 4);
          mma_bf16_ss(tmem + sb * 128, d_q + off, d_k + off, id_qk, kk > 0);
        }
        mma_commit(bar(B_S_FULL + sb));
        if (++sb == kSBufs) {
          sb = 0;
          s_ph ^= 1;
        }
      };
      uint32_t n_taken = 0;
      while (!failed) {
        int u;
        if (!take_unit<MODE>(p, n_taken, u, uring, bars, abort, true)) {
          failed = true;
          break;
        }
        if (u >= p.n_units) break;
        const Unit w = load_unit(p, u);
        const int n = count_tiles(p, w);
        if (n == 0) continue;
        // S runs two key tiles ahead of P V; Q is free once the unit's last S has run
        if (!mbar_wait_relaxed(bar(B_QK0_FULL), item_it & 1, abort)) { failed = true; break; }
        issue_s();
        if (n > 1) {
          if (!mbar_wait_relaxed(bar(B_K1_FULL), k1_it & 1, abort)) { failed = true; break; }
          ++k1_it;
          issue_s();
        }
        if (n <= 2) mma_commit(bar(B_Q_EMPTY));
        for (int j = 0; j < n; ++j) {
          // P and V of tile j and K of tile j+2 land on one per-buffer
          // barrier (the softmax may run up to two tiles ahead).  The first P
          // of a unit is written after the softmax's epilogue read O, so P V
          // may then overwrite O.
          if (!mbar_wait_relaxed(bar(B_P_FULL + pb), p_ph, abort)) { failed = true; break; }
          tc_fence_after();
          if (j + 2 < n) {
            issue_s();
            if (j + 3 == n) mma_commit(bar(B_Q_EMPTY));
          }
          const uint32_t pt = tmem + pb * 128;  // P (bf16 pairs) over S of this tile
          const uint64_t d_v = sdesc_sw128(sbase + SM_V + pb * 2 * kHalf, kHalf, 1024);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16_ts(t_o, pt + kk * 8, d_v + static_cast<uint64_t>(kk * (2048 >> 4)), id_pv,
                        (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(bar(B_O_DONE + pb));
          if (++pb == kSBufs) {
            pb = 0;
            p_ph ^= 1;
          }
        }
        ++item_it;
      }
      if (failed) raise_abort(abort, 0x4);
    }
  } else {
    // ------------------------------------------------------------ softmax (warps 0-3)
    const int r = threadIdx.x;  // query row == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    uint32_t s_it = 0, p_it = 0, pv_base = 0;
    bool failed = false;
    uint32_t n_taken = 0;
    while (!failed) {
      int u;
      if (!take_unit<MODE>(p, n_taken, u, uring, bars, abort, false)) {
        failed = true;
        break;
      }
      if (u >= p.n_units) break;
      const Unit w = load_unit(p, u);
      const int n = count_tiles(p, w);
      if (n == 0) continue;
      // this thread's row
      bool valid;
      int32_t head, limit;  // limit: keys at positions >= limit are hidden (prefix) / causal bound (fwd)
      int64_t qpos = 0;
      if (MODE == MODE_FWD) {
        const int tt = p.plan.tile_tokens;
        const int hh = r / tt;
        qpos = w.tile_start + (r % tt);
        valid = qpos < w.q_end;
        head = w.g * G + hh;
        limit = static_cast<int32_t>(qpos) + 1;
      } else if (MODE == MODE_OWN) {
        valid = r < w.rows;
        head = w.g * G + r % G;
        qpos = w.q_first + r / G;
        limit = w.own_len;
      } else {
        valid = r < w.rows;
        const int R = w.tile * kTileRows + r;
        head = w.g * G + R % G;
        qpos = w.q_first + R / G;
        limit = valid ? p.q_plen[qpos] : 0;
      }
      // fused verify: this row's branch, and bit c of qvis[c / 32] set when
      // key c of the query-block tile (query token tok_lo + c) is the row's
      // draft-tree ancestor or the row's own token
      int32_t qbr = -1;
      uint32_t qvis[4] = {0u, 0u, 0u, 0u};
      if (MODE == MODE_VERIFY && valid) {
        qbr = p.q_branch[qpos];
        const DecBranch brq = p.branches[qbr];
        const int qi = static_cast<int>(qpos) - brq.q_first;
        uint32_t bits = p.tree_bits ? static_cast<uint32_t>(p.tree_bits[qpos]) : ((2u << qi) - 1u);
        bits &= (1u << brq.q_len) - 1u;
        const int rel = brq.q_first - w.tok_lo;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int sh = rel - 32 * k;
          qvis[k] = sh >= 0 ? (sh < 32 ? bits << sh : 0u) : (sh > -32 ? bits >> -sh : 0u);
        }
      }
      float m_run = -INFINITY, l_run = 0.f;
      TileIter t;
      int j = 0;
      for (bool ok = tiles_begin(p, w, t); ok; ok = tiles_next(p, w, t), ++j) {
        const int sb = s_it % kSBufs;
        // relaxed: only tensor-memory reads follow, ordered by the tcgen05 fence
        if (!__all_sync(0xffffffffu, mbar_wait_relaxed(bar(B_S_FULL + sb), (s_it / kSBufs) & 1, abort))) {
          failed = true;
          break;
        }
        tc_fence_after();
        float s[128];
        {
          // all four loads in flight before one wait
          uint32_t v0[32], v1[32], v2[32], v3[32];
          tmem_ld32(tmem + lane_base + sb * 128 + 0, v0);
          tmem_ld32(tmem + lane_base + sb * 128 + 32, v1);
          tmem_ld32(tmem + lane_base + sb * 128 + 64, v2);
          tmem_ld32(tmem + lane_base + sb * 128 + 96, v3);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            s[i] = __uint_as_float(v0[i]);
            s[32 + i] = __uint_as_float(v1[i]);
            s[64 + i] = __uint_as_float(v2[i]);
            s[96 + i] = __uint_as_float(v3[i]);
          }
        }
        ++s_it;
        // mask keys this row may not see
        const int32_t klen = min(kTileKeys, t.end - t.ks);
        int32_t vis = klen;  // keys [0, vis) of the tile are visible
        if (MODE == MODE_FWD) {
          if (t.causal) vis = min(vis, limit - t.ks);
        } else if (MODE == MODE_PREFIX || (MODE == MODE_VERIFY && t.s == 0)) {
          vis = min(vis, limit - t.ks);
        } else if (MODE == MODE_VERIFY && t.s <= w.b_count) {
          if (qbr != w.b_first + t.s - 1) vis = 0;  // another branch's own keys
        }
        // A row that sees no key of the tile takes P = 0 through an infinite
        // exponent offset; it still masks keys past the tile's end (stale or
        // unwritten bytes), but needs no per-key mask below that.
        const bool row_dead = vis <= 0 && !((MODE == MODE_VERIFY && t.s == w.b_count + 1) || (MODE == MODE_OWN && t.s == 1));
        if (row_dead) vis = klen;
        if (MODE == MODE_VERIFY && t.s == w.b_count + 1) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (!((qvis[c >> 5] >> (c & 31)) & 1u)) s[c] = -INFINITY;
        } else if (MODE == MODE_OWN && t.s == 1) {
          // query block: key c is query token c of this branch, visible iff it
          // is this token's draft-tree ancestor or the token itself
          const int qi = r / G;
          uint32_t bits = 0;
          if (valid) bits = p.tree_bits ? static_cast<uint32_t>(p.tree_bits[qpos]) : ((2u << qi) - 1u);
          bits &= (1u << w.q_len) - 1u;
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= 16 || !((bits >> c) & 1u)) s[c] = -INFINITY;
        } else if (vis < kTileKeys) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= vis) s[c] = -INFINITY;
        }
        float tmax;
        {
          float m8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) m8[i] = s[i];
#pragma unroll
          for (int c = 8; c < 120; c += 16)
#pragma unroll
            for (int i = 0; i < 8; ++i) m8[i] = max3f(m8[i], s[c + i], s[c + 8 + i]);
#pragma unroll
          for (int i = 0; i < 8; ++i) m8[i] = fmaxf(m8[i], s[120 + i]);
          tmax = max3f(max3f(m8[0], m8[1], m8[2]), max3f(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
          if (row_dead) tmax = -INFINITY;
        }
        const float mt = tmax * p.sl2;
        const bool grow = mt > m_run + kRescaleThreshold;
        const float alpha = grow ? fast_exp2(m_run - mt) : 1.f;  // 0 while m_run is -inf
        if (grow) {
          l_run *= alpha;
          m_run = mt;
        }
        const float m_use = row_dead ? INFINITY : ((m_run == -INFINITY) ? 0.f : m_run);
        {
          // x = s * sl2 - m two lanes per instruction; the same partial sums
          // (lane k of the row sum takes columns c with c % 8 == k)
          const uint64_t sl2x2 = f2pack(p.sl2, p.sl2), negm = f2pack(-m_use, -m_use);
          uint64_t l2[4] = {0, 0, 0, 0};
#pragma unroll
          for (int c = 0; c < 128; c += 2) {
            float x0, x1;
            f2unpack(fma2(f2pack(s[c], s[c + 1]), sl2x2, negm), x0, x1);
            s[c] = fast_exp2(x0);
            s[c + 1] = fast_exp2(x1);
            l2[(c >> 1) & 3] = add2(l2[(c >> 1) & 3], f2pack(s[c], s[c + 1]));
          }
          float l8[8];
#pragma unroll
          for (int k = 0; k < 4; ++k) f2unpack(l2[k], l8[2 * k], l8[2 * k + 1]);
          l_run += ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
        }
        // Only a rescale of O waits for P V of tile j-1.  P V number q
        // completes a phase of O_DONE + q % 3 (phase q / 3); the barrier
        // cannot run a phase ahead of this wait, because P V q + 3 needs a P
        // this warp has not written yet.  Writing P needs no wait: its S
        // buffer last held P of tile j-3, whose P V ran before S of tile j.
        if (j > 0 && __any_sync(0xffffffffu, grow)) {
          const uint32_t q = pv_base + j - 1;
          if (!__all_sync(0xffffffffu, mbar_wait_relaxed(bar(B_O_DONE + q % kSBufs), (q / kSBufs) & 1, abort))) {
            failed = true;
            break;
          }
          tc_fence_after();
          {
            // O holds sums taken against the old max: rescale before P V of tile j
            uint32_t v[32];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              tmem_ld32(tmem + kTmemO + lane_base + c * 32, v);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
              tmem_st32(tmem + kTmemO + lane_base + c * 32, v);
            }
            tmem_wait_st();
          }
        }
        {
          // P as bf16 pairs into the first 64 columns of this tile's S buffer
          uint32_t pk[64];
#pragma unroll
          for (int c = 0; c < 64; ++c) pk[c] = pack_bf16x2(s[2 * c], s[2 * c + 1]);
          tmem_st64(tmem + lane_base + sb * 128, pk);
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_P_FULL + sb));
        ++p_it;
      }
      if (failed) break;
      // epilogue: O / l and LSE
      {
        // the unit's last P V (its commit covers all earlier ones)
        const uint32_t q = pv_base + n - 1;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(B_O_DONE + q % kSBufs), (q / kSBufs) & 1, abort))) {
          failed = true;
          break;
        }
      }
      tc_fence_after();
      if (MODE == MODE_OWN) {
        // merge with the prefix pass's partial rows of this (query, head) by
        // log-sum-exp, then write the final O and LSE
        const DecPage pg = p.pages[w.page];
        const int R = (w.q_in_page + r / G) * G + r % G;
        const int ptile = R / kTileRows, prr = R % kTileRows;
        float M = l_run > 0.f ? m_run : -INFINITY;
        for (int c = 0; c < pg.n_chunks && valid; ++c) {
          const DecItem it = p.items[pg.item_base + ptile * pg.n_chunks + c];
          M = fmaxf(M, p.part_lse[static_cast<int64_t>(it.row_base) + static_cast<int64_t>(w.g) * it.rows + prr] * kLog2e);
        }
        const float Mu = M == -INFINITY ? 0.f : M;
        const float w_own = l_run > 0.f ? fast_exp2(m_run - Mu) : 0.f;
        float L = l_run * w_own;
        for (int c = 0; c < pg.n_chunks && valid; ++c) {
          const DecItem it = p.items[pg.item_base + ptile * pg.n_chunks + c];
          L += fast_exp2(p.part_lse[static_cast<int64_t>(it.row_base) + static_cast<int64_t>(w.g) * it.rows + prr] *
                             kLog2e - Mu);
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t v[32];
          tmem_ld32(tmem + kTmemO + lane_base + cc * 32, v);
          tmem_wait_ld();
          if (valid) {
            float acc[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] = __uint_as_float(v[i]) * w_own;
            for (int c = 0; c < pg.n_chunks; ++c) {
              const DecItem it = p.items[pg.item_base + ptile * pg.n_chunks + c];
              const int64_t prow = static_cast<int64_t>(it.row_base) + static_cast<int64_t>(w.g) * it.rows + prr;
              const float wc = fast_exp2(p.part_lse[prow] * kLog2e - Mu);
              const float4* src = reinterpret_cast<const float4*>(p.part_o + prow * kHeadDim + cc * 32);
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float4 x = src[i];
                acc[4 * i + 0] = fmaf(x.x, wc, acc[4 * i + 0]);
                acc[4 * i + 1] = fmaf(x.y, wc, acc[4 * i + 1]);
                acc[4 * i + 2] = fmaf(x.z, wc, acc[4 * i + 2]);
                acc[4 * i + 3] = fmaf(x.w, wc, acc[4 * i + 3]);
              }
            }
            uint4* dst = reinterpret_cast<uint4*>(p.o + (qpos * p.Hq + head) * kHeadDim + cc * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(pack_bf16x2(acc[8 * i + 0] * inv, acc[8 * i + 1] * inv),
                                  pack_bf16x2(acc[8 * i + 2] * inv, acc[8 * i + 3] * inv),
                                  pack_bf16x2(acc[8 * i + 4] * inv, acc[8 * i + 5] * inv),
                                  pack_bf16x2(acc[8 * i + 6] * inv, acc[8 * i + 7] * inv));
          }
        }
        // O is read: this warp's next P_FULL arrival (after its own
        // tcgen05.fence::before_thread_sync) lets P V overwrite it
        if (valid) p.lse[qpos * p.Hq + head] = L > 0.f ? (Mu + __log2f(L)) * kLn2 : -INFINITY;
        pv_base += n;
        continue;
      }
      const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
      const float lse_v = l_run > 0.f ? (m_run + __log2f(l_run)) * kLn2 : -INFINITY;
      {
        // all of O's row in flight before one wait, then 32-byte stores
        uint32_t v[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tmem + kTmemO + lane_base + c * 32, v[c]);
        tmem_wait_ld();
        if (valid) {
          if (MODE == MODE_FWD || MODE == MODE_VERIFY) {
            uint32_t* dst = reinterpret_cast<uint32_t*>(p.o + (qpos * p.Hq + head) * kHeadDim);
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                uint32_t pk[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                  pk[i] = pack_bf16x2(__uint_as_float(v[c][16 * h + 2 * i]) * inv_l,
                                      __uint_as_float(v[c][16 * h + 2 * i + 1]) * inv_l);
                if (p.o_v8) {
                  st_global_v8(dst + c * 16 + h * 8, pk);
                } else {
                  uint4* d4 = reinterpret_cast<uint4*>(dst + c * 16 + h * 8);
                  d4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                  d4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                }
              }
          } else {
            float* dst = p.part_o + (static_cast<int64_t>(w.row_base) + static_cast<int64_t>(w.g) * w.rows + r) * kHeadDim;
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                uint32_t x[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) x[i] = __float_as_uint(__uint_as_float(v[c][8 * h + i]) * inv_l);
                st_global_v8(dst + c * 32 + h * 8, x);
              }
          }
        }
      }
      // O is read: this warp's next P_FULL arrival (after its own
      // tcgen05.fence::before_thread_sync) lets P V overwrite it
      if (valid) {
        if (MODE == MODE_FWD)
          p.lse[static_cast<int64_t>(head) * p.T + qpos] = lse_v;
        else if (MODE == MODE_VERIFY)
          p.lse[qpos * p.Hq + head] = lse_v;
        else
          p.part_lse[static_cast<int64_t>(w.row_base) + static_cast<int64_t>(w.g) * w.rows + r] = lse_v;
      }
      pv_base += n;
    }
    if (failed && lane == 0) raise_abort(abort, 0x8);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

int make_map(EncodeTiledFn enc, CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims,
             const cuuint64_t* strides, const cuuint32_t* box, std::string* err) {
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(ptr), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *err = "cuTensorMapEncodeTiled failed with code " + std::to_string(static_cast<int>(r));
    return PADOC_ERR_CUDA;
  }
  return PADOC_OK;
}

// The K / V pools viewed as [num_blocks][Hkv][16][d] with a box of eight
// consecutive blocks of one kv head (16 KB, one half of a key tile).
int make_pool8_maps(EncodeTiledFn enc, const DecodeArgs& a, CUtensorMap* mk8, CUtensorMap* mv8, std::string* err) {
  const cuuint64_t d8[4] = {128, 16, static_cast<cuuint64_t>(a.Hkv), static_cast<cuuint64_t>(a.num_blocks)};
  const cuuint64_t s8[3] = {256, 4096, static_cast<cuuint64_t>(a.Hkv) * 4096};
  const cuuint32_t b8[4] = {64, 16, 1, 8};
  int rc = make_map(enc, mk8, a.k_pool, 4, d8, s8, b8, err);
  if (!rc) rc = make_map(enc, mv8, a.v_pool, 4, d8, s8, b8, err);
  return rc;
}

template <int MODE>
int launch(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mkn,
           const CUtensorMap& mvn, const CUtensorMap& mk8, const CUtensorMap& mv8, const Params& prm, cudaStream_t s,
           std::string* err) {
  static bool attr_set[4] = {false, false, false, false};
  if (!attr_set[MODE]) {
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) {
      *err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
      return PADOC_ERR_CUDA;
    }
    attr_set[MODE] = true;
  }
  const int grid = std::min(prm.n_units, num_sms());
  attn_tc_kernel<MODE><<<grid, kThreads, kSmemBytes, s>>>(mq, mk, mv, mkn, mvn, mk8, mv8, prm);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *err = std::string("attention kernel launch: ") + cudaGetErrorString(e);
    return PADOC_ERR_CUDA;
  }
  return PADOC_OK;
}

}  // namespace

int launch_fwd_bf16(const FwdArgs& a, cudaStream_t s, std::string* err) {
  if (a.plan.n_items == 0) return PADOC_OK;
  EncodeTiledFn enc = get_encode_fn(err);
  if (!enc) return PADOC_ERR_CUDA;
  CUtensorMap mq, mk, mv;
  const cuuint64_t dq[3] = {128, static_cast<cuuint64_t>(a.Hq), static_cast<cuuint64_t>(a.T)};
  const cuuint64_t sq[2] = {256, static_cast<cuuint64_t>(a.Hq) * 256};
  const cuuint32_t bq[3] = {64, 1, static_cast<cuuint32_t>(a.plan.tile_tokens)};
  const cuuint64_t dk[3] = {128, static_cast<cuuint64_t>(a.Hkv), static_cast<cuuint64_t>(a.T)};
  const cuuint64_t sk[2] = {256, static_cast<cuuint64_t>(a.Hkv) * 256};
  const cuuint32_t bk[3] = {64, 1, 128};
  int rc = make_map(enc, &mq, a.q, 3, dq, sq, bq, err);
  if (!rc) rc = make_map(enc, &mk, a.k, 3, dk, sk, bk, err);
  if (!rc) rc = make_map(enc, &mv, a.v, 3, dk, sk, bk, err);
  if (rc) return rc;
  Params p{};
  p.mode = MODE_FWD;
  p.n_units = a.plan.n_items * a.Hkv;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.group = a.plan.group;
  p.sl2 = a.scale * kLog2e;
  p.plan = a.plan;
  p.T = a.T;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.o_v8 = (reinterpret_cast<uintptr_t>(a.o) & 31u) == 0;
  p.lse = a.lse;
  return launch<MODE_FWD>(mq, mk, mv, mk, mv, mk, mv, p, s, err);
}

int launch_decode_prefix(const DecodeArgs& a, cudaStream_t s, std::string* err) {
  if (a.n_items == 0) return PADOC_OK;
  EncodeTiledFn enc = get_encode_fn(err);
  if (!enc) return PADOC_ERR_CUDA;
  CUtensorMap mq, mk, mv;
  // q viewed as [nq][Hkv][G][d]; box {64, G, 1, 128/G}
  const cuuint64_t dq[4] = {128, static_cast<cuuint64_t>(a.group), static_cast<cuuint64_t>(a.Hkv),
                            static_cast<cuuint64_t>(a.nq)};
  const cuuint64_t sq[3] = {256, static_cast<cuuint64_t>(a.group) * 256, static_cast<cuuint64_t>(a.Hq) * 256};
  const cuuint32_t bq[4] = {64, static_cast<cuuint32_t>(a.group), 1, static_cast<cuuint32_t>(kTileRows / a.group)};
  const cuuint64_t dk[2] = {128, static_cast<cuuint64_t>(a.num_blocks) * a.Hkv * 16};
  const cuuint64_t sk[1] = {256};
  const cuuint32_t bk[2] = {64, 16};
  int rc = make_map(enc, &mq, a.q, 4, dq, sq, bq, err);
  if (!rc) rc = make_map(enc, &mk, a.k_pool, 2, dk, sk, bk, err);
  if (!rc) rc = make_map(enc, &mv, a.v_pool, 2, dk, sk, bk, err);
  if (rc) return rc;
  Params p{};
  p.mode = MODE_PREFIX;
  p.n_units = a.n_items * a.Hkv;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.group = a.group;
  p.sl2 = a.scale * kLog2e;
  p.pages = a.pages;
  p.items = a.items;
  p.q_plen = a.q_plen;
  p.table = a.table;
  p.max_bps = a.max_bps;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.part_o = a.part_o;
  p.part_lse = a.part_lse;
  CUtensorMap mk8, mv8;
  rc = make_pool8_maps(enc, a, &mk8, &mv8, err);
  if (rc) return rc;
  p.work = a.work;
  {
    // units are drawn from this counter in order
    const cudaError_t e = cudaMemsetAsync(a.work, 0, sizeof(int32_t), s);
    if (e != cudaSuccess) {
      *err = std::string("cudaMemsetAsync of the unit counter: ") + cudaGetErrorString(e);
      return PADOC_ERR_CUDA;
    }
  }
  return launch<MODE_PREFIX>(mq, mk, mv, mk, mv, mk8, mv8, p, s, err);
}

int launch_decode_own_tc(const DecodeArgs& a, cudaStream_t s, std::string* err) {
  if (a.n_branches == 0) return PADOC_OK;
  EncodeTiledFn enc = get_encode_fn(err);
  if (!enc) return PADOC_ERR_CUDA;
  CUtensorMap mq, mk, mv, mkn, mvn;
  const cuuint64_t dq[4] = {128, static_cast<cuuint64_t>(a.group), static_cast<cuuint64_t>(a.Hkv),
                            static_cast<cuuint64_t>(a.nq)};
  const cuuint64_t sq[3] = {256, static_cast<cuuint64_t>(a.group) * 256, static_cast<cuuint64_t>(a.Hq) * 256};
  const cuuint32_t bq[4] = {64, static_cast<cuuint32_t>(a.group), 1, static_cast<cuuint32_t>(kTileRows / a.group)};
  const cuuint64_t dk[2] = {128, static_cast<cuuint64_t>(a.num_blocks) * a.Hkv * 16};
  const cuuint64_t sk[1] = {256};
  const cuuint32_t bk[2] = {64, 16};
  // k_new / v_new viewed as [nq][Hkv][d]; box: 16 query tokens of one kv head
  const cuuint64_t dn[3] = {128, static_cast<cuuint64_t>(a.Hkv), static_cast<cuuint64_t>(a.nq)};
  const cuuint64_t sn[2] = {256, static_cast<cuuint64_t>(a.Hkv) * 256};
  const cuuint32_t bn[3] = {64, 1, 16};
  int rc = make_map(enc, &mq, a.q, 4, dq, sq, bq, err);
  if (!rc) rc = make_map(enc, &mk, a.k_pool, 2, dk, sk, bk, err);
  if (!rc) rc = make_map(enc, &mv, a.v_pool, 2, dk, sk, bk, err);
  if (!rc) rc = make_map(enc, &mkn, a.k_new, 3, dn, sn, bn, err);
  if (!rc) rc = make_map(enc, &mvn, a.v_new, 3, dn, sn, bn, err);
  if (rc) return rc;
  Params p{};
  p.mode = MODE_OWN;
  p.n_units = a.n_branches * a.Hkv;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.group = a.group;
  p.sl2 = a.scale * kLog2e;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.o_v8 = (reinterpret_cast<uintptr_t>(a.o) & 31u) == 0;
  p.lse = a.lse;
  p.pages = a.pages;
  p.items = a.items;
  p.table = a.table;
  p.max_bps = a.max_bps;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.part_o = a.part_o;
  p.part_lse = a.part_lse;
  p.branches = a.branches;
  p.tree_bits = a.tree_bits;
  CUtensorMap mk8, mv8;
  rc = make_pool8_maps(enc, a, &mk8, &mv8, err);
  if (rc) return rc;
  p.work = a.work;
  {
    // units are drawn from this counter in order
    const cudaError_t e = cudaMemsetAsync(a.work, 0, sizeof(int32_t), s);
    if (e != cudaSuccess) {
      *err = std::string("cudaMemsetAsync of the unit counter: ") + cudaGetErrorString(e);
      return PADOC_ERR_CUDA;
    }
  }
  return launch<MODE_OWN>(mq, mk, mv, mkn, mvn, mk8, mv8, p, s, err);
}

int launch_decode_verify_fused(const DecodeArgs& a, cudaStream_t s, std::string* err) {
  if (a.n_items == 0) return PADOC_OK;
  EncodeTiledFn enc = get_encode_fn(err);
  if (!enc) return PADOC_ERR_CUDA;
  CUtensorMap mq, mk, mv, mkn, mvn;
  // q viewed as [nq][Hkv][G][d]; box {64, G, 1, 128/G}
  const cuuint64_t dq[4] = {128, static_cast<cuuint64_t>(a.group), static_cast<cuuint64_t>(a.Hkv),
                            static_cast<cuuint64_t>(a.nq)};
  const cuuint64_t sq[3] = {256, static_cast<cuuint64_t>(a.group) * 256, static_cast<cuuint64_t>(a.Hq) * 256};
  const cuuint32_t bq[4] = {64, static_cast<cuuint32_t>(a.group), 1, static_cast<cuuint32_t>(kTileRows / a.group)};
  const cuuint64_t dk[2] = {128, static_cast<cuuint64_t>(a.num_blocks) * a.Hkv * 16};
  const cuuint64_t sk[1] = {256};
  const cuuint32_t bk[2] = {64, 16};
  // k_new / v_new viewed as [nq][Hkv][d]; box: 128 query tokens of one kv head
  const cuuint64_t dn[3] = {128, static_cast<cuuint64_t>(a.Hkv), static_cast<cuuint64_t>(a.nq)};
  const cuuint64_t sn[2] = {256, static_cast<cuuint64_t>(a.Hkv) * 256};
  const cuuint32_t bn[3] = {64, 1, 128};
  int rc = make_map(enc, &mq, a.q, 4, dq, sq, bq, err);
  if (!rc) rc = make_map(enc, &mk, a.k_pool, 2, dk, sk, bk, err);
  if (!rc) rc = make_map(enc, &mv, a.v_pool, 2, dk, sk, bk, err);
  if (!rc) rc = make_map(enc, &mkn, a.k_new, 3, dn, sn, bn, err);
  if (!rc) rc = make_map(enc, &mvn, a.v_new, 3, dn, sn, bn, err);
  if (rc) return rc;
  Params p{};
  p.mode = MODE_VERIFY;
  p.n_units = a.n_items * a.Hkv;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.group = a.group;
  p.sl2 = a.scale * kLog2e;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.o_v8 = (reinterpret_cast<uintptr_t>(a.o) & 31u) == 0;
  p.lse = a.lse;
  p.pages = a.pages;
  p.items = a.items;
  p.q_plen = a.q_plen;
  p.table = a.table;
  p.max_bps = a.max_bps;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.branches = a.branches;
  p.tree_bits = a.tree_bits;
  p.q_branch = a.q_branch;
  CUtensorMap mk8, mv8;
  rc = make_pool8_maps(enc, a, &mk8, &mv8, err);
  if (rc) return rc;
  p.work = a.work;
  {
    // units are drawn from this counter in order
    const cudaError_t e = cudaMemsetAsync(a.work, 0, sizeof(int32_t), s);
    if (e != cudaSuccess) {
      *err = std::string("cudaMemsetAsync of the unit counter: ") + cudaGetErrorString(e);
      return PADOC_ERR_CUDA;
    }
  }
  return launch<MODE_VERIFY>(mq, mk, mv, mkn, mvn, mk8, mv8, p, s, err);
}

int read_and_clear_tc_error(cudaStream_t s, unsigned* word) {
  unsigned zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(word, g_tc_err, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpyToSymbolAsync(g_tc_err, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e == cudaSuccess ? PADOC_OK : PADOC_ERR_CUDA;
}

}  // namespace padoc
