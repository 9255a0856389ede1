// Own pass of a speculative-verify step on tensor cores, keys on the MMA's M
// side (sm_103a: tcgen05 + TMEM + TMA).
//
// In a verify step every live branch queries a small draft-token tree (HSD,
// "prefix-tree batching"; HPD-Parsing, parallel verify of drafted tokens):
// after the cascade prefix pass, each query still has to attend to its
// branch's own cached suffix and to its draft-tree ancestors inside the query
// block, and the two partial results are merged by log-sum-exp.  A work unit
// is one (branch, kv head): at most 16 query tokens times the G query heads
// of the group, i.e. at most 32 rows for G <= 2, against a few hundred keys.
//
// With the query rows on M (the engine of attn_tc.cu) a unit fills 17 of 128
// rows and its two or three key tiles never fill the pipeline.  Here the
// keys go on M instead:
//     S^T[key][row]  = K  Q^T    M = 128 keys, N = 32 rows, K = d = 128
//     O^T[d][row]   += V^T P^T   M = d = 128,  N = 32 rows, K = 128 keys
// so every MMA is dense in the keys and the kernel is a stream of K/V tiles
// from HBM.  TMEM lane = key for S^T (lane = head dim for O^T); the softmax
// thread t owns lane t and holds that key's scores for all 32 rows.  Row
// maxima are kept lazily: a tile needs a cross-thread reduction only when some
// score exceeds its row's running maximum by more than 2^8 (a vote), which
// after a unit's first tile is rare; the row sums stay per thread until the
// unit ends.
//
// Roles (384 threads, one persistent CTA per SM):
//   warps 0-7  softmax and epilogue: warp w reads TMEM lanes 32 (w % 4) ..
//              + 31 (thread t = lane = key of the tile for S^T, head dim
//              for O^T) and takes the rows 16 (w / 4) .. + 15, so each
//              scheduler runs two of them and each thread holds 16 rows;
//   warp 8     TMA producer of Q and K tiles (paged own blocks, then the
//              query block's k_new rows);
//   warp 9     MMA issuer (one thread);
//   warp 10    TMA producer of V tiles;
//   warp 11    row data: the combined prefix LSE of each row and where its
//              prefix partials are, staged a unit or two ahead.
// Shared memory (1024-byte aligned, 128-byte swizzle):
//   Q 2 x 8 KB | K 3 x 32 KB | V 3 x 32 KB | P 2 x 8 KB | reduction | barriers
// TMEM (128 columns): S^T buffers [0, 64) (2 x 32), O^T buffers [64, 128).
// Every wait is bounded; a role that gives up raises the CTA's abort flag and
// the device error word, and all roles leave their loops.
#include <cuda_bf16.h>

#include "../../include/padoc.h"
#include "padoc_internal.h"
#include "ptx_sm103.cuh"

namespace padoc {

__device__ unsigned int g_own_err;
// Longest time one wait of this kernel may take before it gives up
// (nanoseconds of the global timer); settable for tests, read at launch.
__device__ unsigned long long g_own_wait_limit_ns = ptx::kWaitLimitNs;

namespace {

using namespace ptx;

constexpr int kThreads = 384;
constexpr int kHalfRows = 16;  // rows per softmax warpgroup
constexpr int kRows = 32;          // N of both products: query rows of a unit (padded)
constexpr int kStages = 3;         // K and V rings
constexpr int kKHalf = 16384;      // one 64-column half of a 128-key tile
constexpr int kRHalf = kRows * 128;  // one 64-column half of a 32-row tile (Q or P)
constexpr int SM_Q = 0;
constexpr int SM_K = SM_Q + 2 * 2 * kRHalf;
constexpr int SM_V = SM_K + kStages * 2 * kKHalf;
constexpr int SM_P = SM_V + kStages * 2 * kKHalf;
constexpr int SM_RED = SM_P + 2 * 2 * kRHalf;  // [2 row halves][4 lane quadrants][16 rows] f32
// Row data, two buffers (unit parity): per row of the unit, the combined
// LSE of the prefix pass's partial results (log2 units), the partial row of
// the page's first prefix chunk and that chunk's share of the prefix mass.
// Then the row maxima published by the epilogue.
constexpr int kRowBuf = 3 * 32 * 4;
constexpr int SM_ROW = SM_RED + 4 * 32 * 4;
constexpr int SM_BAR = SM_ROW + 2 * kRowBuf + 32 * 4;
enum {
  B_K_FULL = 0,    // +stage (3)
  B_K_EMPTY = 3,   // +stage
  B_V_FULL = 6,    // +stage
  B_V_EMPTY = 9,   // +stage
  B_Q_FULL = 12,   // +buffer (2)
  B_Q_EMPTY = 14,  // +buffer: the unit's last S^T has run
  B_S_FULL = 16,   // +buffer: S^T of the tile is in TMEM
  B_S_FREE = 18,   // +buffer, count 8: the softmax warps have read it
  B_P_FULL = 20,   // +buffer, count 8: P of the tile is in shared memory
  B_P_FREE = 22,   // +buffer: P V of the tile has run
  B_O_FULL = 24,   // +buffer: the unit's last P V has run
  B_O_FREE = 26,   // +buffer, count 8: the epilogue has read O^T
  B_DRAIN = 28,    // the MMA thread's last commit at exit
  B_ROW_FULL = 29,  // +buffer (2): the unit's row data is staged
  B_ROW_FREE = 31,  // +buffer, count 8: the unit's epilogue has read it
  N_BARS = 33
};
constexpr int SM_MISC = SM_BAR + N_BARS * 8;  // tmem slot, abort flag
constexpr int SM_TOTAL = SM_MISC + 16;
constexpr int kSmemBytes = SM_TOTAL + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");
constexpr uint32_t kTmemS = 0, kTmemO = 64, kTmemCols = 128;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

struct Params {
  int n_units;
  int32_t Hq, Hkv, group;
  float sl2;
  const DecPage* pages;
  const DecItem* items;
  const DecBranch* branches;
  const int32_t* table;
  int32_t max_bps;
  const uint16_t* tree_bits;
  const float* part_o;
  const float* part_lse;
  __nv_bfloat16* o;
  float* lse;
};

struct Unit {
  int32_t g, page, seq, q_first, q_len, own_len, n_shared, q_in_page, rows, n_tiles;
};

__device__ __forceinline__ Unit load_unit(const Params& p, int u) {
  Unit w;
  const DecBranch br = p.branches[u / p.Hkv];
  w.g = u % p.Hkv;
  w.page = br.page;
  w.seq = br.seq;
  w.q_first = br.q_first;
  w.q_len = br.q_len;
  w.own_len = br.own_len;
  w.n_shared = br.n_shared;
  w.q_in_page = br.q_in_page;
  w.rows = br.q_len * p.group;
  // the own cached tokens in tiles of 128, then one tile for the query block
  w.n_tiles = (br.own_len + kTileKeys - 1) / kTileKeys + 1;
  return w;
}

__device__ __forceinline__ void raise_abort(volatile int* abort, unsigned site) {
  *abort = 1;
  atomicOr(&g_own_err, site);
}

// The pipeline's waits, with the limit read at launch.
__device__ __forceinline__ bool wait_l(uint32_t bar, uint32_t parity, volatile int* abort, uint64_t limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (global_timer() - t0 > limit) return false;
  }
}
__device__ __forceinline__ bool wait_relaxed_l(uint32_t bar, uint32_t parity, volatile int* abort, uint64_t limit) {
  if (mbar_try_wait_relaxed(bar, parity)) return true;
  const uint64_t t0 = global_timer();
  while (true) {
    if (mbar_try_wait_relaxed(bar, parity)) return true;
    if (*abort) return false;
    if (global_timer() - t0 > limit) return false;
  }
}

// A wait that ignores the abort flag but keeps the default time limit: used at exit
// to let copies and products already issued land before the CTA leaves.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
  int never = 0;
  return mbar_wait(bar, parity, &never);
}

// Named barriers 1 and 2: the four warps of one row half of the softmax.
__device__ __forceinline__ void bar_sync_half(int hf) {
  asm volatile("bar.sync %0, 128;" ::"r"(1 + hf) : "memory");
}
// OR of pred over the 128 threads of a row half.
__device__ __forceinline__ bool bar_or_half(int hf, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(1 + hf)
      : "memory");
  return r != 0;
}

// OR of pred over all 256 softmax threads (named barrier 3).  Every failed
// wait goes through this vote, so both row halves leave at the same step;
// it also keeps the halves in step at each tile, so a half writes the next
// unit's P only after the other half is done with the staging area.
__device__ __forceinline__ bool bar_or_all(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 3, 256, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred))
      : "memory");
  return r != 0;
}

// Reduces 16 per-row values over the 32 lanes of a warp (max or sum); lane
// l returns row (l % 16)'s result.  Lanes l and l ^ 16 combine first, then
// each step hands half of the rows to the partner lane: 31 shuffles.
template <bool MAX>
__device__ __forceinline__ float warp_rows_reduce16(float (&v)[16], int lane) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float o = __shfl_xor_sync(0xffffffffu, v[i], 16);
    v[i] = MAX ? fmaxf(v[i], o) : v[i] + o;
  }
#pragma unroll
  for (int s = 8; s >= 1; s >>= 1) {
    const bool up = (lane & s) != 0;
#pragma unroll
    for (int i = 0; i < s; ++i) {
      const float send = up ? v[i] : v[i + s];
      const float keep = up ? v[i + s] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, s);
      v[i] = MAX ? fmaxf(keep, recv) : keep + recv;
    }
  }
  return v[0];
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    own_kmajor_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_kn,
                      const __grid_constant__ CUtensorMap tm_vn, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM_MISC);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + SM_MISC + 4);
  float* red = reinterpret_cast<float*>(smem + SM_RED);
  // row data of buffer rb: lpre [32] f32 | prow [32] i32 | share [32] f32
  auto row_lpre = [&](int rb) { return reinterpret_cast<float*>(smem + SM_ROW + rb * kRowBuf); };
  auto row_prow = [&](int rb) { return reinterpret_cast<int32_t*>(smem + SM_ROW + rb * kRowBuf + 128); };
  auto row_share = [&](int rb) { return reinterpret_cast<float*>(smem + SM_ROW + rb * kRowBuf + 256); };
  float* row_m = reinterpret_cast<float*>(smem + SM_ROW + 2 * kRowBuf);  // [32]
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const int G = p.group;
  const uint64_t wlim = g_own_wait_limit_ns;
  const int gsh = G == 2 ? 1 : 0;  // row r is query token r >> gsh, head r & gsh of the group (G is 1 or 2)

  if (threadIdx.x == 0) {
    for (int i = 0; i < N_BARS; ++i) {
      uint32_t cnt = 1;
      if ((i >= B_S_FREE && i < B_S_FREE + 2) || (i >= B_P_FULL && i < B_P_FULL + 2) ||
          (i >= B_O_FREE && i < B_O_FREE + 2) || (i >= B_ROW_FREE && i < B_ROW_FREE + 2))
        cnt = 8;
      mbar_init(bar(i), cnt);
    }
    *abort = 0;
    fence_mbar_init();
  }
  {
    // Rows of a tile that a unit does not fill keep older bytes: zero them
    // once so that they are finite (they are masked, or multiplied by P = 0).
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int i = threadIdx.x; i < (SM_P - SM_Q) / 16; i += kThreads) reinterpret_cast<uint4*>(smem + SM_Q)[i] = z;
    fence_proxy_async_smem();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8 || warp == 10) {
    // ------------------------------------------------------------ producers
    const bool is_k = warp == 8;
    const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
    const CUtensorMap* tmn = is_k ? &tm_kn : &tm_vn;
    const int b_full = is_k ? B_K_FULL : B_V_FULL;
    const int b_empty = is_k ? B_K_EMPTY : B_V_EMPTY;
    const uint32_t ring = sbase + (is_k ? SM_K : SM_V);
    if (lane == 0) {
      if (is_k) tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(tm);
      tma_prefetch_desc(tmn);
    }
    uint32_t kt = 0;  // tiles whose copies were issued
    int iu = 0;       // units whose Q copy was issued (K producer)
    bool failed = false;
    // the next unit and its first 32 own block ids, read one unit ahead
    Unit w_next{};
    int32_t id_next = 0;
    auto prefetch = [&](int un) {
      if (un >= p.n_units) return;
      w_next = load_unit(p, un);
      const int nb = (w_next.own_len + 15) >> 4;
      id_next = lane < nb ? p.table[static_cast<int64_t>(w_next.seq) * p.max_bps + w_next.n_shared + lane] : 0;
    };
    prefetch(blockIdx.x);
    for (int u = blockIdx.x; u < p.n_units && !failed; u += gridDim.x) {
      const Unit w = w_next;
      int32_t idreg = id_next;  // lane l: id of own block l (32 at a time)
      prefetch(u + gridDim.x);
      if (is_k) {
        const int qb = iu & 1;
        if (!__all_sync(0xffffffffu, wait_l(bar(B_Q_EMPTY + qb), ((iu >> 1) & 1) ^ 1, abort, wlim))) {
          failed = true;
          break;
        }
        if (lane == 0) {
          // rows token * G + head of the unit's 16 query tokens: a 4-D box
          // {64, G, 1, 16} of q viewed as [nq][Hkv][G][d]
          mbar_arrive_expect_tx(bar(B_Q_FULL + qb), 2 * 16 * G * 128);
          for (int h = 0; h < 2; ++h)
            tma_load_4d(sbase + SM_Q + qb * 2 * kRHalf + h * kRHalf, &tm_q, bar(B_Q_FULL + qb), h * 64, 0, w.g,
                        w.q_first);
        }
        ++iu;
      }
      const int32_t* trow = p.table + static_cast<int64_t>(w.seq) * p.max_bps + w.n_shared;
      const int n_own_blocks = (w.own_len + 15) >> 4;
      for (int j = 0; j < w.n_tiles; ++j) {
        const int st = kt % kStages;
        if (!__all_sync(0xffffffffu, wait_l(bar(b_empty + st), ((kt / kStages) & 1) ^ 1, abort, wlim))) {
          failed = true;
          break;
        }
        const uint32_t dst = ring + st * 2 * kKHalf;
        ++kt;
        if (j + 1 == w.n_tiles) {
          // the query block's own keys: 16 rows of k_new / v_new for kv head g
          if (lane == 0) {
            mbar_arrive_expect_tx(bar(b_full + st), 2 * 2048);
            for (int h = 0; h < 2; ++h) tma_load_3d(dst + h * kKHalf, tmn, bar(b_full + st), h * 64, w.g, w.q_first);
          }
        } else {
          if (j > 0 && (j & 3) == 0) {
            const int bi = (j << 3) + lane;
            idreg = bi < n_own_blocks ? trow[bi] : 0;
          }
          const int nblk = min(8, (w.own_len - j * kTileKeys + 15) >> 4);
          const int32_t blk = __shfl_sync(0xffffffffu, idreg, ((j & 3) << 3) + (lane & 7));
          if (lane == 0) mbar_arrive_expect_tx(bar(b_full + st), nblk * 2 * 2048);
          __syncwarp();
          if (lane < nblk) {
            const int32_t row = (blk * p.Hkv + w.g) * 16;
            for (int h = 0; h < 2; ++h) tma_load_2d(dst + h * kKHalf + lane * 2048, tm, bar(b_full + st), h * 64, row);
          }
        }
      }
    }
    if (failed && lane == 0) raise_abort(abort, is_k ? 0x100 : 0x200);
    // every copy this warp issued has landed before the CTA may exit (a
    // no-op on the normal path, where the consumers waited for all of them)
    for (uint32_t k = kt > kStages ? kt - kStages : 0; k < kt; ++k)
      mbar_wait_drain(bar(b_full + k % kStages), (k / kStages) & 1);
    if (is_k)
      for (int i = iu > 2 ? iu - 2 : 0; i < iu; ++i) mbar_wait_drain(bar(B_Q_FULL + (i & 1)), (i >> 1) & 1);
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16_f32(128, kRows, false, false);  // K (K-major) x Q^T (K-major)
      constexpr uint32_t id_o = idesc_bf16_f32(128, kRows, true, false);   // V^T (MN-major) x P^T (K-major)
      uint32_t kt_s = 0, kt_p = 0;  // tiles whose S^T / P V have been issued
      int iu = 0;
      bool failed = false;
      auto issue_s = [&](uint32_t qaddr) -> bool {
        const int st = kt_s % kStages, sb = kt_s & 1;
        if (!wait_relaxed_l(bar(B_K_FULL + st), (kt_s / kStages) & 1, abort, wlim)) return false;
        if (!wait_relaxed_l(bar(B_S_FREE + sb), ((kt_s >> 1) & 1) ^ 1, abort, wlim)) return false;
        tc_fence_after();
        const uint64_t d_k = sdesc_sw128(sbase + SM_K + st * 2 * kKHalf, 16, 1024);
        const uint64_t d_q = sdesc_sw128(qaddr, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t ok = static_cast<uint64_t>(((kk >> 2) * kKHalf + (kk & 3) * 32) >> 4);
          const uint64_t oq = static_cast<uint64_t>(((kk >> 2) * kRHalf + (kk & 3) * 32) >> 4);
          mma_bf16_ss(tmem + kTmemS + sb * kRows, d_k + ok, d_q + oq, id_s, kk > 0);
        }
        mma_commit(bar(B_S_FULL + sb));
        mma_commit(bar(B_K_EMPTY + st));
        ++kt_s;
        return true;
      };
      Unit w_next = load_unit(p, blockIdx.x);
      for (int u = blockIdx.x; u < p.n_units && !failed; u += gridDim.x, ++iu) {
        const Unit w = w_next;
        if (u + static_cast<int>(gridDim.x) < p.n_units) w_next = load_unit(p, u + gridDim.x);
        const int qb = iu & 1, ob = iu & 1;
        if (!wait_relaxed_l(bar(B_Q_FULL + qb), (iu >> 1) & 1, abort, wlim)) { failed = true; break; }
        const uint32_t qaddr = sbase + SM_Q + qb * 2 * kRHalf;
        if (!issue_s(qaddr)) { failed = true; break; }
        for (int j = 0; j < w.n_tiles; ++j) {
          if (j + 1 < w.n_tiles) {
            if (!issue_s(qaddr)) { failed = true; break; }
          } else {
            mma_commit(bar(B_Q_EMPTY + qb));  // every S^T of the unit is issued
          }
          const int st = kt_p % kStages, pb = kt_p & 1;
          if (!wait_relaxed_l(bar(B_V_FULL + st), (kt_p / kStages) & 1, abort, wlim) ||
              !wait_relaxed_l(bar(B_P_FULL + pb), (kt_p >> 1) & 1, abort, wlim) ||
              (j == 0 && !wait_relaxed_l(bar(B_O_FREE + ob), ((iu >> 1) & 1) ^ 1, abort, wlim))) {
            failed = true;
            break;
          }
          tc_fence_after();
          const uint64_t d_v = sdesc_sw128(sbase + SM_V + st * 2 * kKHalf, kKHalf, 1024);
          const uint64_t d_p = sdesc_sw128(sbase + SM_P + pb * 2 * kRHalf, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t ov = static_cast<uint64_t>((kk * 2048) >> 4);
            const uint64_t op = static_cast<uint64_t>(((kk >> 2) * kRHalf + (kk & 3) * 32) >> 4);
            mma_bf16_ss(tmem + kTmemO + ob * kRows, d_v + ov, d_p + op, id_o, (j > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(bar(B_P_FREE + pb));
          mma_commit(bar(B_V_EMPTY + st));
          ++kt_p;
        }
        if (failed) break;
        mma_commit(bar(B_O_FULL + ob));
      }
      if (failed) raise_abort(abort, 0x400);
      // every product issued has completed before TMEM is released
      mma_commit(bar(B_DRAIN));
      mbar_wait_drain(bar(B_DRAIN), 0);
    }
  } else if (warp == 11) {
    // ------------------------------------------------------------ row data
    // lane r < rows: the combined prefix LSE of row r and where its first
    // partial row is, one or two units ahead of the softmax warps (which
    // start a unit's row maxima at the prefix LSE and merge in its epilogue)
    int iu = 0;
    bool failed = false;
    for (int u = blockIdx.x; u < p.n_units && !failed; u += gridDim.x, ++iu) {
      const Unit w = load_unit(p, u);
      const DecPage pg = p.pages[w.page];
      const int rb = iu & 1;
      if (!__all_sync(0xffffffffu, wait_l(bar(B_ROW_FREE + rb), ((iu >> 1) & 1) ^ 1, abort, wlim))) {
        failed = true;
        break;
      }
      if (lane < w.rows) {
        const int r = lane;
        const int R = (w.q_in_page + (r >> gsh)) * G + (r & gsh);
        const int ptile = R / kTileRows, prr = R % kTileRows;
        // log2 of the prefix mass of each chunk: a first pass for the
        // maximum, a second for the sum (the chunks' LSE reads hit L1)
        auto chunk_l2 = [&](int c, int64_t* prow_out) {
          const DecItem it = p.items[pg.item_base + ptile * pg.n_chunks + c];
          const int64_t prow = static_cast<int64_t>(it.row_base) + static_cast<int64_t>(w.g) * it.rows + prr;
          if (prow_out) *prow_out = prow;
          return p.part_lse[prow] * kLog2e;
        };
        float M = -INFINITY, l0 = -INFINITY;
        int64_t prow0 = 0;
        for (int c = 0; c < pg.n_chunks; ++c) {
          const float l2 = chunk_l2(c, c == 0 ? &prow0 : nullptr);
          if (c == 0) l0 = l2;
          M = fmaxf(M, l2);
        }
        float S = 0.f;
        for (int c = 0; c < pg.n_chunks; ++c) S += fast_exp2((c == 0 ? l0 : chunk_l2(c, nullptr)) - M);
        const float lpre = S > 0.f ? M + __log2f(S) : -INFINITY;
        row_lpre(rb)[r] = lpre;
        row_prow(rb)[r] = static_cast<int32_t>(prow0);
        row_share(rb)[r] = pg.n_chunks > 0 ? fast_exp2(l0 - lpre) : 0.f;
        if (pg.n_chunks > 0) {
          // the epilogue stages this 512-byte partial row: bring it to L2 now
          const char* row = reinterpret_cast<const char*>(p.part_o + prow0 * kHeadDim);
          for (int k = 0; k < 4; ++k) asm volatile("prefetch.global.L2 [%0];" ::"l"(row + k * 128));
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_ROW_FULL + rb));
    }
    if (failed && lane == 0) raise_abort(abort, 0x1000);
  } else {
    // ------------------------------------------------------------ softmax + epilogue (warps 0-7)
    // The four warps of a row half meet at their named barrier (votes and
    // reductions), so a failed wait in one warp is shared through a vote
    // and all four leave together; a warp never waits alone at a barrier
    // the others have left.
    const int qd = warp & 3, hf = warp >> 2;
    const int t = qd * 32 + lane;  // key of the tile (S^T lane) / head dim (O^T lane)
    const int r0 = hf * kHalfRows;  // this warp's rows: r0 .. r0 + 15
    const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
    float* red_h = red + hf * 64;  // [4 quadrants][16 rows] of this half
    uint32_t kt = 0;
    int iu = 0;
    bool failed = false;
    // the next unit's branch, page and draft-tree masks (lane i: query token
    // i), read during the current unit's epilogue
    Unit w_next{};
    DecPage pg_next{};
    uint32_t mine_next = 0;
    auto prefetch = [&](int un) {
      if (un >= p.n_units) return;
      w_next = load_unit(p, un);
      pg_next = p.pages[w_next.page];
      mine_next = 0;
      if (lane < w_next.q_len)
        mine_next = p.tree_bits ? static_cast<uint32_t>(p.tree_bits[w_next.q_first + lane]) : ((2u << lane) - 1u);
    };
    prefetch(blockIdx.x);
    for (int u = blockIdx.x; u < p.n_units && !failed; u += gridDim.x, ++iu) {
      const Unit w = w_next;
      const DecPage pg = pg_next;
      const int ob = iu & 1, rb = iu & 1;
      // bit i: row r0 + i of the unit exists
      const uint32_t my_rows = w.rows - r0 >= 16 ? 0xffffu : (w.rows > r0 ? (1u << (w.rows - r0)) - 1u : 0u);
      const bool ok_r = __all_sync(0xffffffffu, wait_l(bar(B_ROW_FULL + rb), (iu >> 1) & 1, abort, wlim));
      if (bar_or_all(!ok_r)) {
        failed = true;
        break;
      }
      // Row maxima start at the prefix side's LSE: usually above every own
      // score, so the first tile needs no reduction, while P = 2^(x - m)
      // stays within bf16 range (a row far below it contributes nothing
      // visible next to the prefix).
      float m_ref[kHalfRows], l_part[kHalfRows];
#pragma unroll
      for (int i = 0; i < kHalfRows; ++i) {
        m_ref[i] = ((my_rows >> i) & 1u) ? row_lpre(rb)[r0 + i] : -INFINITY;
        l_part[i] = 0.f;
      }
      // bit i: row r0 + i's query token sees key t of the query block
      uint32_t qblock_rows = 0;
      {
        const uint32_t mine = mine_next;  // lane j < q_len: the mask of query token j
        uint32_t vis = 0;                 // bit j: query token j sees key token t
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const uint32_t b = __shfl_sync(0xffffffffu, mine, j);
          if (t < 16) vis |= ((b >> t) & 1u) << j;
        }
        vis &= (1u << w.q_len) - 1u;
        for (int i = 0; i < kHalfRows; ++i) qblock_rows |= ((vis >> ((r0 + i) >> gsh)) & 1u) << i;
        qblock_rows &= my_rows;
      }
      for (int j = 0; j < w.n_tiles; ++j, ++kt) {
        const int sb = kt & 1;
        // a failed wait here is voted on with the P buffer's below (reading
        // an unfinished S^T only gives values that are thrown away)
        const bool ok_s = __all_sync(0xffffffffu, wait_relaxed_l(bar(B_S_FULL + sb), (kt >> 1) & 1, abort, wlim));
        tc_fence_after();
        float x[kHalfRows];
        {
          uint32_t v[16];
          tmem_ld16(tmem + lane_base + kTmemS + sb * kRows + r0, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < kHalfRows; ++i) x[i] = __uint_as_float(v[i]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_S_FREE + sb));
        // scores in log2 units; keys and rows this unit may not use are -inf
        const bool qblock = j + 1 == w.n_tiles;
        const uint32_t okm = qblock ? qblock_rows : (j * kTileKeys + t < w.own_len ? my_rows : 0u);
        bool grow = false;
#pragma unroll
        for (int i = 0; i < kHalfRows; ++i) {
          x[i] = ((okm >> i) & 1u) ? x[i] * p.sl2 : -INFINITY;
          grow |= x[i] > m_ref[i] + kRescaleThreshold;
        }
        bool late = false;  // a wait in the rescale below gave up: voted on with the next one
        if (bar_or_half(hf, grow)) {
          // exact row maxima of this tile; the rows that grew by more than
          // the threshold move their reference and rescale their sums
          float v[kHalfRows];
#pragma unroll
          for (int i = 0; i < kHalfRows; ++i) v[i] = x[i];
          const float mx = warp_rows_reduce16<true>(v, lane);
          if (lane < 16) red_h[qd * 16 + lane] = mx;
          bar_sync_half(hf);
          float alpha[kHalfRows];
          bool any_rescale = false;
#pragma unroll
          for (int i = 0; i < kHalfRows; ++i) {
            const float mt = fmaxf(fmaxf(red_h[i], red_h[16 + i]), fmaxf(red_h[32 + i], red_h[48 + i]));
            alpha[i] = 1.f;
            if (mt > m_ref[i] + kRescaleThreshold) {
              alpha[i] = fast_exp2(m_ref[i] - mt);  // 0 while m_ref is -inf
              any_rescale |= m_ref[i] != -INFINITY;
              m_ref[i] = mt;
            }
            l_part[i] *= alpha[i];
          }
          bar_sync_half(hf);  // red may be overwritten from here on
          if (j > 0 && any_rescale) {
            // O^T (lane t = head dim t) holds sums against the old maxima:
            // rescale this half's columns once P V of the previous tile ran
            const uint32_t q = kt - 1;
            late = !__all_sync(0xffffffffu, wait_relaxed_l(bar(B_P_FREE + (q & 1)), (q >> 1) & 1, abort, wlim));
          }
          if (j > 0 && any_rescale && !late) {
            tc_fence_after();
            uint32_t v2[16];
            tmem_ld16(tmem + lane_base + kTmemO + ob * kRows + r0, v2);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < kHalfRows; ++i) v2[i] = __float_as_uint(__uint_as_float(v2[i]) * alpha[i]);
            asm volatile(
                "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
                    tmem + lane_base + kTmemO + ob * kRows + r0),
                "r"(v2[0]), "r"(v2[1]), "r"(v2[2]), "r"(v2[3]), "r"(v2[4]), "r"(v2[5]), "r"(v2[6]), "r"(v2[7]),
                "r"(v2[8]), "r"(v2[9]), "r"(v2[10]), "r"(v2[11]), "r"(v2[12]), "r"(v2[13]), "r"(v2[14]), "r"(v2[15])
                : "memory");
            tmem_wait_st();
          }
        }
        // P = exp2(x - m_ref) into shared memory as P[row][key] (bf16,
        // K-major with the 128-byte swizzle), once P V two tiles back has
        // released the buffer
        const bool ok_p =
            kt < 2 || __all_sync(0xffffffffu, wait_relaxed_l(bar(B_P_FREE + sb), ((kt >> 1) & 1) ^ 1, abort, wlim));
        if (bar_or_all(!ok_s || !ok_p || late)) {
          failed = true;
          break;
        }
        const uint32_t pbase = sbase + SM_P + sb * 2 * kRHalf + (t >> 6) * kRHalf + (t & 7) * 2;
        const uint32_t chunk = (t & 63) >> 3;
#pragma unroll
        for (int i = 0; i < kHalfRows; ++i) {
          const int r = r0 + i;
          const float mu = m_ref[i] == -INFINITY ? 0.f : m_ref[i];
          const float pr = fast_exp2(x[i] - mu);
          l_part[i] += pr;
          const __nv_bfloat16 hb = __float2bfloat16_rn(pr);
          st_shared_u16(pbase + r * 128 + ((chunk ^ (r & 7)) << 4), *reinterpret_cast<const uint16_t*>(&hb));
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_P_FULL + sb));
      }
      if (failed) break;

      // ---------------------------------------------------------- epilogue
      // Runtime loops keep this code small: it runs once per unit, and
      // instruction fetches of big unrolled blocks cost.  Each row half
      // handles its own rows.
      prefetch(u + gridDim.x);
      const bool ok_e = __all_sync(0xffffffffu, wait_relaxed_l(bar(B_O_FULL + ob), (iu >> 1) & 1, abort, wlim));
      if (bar_or_all(!ok_e)) {
        failed = true;
        break;
      }
      tc_fence_after();
      const float* lpre = row_lpre(rb);
      const int32_t* prow0 = row_prow(rb);
      const float* share0 = row_share(rb);
      const int nr = max(0, min(kHalfRows, w.rows - r0));  // rows of this half
      // (a) the unit's P V have all run, so the P buffers are free: stage the
      // first chunk's partial rows there (row r at +512 r), one round trip
      float* stage = reinterpret_cast<float*>(smem + SM_P);
      const int tq = qd * 32 + lane;  // 0..127 within the half
      if (pg.n_chunks > 0) {
        for (int i = tq; i < nr * 32; i += 128) {
          const int r = r0 + (i >> 5), part = i & 31;
          const float* src = p.part_o + static_cast<int64_t>(prow0[r]) * kHeadDim + part * 4;
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(stage + r * 128 + part * 4)),
                       "l"(src)
                       : "memory");
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
      }
      // (b) row sums over the 128 key lanes; warp qd 0 publishes the maxima
      {
        float v[kHalfRows];
#pragma unroll
        for (int i = 0; i < kHalfRows; ++i) v[i] = l_part[i];
        const float sm = warp_rows_reduce16<false>(v, lane);
        if (lane < 16) red_h[qd * 16 + lane] = sm;
      }
      if (qd == 0 && lane == 0) {
#pragma unroll
        for (int i = 0; i < kHalfRows; ++i) row_m[r0 + i] = m_ref[i];
      }
      bar_sync_half(hf);
      // (c) lane i of warp qd 0: the weights of row r0 + i's own and prefix
      // sides, O = w_own O_own (unnormalised sums) + w_pre sum_c share_c o_c,
      // and its LSE; lane i alone reads red_h[. + i], so the weights reuse it
      float* row_wo = red_h;
      float* row_wp = red_h + 16;
      if (qd == 0 && lane < nr) {
        const int i = lane, r = r0 + i;
        const float lo = (red_h[i] + red_h[16 + i]) + (red_h[32 + i] + red_h[48 + i]);
        const float lp = lpre[r];
        const float own2 = lo > 0.f ? row_m[r] + __log2f(lo) : -INFINITY;  // own mass, log2
        const float M = fmaxf(own2, lp);
        const float Mu = M == -INFINITY ? 0.f : M;
        const float eo = lo > 0.f ? fast_exp2(own2 - Mu) : 0.f, ep = lp == -INFINITY ? 0.f : fast_exp2(lp - Mu);
        const float L = eo + ep;
        const float inv = L > 0.f ? 1.f / L : 0.f;
        row_wo[i] = lo > 0.f ? eo / lo * inv : 0.f;
        row_wp[i] = ep * inv;
        const int64_t qh = static_cast<int64_t>(w.q_first + (r >> gsh)) * p.Hq + w.g * G + (r & gsh);
        p.lse[qh] = L > 0.f ? (Mu + __log2f(L)) * kLn2 : -INFINITY;
      }
      asm volatile("cp.async.wait_all;" ::: "memory");
      bar_sync_half(hf);
      // (d) thread t = head dim t: this half's 16 O^T columns at once
      uint32_t ov[16];
      tmem_ld16(tmem + lane_base + kTmemO + ob * kRows + r0, ov);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_O_FREE + ob));
      // combine in the staging area (this thread's own slots), then further
      // prefix chunks (pages whose prefix the plan split; read row by row),
      // then the rows out as bf16
      const bool has_pre = pg.n_chunks > 0;
#pragma unroll
      for (int i = 0; i < kHalfRows; ++i) {
        if (i < nr) {
          const int r = r0 + i;
          const float own = __uint_as_float(ov[i]) * row_wo[i];
          stage[r * 128 + t] = has_pre ? fmaf(stage[r * 128 + t], row_wp[i] * share0[r], own) : own;
        }
      }
      for (int c = 1; c < pg.n_chunks; ++c) {
        for (int i = 0; i < nr; ++i) {
          const int r = r0 + i;
          const int R = (w.q_in_page + (r >> gsh)) * G + (r & gsh);
          const DecItem it = p.items[pg.item_base + (R / kTileRows) * pg.n_chunks + c];
          const int64_t prow = static_cast<int64_t>(it.row_base) + static_cast<int64_t>(w.g) * it.rows + R % kTileRows;
          const float share = fast_exp2(p.part_lse[prow] * kLog2e - lpre[r]);
          stage[r * 128 + t] = fmaf(p.part_o[prow * kHeadDim + t], row_wp[i] * share, stage[r * 128 + t]);
        }
      }
      {
        __nv_bfloat16* dst = p.o + (static_cast<int64_t>(w.q_first) * p.Hq + w.g * G) * kHeadDim + t;
        for (int i = 0; i < nr; ++i) {
          const int r = r0 + i;
          dst[((r >> gsh) * p.Hq + (r & gsh)) * kHeadDim] = __float2bfloat16_rn(stage[r * 128 + t]);
        }
      }
      // this half's staging rows and red are free again for the next unit
      bar_sync_half(hf);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_ROW_FREE + rb));  // this warp is done with the unit's row data
    }
    if (failed && lane == 0) raise_abort(abort, 0x800);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
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

}  // namespace

int launch_decode_own_kmajor(const DecodeArgs& a, cudaStream_t s, std::string* err) {
  if (a.n_branches == 0) return PADOC_OK;
  if (a.group > 2) {
    *err = "keys-major own pass: Hq/Hkv must be 1 or 2";
    return PADOC_ERR_UNSUPPORTED;
  }
  EncodeTiledFn enc = get_encode_fn(err);
  if (!enc) return PADOC_ERR_CUDA;
  CUtensorMap mq, mk, mv, mkn, mvn;
  // q viewed as [nq][Hkv][G][d]; box {64, G, 1, 16}: 16 query tokens of one
  // kv head's group, rows token * G + head
  const cuuint64_t dq[4] = {128, static_cast<cuuint64_t>(a.group), static_cast<cuuint64_t>(a.Hkv),
                            static_cast<cuuint64_t>(a.nq)};
  const cuuint64_t sq[3] = {256, static_cast<cuuint64_t>(a.group) * 256, static_cast<cuuint64_t>(a.Hq) * 256};
  const cuuint32_t bq[4] = {64, static_cast<cuuint32_t>(a.group), 1, 16};
  const cuuint64_t dk[2] = {128, static_cast<cuuint64_t>(a.num_blocks) * a.Hkv * 16};
  const cuuint64_t sk[1] = {256};
  const cuuint32_t bk[2] = {64, 16};
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
  p.n_units = a.n_branches * a.Hkv;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.group = a.group;
  p.sl2 = a.scale * kLog2e;
  p.pages = a.pages;
  p.items = a.items;
  p.branches = a.branches;
  p.table = a.table;
  p.max_bps = a.max_bps;
  p.tree_bits = a.tree_bits;
  p.part_o = a.part_o;
  p.part_lse = a.part_lse;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(own_kmajor_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) {
      *err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
      return PADOC_ERR_CUDA;
    }
    attr_set = true;
  }
  const int grid = std::min(p.n_units, num_sms());
  own_kmajor_kernel<<<grid, kThreads, kSmemBytes, s>>>(mq, mk, mv, mkn, mvn, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *err = std::string("own pass launch: ") + cudaGetErrorString(e);
    return PADOC_ERR_CUDA;
  }
  return PADOC_OK;
}

}  // namespace padoc

extern "C" int padoc_debug_set_wait_limit(uint64_t ns) {
  const unsigned long long v = ns ? ns : padoc::ptx::kWaitLimitNs;
  const cudaError_t e = cudaMemcpyToSymbol(padoc::g_own_wait_limit_ns, &v, sizeof(v));
  if (e != cudaSuccess)
    return padoc::set_error(PADOC_ERR_CUDA, "debug_set_wait_limit: %s", cudaGetErrorString(e));
  return PADOC_OK;
}

namespace padoc {

int read_and_clear_own_error(cudaStream_t s, unsigned* word) {
  unsigned zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(word, g_own_err, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpyToSymbolAsync(g_own_err, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e == cudaSuccess ? PADOC_OK : PADOC_ERR_CUDA;
}

}  // namespace padoc
