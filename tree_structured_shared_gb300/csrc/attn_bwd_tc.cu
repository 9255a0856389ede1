// Tensor-core backward of the tree-varlen forward (tcgen05 + TMEM + TMA).
//
// The gradients of sum(dO * O) through each token's softmax over its
// ancestor set (PaDoc, "Training paradigm": the model trains through the
// same ancestor-masked attention) are split into two persistent kernels
// that both recompute the probabilities from the forward's LSE:
//
//   bwd_dq_kernel   query-stationary, the forward's work units (128 rows =
//                   query tokens x heads of one GQA group) and key-tile walk:
//                     S = Q K^T, dP = dO V^T            (tensor cores)
//                     dS = P (dP - D), P = exp(S - LSE)  (warps 0-3, row = lane)
//                     dQ += dS K                         (tensor cores, A = dS in TMEM)
//   bwd_dkv_kernel  key-stationary over the transposed segment lists: a CTA
//                   keeps one 128-key tile of K and V and walks the query
//                   tiles that see it:
//                     S^T = K Q^T, dP^T = V dO^T         (tensor cores)
//                     P^T, dS^T                          (warps 0-3, key = lane)
//                     dV += P^T dO, dK += dS^T Q         (tensor cores, A in TMEM)
// Neither kernel needs atomics: every output row belongs to one unit.
//
// Roles (320 threads): warps 0-7 element-wise work and epilogue (two
// warpgroups; warp w reads TMEM lanes 32 (w % 4) .. + 31, warpgroup w / 4
// takes one half of the tile's columns), warp 8 TMA producer, warp 9 MMA
// issuer (one thread).  The MMA thread starts the products of a column half
// as soon as that half's warpgroup is done with it.  Every wait is bounded; a timed
// out wait raises the CTA abort flag and this file's device error word.
#include <cuda_bf16.h>

#include <algorithm>
#include <string>

#include "../../include/padoc.h"
#include "padoc_internal.h"
#include "ptx_sm103.cuh"

namespace padoc {

__device__ unsigned int g_bwd_err;

namespace {

using namespace ptx;

constexpr int kThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kHalf = 16384;  // one 64-column half of a 128-row bf16 tile
constexpr int kTile = 2 * kHalf;
constexpr float kLog2e = 1.44269504088896340736f;

// Descriptors of the 16-wide K steps of a 128-byte-swizzled tile, as
// offsets from the tile's base descriptor (the start address field holds the
// address / 16, and no step carries out of it): K-major operands step 32
// bytes inside a 64-column half and then to the other half; MN-major
// operands step 16 rows of 128 bytes.
__device__ __forceinline__ uint64_t kmajor_step(uint64_t base, int kk) {
  return base + static_cast<uint64_t>(((kk >> 2) * kHalf + (kk & 3) * 32) >> 4);
}
__device__ __forceinline__ uint64_t mnmajor_step(uint64_t base, int kk) {
  return base + static_cast<uint64_t>(kk * (2048 >> 4));
}

__device__ __forceinline__ void raise_abort(volatile int* abort, unsigned site) {
  *abort = 1;
  atomicOr(&g_bwd_err, site);
}

struct DqParams {
  FwdPlan plan;
  int n_units;
  int32_t Hq, Hkv, group;
  int64_t T;
  float sl2, scale;
  const float* lse;
  const float* delta;
  __nv_bfloat16* dq;
  int32_t* work;  // unit counter, zero at launch
};

struct DkvParams {
  BwdPlan plan;
  int n_units;
  int32_t Hq, Hkv, group, tile_tokens;
  int64_t T;
  float sl2, scale;
  const float* lse;
  const float* delta;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int32_t* work;  // unit counter, zero at launch
};

// Both passes draw their units in order from a counter in the workspace as
// CTAs free up: the producer draws the next unit once the current one's
// copies are issued and publishes it in a ring of kURing slots after the
// barriers; the MMA thread and the element-wise warps read it there.
constexpr int kURing = 4;

// The next unit of a role that reads the ring (`single`: one thread runs
// the role; full / empty: the slots' barrier indices); false when a wait
// gave up.
__device__ __forceinline__ bool take_unit(uint32_t& k, int& u, volatile int32_t* uring, uint64_t* bars, int full,
                                          int empty, volatile int* abort, bool single) {
  const int slot = k % kURing;
  const bool ok = mbar_wait(smem_u32(&bars[full + slot]), (k / kURing) & 1, abort);
  if (single ? !ok : !__all_sync(0xffffffffu, ok)) return false;
  u = uring[slot];
  if (!single) __syncwarp();
  if (single || (threadIdx.x & 31) == 0) mbar_arrive(smem_u32(&bars[empty + slot]));
  ++k;
  return true;
}

// ============================================================ dQ pass
// smem: Q | dO | K ring (3) | V ring (2) | barriers
constexpr int Q_SM_Q = 0;
constexpr int Q_SM_DO = kTile;
// K is read by S (early in a tile's period) and by dQ (late), V only by dP:
// a three-stage K ring and a two-stage V ring whose stage frees after dP
// give both a tile's lead over their L2 fetch.
constexpr int kDqKStages = 3, kDqVStages = 2;
constexpr int Q_SM_K = 2 * kTile;
constexpr int Q_SM_V = Q_SM_K + kDqKStages * kTile;
constexpr int Q_SM_BAR = Q_SM_V + kDqVStages * kTile;
constexpr int kDqSmem = Q_SM_BAR + 256 + 1024;
// TMEM columns
constexpr uint32_t Q_T_S = 0, Q_T_DP = 128, Q_T_DS = 256, Q_T_DQ = 384;
enum {
  QB_QD_FULL = 0,
  QB_QD_EMPTY = 1,
  QB_K_FULL = 2,    // +K stage (3): K and V of the tile have landed
  QB_K_EMPTY = 5,   // +stage (3): the tile's dQ has run
  QB_V_EMPTY = 10,  // +stage (2): the tile's dP has run
  QB_SP_FULL = 12,  // S and dP of the tile are in TMEM
  QB_RD = 13,       // count 8: both warpgroups have read them (the columns are free)
  QB_DS_FULL = 14,  // count 8: dS of the tile is in TMEM (both warpgroups)
  QB_DQ_DONE = 16,  // dQ += dS K of the tile has run (the dS columns are free)
  QB_DQ_ALL = 18,   // the unit's dQ is complete
  QB_ACC_FREE = 19,  // count 8: the epilogue has read dQ
  QB_UNIT_FULL = 20,   // +slot (4): the unit ring's slot holds the next unit
  QB_UNIT_EMPTY = 24,  // +slot (4), count 9: the MMA thread and the element-wise warps read it
  QB_N = 28  // slots 8-9, 15 and 17 are unused
};
constexpr int Q_SM_URING = Q_SM_BAR + 240;
static_assert(QB_N * 8 + 8 <= 240, "dQ barrier area");
static_assert(kDqSmem <= 232448, "dQ pass shared memory");

struct DqUnit {
  int32_t g, tile_start, q_end, kv_first, kv_count, tile_last, n_tiles;
  KVSeg kv0;
};

// One record per unit: the plan item carries its query segment's fields,
// its first key segment and its key-tile count.
__device__ __forceinline__ DqUnit dq_unit(const DqParams& p, int u) {
  DqUnit w;
  // head-major: the CTAs at work at one time share one kv head's K/V
  w.g = u / p.plan.n_items;
  const FwdItem it = p.plan.items[u % p.plan.n_items];
  w.tile_start = it.tile_start;
  w.q_end = it.q_end;
  w.kv_first = it.kv_first;
  w.kv_count = it.kv_count;
  w.tile_last = it.tile_last;
  w.n_tiles = it.n_tiles;
  w.kv0 = it.kv0;
  return w;
}

// Key tiles of a dQ unit: each key segment in 128-key steps, causal
// segments cut after the unit's last query.  The next segment's descriptor
// is loaded on entering a segment (t.nx).
struct KeyIter {
  int32_t s, ks, end, causal;
  KVSeg nx;
};
__device__ __forceinline__ bool key_setup(const DqParams& p, const DqUnit& w, KeyIter& t) {
  while (t.s < w.kv_first + w.kv_count) {
    const KVSeg kv = t.nx;
    if (t.s + 1 < w.kv_first + w.kv_count) t.nx = p.plan.kvsegs[t.s + 1];
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
__device__ __forceinline__ bool key_begin(const DqParams& p, const DqUnit& w, KeyIter& t) {
  t.s = w.kv_first;
  t.nx = w.kv0;
  return key_setup(p, w, t);
}
__device__ __forceinline__ bool key_next(const DqParams& p, const DqUnit& w, KeyIter& t) {
  t.ks += kTileKeys;
  if (t.ks < t.end) return true;
  ++t.s;
  return key_setup(p, w, t);
}
__device__ __forceinline__ int key_count(const DqParams&, const DqUnit& w) { return w.n_tiles; }

__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const DqParams p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base; offsetting the shared array itself keeps the
  // compiler aware that every pointer below is a shared-memory pointer
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Q_SM_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Q_SM_BAR + QB_N * 8);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + Q_SM_BAR + QB_N * 8 + 4);
  volatile int32_t* uring = reinterpret_cast<volatile int32_t*>(smem + Q_SM_URING);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  if (threadIdx.x == 0) {
    for (int i = 0; i < QB_N; ++i)
      mbar_init(bar(i), (i == QB_DS_FULL || i == QB_ACC_FREE || i == QB_RD)
                            ? 8u
                            : ((i >= QB_UNIT_EMPTY && i < QB_UNIT_EMPTY + kURing) ? 9u : 1u));
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int G = p.group, tt = p.plan.tile_tokens;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      uint32_t kv_it = 0, unit_it = 0;
      bool failed = false;
      // draw a unit and publish it in the ring (-1 when a wait gave up)
      uint32_t n_pub = 0;
      auto publish = [&]() -> int {
        const int slot = n_pub % kURing;
        if (!mbar_wait(bar(QB_UNIT_EMPTY + slot), ((n_pub / kURing) & 1) ^ 1, abort)) return -1;
        const int v = atomicAdd(p.work, 1);
        uring[slot] = v;
        mbar_arrive(bar(QB_UNIT_FULL + slot));
        ++n_pub;
        return v;
      };
      int u_next = publish();
      if (u_next < 0) failed = true;
      while (!failed) {
        const int u = u_next;
        if (u >= p.n_units) break;
        const DqUnit w = dq_unit(p, u);
        if (key_count(p, w) == 0) {
          u_next = publish();
          if (u_next < 0) failed = true;
          continue;
        }
        if (!mbar_wait(bar(QB_QD_EMPTY), (unit_it & 1) ^ 1, abort)) { failed = true; break; }
        mbar_arrive_expect_tx(bar(QB_QD_FULL), 2 * kTile);
        for (int hh = 0; hh < G; ++hh)
          for (int h = 0; h < 2; ++h) {
            tma_load_3d(sbase + Q_SM_Q + h * kHalf + hh * tt * 128, &tm_q, bar(QB_QD_FULL), h * 64, w.g * G + hh,
                        w.tile_start);
            tma_load_3d(sbase + Q_SM_DO + h * kHalf + hh * tt * 128, &tm_do, bar(QB_QD_FULL), h * 64, w.g * G + hh,
                        w.tile_start);
          }
        KeyIter t;
        for (bool ok = key_begin(p, w, t); ok; ok = key_next(p, w, t), ++kv_it) {
          const int ks = kv_it % kDqKStages, vs = kv_it % kDqVStages;
          // K and V of a tile land on one barrier (one wait for the MMA
          // thread); a V stage frees (after dP) before the K stage of the
          // same tile (after dQ of the tile before)
          if (!mbar_wait(bar(QB_K_EMPTY + ks), ((kv_it / kDqKStages) & 1) ^ 1, abort)) { failed = true; break; }
          if (!mbar_wait(bar(QB_V_EMPTY + vs), ((kv_it / kDqVStages) & 1) ^ 1, abort)) { failed = true; break; }
          mbar_arrive_expect_tx(bar(QB_K_FULL + ks), 2 * kTile);
          for (int h = 0; h < 2; ++h)
            tma_load_3d(sbase + Q_SM_K + ks * kTile + h * kHalf, &tm_k, bar(QB_K_FULL + ks), h * 64, w.g, t.ks);
          for (int h = 0; h < 2; ++h)
            tma_load_3d(sbase + Q_SM_V + vs * kTile + h * kHalf, &tm_v, bar(QB_K_FULL + ks), h * 64, w.g, t.ks);
        }
        if (failed) break;
        u_next = publish();
        if (u_next < 0) {
          failed = true;
          break;
        }
        ++unit_it;
      }
      if (failed) raise_abort(abort, 0x10);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_kk = idesc_bf16_f32(128, 128, false, false);  // both K-major
      constexpr uint32_t id_mn = idesc_bf16_f32(128, 128, false, true);   // B MN-major
      uint32_t kv_it = 0, g_it = 0, unit_it = 0;
      bool failed = false;
      // base descriptors: Q and dO (K-major), K and V of each stage (K-major), K as MN-major B
      const uint64_t d_q = sdesc_sw128(sbase + Q_SM_Q, 16, 1024), d_do = sdesc_sw128(sbase + Q_SM_DO, 16, 1024);
      const uint64_t d_k0 = sdesc_sw128(sbase + Q_SM_K, 16, 1024), d_k1 = sdesc_sw128(sbase + Q_SM_K + kTile, 16, 1024),
                     d_k2 = sdesc_sw128(sbase + Q_SM_K + 2 * kTile, 16, 1024);
      const uint64_t d_v0 = sdesc_sw128(sbase + Q_SM_V, 16, 1024), d_v1 = sdesc_sw128(sbase + Q_SM_V + kTile, 16, 1024);
      const uint64_t d_kmn0 = sdesc_sw128(sbase + Q_SM_K, kHalf, 1024);
      const uint64_t d_kmn1 = sdesc_sw128(sbase + Q_SM_K + kTile, kHalf, 1024);
      const uint64_t d_kmn2 = sdesc_sw128(sbase + Q_SM_K + 2 * kTile, kHalf, 1024);
      auto issue_dq = [&](uint32_t tile_it, bool first, bool last) -> bool {
        // dQ += dS K for tile tile_it (dS in TMEM, K of its stage as MN-major
        // B).  One wait and one commit for the whole tile: every wait, fence
        // and commit between MMA groups leaves the pipe idle once the few
        // queued MMAs have run, and both warpgroups finish dS together.
        if (first && !mbar_wait_relaxed(bar(QB_ACC_FREE), (unit_it & 1) ^ 1, abort)) return false;
        const int st = tile_it % kDqKStages;
        const uint64_t kd = st == 0 ? d_kmn0 : (st == 1 ? d_kmn1 : d_kmn2);
        if (!mbar_wait_relaxed(bar(QB_DS_FULL), tile_it & 1, abort)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16_ts(tmem + Q_T_DQ, tmem + Q_T_DS + kk * 8, mnmajor_step(kd, kk), id_mn,
                      (!first || kk > 0) ? 1u : 0u);
        mma_commit(bar(QB_DQ_DONE));
        mma_commit(bar(QB_K_EMPTY + st));
        if (last) mma_commit(bar(QB_DQ_ALL));
        return true;
      };
      uint32_t n_taken = 0;
      while (!failed) {
        int u;
        if (!take_unit(n_taken, u, uring, bars, QB_UNIT_FULL, QB_UNIT_EMPTY, abort, true)) {
          failed = true;
          break;
        }
        if (u >= p.n_units) break;
        const DqUnit w = dq_unit(p, u);
        const int n = key_count(p, w);
        if (n == 0) continue;
        if (!mbar_wait_relaxed(bar(QB_QD_FULL), unit_it & 1, abort)) { failed = true; break; }
        for (int j = 0; j < n; ++j, ++kv_it, ++g_it) {
          const int ks = kv_it % kDqKStages, vs = kv_it % kDqVStages;
          if (!mbar_wait_relaxed(bar(QB_K_FULL + ks), (kv_it / kDqKStages) & 1, abort)) { failed = true; break; }
          const uint64_t dk = ks == 0 ? d_k0 : (ks == 1 ? d_k1 : d_k2), dv = vs ? d_v1 : d_v0;
          // S and dP go over columns both warpgroups have read (they compute the
          // previous tile's dS from registers meanwhile)
          if (g_it > 0 && !mbar_wait_relaxed(bar(QB_RD), (g_it - 1) & 1, abort)) { failed = true; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16_ss(tmem + Q_T_S, kmajor_step(d_q, kk), kmajor_step(dk, kk), id_kk, kk > 0);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16_ss(tmem + Q_T_DP, kmajor_step(d_do, kk), kmajor_step(dv, kk), id_kk, kk > 0);
          mma_commit(bar(QB_SP_FULL));
          mma_commit(bar(QB_V_EMPTY + vs));  // dP has read V
          if (j == n - 1) mma_commit(bar(QB_QD_EMPTY));
          if (j > 0 && !issue_dq(g_it - 1, j == 1, false)) { failed = true; break; }
        }
        if (failed) break;
        if (!issue_dq(g_it - 1, n == 1, true)) { failed = true; break; }
        ++unit_it;
      }
      if (failed) raise_abort(abort, 0x20);
    }
  } else {
    // ------------------------------------------------------------ element-wise (warps 0-7)
    const int wg = warp >> 2;                    // column half of this warpgroup
    const int r = (warp & 3) * 32 + lane;        // query row == TMEM lane
    const uint32_t lb = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint32_t g_it = 0, unit_it = 0;
    bool failed = false;
    uint32_t n_taken = 0;
    while (!failed) {
      int u;
      if (!take_unit(n_taken, u, uring, bars, QB_UNIT_FULL, QB_UNIT_EMPTY, abort, false)) {
        failed = true;
        break;
      }
      if (u >= p.n_units) break;
      const DqUnit w = dq_unit(p, u);
      const int n = key_count(p, w);
      if (n == 0) continue;
      const int hh = r / tt;
      const int64_t qpos = w.tile_start + (r % tt);
      const bool valid = qpos < w.q_end;
      const int head = w.g * G + hh;
      const float lse2 = valid ? p.lse[static_cast<int64_t>(head) * p.T + qpos] * kLog2e : INFINITY;
      const float Dr = valid ? p.delta[static_cast<int64_t>(head) * p.T + qpos] : 0.f;
      KeyIter t;
      for (bool ok = key_begin(p, w, t); ok; ok = key_next(p, w, t), ++g_it) {
        if (!__all_sync(0xffffffffu, mbar_wait(bar(QB_SP_FULL), g_it & 1, abort))) { failed = true; break; }
        tc_fence_after();
        const int32_t klen = min(kTileKeys, t.end - t.ks);
        int32_t vis = valid ? klen : 0;
        if (t.causal) vis = min(vis, static_cast<int32_t>(qpos + 1 - t.ks));
        vis -= wg * 64;  // in this half's column numbering
        uint32_t sv[2][32], dv[2][32];
        tmem_ld32(tmem + lb + Q_T_S + wg * 64, sv[0]);
        tmem_ld32(tmem + lb + Q_T_DP + wg * 64, dv[0]);
        tmem_ld32(tmem + lb + Q_T_S + wg * 64 + 32, sv[1]);
        tmem_ld32(tmem + lb + Q_T_DP + wg * 64 + 32, dv[1]);
        tmem_wait_ld();
        // the half's S and dP columns may take the next tile's products now
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(QB_RD));
        uint32_t pk[32];
        const uint64_t sl2x2 = f2pack(p.sl2, p.sl2), negl2 = f2pack(-lse2, -lse2), d2 = f2pack(Dr, Dr);
        if (__all_sync(0xffffffffu, vis >= 64)) {  // no masked column in this half for the warp
#pragma unroll
          for (int c = 0; c < 2; ++c) {
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              // two lanes per instruction: x = s * sl2 - LSE2, P = 2^x, dS = P (dP - D)
              float x0, x1;
              f2unpack(fma2(f2pack(__uint_as_float(sv[c][i]), __uint_as_float(sv[c][i + 1])), sl2x2, negl2), x0, x1);
              const uint64_t ds = mul2(f2pack(fast_exp2(x0), fast_exp2(x1)),
                                       sub2(f2pack(__uint_as_float(dv[c][i]), __uint_as_float(dv[c][i + 1])), d2));
              float a, b;
              f2unpack(ds, a, b);
              pk[(c * 32 + i) >> 1] = pack_bf16x2(a, b);
            }
          }
        } else {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const int col = c * 32 + i;
              const float p0 = col < vis ? fast_exp2(fmaf(__uint_as_float(sv[c][i]), p.sl2, -lse2)) : 0.f;
              const float p1 = col + 1 < vis ? fast_exp2(fmaf(__uint_as_float(sv[c][i + 1]), p.sl2, -lse2)) : 0.f;
              pk[col >> 1] =
                  pack_bf16x2(p0 * (__uint_as_float(dv[c][i]) - Dr), p1 * (__uint_as_float(dv[c][i + 1]) - Dr));
            }
          }
        }
        // dS goes over the previous tile's dS once that tile's dQ has read it
        if (g_it > 0) {
          if (!__all_sync(0xffffffffu, mbar_wait(bar(QB_DQ_DONE), (g_it - 1) & 1, abort))) { failed = true; break; }
          tc_fence_after();
        }
        tmem_st32(tmem + lb + Q_T_DS + wg * 32, pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(QB_DS_FULL));
      }
      if (failed) break;
      // epilogue: this warpgroup's half of the row's dQ
      if (!__all_sync(0xffffffffu, mbar_wait(bar(QB_DQ_ALL), unit_it & 1, abort))) { failed = true; break; }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lb + Q_T_DQ + wg * 64 + c * 32, v);
        tmem_wait_ld();
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(p.dq + (qpos * p.Hq + head) * kHeadDim + wg * 64 + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * i + 0]) * p.scale, __uint_as_float(v[8 * i + 1]) * p.scale),
                                pack_bf16x2(__uint_as_float(v[8 * i + 2]) * p.scale, __uint_as_float(v[8 * i + 3]) * p.scale),
                                pack_bf16x2(__uint_as_float(v[8 * i + 4]) * p.scale, __uint_as_float(v[8 * i + 5]) * p.scale),
                                pack_bf16x2(__uint_as_float(v[8 * i + 6]) * p.scale, __uint_as_float(v[8 * i + 7]) * p.scale));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(QB_ACC_FREE));
      ++unit_it;
    }
    if (failed && lane == 0) raise_abort(abort, 0x40);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// ============================================================ dK / dV pass
// smem: K | V | Q ring (3) | dO ring (2) | row data (lse2 128 | D 128) | barriers
constexpr int K_SM_K = 0;
constexpr int K_SM_V = kTile;
// Q is read by S^T (early in a query tile's period) and by dK (late), dO by
// dP^T and dV: a three-stage Q ring and a two-stage dO ring, so that the
// next tile's Q has landed when its S^T is due.  One slot of row data (LSE,
// D) fits beside them: the producer holds a tile's row data in registers
// and writes it once the element-wise warps are done with the tile before.
constexpr int kDkvQStages = 3, kDkvDoStages = 2;
constexpr int K_SM_Q = 2 * kTile;
constexpr int K_SM_DO = K_SM_Q + kDkvQStages * kTile;
constexpr int K_SM_ROW = K_SM_DO + kDkvDoStages * kTile;
constexpr int K_SM_BAR = K_SM_ROW + 1024;
constexpr int kDkvSmem = K_SM_BAR + 256 + 1024;
constexpr uint32_t K_T_S = 0, K_T_DP = 128, K_T_DV = 256, K_T_DK = 384;
// Per query tile i the MMA thread issues dV(i) += P^T(i) dO(i), S^T(i+1),
// dK(i) += dS^T(i) Q(i) once dS^T(i) is in, and dP^T(i+1) right behind it.
// P^T(i) lives over S^T(i)'s columns and dS^T(i) over dP^T(i)'s; S^T(i+1) is
// issued after dV(i) and dP^T(i+1) after dK(i), and tensor operations run in
// issue order, so each overwrites its columns only after they were read.
// The element-wise warps compute P^T(i) (phase 1) and dS^T(i) (phase 2),
// keeping P in registers between the two; dP^T(i) is done by then.
enum {
  KB_KV_FULL = 0,
  KB_KV_EMPTY = 1,
  KB_Q_FULL = 2,    // +stage (3)
  KB_Q_EMPTY = 5,   // +stage (3): the tile's dK has run
  KB_DO_FULL = 8,   // +stage (2)
  KB_DO_EMPTY = 10, // +stage (2): the tile's dV has run
  KB_ROW_FULL = 12, // the tile's row data is in shared memory
  KB_S_FULL = 13,   // S^T of the tile is in TMEM
  KB_P_FULL = 14,   // count 8: P^T of the tile is in TMEM
  KB_DP_FULL = 15,  // dP^T of the tile is in TMEM
  KB_DS_FULL = 16,  // count 8: dS^T of the tile is in TMEM (also: its row data was read)
  KB_ACC_DONE = 17,
  KB_ACC_FREE = 18,   // count 8
  KB_UNIT_FULL = 19,  // +slot (4): the unit ring's slot holds the next unit
  KB_UNIT_EMPTY = 23, // +slot (4), count 9: the MMA thread and the element-wise warps read it
  KB_N = 27
};
// The units (key tile, kv head) vary with how many query tiles see the key
// tile; the ring sits after the barriers.
constexpr int K_SM_URING = K_SM_BAR + 240;
static_assert(KB_N * 8 + 8 <= 240, "dK/dV barrier area");
static_assert(K_SM_BAR + 256 + 1024 <= 232448, "dK/dV shared memory");


// Query tiles of a key tile: each entry's queries in steps of tile_tokens.
// The next entry is prefetched into L1 on entering an entry, so a switch
// does not wait on L2 or DRAM.
struct QIter {
  int32_t e, e_end, t0;
  BwdEntry be;
};
__device__ __forceinline__ bool q_begin(const DkvParams& p, const BwdItem& it, QIter& q) {
  q.e = it.e_first;
  q.e_end = it.e_first + it.e_count;
  if (q.e >= q.e_end) return false;
  q.be = p.plan.entries[q.e];
  if (q.e + 1 < q.e_end) asm volatile("prefetch.global.L1 [%0];" ::"l"(&p.plan.entries[q.e + 1]));
  q.t0 = q.be.q_lo;
  return true;
}
__device__ __forceinline__ bool q_next(const DkvParams& p, QIter& q) {
  q.t0 += p.tile_tokens;
  if (q.t0 < q.be.q_hi) return true;
  if (++q.e >= q.e_end) return false;
  q.be = p.plan.entries[q.e];
  if (q.e + 1 < q.e_end) asm volatile("prefetch.global.L1 [%0];" ::"l"(&p.plan.entries[q.e + 1]));
  q.t0 = q.be.q_lo;
  return true;
}

__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                   const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const DkvParams p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base; offsetting the shared array itself keeps the
  // compiler aware that every pointer below is a shared-memory pointer
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + K_SM_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + K_SM_BAR + KB_N * 8);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + K_SM_BAR + KB_N * 8 + 4);
  float* rowdata = reinterpret_cast<float*>(smem + K_SM_ROW);
  volatile int32_t* uring = reinterpret_cast<volatile int32_t*>(smem + K_SM_URING);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  if (threadIdx.x == 0) {
    for (int i = 0; i < KB_N; ++i)
      mbar_init(bar(i), (i == KB_P_FULL || i == KB_DS_FULL || i == KB_ACC_FREE)
                            ? 8u
                            : ((i >= KB_UNIT_EMPTY && i < KB_UNIT_EMPTY + kURing) ? 9u : 1u));
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int G = p.group, tt = p.tile_tokens;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    uint32_t qd_it = 0, unit_it = 0;
    bool failed = false;
    // draw a unit and publish it in the ring (-1 when a wait gave up)
    uint32_t n_pub = 0;
    auto publish = [&]() -> int {
      const int slot = n_pub % kURing;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(KB_UNIT_EMPTY + slot), ((n_pub / kURing) & 1) ^ 1, abort)))
        return -1;
      int v = 0;
      if (lane == 0) {
        v = atomicAdd(p.work, 1);
        uring[slot] = v;
        mbar_arrive(bar(KB_UNIT_FULL + slot));
      }
      ++n_pub;
      return __shfl_sync(0xffffffffu, v, 0);
    };
    int u_next = publish();
    if (u_next < 0) failed = true;
    while (!failed) {
      const int u = u_next;
      if (u >= p.n_units) break;
      // head-major: the CTAs at work at one time share one kv head's Q / dO
      const BwdItem it = p.plan.items[u % p.plan.n_items];
      const int g = u / p.plan.n_items;
      QIter q;
      if (!q_begin(p, it, q)) {
        u_next = publish();
        if (u_next < 0) failed = true;
        continue;
      }
      if (!__all_sync(0xffffffffu, mbar_wait(bar(KB_KV_EMPTY), (unit_it & 1) ^ 1, abort))) { failed = true; break; }
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(KB_KV_FULL), 2 * kTile);
        for (int h = 0; h < 2; ++h) {
          tma_load_3d(sbase + K_SM_K + h * kHalf, &tm_k, bar(KB_KV_FULL), h * 64, g, it.k_start);
          tma_load_3d(sbase + K_SM_V + h * kHalf, &tm_v, bar(KB_KV_FULL), h * 64, g, it.k_start);
        }
      }
      for (bool ok = true; ok; ok = q_next(p, q), ++qd_it) {
        const int qs = qd_it % kDkvQStages, ds = qd_it % kDkvDoStages;
        // LSE (log2 units) and D of the tile's rows (lane takes rows lane +
        // 32 k); rows past the entry get LSE = +inf so that their
        // probabilities vanish
        float lse4[4], d4[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int c = lane + 32 * k;
          const int64_t tok = q.t0 + (c % tt);
          const int head = g * G + c / tt;
          const bool ok2 = tok < q.be.q_hi;
          lse4[k] = ok2 ? p.lse[static_cast<int64_t>(head) * p.T + tok] * kLog2e : INFINITY;
          d4[k] = ok2 ? p.delta[static_cast<int64_t>(head) * p.T + tok] : 0.f;
        }
        if (!__all_sync(0xffffffffu, mbar_wait(bar(KB_Q_EMPTY + qs), ((qd_it / kDkvQStages) & 1) ^ 1, abort))) {
          failed = true;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(KB_Q_FULL + qs), kTile);
          for (int hh = 0; hh < G; ++hh)
            for (int h = 0; h < 2; ++h)
              tma_load_3d(sbase + K_SM_Q + qs * kTile + h * kHalf + hh * tt * 128, &tm_q, bar(KB_Q_FULL + qs), h * 64,
                          g * G + hh, q.t0);
        }
        if (!__all_sync(0xffffffffu, mbar_wait(bar(KB_DO_EMPTY + ds), ((qd_it / kDkvDoStages) & 1) ^ 1, abort))) {
          failed = true;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(KB_DO_FULL + ds), kTile);
          for (int hh = 0; hh < G; ++hh)
            for (int h = 0; h < 2; ++h)
              tma_load_3d(sbase + K_SM_DO + ds * kTile + h * kHalf + hh * tt * 128, &tm_do, bar(KB_DO_FULL + ds),
                          h * 64, g * G + hh, q.t0);
        }
        // the row slot is free once the element-wise warps are done with the
        // tile before (its dS^T is in, after both of their phases read it)
        if (qd_it > 0 &&
            !__all_sync(0xffffffffu, mbar_wait(bar(KB_DS_FULL), (qd_it - 1) & 1, abort))) {
          failed = true;
          break;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          rowdata[lane + 32 * k] = lse4[k];
          rowdata[128 + lane + 32 * k] = d4[k];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(KB_ROW_FULL));
      }
      if (failed) break;
      u_next = publish();
      if (u_next < 0) {
        failed = true;
        break;
      }
      ++unit_it;
    }
    if (failed && lane == 0) raise_abort(abort, 0x100);
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_kk = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t id_mn = idesc_bf16_f32(128, 128, false, true);
      uint32_t qd_it = 0, unit_it = 0;
      bool failed = false;
      // base descriptors: K and V (K-major A), Q and dO of each stage as
      // K-major B (for S^T, dP^T) and as MN-major B (for dK, dV)
      const uint64_t d_k = sdesc_sw128(sbase + K_SM_K, 16, 1024), d_v = sdesc_sw128(sbase + K_SM_V, 16, 1024);
      // descriptors of the Q stages (K-major B for S^T, MN-major B for dK) and
      // of the dO stages (K-major for dP^T, MN-major for dV)
      const uint32_t qa0 = sbase + K_SM_Q, da0 = sbase + K_SM_DO;
      const uint64_t d_q0 = sdesc_sw128(qa0, 16, 1024), d_q1 = sdesc_sw128(qa0 + kTile, 16, 1024),
                     d_q2 = sdesc_sw128(qa0 + 2 * kTile, 16, 1024);
      const uint64_t d_qm0 = sdesc_sw128(qa0, kHalf, 1024), d_qm1 = sdesc_sw128(qa0 + kTile, kHalf, 1024),
                     d_qm2 = sdesc_sw128(qa0 + 2 * kTile, kHalf, 1024);
      const uint64_t d_do0 = sdesc_sw128(da0, 16, 1024), d_do1 = sdesc_sw128(da0 + kTile, 16, 1024);
      const uint64_t d_dom0 = sdesc_sw128(da0, kHalf, 1024), d_dom1 = sdesc_sw128(da0 + kTile, kHalf, 1024);
      // S^T = K Q^T for tile i (its Q landed)
      auto issue_s = [&](uint32_t i) {
        const uint32_t qs = i % kDkvQStages;
        const uint64_t dq = qs == 0 ? d_q0 : (qs == 1 ? d_q1 : d_q2);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_bf16_ss(tmem + K_T_S, kmajor_step(d_k, kk), kmajor_step(dq, kk), id_kk, kk > 0);
        mma_commit(bar(KB_S_FULL));
      };
      // dP^T = V dO^T for tile i (its dO landed), over the columns of the
      // previous tile's dS^T (read by its dK, issued earlier)
      auto issue_dp = [&](uint32_t i) {
        const uint64_t ddo = (i % kDkvDoStages) ? d_do1 : d_do0;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16_ss(tmem + K_T_DP, kmajor_step(d_v, kk), kmajor_step(ddo, kk), id_kk, kk > 0);
        mma_commit(bar(KB_DP_FULL));
      };
      auto wait_q = [&](uint32_t i) {
        return mbar_wait_relaxed(bar(KB_Q_FULL + i % kDkvQStages), (i / kDkvQStages) & 1, abort);
      };
      auto wait_do = [&](uint32_t i) {
        return mbar_wait_relaxed(bar(KB_DO_FULL + i % kDkvDoStages), (i / kDkvDoStages) & 1, abort);
      };
      uint32_t n_taken = 0;
      while (!failed) {
        int u;
        if (!take_unit(n_taken, u, uring, bars, KB_UNIT_FULL, KB_UNIT_EMPTY, abort, true)) {
          failed = true;
          break;
        }
        if (u >= p.n_units) break;
        const BwdItem it = p.plan.items[u % p.plan.n_items];
        QIter q;
        if (!q_begin(p, it, q)) continue;
        if (!mbar_wait_relaxed(bar(KB_KV_FULL), unit_it & 1, abort)) { failed = true; break; }
        if (!wait_q(qd_it)) { failed = true; break; }
        tc_fence_after();
        issue_s(qd_it);
        if (!wait_do(qd_it)) { failed = true; break; }
        tc_fence_after();
        issue_dp(qd_it);
        bool first = true;
        for (bool ok = true; ok; ++qd_it) {
          const uint32_t qs = qd_it % kDkvQStages, ds = qd_it % kDkvDoStages;
          const uint64_t dqm = qs == 0 ? d_qm0 : (qs == 1 ? d_qm1 : d_qm2), ddom = ds ? d_dom1 : d_dom0;
          const bool more = q_next(p, q);
          if (first && !mbar_wait_relaxed(bar(KB_ACC_FREE), (unit_it & 1) ^ 1, abort)) { failed = true; break; }
          if (!mbar_wait_relaxed(bar(KB_P_FULL), qd_it & 1, abort)) { failed = true; break; }
          tc_fence_after();
          // dV += P^T dO (warpgroup h packed query rows 64h .. 64h + 63 into
          // columns 64h .. 64h + 31)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16_ts(tmem + K_T_DV, tmem + K_T_S + (kk >> 2) * 64 + (kk & 3) * 8, mnmajor_step(ddom, kk), id_mn,
                        (!first || kk > 0) ? 1u : 0u);
          mma_commit(bar(KB_DO_EMPTY + ds));  // dP^T and dV have read dO
          // The next tile's S^T over the columns dV has just read: now, so
          // that it runs while the element-wise warps compute dS^T, when its
          // Q has landed; otherwise after dK, so as not to hold dK up.
          const uint32_t nb = KB_Q_FULL + (qd_it + 1) % kDkvQStages, nph = ((qd_it + 1) / kDkvQStages) & 1;
          const bool s_early = more && mbar_test_wait(bar(nb), nph);
          if (s_early) {
            tc_fence_after();
            issue_s(qd_it + 1);
          }
          if (!mbar_wait_relaxed(bar(KB_DS_FULL), qd_it & 1, abort)) { failed = true; break; }
          tc_fence_after();
          // dK += dS^T Q
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16_ts(tmem + K_T_DK, tmem + K_T_DP + (kk >> 2) * 64 + (kk & 3) * 8, mnmajor_step(dqm, kk), id_mn,
                        (!first || kk > 0) ? 1u : 0u);
          mma_commit(bar(KB_Q_EMPTY + qs));  // S^T and dK have read Q
          if (more) {
            if (!s_early) {
              if (!mbar_wait_relaxed(bar(nb), nph, abort)) {
                failed = true;
                break;
              }
              tc_fence_after();
              issue_s(qd_it + 1);
            }
            // the next tile's dP^T right behind dK: the element-wise warps
            // find it done when they reach its dS^T
            if (!wait_do(qd_it + 1)) {
              failed = true;
              break;
            }
            tc_fence_after();
            issue_dp(qd_it + 1);
          }
          first = false;
          ok = more;
        }
        if (failed) break;
        mma_commit(bar(KB_KV_EMPTY));
        mma_commit(bar(KB_ACC_DONE));
        ++unit_it;
      }
      if (failed) raise_abort(abort, 0x200);
    }
  } else {
    // ------------------------------------------------------------ element-wise (warps 0-7)
    const int wg = warp >> 2;                    // query-row half of this warpgroup
    const int r = (warp & 3) * 32 + lane;        // key of the tile == TMEM lane
    const uint32_t lb = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint32_t qd_it = 0, g_it = 0, unit_it = 0;
    bool failed = false;
    uint32_t n_taken = 0;
    while (!failed) {
      int u;
      if (!take_unit(n_taken, u, uring, bars, KB_UNIT_FULL, KB_UNIT_EMPTY, abort, false)) {
        failed = true;
        break;
      }
      if (u >= p.n_units) break;
      // head-major: the CTAs at work at one time share one kv head's Q / dO
      const BwdItem it = p.plan.items[u % p.plan.n_items];
      const int g = u / p.plan.n_items;
      QIter q;
      if (!q_begin(p, it, q)) continue;
      const int32_t key = it.k_start + r;
      for (bool ok = true; ok; ok = q_next(p, q), ++qd_it, ++g_it) {
        // the tile's row data (the producer writes it once this warp's
        // previous tile is done)
        if (!__all_sync(0xffffffffu, mbar_wait(bar(KB_ROW_FULL), qd_it & 1, abort))) {
          failed = true;
          break;
        }
        if (!__all_sync(0xffffffffu, mbar_wait(bar(KB_S_FULL), qd_it & 1, abort))) { failed = true; break; }
        tc_fence_after();
        const float* rd = rowdata + wg * 64;
        // row c (token t0 + c % tt) sees this key iff the token index i = c % tt
        // lies in [i_lo, i_hi)
        const bool key_ok = key >= q.be.k_lo && key < q.be.k_hi;
        const int i_lo = q.be.causal ? max(0, key - q.t0) : 0;
        const int i_hi = key_ok ? min(tt, q.be.q_hi - q.t0) : 0;
        // every row of the tile sees every key of the warp: no masks
        const bool all_visible = __all_sync(0xffffffffu, i_lo == 0 && i_hi == tt);
        // phase 1: P^T = 2^(S^T sl2 - LSE2) over this warpgroup's 64 query
        // rows, kept in registers for phase 2 and written as bf16 pairs over
        // the first 32 of those columns
        float pf[64];
        {
          uint32_t sv[2][32];
          tmem_ld32(tmem + lb + K_T_S + wg * 64, sv[0]);
          tmem_ld32(tmem + lb + K_T_S + wg * 64 + 32, sv[1]);
          tmem_wait_ld();
          const float4* l4 = reinterpret_cast<const float4*>(rd);  // LSE (log2) of the rows
          if (all_visible) {
            const uint64_t sl2x2 = f2pack(p.sl2, p.sl2);
#pragma unroll
            for (int i = 0; i < 64; i += 4) {
              const float4 l = l4[i >> 2];
              float x0, x1, x2, x3;
              f2unpack(fma2(f2pack(__uint_as_float(sv[i >> 5][(i & 31) + 0]), __uint_as_float(sv[i >> 5][(i & 31) + 1])),
                            sl2x2, f2pack(-l.x, -l.y)),
                       x0, x1);
              f2unpack(fma2(f2pack(__uint_as_float(sv[i >> 5][(i & 31) + 2]), __uint_as_float(sv[i >> 5][(i & 31) + 3])),
                            sl2x2, f2pack(-l.z, -l.w)),
                       x2, x3);
              pf[i + 0] = fast_exp2(x0);
              pf[i + 1] = fast_exp2(x1);
              pf[i + 2] = fast_exp2(x2);
              pf[i + 3] = fast_exp2(x3);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 64; i += 4) {
              const float4 l = l4[i >> 2];
              const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int ie = (wg * 64 + i + e) & (tt - 1);
                pf[i + e] = (ie >= i_lo && ie < i_hi)
                                ? fast_exp2(fmaf(__uint_as_float(sv[i >> 5][(i & 31) + e]), p.sl2, -lv[e]))
                                : 0.f;
              }
            }
          }
          uint32_t pp[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) pp[i] = pack_bf16x2(pf[2 * i], pf[2 * i + 1]);
          tmem_st16(tmem + lb + K_T_S + wg * 64, *reinterpret_cast<const uint32_t(*)[16]>(&pp[0]));
          tmem_st16(tmem + lb + K_T_S + wg * 64 + 16, *reinterpret_cast<const uint32_t(*)[16]>(&pp[16]));
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(KB_P_FULL));
        // phase 2: dS^T = P^T (dP^T - D), as bf16 pairs over dP^T's columns
        if (!__all_sync(0xffffffffu, mbar_wait(bar(KB_DP_FULL), qd_it & 1, abort))) { failed = true; break; }
        tc_fence_after();
        {
          uint32_t dv[2][32];
          tmem_ld32(tmem + lb + K_T_DP + wg * 64, dv[0]);
          tmem_ld32(tmem + lb + K_T_DP + wg * 64 + 32, dv[1]);
          tmem_wait_ld();
          const float4* d4 = reinterpret_cast<const float4*>(rd + 128);  // D of the rows
          uint32_t dd[32];
#pragma unroll
          for (int i = 0; i < 64; i += 4) {
            const float4 dl = d4[i >> 2];
            const uint64_t d01 = mul2(f2pack(pf[i + 0], pf[i + 1]),
                                      sub2(f2pack(__uint_as_float(dv[i >> 5][(i & 31) + 0]), __uint_as_float(dv[i >> 5][(i & 31) + 1])),
                                           f2pack(dl.x, dl.y)));
            const uint64_t d23 = mul2(f2pack(pf[i + 2], pf[i + 3]),
                                      sub2(f2pack(__uint_as_float(dv[i >> 5][(i & 31) + 2]), __uint_as_float(dv[i >> 5][(i & 31) + 3])),
                                           f2pack(dl.z, dl.w)));
            float a, b;
            f2unpack(d01, a, b);
            dd[(i >> 1) + 0] = pack_bf16x2(a, b);
            f2unpack(d23, a, b);
            dd[(i >> 1) + 1] = pack_bf16x2(a, b);
          }
          tmem_st16(tmem + lb + K_T_DP + wg * 64, *reinterpret_cast<const uint32_t(*)[16]>(&dd[0]));
          tmem_st16(tmem + lb + K_T_DP + wg * 64 + 16, *reinterpret_cast<const uint32_t(*)[16]>(&dd[16]));
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(KB_DS_FULL));
      }
      if (failed) break;
      // epilogue: this warpgroup's half of the key's dV and dK
      if (!__all_sync(0xffffffffu, mbar_wait(bar(KB_ACC_DONE), unit_it & 1, abort))) { failed = true; break; }
      tc_fence_after();
      const bool valid = r < it.k_len;
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        __nv_bfloat16* out = part == 0 ? p.dv : p.dk;
        const float mul = part == 0 ? 1.f : p.scale;
        const uint32_t col0 = (part == 0 ? K_T_DV : K_T_DK) + wg * 64;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + lb + col0 + c * 32, v);
          tmem_wait_ld();
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(out + (static_cast<int64_t>(key) * p.Hkv + g) * kHeadDim + wg * 64 +
                                                  c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * i + 0]) * mul, __uint_as_float(v[8 * i + 1]) * mul),
                                  pack_bf16x2(__uint_as_float(v[8 * i + 2]) * mul, __uint_as_float(v[8 * i + 3]) * mul),
                                  pack_bf16x2(__uint_as_float(v[8 * i + 4]) * mul, __uint_as_float(v[8 * i + 5]) * mul),
                                  pack_bf16x2(__uint_as_float(v[8 * i + 6]) * mul, __uint_as_float(v[8 * i + 7]) * mul));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(KB_ACC_FREE));
      ++unit_it;
    }
    if (failed && lane == 0) raise_abort(abort, 0x400);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

int make_map(EncodeTiledFn enc, CUtensorMap* m, const void* ptr, cuuint64_t heads, cuuint64_t T, cuuint32_t rows,
             std::string* err) {
  const cuuint64_t dims[3] = {128, heads, T};
  const cuuint64_t strides[2] = {256, heads * 256};
  const cuuint32_t box[3] = {64, 1, rows};
  const cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *err = "cuTensorMapEncodeTiled failed with code " + std::to_string(static_cast<int>(r));
    return PADOC_ERR_CUDA;
  }
  return PADOC_OK;
}

}  // namespace

int launch_bwd_tc(const BwdArgs& a, cudaStream_t s, std::string* err) {
  int rc = launch_bwd_delta(a, PADOC_BF16, s, err);
  if (rc) return rc;
  EncodeTiledFn enc = get_encode_fn(err);
  if (!enc) return PADOC_ERR_CUDA;
  const int tt = a.fwd.tile_tokens;
  CUtensorMap mq, mdo, mk, mv;
  rc = make_map(enc, &mq, a.q, a.Hq, a.T, tt, err);
  if (!rc) rc = make_map(enc, &mdo, a.dout, a.Hq, a.T, tt, err);
  if (!rc) rc = make_map(enc, &mk, a.k, a.Hkv, a.T, 128, err);
  if (!rc) rc = make_map(enc, &mv, a.v, a.Hkv, a.T, 128, err);
  if (rc) return rc;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDqSmem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(bwd_dkv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDkvSmem);
    if (e != cudaSuccess) {
      *err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
      return PADOC_ERR_CUDA;
    }
    attr = true;
  }
  const float sl2 = a.scale * kLog2e;
  if (a.fwd.n_items > 0) {
    DqParams p{};
    p.work = a.work + 1;  // the dK/dV pass counts in a.work[0]
    {
      const cudaError_t e = cudaMemsetAsync(p.work, 0, sizeof(int32_t), s);
      if (e != cudaSuccess) {
        *err = std::string("cudaMemsetAsync of the unit counter: ") + cudaGetErrorString(e);
        return PADOC_ERR_CUDA;
      }
    }
    p.plan = a.fwd;
    p.n_units = a.fwd.n_items * a.Hkv;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.group = a.fwd.group;
    p.T = a.T;
    p.sl2 = sl2;
    p.scale = a.scale;
    p.lse = a.lse;
    p.delta = a.delta;
    p.dq = static_cast<__nv_bfloat16*>(a.dq);
    bwd_dq_kernel<<<std::min(p.n_units, num_sms()), kThreads, kDqSmem, s>>>(mq, mdo, mk, mv, p);
  }
  if (a.bwd.n_items > 0) {
    DkvParams p{};
    p.work = a.work;
    {
      // units are drawn from this counter in order
      const cudaError_t e = cudaMemsetAsync(a.work, 0, sizeof(int32_t), s);
      if (e != cudaSuccess) {
        *err = std::string("cudaMemsetAsync of the unit counter: ") + cudaGetErrorString(e);
        return PADOC_ERR_CUDA;
      }
    }
    p.plan = a.bwd;
    p.n_units = a.bwd.n_items * a.Hkv;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.group = a.fwd.group;
    p.tile_tokens = tt;
    p.T = a.T;
    p.sl2 = sl2;
    p.scale = a.scale;
    p.lse = a.lse;
    p.delta = a.delta;
    p.dk = static_cast<__nv_bfloat16*>(a.dk);
    p.dv = static_cast<__nv_bfloat16*>(a.dv);
    bwd_dkv_kernel<<<std::min(p.n_units, num_sms()), kThreads, kDkvSmem, s>>>(mq, mdo, mk, mv, p);
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *err = std::string("backward kernel launch: ") + cudaGetErrorString(e);
    return PADOC_ERR_CUDA;
  }
  return PADOC_OK;
}

int read_and_clear_bwd_error(cudaStream_t s, unsigned* word) {
  unsigned zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(word, g_bwd_err, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpyToSymbolAsync(g_bwd_err, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e == cudaSuccess ? PADOC_OK : PADOC_ERR_CUDA;
}

}  // namespace padoc
