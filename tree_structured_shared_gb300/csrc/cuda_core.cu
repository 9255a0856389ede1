// CUDA-core kernels:
//  * fwd_f32_kernel   tree-varlen forward in f32 (the f32 workload; no tensor
//                     core format holds f32 exactly);
//  * own_pass_kernel  second half of branch decode: each (branch, kv head)
//                     streams its own cached suffix with 16-byte coalesced
//                     loads, adds the query-block tokens its draft-tree mask
//                     allows, and merges everything with the prefix partials
//                     by log-sum-exp into the final O and LSE;
//  * kv_append_kernel scatter of new K/V rows into pool blocks.
#include <cuda_bf16.h>

#include <algorithm>
#include <string>

#include "../../include/padoc.h"
#include "padoc_internal.h"

namespace padoc {

namespace {

constexpr float kLog2e = 1.44269504088896340736f;
constexpr float kLn2 = 0.69314718055994530942f;

__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// ------------------------------------------------------------------ f32 forward
// One block per (query tile, kv head); warp w handles rows w, w+4, ...; a row
// walks its key segments one key at a time with an online softmax.
template <int D>
__global__ void __launch_bounds__(128) fwd_f32_kernel(FwdPlan plan, const float* __restrict__ q,
                                                      const float* __restrict__ k, const float* __restrict__ v,
                                                      float* __restrict__ o, float* __restrict__ lse, int64_t T,
                                                      int Hq, int Hkv, float sl2) {
  constexpr int E = D / 32;
  const int item = blockIdx.x / Hkv;
  const int g = blockIdx.x % Hkv;
  const FwdItem it = plan.items[item];
  const QSeg qs = plan.qsegs[it.qseg];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = plan.group, tt = plan.tile_tokens;
  for (int r = warp; r < tt * G; r += 4) {
    const int64_t qpos = it.tile_start + r % tt;
    if (qpos >= qs.q_start + qs.q_len) continue;
    const int head = g * G + r / tt;
    float qr[E], acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      qr[e] = q[(qpos * Hq + head) * D + lane + 32 * e];
      acc[e] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    for (int s = 0; s < qs.kv_count; ++s) {
      const KVSeg kv = plan.kvsegs[qs.kv_first + s];
      int64_t end = kv.start + kv.len;
      if (kv.causal && end > qpos + 1) end = qpos + 1;
      for (int64_t j = kv.start; j < end; ++j) {
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) dot += qr[e] * k[(j * Hkv + g) * D + lane + 32 * e];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
        const float sc = dot * sl2;
        const float mn = fmaxf(m, sc);
        const float corr = exp2f(m - mn);
        const float pj = exp2f(sc - mn);
        l = l * corr + pj;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = acc[e] * corr + pj * v[(j * Hkv + g) * D + lane + 32 * e];
        m = mn;
      }
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) o[(qpos * Hq + head) * D + lane + 32 * e] = acc[e] * inv;
    if (lane == 0) lse[static_cast<int64_t>(head) * T + qpos] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
  }
}

// ------------------------------------------------------------------ own pass
// Lane layout for a 16-token block of one kv head (16 rows x 256 bytes):
// half-warp h reads token rows with (row & 1) == h; lane s of the half reads
// bytes [16 s, 16 s + 16) of the row, i.e. head dims [8 s, 8 s + 8).
template <int G>
struct OwnState {
  float m[G], l[G], acc[G][8];
};

template <int G>
__device__ __forceinline__ void own_init(OwnState<G>& st) {
#pragma unroll
  for (int h = 0; h < G; ++h) {
    st.m[h] = -INFINITY;
    st.l[h] = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) st.acc[h][e] = 0.f;
  }
}

// Folds up to 8 keys (one per step for this half-warp) into the state.
// kr/vr hold each key's 8 head dims for this lane; ok[i] says key i is visible.
template <int G>
__device__ __forceinline__ void own_fold(OwnState<G>& st, const float (&qr)[G][8], const uint4 (&kr)[8],
                                         const uint4 (&vr)[8], const bool (&ok)[8], float sl2) {
  float s[G][8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t w[4] = {kr[i].x, kr[i].y, kr[i].z, kr[i].w};
    float kf[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      kf[2 * e] = bf_lo(w[e]);
      kf[2 * e + 1] = bf_hi(w[e]);
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float d = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) d = fmaf(qr[h][e], kf[e], d);
      s[h][i] = d;
    }
  }
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float d = s[h][i];
      d += __shfl_xor_sync(0xffffffffu, d, 1);
      d += __shfl_xor_sync(0xffffffffu, d, 2);
      d += __shfl_xor_sync(0xffffffffu, d, 4);
      d += __shfl_xor_sync(0xffffffffu, d, 8);
      s[h][i] = ok[i] ? d * sl2 : -INFINITY;
    }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float mx = st.m[h];
#pragma unroll
    for (int i = 0; i < 8; ++i) mx = fmaxf(mx, s[h][i]);
    const float mu = (mx == -INFINITY) ? 0.f : mx;
    const float corr = exp2f(st.m[h] - mu);
    st.l[h] *= corr;
#pragma unroll
    for (int e = 0; e < 8; ++e) st.acc[h][e] *= corr;
    st.m[h] = mx;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float pj = exp2f(s[h][i] - mu);
      st.l[h] += pj;
      const uint32_t w[4] = {vr[i].x, vr[i].y, vr[i].z, vr[i].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        st.acc[h][2 * e] = fmaf(pj, bf_lo(w[e]), st.acc[h][2 * e]);
        st.acc[h][2 * e + 1] = fmaf(pj, bf_hi(w[e]), st.acc[h][2 * e + 1]);
      }
    }
  }
}

template <int G>
__global__ void __launch_bounds__(128) own_pass_kernel(DecodeArgs a) {
  const int b = blockIdx.x / a.Hkv;
  const int g = blockIdx.x % a.Hkv;
  const DecBranch br = a.branches[b];
  const DecPage pg = a.pages[br.page];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = lane >> 4, sub = lane & 15;
  // partial states of the 8 half-warps, per head: m, l, acc[128]
  __shared__ float sm_m[8][G], sm_l[8][G];
  __shared__ float sm_acc[8][G][128];
  const uint4* kp = reinterpret_cast<const uint4*>(a.k_pool);
  const uint4* vp = reinterpret_cast<const uint4*>(a.v_pool);
  const uint4* kn = reinterpret_cast<const uint4*>(a.k_new);
  const uint4* vn = reinterpret_cast<const uint4*>(a.v_new);
  const uint4* q4 = reinterpret_cast<const uint4*>(a.q);
  const int32_t* trow = a.table + static_cast<int64_t>(br.seq) * a.max_bps + br.n_shared;
  const int n_blocks = (br.own_len + 15) >> 4;
  const float sl2 = a.scale * kLog2e;

  for (int qi = 0; qi < br.q_len; ++qi) {
    const int64_t qrow = br.q_first + qi;
    float qr[G][8];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const uint4 x = q4[(qrow * a.Hq + g * G + h) * 16 + sub];
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        qr[h][2 * e] = bf_lo(w[e]);
        qr[h][2 * e + 1] = bf_hi(w[e]);
      }
    }
    OwnState<G> st;
    own_init(st);
    // own cached suffix: warp w takes blocks w, w + 4, ...
    for (int bi = warp; bi < n_blocks; bi += 4) {
      const int64_t blk = trow[bi];
      const int64_t base = ((blk * a.Hkv + g) * 16) * 16;  // in uint4 units
      uint4 kr[8], vr[8];
      bool ok[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int slot = 2 * i + half;
        ok[i] = bi * 16 + slot < br.own_len;
        kr[i] = kp[base + slot * 16 + sub];
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) vr[i] = vp[base + (2 * i + half) * 16 + sub];
      own_fold(st, qr, kr, vr, ok, sl2);
    }
    // query-block tokens of this branch (draft-tree ancestors and itself)
    if (warp == 0) {
      const uint32_t bits = a.tree_bits ? a.tree_bits[qrow] : ((2u << qi) - 1u);
      uint4 kr[8], vr[8];
      bool ok[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int j = 2 * i + half;
        ok[i] = j < br.q_len && ((bits >> j) & 1u);
        const int64_t src = ((br.q_first + min(j, br.q_len - 1)) * a.Hkv + g) * 16 + sub;
        kr[i] = kn[src];
        vr[i] = vn[src];
      }
      own_fold(st, qr, kr, vr, ok, sl2);
    }
    // combine lanes of each half-warp: every lane holds m, l; acc is per lane
    const int slot = warp * 2 + half;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      if (sub == 0) {
        sm_m[slot][h] = st.m[h];
        sm_l[slot][h] = st.l[h];
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) sm_acc[slot][h][sub * 8 + e] = st.acc[h][e];
    }
    __syncthreads();
    // final merge: thread t handles (head h, dims) pairs
    for (int x = threadIdx.x; x < G * 128; x += 128) {
      const int h = x >> 7, dd = x & 127;
      const int head = g * G + h;
      float M = -INFINITY;
#pragma unroll
      for (int s2 = 0; s2 < 8; ++s2) M = fmaxf(M, sm_m[s2][h]);
      // prefix partials of this row (natural-log LSE, normalised O)
      const int R = (br.q_in_page + qi) * G + h;
      const int tile = R / kTileRows, rr = R % kTileRows;
      for (int c = 0; c < pg.n_chunks; ++c) {
        const DecItem it = a.items[pg.item_base + tile * pg.n_chunks + c];
        const float ls = a.part_lse[static_cast<int64_t>(it.row_base) + static_cast<int64_t>(g) * it.rows + rr];
        M = fmaxf(M, ls * kLog2e);
      }
      const float Mu = (M == -INFINITY) ? 0.f : M;
      float L = 0.f, O = 0.f;
#pragma unroll
      for (int s2 = 0; s2 < 8; ++s2) {
        const float w = exp2f(sm_m[s2][h] - Mu);
        L += sm_l[s2][h] * w;
        O += sm_acc[s2][h][dd] * w;
      }
      for (int c = 0; c < pg.n_chunks; ++c) {
        const DecItem it = a.items[pg.item_base + tile * pg.n_chunks + c];
        const int64_t prow = static_cast<int64_t>(it.row_base) + static_cast<int64_t>(g) * it.rows + rr;
        const float w = exp2f(a.part_lse[prow] * kLog2e - Mu);
        L += w;
        O += a.part_o[prow * kHeadDim + dd] * w;
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
      reinterpret_cast<__nv_bfloat16*>(a.o)[(qrow * a.Hq + head) * kHeadDim + dd] = __float2bfloat16_rn(O * inv);
      if (dd == 0) a.lse[qrow * a.Hq + head] = L > 0.f ? (Mu + log2f(L)) * kLn2 : -INFINITY;
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ append
__global__ void kv_append_kernel(uint4* __restrict__ kpool, uint4* __restrict__ vpool,
                                 const int32_t* __restrict__ table_row, int32_t first_own, int32_t n, int32_t Hkv,
                                 const uint4* __restrict__ k, const uint4* __restrict__ v) {
  const int64_t total = static_cast<int64_t>(n) * Hkv * 16;
  for (int64_t x = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; x < total;
       x += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(x & 15);
    const int h = static_cast<int>((x >> 4) % Hkv);
    const int64_t i = (x >> 4) / Hkv;
    const int64_t j = first_own + i;
    const int64_t blk = table_row[j >> 4];
    const int64_t dst = ((blk * Hkv + h) * 16 + (j & 15)) * 16 + c;
    kpool[dst] = k[x];
    vpool[dst] = v[x];
  }
}

}  // namespace

int launch_fwd_f32(const FwdArgs& a, cudaStream_t s, std::string* err) {
  if (a.plan.n_items == 0) return PADOC_OK;
  const int grid = a.plan.n_items * a.Hkv;
  const float sl2 = a.scale * kLog2e;
  if (a.d == 64)
    fwd_f32_kernel<64><<<grid, 128, 0, s>>>(a.plan, static_cast<const float*>(a.q), static_cast<const float*>(a.k),
                                            static_cast<const float*>(a.v), static_cast<float*>(a.o), a.lse, a.T,
                                            a.Hq, a.Hkv, sl2);
  else
    fwd_f32_kernel<128><<<grid, 128, 0, s>>>(a.plan, static_cast<const float*>(a.q), static_cast<const float*>(a.k),
                                             static_cast<const float*>(a.v), static_cast<float*>(a.o), a.lse, a.T,
                                             a.Hq, a.Hkv, sl2);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *err = std::string("f32 forward launch: ") + cudaGetErrorString(e);
    return PADOC_ERR_CUDA;
  }
  return PADOC_OK;
}

int launch_decode_own(const DecodeArgs& a, cudaStream_t s, std::string* err) {
  if (a.n_branches == 0) return PADOC_OK;
  const int grid = a.n_branches * a.Hkv;
  switch (a.group) {
    case 1: own_pass_kernel<1><<<grid, 128, 0, s>>>(a); break;
    case 2: own_pass_kernel<2><<<grid, 128, 0, s>>>(a); break;
    case 4: own_pass_kernel<4><<<grid, 128, 0, s>>>(a); break;
    case 8: own_pass_kernel<8><<<grid, 128, 0, s>>>(a); break;
    default:
      *err = "own pass: Hq/Hkv must be 1, 2, 4 or 8";
      return PADOC_ERR_UNSUPPORTED;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *err = std::string("own pass launch: ") + cudaGetErrorString(e);
    return PADOC_ERR_CUDA;
  }
  return PADOC_OK;
}

int launch_kv_append(void* k_pool, void* v_pool, const int32_t* table_row, int32_t first_own, int32_t n, int32_t Hkv,
                     int32_t d, const void* k, const void* v, cudaStream_t s, std::string* err) {
  if (d != kHeadDim) {
    *err = "append: d must be 128";
    return PADOC_ERR_UNSUPPORTED;
  }
  const int64_t total = static_cast<int64_t>(n) * Hkv * 16;
  const int grid = static_cast<int>(std::min<int64_t>((total + 255) / 256, 8 * 1024));
  kv_append_kernel<<<grid, 256, 0, s>>>(static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), table_row, first_own,
                                        n, Hkv, static_cast<const uint4*>(k), static_cast<const uint4*>(v));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *err = std::string("append launch: ") + cudaGetErrorString(e);
    return PADOC_ERR_CUDA;
  }
  return PADOC_OK;
}

}  // namespace padoc
