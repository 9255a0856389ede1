// Backward of the tree-varlen forward on CUDA cores (f32 arithmetic).
//
// For every (query t, visible key j, query head h) the chain rule through
// the forward's softmax gives (PaDoc, "Training paradigm": the forward is a
// softmax over each token's ancestor set):
//   P = exp(scale q.k - LSE_t),  dP = dO_t . v_j,  dS = P (dP - D_t),
//   dq_t += scale dS k_j,  dk_j += scale dS q_t,  dv_j += P dO_t,
// with D_t = dO_t . O_t.  Three launches:
//   delta_kernel     D for every (token, head), into the workspace;
//   dq_core_kernel   query-stationary: one warp per (token, head) of a forward
//                    query tile walks that tile's key segments;
//   dkv_core_kernel  key-stationary: one warp per key of a key tile walks the
//                    tile's entries (the transposed key lists), summing over
//                    the query heads of the key's group.
// Each output element is written by exactly one warp, in a fixed order, so
// results are deterministic.
#include <cuda_bf16.h>

#include <string>

#include "../../include/padoc.h"
#include "padoc_internal.h"

namespace padoc {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

template <typename T, int D>
__device__ __forceinline__ void load_row(const T* p, int lane, float (&x)[D / 32]) {
#pragma unroll
  for (int e = 0; e < D / 32; ++e) x[e] = to_f(p[lane * (D / 32) + e]);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <typename T, int D>
__global__ void __launch_bounds__(256) delta_kernel(const T* __restrict__ o, const T* __restrict__ dout,
                                                   float* __restrict__ delta, int64_t T_, int32_t Hq) {
  const int64_t w = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= T_ * Hq) return;
  const int64_t t = w / Hq;
  const int h = static_cast<int>(w % Hq);
  float a[D / 32], b[D / 32];
  load_row<T, D>(o + (t * Hq + h) * D, lane, a);
  load_row<T, D>(dout + (t * Hq + h) * D, lane, b);
  float acc = 0.f;
#pragma unroll
  for (int e = 0; e < D / 32; ++e) acc += a[e] * b[e];
  acc = warp_sum(acc);
  if (lane == 0) delta[h * T_ + t] = acc;
}

// grid (forward query tiles, Hkv); the block's warps take the tile's
// (token, head-in-group) rows in turn.
template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) dq_core_kernel(FwdPlan plan, const T* __restrict__ q,
                                                              const T* __restrict__ k, const T* __restrict__ v,
                                                              const T* __restrict__ dout,
                                                              const float* __restrict__ lse,
                                                              const float* __restrict__ delta, T* __restrict__ dq,
                                                              int64_t T_, int32_t Hq, int32_t Hkv, float scale) {
  const FwdItem it = plan.items[blockIdx.x];
  const QSeg qs = plan.qsegs[it.qseg];
  const int g = blockIdx.y, G = plan.group;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tend = min(it.tile_start + plan.tile_tokens, qs.q_start + qs.q_len);
  const int rows = (tend - it.tile_start) * G;
  for (int r = warp; r < rows; r += kWarps) {
    const int64_t t = it.tile_start + r / G;
    const int h = g * G + r % G;
    float qr[D / 32], dor[D / 32], acc[D / 32];
    load_row<T, D>(q + (t * Hq + h) * D, lane, qr);
    load_row<T, D>(dout + (t * Hq + h) * D, lane, dor);
#pragma unroll
    for (int e = 0; e < D / 32; ++e) acc[e] = 0.f;
    const float L = lse[h * T_ + t], Dt = delta[h * T_ + t];
    for (int s = 0; s < qs.kv_count; ++s) {
      const KVSeg kv = plan.kvsegs[qs.kv_first + s];
      const int64_t jend = kv.causal ? min(static_cast<int64_t>(kv.start) + kv.len, t + 1)
                                     : static_cast<int64_t>(kv.start) + kv.len;
      for (int64_t j = kv.start; j < jend; ++j) {
        float kr[D / 32], vr[D / 32];
        load_row<T, D>(k + (j * Hkv + g) * D, lane, kr);
        load_row<T, D>(v + (j * Hkv + g) * D, lane, vr);
        float sd = 0.f, pd = 0.f;
#pragma unroll
        for (int e = 0; e < D / 32; ++e) {
          sd += qr[e] * kr[e];
          pd += dor[e] * vr[e];
        }
        sd = warp_sum(sd);
        pd = warp_sum(pd);
        const float p = expf(sd * scale - L);
        const float ds = p * (pd - Dt);
#pragma unroll
        for (int e = 0; e < D / 32; ++e) acc[e] += ds * kr[e];
      }
    }
#pragma unroll
    for (int e = 0; e < D / 32; ++e) dq[(t * Hq + h) * D + lane * (D / 32) + e] = from_f<T>(acc[e] * scale);
  }
}

// grid (key tiles, Hkv); warp w takes keys k_start + w, + kWarps, ...
template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) dkv_core_kernel(BwdPlan plan, int32_t G, const T* __restrict__ q,
                                                               const T* __restrict__ k, const T* __restrict__ v,
                                                               const T* __restrict__ dout,
                                                               const float* __restrict__ lse,
                                                               const float* __restrict__ delta, T* __restrict__ dk,
                                                               T* __restrict__ dv, int64_t T_, int32_t Hq,
                                                               int32_t Hkv, float scale) {
  const BwdItem it = plan.items[blockIdx.x];
  const int g = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int64_t j = it.k_start + warp; j < it.k_start + it.k_len; j += kWarps) {
    float kr[D / 32], vr[D / 32], dka[D / 32], dva[D / 32];
    load_row<T, D>(k + (j * Hkv + g) * D, lane, kr);
    load_row<T, D>(v + (j * Hkv + g) * D, lane, vr);
#pragma unroll
    for (int e = 0; e < D / 32; ++e) dka[e] = dva[e] = 0.f;
    for (int ei = 0; ei < it.e_count; ++ei) {
      const BwdEntry be = plan.entries[it.e_first + ei];
      if (j < be.k_lo || j >= be.k_hi) continue;
      const int64_t t0 = be.causal ? max(static_cast<int64_t>(be.q_lo), j) : be.q_lo;
      for (int64_t t = t0; t < be.q_hi; ++t) {
        for (int hh = 0; hh < G; ++hh) {
          const int h = g * G + hh;
          float qr[D / 32], dor[D / 32];
          load_row<T, D>(q + (t * Hq + h) * D, lane, qr);
          load_row<T, D>(dout + (t * Hq + h) * D, lane, dor);
          float sd = 0.f, pd = 0.f;
#pragma unroll
          for (int e = 0; e < D / 32; ++e) {
            sd += qr[e] * kr[e];
            pd += dor[e] * vr[e];
          }
          sd = warp_sum(sd);
          pd = warp_sum(pd);
          const float p = expf(sd * scale - lse[h * T_ + t]);
          const float ds = p * (pd - delta[h * T_ + t]);
#pragma unroll
          for (int e = 0; e < D / 32; ++e) {
            dka[e] += ds * qr[e];
            dva[e] += p * dor[e];
          }
        }
      }
    }
#pragma unroll
    for (int e = 0; e < D / 32; ++e) {
      dk[(j * Hkv + g) * D + lane * (D / 32) + e] = from_f<T>(dka[e] * scale);
      dv[(j * Hkv + g) * D + lane * (D / 32) + e] = from_f<T>(dva[e]);
    }
  }
}

template <typename T, int D>
int launch_delta(const BwdArgs& a, cudaStream_t s, std::string* err) {
  const int64_t warps = a.T * a.Hq;
  delta_kernel<T, D><<<static_cast<unsigned>((warps * 32 + 255) / 256), 256, 0, s>>>(
      static_cast<const T*>(a.o), static_cast<const T*>(a.dout), a.delta, a.T, a.Hq);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *err = std::string("delta launch: ") + cudaGetErrorString(e);
    return PADOC_ERR_CUDA;
  }
  return PADOC_OK;
}

template <typename T, int D>
int launch_typed(const BwdArgs& a, cudaStream_t s, std::string* err) {
  const T* q = static_cast<const T*>(a.q);
  const T* k = static_cast<const T*>(a.k);
  const T* v = static_cast<const T*>(a.v);
  const T* o = static_cast<const T*>(a.o);
  const T* dout = static_cast<const T*>(a.dout);
  const int64_t warps = a.T * a.Hq;
  delta_kernel<T, D><<<static_cast<unsigned>((warps * 32 + 255) / 256), 256, 0, s>>>(o, dout, a.delta, a.T, a.Hq);
  if (a.fwd.n_items > 0)
    dq_core_kernel<T, D><<<dim3(a.fwd.n_items, a.Hkv), kWarps * 32, 0, s>>>(
        a.fwd, q, k, v, dout, a.lse, a.delta, static_cast<T*>(a.dq), a.T, a.Hq, a.Hkv, a.scale);
  if (a.bwd.n_items > 0)
    dkv_core_kernel<T, D><<<dim3(a.bwd.n_items, a.Hkv), kWarps * 32, 0, s>>>(
        a.bwd, a.Hq / a.Hkv, q, k, v, dout, a.lse, a.delta, static_cast<T*>(a.dk), static_cast<T*>(a.dv), a.T,
        a.Hq, a.Hkv, a.scale);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *err = std::string("backward launch: ") + cudaGetErrorString(e);
    return PADOC_ERR_CUDA;
  }
  return PADOC_OK;
}

}  // namespace

int launch_bwd_delta(const BwdArgs& a, int32_t dtype, cudaStream_t s, std::string* err) {
  if (dtype == PADOC_BF16)
    return a.d == 128 ? launch_delta<__nv_bfloat16, 128>(a, s, err) : launch_delta<__nv_bfloat16, 64>(a, s, err);
  return a.d == 128 ? launch_delta<float, 128>(a, s, err) : launch_delta<float, 64>(a, s, err);
}

int launch_bwd_core(const BwdArgs& a, int32_t dtype, cudaStream_t s, std::string* err) {
  if (dtype == PADOC_BF16)
    return a.d == 128 ? launch_typed<__nv_bfloat16, 128>(a, s, err) : launch_typed<__nv_bfloat16, 64>(a, s, err);
  return a.d == 128 ? launch_typed<float, 128>(a, s, err) : launch_typed<float, 64>(a, s, err);
}

}  // namespace padoc
