// Accept step of speculative verify, and the commit of accepted keys/values.
//
// The verify step leaves, for every query row (draft node) of every branch,
// the model's next-token logits.  Accepting is two launches:
//
//  1. row_argmax_kernel, one CTA per (branch, node): the argmax u_hat of the
//     node's logit row, lowest token index on ties.  The row is streamed once
//     from HBM with 16-byte loads; each thread keeps the packed-bf16 maximum
//     of every 8-token chunk and remembers the first chunk that holds its
//     running maximum, so only one chunk per thread is searched for the exact
//     index.  The index is parked in the branch's slot of `path`.
//  2. accept_walk_kernel, one thread per branch: the greedy tree traversal of
//     the HSD page.  From the anchor (node 0), among the children of the
//     current node take the one whose token has the largest logit (lowest node
//     index on ties) and accept it when
//         logit(child) - logit(u_hat) >= log(tau)
//     (the log-probability difference of the page: the softmax normaliser
//     cancels); stop otherwise or at a leaf.  The free token is u_hat at the
//     last accepted node.  tau = 1 is HPD-Parsing's greedy chain rule: a
//     drafted token is kept while it is the target's argmax.
//
// commit_kernel scatters listed rows of k_new / v_new into pool blocks chosen
// on the host (one thread per 16-byte chunk).
#include <cuda_bf16.h>

#include <algorithm>
#include <string>

#include "../../include/padoc.h"
#include "padoc_internal.h"

namespace padoc {
namespace {

constexpr int kArgThreads = 256;
constexpr int kArgUnroll = 4;
constexpr int kWalkThreads = 128;
constexpr int kMaxNodes = 16;

__device__ __forceinline__ void take_better(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

__device__ __forceinline__ float chunk_max(const uint4& u) {
  __nv_bfloat162 a = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&u.x),
                             *reinterpret_cast<const __nv_bfloat162*>(&u.y));
  const __nv_bfloat162 c = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&u.z),
                                   *reinterpret_cast<const __nv_bfloat162*>(&u.w));
  a = __hmax2(a, c);
  return fmaxf(__low2float(a), __high2float(a));
}

__device__ __forceinline__ float bf16_at(const uint4& u, int e) {
  const uint32_t w = e < 2 ? u.x : e < 4 ? u.y : e < 6 ? u.z : u.w;
  return __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
}

// grid (n_branches, max_nodes); CTA (b, i) takes row q_offsets[b] + i.
__global__ void __launch_bounds__(kArgThreads) row_argmax_kernel(const __nv_bfloat16* __restrict__ logits, int64_t V,
                                                                 int32_t nq, const int32_t* __restrict__ q_offsets,
                                                                 int32_t* __restrict__ path) {
  const int b = blockIdx.x, i = blockIdx.y;
  const int64_t q0 = q_offsets[b], q1 = q_offsets[b + 1];
  if (q0 < 0 || i >= q1 - q0 || q0 + i >= nq) return;
  const __nv_bfloat16* row = logits + (q0 + i) * V;
  float best = -INFINITY;
  int arg = 0x7fffffff;
  if ((V & 7) == 0 && (reinterpret_cast<uintptr_t>(logits) & 15) == 0) {
    const uint4* r4 = reinterpret_cast<const uint4*>(row);
    const int64_t n4 = V >> 3;
    int64_t bx = -1;
    uint4 bu = make_uint4(0, 0, 0, 0);
    for (int64_t x = threadIdx.x; x < n4; x += kArgThreads * kArgUnroll) {
      uint4 u[kArgUnroll];
#pragma unroll
      for (int k = 0; k < kArgUnroll; ++k)
        if (x + k * kArgThreads < n4) u[k] = __ldcs(r4 + x + k * kArgThreads);
#pragma unroll
      for (int k = 0; k < kArgUnroll; ++k) {
        if (x + k * kArgThreads >= n4) break;
        const float m = chunk_max(u[k]);
        if (bx < 0 || m > best) {  // strict: keep this thread's first chunk holding its maximum
          best = m;
          bx = x + k * kArgThreads;
          bu = u[k];
        }
      }
    }
    if (bx >= 0) {
      int e = 0;
      while (e < 7 && bf16_at(bu, e) != best) ++e;
      arg = static_cast<int>(8 * bx + e);
    }
  } else {
    for (int64_t x = threadIdx.x; x < V; x += kArgThreads) take_better(best, arg, __bfloat162float(row[x]), static_cast<int>(x));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, best, off);
    const int i2 = __shfl_xor_sync(0xffffffffu, arg, off);
    take_better(best, arg, v2, i2);
  }
  __shared__ float s_v[kArgThreads / 32];
  __shared__ int s_i[kArgThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    s_v[warp] = best;
    s_i[warp] = arg;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kArgThreads / 32; ++w) take_better(best, arg, s_v[w], s_i[w]);
    path[static_cast<int64_t>(b) * kMaxNodes + i] = arg;
  }
}

__global__ void __launch_bounds__(kWalkThreads) accept_walk_kernel(
    const __nv_bfloat16* __restrict__ logits, int64_t V, int32_t nq, const int32_t* __restrict__ tokens,
    const int32_t* __restrict__ parents, const int32_t* __restrict__ q_offsets, int32_t n_branches, int32_t max_nodes,
    float log_tau, int32_t* __restrict__ n_acc, int32_t* __restrict__ path, int32_t* __restrict__ free_token) {
  const int b = blockIdx.x * kWalkThreads + threadIdx.x;
  if (b >= n_branches) return;
  int32_t* pb = path + static_cast<int64_t>(b) * kMaxNodes;
  const int64_t q0 = q_offsets[b], n = q_offsets[b + 1] - q0;
  bool ok = q0 >= 0 && n >= 1 && n <= max_nodes && q0 + n <= nq && parents[q0] == -1;
  for (int c = 1; ok && c < n; ++c) {
    const int p = parents[q0 + c], t = tokens[q0 + c];
    ok = p >= 0 && p < c && t >= 0 && t < V;
  }
  for (int c = 0; ok && c < n; ++c) ok = pb[c] >= 0 && pb[c] < V;  // argmaxes parked by row_argmax_kernel
  if (!ok) {
    for (int k = 0; k < kMaxNodes; ++k) pb[k] = -1;
    n_acc[b] = -1;
    free_token[b] = -1;
    return;
  }
  // The walk writes accepted node indices into pb[0..cnt) while the argmax of
  // node s still sits in pb[s]; s >= cnt at every read, so no parked value
  // is read after it has been overwritten.
  int cnt = 0, s = 0;
  int u_hat = pb[0];
  while (true) {
    const __nv_bfloat16* row = logits + (q0 + s) * V;
    int bestc = -1;
    float bestv = -INFINITY;
    for (int c = s + 1; c < n; ++c) {
      if (parents[q0 + c] != s) continue;
      const float v = __bfloat162float(row[tokens[q0 + c]]);
      if (bestc < 0 || v > bestv) {
        bestc = c;
        bestv = v;
      }
    }
    if (bestc < 0 || !(bestv - __bfloat162float(row[u_hat]) >= log_tau)) break;
    pb[cnt++] = bestc;
    s = bestc;
    u_hat = pb[s];
  }
  for (int k = cnt; k < kMaxNodes; ++k) pb[k] = -1;
  n_acc[b] = cnt;
  free_token[b] = u_hat;
}

__global__ void commit_kernel(uint4* __restrict__ kpool, uint4* __restrict__ vpool, const int4* __restrict__ plan,
                              int64_t n_rows, int32_t Hkv, const uint4* __restrict__ k, const uint4* __restrict__ v) {
  const int64_t total = n_rows * Hkv * 16;
  for (int64_t x = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; x < total;
       x += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(x & 15);
    const int h = static_cast<int>((x >> 4) % Hkv);
    const int64_t e = (x >> 4) / Hkv;
    const int4 pe = plan[e];  // source row, block, slot
    const int64_t src = (static_cast<int64_t>(pe.x) * Hkv + h) * 16 + c;
    const int64_t dst = ((static_cast<int64_t>(pe.y) * Hkv + h) * 16 + pe.z) * 16 + c;
    kpool[dst] = k[src];
    vpool[dst] = v[src];
  }
}

int launch_error(const char* what, std::string* err) {
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) return PADOC_OK;
  *err = std::string(what) + ": " + cudaGetErrorString(e);
  return PADOC_ERR_CUDA;
}

}  // namespace

int launch_accept(const void* logits, int64_t V, int32_t nq, const int32_t* tokens, const int32_t* parents,
                  const int32_t* q_offsets, int32_t n_branches, int32_t max_nodes, float log_tau, int32_t* n_acc,
                  int32_t* path, int32_t* free_token, cudaStream_t s, std::string* err) {
  if (n_branches == 0) return PADOC_OK;
  const __nv_bfloat16* lg = static_cast<const __nv_bfloat16*>(logits);
  row_argmax_kernel<<<dim3(n_branches, max_nodes), kArgThreads, 0, s>>>(lg, V, nq, q_offsets, path);
  int rc = launch_error("row_argmax launch", err);
  if (rc) return rc;
  accept_walk_kernel<<<(n_branches + kWalkThreads - 1) / kWalkThreads, kWalkThreads, 0, s>>>(
      lg, V, nq, tokens, parents, q_offsets, n_branches, max_nodes, log_tau, n_acc, path, free_token);
  return launch_error("accept_walk launch", err);
}

int launch_commit(void* k_pool, void* v_pool, const void* plan, int64_t n_rows, int32_t Hkv, const void* k,
                  const void* v, cudaStream_t s, std::string* err) {
  if (n_rows == 0) return PADOC_OK;
  const int64_t total = n_rows * Hkv * 16;
  const int grid = static_cast<int>(std::min<int64_t>((total + 255) / 256, 8 * 1024));
  commit_kernel<<<grid, 256, 0, s>>>(static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool),
                                     static_cast<const int4*>(plan), n_rows, Hkv, static_cast<const uint4*>(k),
                                     static_cast<const uint4*>(v));
  return launch_error("commit launch", err);
}

}  // namespace padoc
