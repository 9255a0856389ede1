// libpadoc host side: error reporting, the tree-descriptor builder, the
// refcounted paged KV pool, decode planning and the C ABI entry points.
#include "../../include/padoc.h"
#include "padoc_internal.h"

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <memory>
#include <new>
#include <numeric>
#include <string>
#include <vector>

using namespace padoc;

// ============================================================== errors

static thread_local std::string g_last_error;

static int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

static int cuda_fail(cudaError_t e, const char* what) {
  return fail(PADOC_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define PADOC_TRY(...)                                                      \
  try {                                                                     \
    __VA_ARGS__;                                                            \
  } catch (const std::bad_alloc&) {                                         \
    return fail(PADOC_ERR_OOM, "host allocation failed");                   \
  } catch (...) {                                                           \
    return fail(PADOC_ERR_INVALID, "unexpected host exception");            \
  }

extern "C" const char* padoc_last_error(void) { return g_last_error.c_str(); }
extern "C" int padoc_version(void) { return 100; }

namespace padoc {

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
  return n > 0 ? n : 148;
}

EncodeTiledFn get_encode_fn(std::string* err) {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  if (!fn && err) *err = "cuTensorMapEncodeTiled is not available from the driver";
  return fn;
}

}  // namespace padoc

// ============================================================== tree descriptor

struct Run {
  int64_t start, len;
  bool causal;
};

struct DevPlan {
  int device = -1;
  int group = 0;
  int tile_tokens = 0;
  QSeg* qsegs = nullptr;
  KVSeg* kvsegs = nullptr;
  FwdItem* items = nullptr;
  int32_t n_items = 0;
  BwdItem* bitems = nullptr;
  BwdEntry* bentries = nullptr;
};

struct padoc_tree_desc {
  int64_t T = 0;
  int64_t pairs = 0;
  std::vector<QSeg> qsegs;
  std::vector<KVSeg> kvsegs;
  std::vector<BwdItem> bitems;
  std::vector<BwdEntry> bentries;
  std::vector<DevPlan> dev;
  ~padoc_tree_desc() {
    for (auto& d : dev) {
      int cur = -1;
      cudaGetDevice(&cur);
      if (d.device >= 0) cudaSetDevice(d.device);
      cudaFree(d.qsegs);
      cudaFree(d.kvsegs);
      cudaFree(d.items);
      cudaFree(d.bitems);
      cudaFree(d.bentries);
      if (cur >= 0) cudaSetDevice(cur);
    }
  }
};

// Transposes the query segments' key lists onto the global key-tile grid
// (the key-stationary half of the backward).  Tiles stay in position order:
// the kernel draws them in order as CTAs free up, so the CTAs at work at one
// time hold key tiles of one page and share its queries' Q and dO in L2
// (a kv head's Q and dO exceed L2); a page's prefix tiles, seen by the most
// queries, come before its content tiles.
static void build_bwd(padoc_tree_desc* desc) {
  const int64_t ntiles = (desc->T + kTileKeys - 1) / kTileKeys;
  std::vector<std::vector<BwdEntry>> per(ntiles);
  for (const QSeg& s : desc->qsegs) {
    for (int32_t j = 0; j < s.kv_count; ++j) {
      const KVSeg& e = desc->kvsegs[s.kv_first + j];
      if (e.len <= 0) continue;
      for (int64_t i = e.start / kTileKeys; i <= (static_cast<int64_t>(e.start) + e.len - 1) / kTileKeys; ++i) {
        BwdEntry b{};
        b.k_lo = static_cast<int32_t>(std::max<int64_t>(e.start, i * kTileKeys));
        b.k_hi = static_cast<int32_t>(std::min<int64_t>(static_cast<int64_t>(e.start) + e.len, (i + 1) * kTileKeys));
        b.causal = e.causal;
        b.q_lo = e.causal ? std::max(s.q_start, b.k_lo) : s.q_start;
        b.q_hi = s.q_start + s.q_len;
        if (b.q_lo >= b.q_hi) continue;
        per[i].push_back(b);
      }
    }
  }
  std::vector<int64_t> order;
  for (int64_t i = 0; i < ntiles; ++i)
    if (!per[i].empty()) order.push_back(i);
  desc->bitems.clear();
  desc->bentries.clear();
  for (int64_t i : order) {
    BwdItem it;
    it.k_start = static_cast<int32_t>(i * kTileKeys);
    it.k_len = static_cast<int32_t>(std::min<int64_t>(kTileKeys, desc->T - i * kTileKeys));
    it.e_first = static_cast<int32_t>(desc->bentries.size());
    it.e_count = static_cast<int32_t>(per[i].size());
    desc->bitems.push_back(it);
    desc->bentries.insert(desc->bentries.end(), per[i].begin(), per[i].end());
  }
}

namespace {

// Query region with its key runs, in packing order.
struct Region {
  int64_t q_start, q_len;
  std::vector<Run> runs;  // ordered; the last is causal and contains the queries
};

// Merges position-adjacent runs; a full run directly before the causal run
// joins it (all of its keys precede every query of the region).
std::vector<Run> merge_runs(const std::vector<Run>& in) {
  std::vector<Run> out;
  for (const Run& r : in) {
    if (r.len <= 0 && !r.causal) continue;
    if (!out.empty() && out.back().start + out.back().len == r.start && !out.back().causal) {
      out.back().len += r.len;
      out.back().causal = r.causal;
    } else {
      out.push_back(r);
    }
  }
  return out;
}

// Region B may extend region A (same key runs, causal run grown to cover B).
bool extends(const Region& a, const Region& b) {
  if (a.q_start + a.q_len != b.q_start || a.runs.size() != b.runs.size()) return false;
  for (size_t i = 0; i + 1 < a.runs.size(); ++i)
    if (a.runs[i].start != b.runs[i].start || a.runs[i].len != b.runs[i].len ||
        a.runs[i].causal != b.runs[i].causal)
      return false;
  const Run& ra = a.runs.back();
  const Run& rb = b.runs.back();
  return ra.causal && rb.causal && ra.start == rb.start && ra.start + ra.len == a.q_start + a.q_len &&
         rb.start + rb.len == b.q_start + b.q_len;
}

}  // namespace

extern "C" int padoc_tree_desc_build(const padoc_tree_spec* spec, padoc_tree_desc** out) {
  if (!spec || !out) return fail(PADOC_ERR_INVALID, "tree_desc_build: null argument");
  *out = nullptr;
  if (spec->n_pages < 0) return fail(PADOC_ERR_INVALID, "tree_desc_build: n_pages < 0");
  if (spec->order != PADOC_PACK_CANONICAL && spec->order != PADOC_PACK_DOCUMENT)
    return fail(PADOC_ERR_INVALID, "tree_desc_build: unknown packing order %d", spec->order);
  if (spec->n_pages > 0 && (!spec->prefix_len || !spec->n_regions))
    return fail(PADOC_ERR_INVALID, "tree_desc_build: null page arrays");
  padoc_tree_desc* d = nullptr;
  PADOC_TRY({
    std::unique_ptr<padoc_tree_desc> desc(new padoc_tree_desc());
    int64_t off = 0;
    int64_t ridx = 0;
    std::vector<Region> regions;
    for (int32_t p = 0; p < spec->n_pages; ++p) {
      const int64_t P = spec->prefix_len[p];
      const int32_t N = spec->n_regions[p];
      if (P < 0 || N < 0) return fail(PADOC_ERR_INVALID, "tree_desc_build: page %d negative size", p);
      if (N > 0 && (!spec->layout_len || !spec->content_len))
        return fail(PADOC_ERR_INVALID, "tree_desc_build: null region arrays");
      std::vector<int64_t> lay(N), con(N), bpos(N), ypos(N);
      int64_t total = P;
      for (int32_t k = 0; k < N; ++k) {
        lay[k] = spec->layout_len[ridx + k];
        con[k] = spec->content_len[ridx + k];
        if (lay[k] < 0 || con[k] < 0)
          return fail(PADOC_ERR_INVALID, "tree_desc_build: page %d region %d negative length", p, k);
        total += lay[k] + con[k];
      }
      ridx += N;
      if (off + total >= (int64_t(1) << 31))
        return fail(PADOC_ERR_INVALID, "tree_desc_build: more than 2^31 - 1 tokens");
      // positions
      int64_t cur = off + P;
      if (spec->order == PADOC_PACK_CANONICAL) {
        for (int32_t k = 0; k < N; ++k) { bpos[k] = cur; cur += lay[k]; }
        for (int32_t k = 0; k < N; ++k) { ypos[k] = cur; cur += con[k]; }
      } else {
        for (int32_t k = 0; k < N; ++k) {
          bpos[k] = cur; cur += lay[k];
          ypos[k] = cur; cur += con[k];
        }
      }
      // regions in packing order: X, then B/Y by position
      std::vector<Region> page_regions;
      if (P > 0) page_regions.push_back({off, P, {{off, P, true}}});
      for (int32_t k = 0; k < N; ++k) {
        if (lay[k] > 0) {  // Anc(B_k) = {X, B<k} plus B_k up to the query
          std::vector<Run> r{{off, P, false}};
          for (int32_t i = 0; i < k; ++i) r.push_back({bpos[i], lay[i], false});
          r.push_back({bpos[k], lay[k], true});
          page_regions.push_back({bpos[k], lay[k], merge_runs(r)});
        }
        if (con[k] > 0) {  // Anc(Y_k) = {X, B<=k} plus Y_k up to the query
          std::vector<Run> r{{off, P, false}};
          for (int32_t i = 0; i <= k; ++i) r.push_back({bpos[i], lay[i], false});
          r.push_back({ypos[k], con[k], true});
          page_regions.push_back({ypos[k], con[k], merge_runs(r)});
        }
      }
      std::sort(page_regions.begin(), page_regions.end(),
                [](const Region& a, const Region& b) { return a.q_start < b.q_start; });
      for (Region& r : page_regions) {
        if (!regions.empty() && extends(regions.back(), r)) {
          Region& a = regions.back();
          a.q_len += r.q_len;
          a.runs.back().len = r.runs.back().len;
        } else {
          regions.push_back(std::move(r));
        }
      }
      off += total;
    }
    desc->T = off;
    int64_t pairs = 0;
    for (const Region& r : regions) {
      QSeg q;
      q.q_start = static_cast<int32_t>(r.q_start);
      q.q_len = static_cast<int32_t>(r.q_len);
      q.kv_first = static_cast<int32_t>(desc->kvsegs.size());
      q.kv_count = static_cast<int32_t>(r.runs.size());
      desc->qsegs.push_back(q);
      for (const Run& run : r.runs) {
        desc->kvsegs.push_back({static_cast<int32_t>(run.start), static_cast<int32_t>(run.len),
                                run.causal ? 1 : 0, 0});
        if (run.causal) {
          const int64_t a = r.q_start - run.start + 1;  // keys seen by the first query
          pairs += r.q_len * a + r.q_len * (r.q_len - 1) / 2;
        } else {
          pairs += r.q_len * run.len;
        }
      }
    }
    desc->pairs = pairs;
    build_bwd(desc.get());
    d = desc.release();
  });
  *out = d;
  return PADOC_OK;
}

extern "C" int padoc_tree_desc_free(padoc_tree_desc* desc) {
  delete desc;
  return PADOC_OK;
}

extern "C" int padoc_tree_desc_info(const padoc_tree_desc* desc, int64_t* n_tokens, int64_t* n_qsegs,
                                    int64_t* n_kvsegs, int64_t* ancestor_pairs) {
  if (!desc) return fail(PADOC_ERR_INVALID, "tree_desc_info: null descriptor");
  if (n_tokens) *n_tokens = desc->T;
  if (n_qsegs) *n_qsegs = static_cast<int64_t>(desc->qsegs.size());
  if (n_kvsegs) *n_kvsegs = static_cast<int64_t>(desc->kvsegs.size());
  if (ancestor_pairs) *ancestor_pairs = desc->pairs;
  return PADOC_OK;
}

extern "C" int padoc_tree_desc_segments(const padoc_tree_desc* desc, int32_t* qseg, int32_t* kvseg) {
  if (!desc) return fail(PADOC_ERR_INVALID, "tree_desc_segments: null descriptor");
  if (qseg)
    for (size_t i = 0; i < desc->qsegs.size(); ++i) {
      qseg[4 * i + 0] = desc->qsegs[i].q_start;
      qseg[4 * i + 1] = desc->qsegs[i].q_len;
      qseg[4 * i + 2] = desc->qsegs[i].kv_first;
      qseg[4 * i + 3] = desc->qsegs[i].kv_count;
    }
  if (kvseg)
    for (size_t i = 0; i < desc->kvsegs.size(); ++i) {
      kvseg[3 * i + 0] = desc->kvsegs[i].start;
      kvseg[3 * i + 1] = desc->kvsegs[i].len;
      kvseg[3 * i + 2] = desc->kvsegs[i].causal;
    }
  return PADOC_OK;
}

// Query tiles of tile_tokens tokens, longest key walk first (LPT order).
static std::vector<FwdItem> build_items(const padoc_tree_desc* desc, int tile_tokens) {
  struct Cost {
    int64_t cost;
    FwdItem it;
  };
  std::vector<Cost> v;
  for (size_t s = 0; s < desc->qsegs.size(); ++s) {
    const QSeg& q = desc->qsegs[s];
    for (int32_t t0 = q.q_start; t0 < q.q_start + q.q_len; t0 += tile_tokens) {
      const int32_t t1 = std::min(t0 + tile_tokens, q.q_start + q.q_len);
      int64_t c = 0;
      for (int32_t j = 0; j < q.kv_count; ++j) {
        const KVSeg& kv = desc->kvsegs[q.kv_first + j];
        int64_t len = kv.len;
        if (kv.causal) len = std::min<int64_t>(kv.len, t1 - kv.start);
        c += (len + kTileKeys - 1) / kTileKeys;
      }
      FwdItem it{};
      it.qseg = static_cast<int32_t>(s);
      it.tile_start = t0;
      it.n_tiles = static_cast<int32_t>(c);
      it.q_end = q.q_start + q.q_len;
      it.kv_first = q.kv_first;
      it.kv_count = q.kv_count;
      it.tile_last = t1 - 1;
      if (q.kv_count > 0) it.kv0 = desc->kvsegs[q.kv_first];
      v.push_back({c, it});
    }
  }
  std::stable_sort(v.begin(), v.end(), [](const Cost& a, const Cost& b) { return a.cost > b.cost; });
  std::vector<FwdItem> out(v.size());
  for (size_t i = 0; i < v.size(); ++i) out[i] = v[i].it;
  return out;
}

static int upload_desc(padoc_tree_desc* desc, int group, DevPlan** plan_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  for (auto& p : desc->dev)
    if (p.device == dev && p.group == group) {
      *plan_out = &p;
      return PADOC_OK;
    }
  DevPlan p;
  p.device = dev;
  p.group = group;
  p.tile_tokens = kTileRows / group;
  std::vector<FwdItem> items;
  PADOC_TRY(items = build_items(desc, p.tile_tokens));
  p.n_items = static_cast<int32_t>(items.size());
  auto alloc_copy = [](void** dst, const void* src, size_t bytes) -> cudaError_t {
    if (bytes == 0) bytes = 16;
    cudaError_t e2 = cudaMalloc(dst, bytes);
    if (e2 != cudaSuccess) return e2;
    if (src) return cudaMemcpy(*dst, src, bytes, cudaMemcpyHostToDevice);
    return cudaSuccess;
  };
  e = alloc_copy(reinterpret_cast<void**>(&p.qsegs), desc->qsegs.data(), desc->qsegs.size() * sizeof(QSeg));
  if (e == cudaSuccess)
    e = alloc_copy(reinterpret_cast<void**>(&p.kvsegs), desc->kvsegs.data(), desc->kvsegs.size() * sizeof(KVSeg));
  if (e == cudaSuccess)
    e = alloc_copy(reinterpret_cast<void**>(&p.items), items.data(), items.size() * sizeof(FwdItem));
  if (e == cudaSuccess)
    e = alloc_copy(reinterpret_cast<void**>(&p.bitems), desc->bitems.data(), desc->bitems.size() * sizeof(BwdItem));
  if (e == cudaSuccess)
    e = alloc_copy(reinterpret_cast<void**>(&p.bentries), desc->bentries.data(),
                   desc->bentries.size() * sizeof(BwdEntry));
  if (e != cudaSuccess) {
    cudaFree(p.qsegs);
    cudaFree(p.kvsegs);
    cudaFree(p.items);
    cudaFree(p.bitems);
    cudaFree(p.bentries);
    return cuda_fail(e, "tree descriptor upload");
  }
  desc->dev.push_back(p);
  *plan_out = &desc->dev.back();
  return PADOC_OK;
}

static bool valid_group(int g) { return g == 1 || g == 2 || g == 4 || g == 8 || g == 16; }

extern "C" int padoc_tree_desc_upload(padoc_tree_desc* desc, int32_t group) {
  if (!desc) return fail(PADOC_ERR_INVALID, "tree_desc_upload: null descriptor");
  if (!valid_group(group)) return fail(PADOC_ERR_INVALID, "tree_desc_upload: group %d not in {1,2,4,8,16}", group);
  DevPlan* p = nullptr;
  return upload_desc(desc, group, &p);
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

extern "C" int padoc_tree_attn_varlen(padoc_tree_desc* desc, const void* q, const void* k, const void* v,
                                      void* o, float* lse, int32_t dtype, int32_t Hq, int32_t Hkv,
                                      int32_t d, float scale, padoc_stream_t stream) {
  if (!desc) return fail(PADOC_ERR_INVALID, "tree_attn_varlen: null descriptor");
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0)
    return fail(PADOC_ERR_INVALID, "tree_attn_varlen: Hq=%d must be a positive multiple of Hkv=%d", Hq, Hkv);
  const int group = Hq / Hkv;
  if (!valid_group(group)) return fail(PADOC_ERR_UNSUPPORTED, "tree_attn_varlen: Hq/Hkv=%d not in {1,2,4,8,16}", group);
  if (dtype == PADOC_BF16) {
    if (d != kHeadDim) return fail(PADOC_ERR_UNSUPPORTED, "tree_attn_varlen: bf16 path needs d=128 (got %d)", d);
  } else if (dtype == PADOC_F32) {
    if (d != 64 && d != 128) return fail(PADOC_ERR_UNSUPPORTED, "tree_attn_varlen: f32 path needs d in {64,128}");
  } else {
    return fail(PADOC_ERR_INVALID, "tree_attn_varlen: unknown dtype %d", dtype);
  }
  if (desc->T == 0) return PADOC_OK;
  if (!q || !k || !v || !o || !lse) return fail(PADOC_ERR_INVALID, "tree_attn_varlen: null tensor");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return fail(PADOC_ERR_INVALID, "tree_attn_varlen: tensors must be 16-byte aligned");
  DevPlan* plan = nullptr;
  int rc = upload_desc(desc, group, &plan);
  if (rc) return rc;
  FwdArgs a;
  a.plan = {plan->qsegs, plan->kvsegs, plan->items, plan->n_items, group, plan->tile_tokens};
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.T = desc->T;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = d;
  a.scale = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(d));
  std::string err;
  rc = dtype == PADOC_BF16 ? launch_fwd_bf16(a, reinterpret_cast<cudaStream_t>(stream), &err)
                           : launch_fwd_f32(a, reinterpret_cast<cudaStream_t>(stream), &err);
  if (rc) return fail(rc, "tree_attn_varlen: %s", err.c_str());
  return PADOC_OK;
}

// rowsum(dO * O) [Hq, T] f32, then the dK/dV pass's unit counter
static size_t bwd_delta_bytes(const padoc_tree_desc* desc, int32_t Hq) {
  return (static_cast<size_t>(Hq) * desc->T * sizeof(float) + 255) / 256 * 256;
}
static size_t bwd_ws_bytes(const padoc_tree_desc* desc, int32_t Hq) { return bwd_delta_bytes(desc, Hq) + 256; }

extern "C" int padoc_tree_attn_varlen_bwd_ws_size(const padoc_tree_desc* desc, int32_t Hq, size_t* bytes) {
  if (!desc || !bytes) return fail(PADOC_ERR_INVALID, "tree_attn_varlen_bwd_ws_size: null argument");
  if (Hq <= 0) return fail(PADOC_ERR_INVALID, "tree_attn_varlen_bwd_ws_size: Hq must be positive");
  *bytes = bwd_ws_bytes(desc, Hq);
  return PADOC_OK;
}

extern "C" int padoc_tree_attn_varlen_bwd(padoc_tree_desc* desc, const void* q, const void* k, const void* v,
                                          const void* o, const float* lse, const void* d_o, void* dq, void* dk,
                                          void* dv, int32_t dtype, int32_t Hq, int32_t Hkv, int32_t d, float scale,
                                          void* ws, size_t ws_bytes, padoc_stream_t stream) {
  if (!desc) return fail(PADOC_ERR_INVALID, "tree_attn_varlen_bwd: null descriptor");
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0)
    return fail(PADOC_ERR_INVALID, "tree_attn_varlen_bwd: Hq=%d must be a positive multiple of Hkv=%d", Hq, Hkv);
  const int group = Hq / Hkv;
  if (!valid_group(group))
    return fail(PADOC_ERR_UNSUPPORTED, "tree_attn_varlen_bwd: Hq/Hkv=%d not in {1,2,4,8,16}", group);
  if (dtype != PADOC_BF16 && dtype != PADOC_F32) return fail(PADOC_ERR_INVALID, "tree_attn_varlen_bwd: unknown dtype %d", dtype);
  if (d != 64 && d != 128) return fail(PADOC_ERR_UNSUPPORTED, "tree_attn_varlen_bwd: d must be 64 or 128");
  if (desc->T == 0) return PADOC_OK;
  if (!q || !k || !v || !o || !lse || !d_o || !dq || !dk || !dv)
    return fail(PADOC_ERR_INVALID, "tree_attn_varlen_bwd: null tensor");
  for (const void* p : {q, k, v, o, static_cast<const void*>(lse), d_o, static_cast<const void*>(dq),
                        static_cast<const void*>(dk), static_cast<const void*>(dv)})
    if (!aligned16(p)) return fail(PADOC_ERR_INVALID, "tree_attn_varlen_bwd: tensors must be 16-byte aligned");
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < bwd_ws_bytes(desc, Hq))
    return fail(PADOC_ERR_INVALID, "tree_attn_varlen_bwd: ws must be 256-byte aligned and hold %zu bytes",
                bwd_ws_bytes(desc, Hq));
  DevPlan* plan = nullptr;
  int rc = upload_desc(desc, group, &plan);
  if (rc) return rc;
  BwdArgs a;
  a.fwd = {plan->qsegs, plan->kvsegs, plan->items, plan->n_items, group, plan->tile_tokens};
  a.bwd = {plan->bitems, plan->bentries, static_cast<int32_t>(desc->bitems.size())};
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.dout = d_o;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.delta = static_cast<float*>(ws);
  a.work = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + bwd_delta_bytes(desc, Hq));
  a.T = desc->T;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = d;
  a.scale = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(d));
  std::string err;
  // bf16 at d = 128 runs on the tensor cores; PADOC_BWD_CORE=1 selects the
  // CUDA-core kernels instead (a second implementation to compare against)
  static const bool force_core = std::getenv("PADOC_BWD_CORE") && std::atoi(std::getenv("PADOC_BWD_CORE")) != 0;
  if (dtype == PADOC_BF16 && d == kHeadDim && !force_core)
    rc = launch_bwd_tc(a, reinterpret_cast<cudaStream_t>(stream), &err);
  else
    rc = launch_bwd_core(a, dtype, reinterpret_cast<cudaStream_t>(stream), &err);
  if (rc) return fail(rc, "tree_attn_varlen_bwd: %s", err.c_str());
  return PADOC_OK;
}

extern "C" int padoc_tree_desc_bwd_plan(const padoc_tree_desc* desc, int32_t* items, int32_t* entries,
                                        int64_t* n_items, int64_t* n_entries) {
  if (!desc) return fail(PADOC_ERR_INVALID, "tree_desc_bwd_plan: null descriptor");
  if (n_items) *n_items = static_cast<int64_t>(desc->bitems.size());
  if (n_entries) *n_entries = static_cast<int64_t>(desc->bentries.size());
  if (items)
    for (size_t i = 0; i < desc->bitems.size(); ++i) {
      const BwdItem& it = desc->bitems[i];
      int32_t* r = items + 4 * i;
      r[0] = it.k_start;
      r[1] = it.k_len;
      r[2] = it.e_first;
      r[3] = it.e_count;
    }
  if (entries)
    for (size_t i = 0; i < desc->bentries.size(); ++i) {
      const BwdEntry& b = desc->bentries[i];
      int32_t* r = entries + 5 * i;
      r[0] = b.k_lo;
      r[1] = b.k_hi;
      r[2] = b.causal;
      r[3] = b.q_lo;
      r[4] = b.q_hi;
    }
  return PADOC_OK;
}

// ============================================================== KV pool

struct Seq {
  bool live = false;
  int32_t len = 0;       // tokens
  int32_t fork_len = 0;  // leading tokens shared from the fork parent
  int32_t n_shared = 0;  // leading blocks shared from the fork parent
  std::vector<int32_t> blocks;
};

struct padoc_kv_pool {
  void* k = nullptr;
  void* v = nullptr;
  int32_t nb = 0, bs = 16, Hkv = 0, d = 0, dtype = 0, max_seqs = 0, max_bps = 0;
  std::vector<int32_t> refcnt;
  // Free blocks as a stack, lowest id on top at creation.  Blocks go back
  // last first, so a freed run comes out again in ascending order: the
  // decode kernels load 8 physically consecutive blocks of a key tile with
  // one copy.
  std::vector<int32_t> free_blocks;
  std::vector<Seq> seqs;
  std::vector<int32_t> free_seqs;    // stack
  int64_t fault_after = -1;          // fail the allocation that would exceed this count
  int64_t allocated = 0;             // blocks handed out so far
  // device mirror of the block table
  int device = -1;
  int32_t* d_table = nullptr;
  std::vector<int32_t> h_table;
  std::vector<uint8_t> dirty;
  int64_t n_dirty = 0;
  bool zeroed = false;

  ~padoc_kv_pool() {
    if (d_table) {
      int cur = -1;
      cudaGetDevice(&cur);
      cudaSetDevice(device);
      cudaFree(d_table);
      if (cur >= 0) cudaSetDevice(cur);
    }
  }
  bool seq_ok(int32_t s) const { return s >= 0 && s < max_seqs && seqs[s].live; }
  int32_t own_blocks(const Seq& s) const { return static_cast<int32_t>(s.blocks.size()) - s.n_shared; }
  void mark(int32_t s) {
    if (!dirty[s]) {
      dirty[s] = 1;
      ++n_dirty;
    }
    int32_t* row = &h_table[static_cast<size_t>(s) * max_bps];
    const Seq& q = seqs[s];
    std::fill(row, row + max_bps, 0);
    std::copy(q.blocks.begin(), q.blocks.end(), row);
  }
  // Takes n blocks or nothing.
  bool take_blocks(int32_t n, std::vector<int32_t>* out) {
    if (n < 0 || static_cast<size_t>(n) > free_blocks.size()) return false;
    if (fault_after >= 0 && allocated + n > fault_after) return false;
    for (int32_t i = 0; i < n; ++i) {
      const int32_t b = free_blocks.back();
      free_blocks.pop_back();
      refcnt[b] = 1;
      out->push_back(b);
    }
    allocated += n;
    return true;
  }
  void drop_block(int32_t b) {
    if (--refcnt[b] == 0) free_blocks.push_back(b);
  }
  int32_t new_seq() {
    if (free_seqs.empty()) return -1;
    const int32_t s = free_seqs.back();
    free_seqs.pop_back();
    seqs[s] = Seq();
    seqs[s].live = true;
    return s;
  }
};

extern "C" int padoc_kv_pool_create(padoc_kv_pool** out, void* k_pool, void* v_pool, int32_t num_blocks,
                                    int32_t block_size, int32_t Hkv, int32_t d, int32_t dtype,
                                    int32_t max_seqs, int32_t max_blocks_per_seq) {
  if (!out) return fail(PADOC_ERR_INVALID, "kv_pool_create: null out");
  *out = nullptr;
  if (block_size != 16) return fail(PADOC_ERR_UNSUPPORTED, "kv_pool_create: block_size must be 16");
  if (d != 128) return fail(PADOC_ERR_UNSUPPORTED, "kv_pool_create: d must be 128");
  if (dtype != PADOC_BF16) return fail(PADOC_ERR_UNSUPPORTED, "kv_pool_create: dtype must be bf16");
  if (num_blocks <= 0 || Hkv <= 0 || max_seqs <= 0 || max_blocks_per_seq <= 0)
    return fail(PADOC_ERR_INVALID, "kv_pool_create: sizes must be positive");
  if (static_cast<int64_t>(num_blocks) * Hkv * block_size >= (int64_t(1) << 31))
    return fail(PADOC_ERR_UNSUPPORTED, "kv_pool_create: num_blocks * Hkv * 16 must stay below 2^31");
  if ((k_pool && !aligned16(k_pool)) || (v_pool && !aligned16(v_pool)))
    return fail(PADOC_ERR_INVALID, "kv_pool_create: storage must be 16-byte aligned");
  padoc_kv_pool* p = nullptr;
  PADOC_TRY({
    std::unique_ptr<padoc_kv_pool> pool(new padoc_kv_pool());
    pool->k = k_pool;
    pool->v = v_pool;
    pool->nb = num_blocks;
    pool->bs = block_size;
    pool->Hkv = Hkv;
    pool->d = d;
    pool->dtype = dtype;
    pool->max_seqs = max_seqs;
    pool->max_bps = max_blocks_per_seq;
    pool->refcnt.assign(num_blocks, 0);
    pool->free_blocks.resize(num_blocks);
    for (int32_t i = 0; i < num_blocks; ++i) pool->free_blocks[i] = num_blocks - 1 - i;
    pool->seqs.resize(max_seqs);
    pool->free_seqs.resize(max_seqs);
    for (int32_t i = 0; i < max_seqs; ++i) pool->free_seqs[i] = max_seqs - 1 - i;
    pool->h_table.assign(static_cast<size_t>(max_seqs) * max_blocks_per_seq, 0);
    pool->dirty.assign(max_seqs, 0);
    if (const char* f = std::getenv("PADOC_FAULT_ALLOC_AFTER")) pool->fault_after = std::atoll(f);
    p = pool.release();
  });
  *out = p;
  return PADOC_OK;
}

extern "C" int padoc_kv_pool_destroy(padoc_kv_pool* pool) {
  delete pool;
  return PADOC_OK;
}

extern "C" int padoc_kv_alloc(padoc_kv_pool* pool, int32_t n_tokens, int32_t* seq) {
  if (!pool || !seq) return fail(PADOC_ERR_INVALID, "kv_alloc: null argument");
  if (n_tokens < 0) return fail(PADOC_ERR_INVALID, "kv_alloc: n_tokens < 0");
  const int32_t nblk = (n_tokens + pool->bs - 1) / pool->bs;
  if (nblk > pool->max_bps) return fail(PADOC_ERR_INVALID, "kv_alloc: %d blocks exceed max_blocks_per_seq %d", nblk, pool->max_bps);
  if (pool->free_seqs.empty()) return fail(PADOC_ERR_OOM, "kv_alloc: no free sequence slot");
  std::vector<int32_t> blocks;
  PADOC_TRY({
    if (!pool->take_blocks(nblk, &blocks)) return fail(PADOC_ERR_OOM, "kv_alloc: out of blocks (%d wanted)", nblk);
    const int32_t s = pool->new_seq();
    pool->seqs[s].blocks = std::move(blocks);
    pool->mark(s);
    *seq = s;
  });
  return PADOC_OK;
}

extern "C" int padoc_kv_fork(padoc_kv_pool* pool, int32_t parent, int32_t fork_len, int32_t* child) {
  if (!pool || !child) return fail(PADOC_ERR_INVALID, "kv_fork: null argument");
  if (!pool->seq_ok(parent)) return fail(PADOC_ERR_INVALID, "kv_fork: parent %d is not a live sequence", parent);
  const Seq& par = pool->seqs[parent];
  if (fork_len < 0 || fork_len > par.len)
    return fail(PADOC_ERR_INVALID, "kv_fork: fork_len %d outside [0, %d]", fork_len, par.len);
  // token t of the child (t < fork_len) must sit at block t/16, slot t%16 of the parent
  if (fork_len > par.fork_len && par.fork_len % pool->bs != 0)
    return fail(PADOC_ERR_UNSUPPORTED, "kv_fork: parent's own tokens do not start on a block boundary");
  if (pool->free_seqs.empty()) return fail(PADOC_ERR_OOM, "kv_fork: no free sequence slot");
  PADOC_TRY({
    const int32_t nsh = (fork_len + pool->bs - 1) / pool->bs;
    std::vector<int32_t> blocks(par.blocks.begin(), par.blocks.begin() + nsh);
    const int32_t s = pool->new_seq();
    for (int32_t b : blocks) ++pool->refcnt[b];
    Seq& c = pool->seqs[s];
    c.blocks = std::move(blocks);
    c.len = fork_len;
    c.fork_len = fork_len;
    c.n_shared = nsh;
    pool->mark(s);
    *child = s;
  });
  return PADOC_OK;
}

extern "C" int padoc_kv_reserve(padoc_kv_pool* pool, int32_t seq, int32_t n_tokens) {
  if (!pool) return fail(PADOC_ERR_INVALID, "kv_reserve: null pool");
  if (!pool->seq_ok(seq)) return fail(PADOC_ERR_INVALID, "kv_reserve: %d is not a live sequence", seq);
  if (n_tokens < 0) return fail(PADOC_ERR_INVALID, "kv_reserve: n_tokens < 0");
  Seq& s = pool->seqs[seq];
  const int64_t need = (static_cast<int64_t>(s.len - s.fork_len) + n_tokens + pool->bs - 1) / pool->bs;
  const int64_t have = pool->own_blocks(s);
  if (s.n_shared + need > pool->max_bps)
    return fail(PADOC_ERR_INVALID, "kv_reserve: sequence would exceed max_blocks_per_seq");
  if (need > have) {
    std::vector<int32_t> extra;
    PADOC_TRY({
      if (!pool->take_blocks(static_cast<int32_t>(need - have), &extra))
        return fail(PADOC_ERR_OOM, "kv_reserve: out of blocks");
      s.blocks.insert(s.blocks.end(), extra.begin(), extra.end());
      pool->mark(seq);
    });
  }
  return PADOC_OK;
}

extern "C" int padoc_kv_advance(padoc_kv_pool* pool, int32_t seq, int32_t n) {
  if (!pool) return fail(PADOC_ERR_INVALID, "kv_advance: null pool");
  if (!pool->seq_ok(seq)) return fail(PADOC_ERR_INVALID, "kv_advance: %d is not a live sequence", seq);
  if (n < 0) return fail(PADOC_ERR_INVALID, "kv_advance: n < 0");
  Seq& s = pool->seqs[seq];
  if (static_cast<int64_t>(s.len - s.fork_len) + n > static_cast<int64_t>(pool->own_blocks(s)) * pool->bs)
    return fail(PADOC_ERR_INVALID, "kv_advance: %d tokens exceed the reserved slots", n);
  s.len += n;
  return PADOC_OK;
}

extern "C" int padoc_kv_trim(padoc_kv_pool* pool, int32_t seq) {
  if (!pool) return fail(PADOC_ERR_INVALID, "kv_trim: null pool");
  if (!pool->seq_ok(seq)) return fail(PADOC_ERR_INVALID, "kv_trim: %d is not a live sequence", seq);
  Seq& s = pool->seqs[seq];
  const size_t keep = static_cast<size_t>(s.n_shared) + (s.len - s.fork_len + pool->bs - 1) / pool->bs;
  if (s.blocks.size() > keep) {
    for (size_t i = s.blocks.size(); i-- > keep;) pool->drop_block(s.blocks[i]);
    s.blocks.resize(keep);
    pool->mark(seq);
  }
  return PADOC_OK;
}

extern "C" int padoc_kv_release(padoc_kv_pool* pool, int32_t seq) {
  if (!pool) return fail(PADOC_ERR_INVALID, "kv_release: null pool");
  if (!pool->seq_ok(seq)) return fail(PADOC_ERR_INVALID, "kv_release: %d is not a live sequence", seq);
  Seq& s = pool->seqs[seq];
  for (size_t i = s.blocks.size(); i-- > 0;) pool->drop_block(s.blocks[i]);
  s = Seq();
  pool->mark(seq);
  pool->free_seqs.push_back(seq);
  return PADOC_OK;
}

extern "C" int padoc_kv_seq_info(const padoc_kv_pool* pool, int32_t seq, int32_t* length, int32_t* fork_len,
                                 int32_t* n_blocks) {
  if (!pool) return fail(PADOC_ERR_INVALID, "kv_seq_info: null pool");
  if (!pool->seq_ok(seq)) return fail(PADOC_ERR_INVALID, "kv_seq_info: %d is not a live sequence", seq);
  const Seq& s = pool->seqs[seq];
  if (length) *length = s.len;
  if (fork_len) *fork_len = s.fork_len;
  if (n_blocks) *n_blocks = static_cast<int32_t>(s.blocks.size());
  return PADOC_OK;
}

extern "C" int padoc_kv_seq_blocks(const padoc_kv_pool* pool, int32_t seq, int32_t* out, int32_t cap) {
  if (!pool || !out) return fail(PADOC_ERR_INVALID, "kv_seq_blocks: null argument");
  if (!pool->seq_ok(seq)) return fail(PADOC_ERR_INVALID, "kv_seq_blocks: %d is not a live sequence", seq);
  const Seq& s = pool->seqs[seq];
  if (cap < static_cast<int32_t>(s.blocks.size())) return fail(PADOC_ERR_INVALID, "kv_seq_blocks: capacity too small");
  std::copy(s.blocks.begin(), s.blocks.end(), out);
  return PADOC_OK;
}

extern "C" int padoc_kv_block_refcount(const padoc_kv_pool* pool, int32_t block, int32_t* refcount) {
  if (!pool || !refcount) return fail(PADOC_ERR_INVALID, "kv_block_refcount: null argument");
  if (block < 0 || block >= pool->nb) return fail(PADOC_ERR_INVALID, "kv_block_refcount: block out of range");
  *refcount = pool->refcnt[block];
  return PADOC_OK;
}

extern "C" int padoc_kv_pool_stats(const padoc_kv_pool* pool, int32_t* free_blocks, int32_t* live_seqs) {
  if (!pool) return fail(PADOC_ERR_INVALID, "kv_pool_stats: null pool");
  if (free_blocks) *free_blocks = static_cast<int32_t>(pool->free_blocks.size());
  if (live_seqs) *live_seqs = pool->max_seqs - static_cast<int32_t>(pool->free_seqs.size());
  return PADOC_OK;
}

static int pool_sync(padoc_kv_pool* pool, cudaStream_t stream) {
  cudaError_t e;
  if (!pool->d_table) {
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    e = cudaMalloc(&pool->d_table, pool->h_table.size() * sizeof(int32_t));
    if (e != cudaSuccess) {
      pool->d_table = nullptr;
      return cuda_fail(e, "kv pool table allocation");
    }
    pool->device = dev;
    std::fill(pool->dirty.begin(), pool->dirty.end(), 1);
    pool->n_dirty = pool->max_seqs;
  }
  if (!pool->zeroed && pool->k && pool->v) {
    // Unwritten slots of a partly filled block are read (and masked) by the
    // kernels; zeroing once keeps them finite.
    const size_t bytes = static_cast<size_t>(pool->nb) * pool->Hkv * pool->bs * pool->d * 2;
    e = cudaMemsetAsync(pool->k, 0, bytes, stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(pool->v, 0, bytes, stream);
    if (e != cudaSuccess) return cuda_fail(e, "kv pool zero fill");
    pool->zeroed = true;
  }
  if (pool->n_dirty == 0) return PADOC_OK;
  const size_t row = static_cast<size_t>(pool->max_bps);
  if (pool->n_dirty > 64) {
    int32_t lo = pool->max_seqs, hi = -1;
    for (int32_t s = 0; s < pool->max_seqs; ++s)
      if (pool->dirty[s]) {
        lo = std::min(lo, s);
        hi = std::max(hi, s);
      }
    e = cudaMemcpyAsync(pool->d_table + lo * row, pool->h_table.data() + lo * row,
                        (hi - lo + 1) * row * sizeof(int32_t), cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return cuda_fail(e, "kv pool table upload");
  } else {
    for (int32_t s = 0; s < pool->max_seqs; ++s)
      if (pool->dirty[s]) {
        e = cudaMemcpyAsync(pool->d_table + s * row, pool->h_table.data() + s * row, row * sizeof(int32_t),
                            cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess) return cuda_fail(e, "kv pool table upload");
      }
  }
  std::fill(pool->dirty.begin(), pool->dirty.end(), 0);
  pool->n_dirty = 0;
  return PADOC_OK;
}

extern "C" int padoc_kv_pool_device(const padoc_kv_pool* pool, int32_t* device) {
  if (!pool || !device) return fail(PADOC_ERR_INVALID, "kv_pool_device: null argument");
  *device = pool->d_table ? pool->device : -1;
  return PADOC_OK;
}

extern "C" int padoc_debug_kv_pool_rehome(padoc_kv_pool* pool, int32_t device) {
  if (!pool) return fail(PADOC_ERR_INVALID, "debug_kv_pool_rehome: null pool");
  if (!pool->d_table) return fail(PADOC_ERR_INVALID, "debug_kv_pool_rehome: the pool has no device table yet");
  pool->device = device;
  return PADOC_OK;
}

extern "C" int padoc_kv_pool_sync(padoc_kv_pool* pool, padoc_stream_t stream) {
  if (!pool) return fail(PADOC_ERR_INVALID, "kv_pool_sync: null pool");
  return pool_sync(pool, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int padoc_kv_append(padoc_kv_pool* pool, int32_t seq, const void* k, const void* v, int32_t n,
                               padoc_stream_t stream) {
  if (!pool) return fail(PADOC_ERR_INVALID, "kv_append: null pool");
  if (!pool->seq_ok(seq)) return fail(PADOC_ERR_INVALID, "kv_append: %d is not a live sequence", seq);
  if (n < 0) return fail(PADOC_ERR_INVALID, "kv_append: n < 0");
  if (n == 0) return PADOC_OK;
  if (!k || !v || !aligned16(k) || !aligned16(v)) return fail(PADOC_ERR_INVALID, "kv_append: k/v must be 16-byte aligned device pointers");
  if (!pool->k || !pool->v) return fail(PADOC_ERR_INVALID, "kv_append: pool has no storage");
  Seq& s = pool->seqs[seq];
  const int32_t own = s.len - s.fork_len;
  const int64_t need_tokens = static_cast<int64_t>(own) + n;
  const int64_t need_blocks = (need_tokens + pool->bs - 1) / pool->bs;
  const int64_t have = pool->own_blocks(s);
  if (s.n_shared + need_blocks > pool->max_bps)
    return fail(PADOC_ERR_INVALID, "kv_append: sequence would exceed max_blocks_per_seq");
  if (need_blocks > have) {
    std::vector<int32_t> extra;
    PADOC_TRY({
      if (!pool->take_blocks(static_cast<int32_t>(need_blocks - have), &extra))
        return fail(PADOC_ERR_OOM, "kv_append: out of blocks");
      s.blocks.insert(s.blocks.end(), extra.begin(), extra.end());
    });
  }
  s.len += n;
  pool->mark(seq);
  int rc = pool_sync(pool, reinterpret_cast<cudaStream_t>(stream));
  if (rc) return rc;
  std::string err;
  rc = launch_kv_append(pool->k, pool->v, pool->d_table + static_cast<size_t>(seq) * pool->max_bps + s.n_shared, own, n,
                        pool->Hkv, pool->d, k, v, reinterpret_cast<cudaStream_t>(stream), &err);
  if (rc) return fail(rc, "kv_append: %s", err.c_str());
  return PADOC_OK;
}

extern "C" int padoc_kv_commit(padoc_kv_pool* pool, int32_t n_seqs, const int32_t* seqs, const int32_t* row_offsets,
                               const int32_t* rows, int32_t n_src_rows, const void* k_new, const void* v_new,
                               void* ws, size_t ws_bytes, padoc_stream_t stream) {
  if (!pool) return fail(PADOC_ERR_INVALID, "kv_commit: null pool");
  if (n_seqs < 0) return fail(PADOC_ERR_INVALID, "kv_commit: n_seqs < 0");
  if (n_seqs == 0) return PADOC_OK;
  if (!seqs || !row_offsets) return fail(PADOC_ERR_INVALID, "kv_commit: null seqs / row_offsets");
  if (row_offsets[0] != 0) return fail(PADOC_ERR_INVALID, "kv_commit: row_offsets[0] must be 0");
  for (int32_t i = 0; i < n_seqs; ++i)
    if (row_offsets[i + 1] < row_offsets[i]) return fail(PADOC_ERR_INVALID, "kv_commit: row_offsets decrease at %d", i);
  const int64_t total = row_offsets[n_seqs];
  if (total > 0 && !rows) return fail(PADOC_ERR_INVALID, "kv_commit: null rows");
  for (int64_t j = 0; j < total; ++j)
    if (rows[j] < 0 || rows[j] >= n_src_rows)
      return fail(PADOC_ERR_INVALID, "kv_commit: rows[%lld] = %d outside [0, %d)", static_cast<long long>(j), rows[j],
                  n_src_rows);
  std::vector<int64_t> extra(n_seqs, 0);
  int64_t extra_total = 0;
  PADOC_TRY({
    std::vector<uint8_t> seen(pool->max_seqs, 0);
    for (int32_t i = 0; i < n_seqs; ++i) {
      const int32_t q = seqs[i];
      if (!pool->seq_ok(q)) return fail(PADOC_ERR_INVALID, "kv_commit: %d is not a live sequence", q);
      if (seen[q]) return fail(PADOC_ERR_INVALID, "kv_commit: sequence %d listed twice", q);
      seen[q] = 1;
      const Seq& s = pool->seqs[q];
      const int64_t need = (static_cast<int64_t>(s.len - s.fork_len) + row_offsets[i + 1] - row_offsets[i] + pool->bs - 1) /
                           pool->bs;
      if (s.n_shared + need > pool->max_bps)
        return fail(PADOC_ERR_INVALID, "kv_commit: sequence %d would exceed max_blocks_per_seq", q);
      extra[i] = std::max<int64_t>(0, need - pool->own_blocks(s));
      extra_total += extra[i];
    }
  });
  if (total == 0) return PADOC_OK;
  if (!pool->k || !pool->v) return fail(PADOC_ERR_INVALID, "kv_commit: pool has no storage");
  if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new))
    return fail(PADOC_ERR_INVALID, "kv_commit: k_new/v_new must be 16-byte aligned device pointers");
  if (!ws || !aligned16(ws) || ws_bytes < static_cast<size_t>(total) * 16)
    return fail(PADOC_ERR_INVALID, "kv_commit: ws must be 16-byte aligned and hold %lld bytes",
                static_cast<long long>(total) * 16);
  std::vector<int32_t> plan;
  PADOC_TRY({
    std::vector<int32_t> fresh;
    if (extra_total > 0 && (extra_total > static_cast<int64_t>(pool->free_blocks.size()) ||
                            !pool->take_blocks(static_cast<int32_t>(extra_total), &fresh)))
      return fail(PADOC_ERR_OOM, "kv_commit: out of blocks (%lld wanted)", static_cast<long long>(extra_total));
    plan.resize(static_cast<size_t>(total) * 4, 0);
    size_t next = 0;
    for (int32_t i = 0; i < n_seqs; ++i) {
      Seq& s = pool->seqs[seqs[i]];
      s.blocks.insert(s.blocks.end(), fresh.begin() + next, fresh.begin() + next + extra[i]);
      next += extra[i];
      const int32_t own = s.len - s.fork_len;
      for (int32_t j = row_offsets[i]; j < row_offsets[i + 1]; ++j) {
        const int32_t t = own + (j - row_offsets[i]);
        int32_t* e = &plan[static_cast<size_t>(j) * 4];
        e[0] = rows[j];
        e[1] = s.blocks[s.n_shared + t / pool->bs];
        e[2] = t % pool->bs;
      }
      s.len += row_offsets[i + 1] - row_offsets[i];
      pool->mark(seqs[i]);
    }
  });
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int rc = pool_sync(pool, st);
  if (rc) return rc;
  // Pageable source: the call returns once the bytes are staged, so plan may go.
  const cudaError_t e = cudaMemcpyAsync(ws, plan.data(), plan.size() * sizeof(int32_t), cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_fail(e, "kv_commit: row list upload");
  std::string err;
  rc = launch_commit(pool->k, pool->v, ws, total, pool->Hkv, k_new, v_new, st, &err);
  if (rc) return fail(rc, "kv_commit: %s", err.c_str());
  return PADOC_OK;
}

// ============================================================== decode planning

namespace {

struct DecodePlan {
  std::vector<DecPage> pages;
  std::vector<DecItem> items;
  std::vector<DecBranch> branches;
  std::vector<int32_t> q_plen;
  std::vector<int32_t> q_branch;  // branch of each query row
  int64_t part_rows = 0;
  bool tc_own = false;  // own pass on tensor cores (several query rows per branch and kv head)
  bool fused = false;   // verify: own suffix and query block walked by the prefix pass's units
  size_t off_pages = 0, off_items = 0, off_branches = 0, off_qplen = 0, off_qbranch = 0, off_part_o = 0, off_part_lse = 0,
         off_work = 0, total = 0;
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int plan_decode(const padoc_kv_pool* pool, const padoc_decode_batch* b, int32_t Hq, int n_sms, DecodePlan* pl) {
  if (!pool || !b) return fail(PADOC_ERR_INVALID, "branch_decode: null argument");
  if (Hq <= 0 || Hq % pool->Hkv != 0)
    return fail(PADOC_ERR_INVALID, "branch_decode: Hq=%d must be a positive multiple of Hkv=%d", Hq, pool->Hkv);
  const int G = Hq / pool->Hkv;
  if (G > 8) return fail(PADOC_ERR_UNSUPPORTED, "branch_decode: Hq/Hkv=%d above 8", G);
  if (b->n_pages < 0 || b->n_branches < 0) return fail(PADOC_ERR_INVALID, "branch_decode: negative counts");
  if (b->n_pages > 0 && (!b->page_seq || !b->branch_offsets))
    return fail(PADOC_ERR_INVALID, "branch_decode: null page arrays");
  if (b->n_branches > 0 && (!b->branch_seq || !b->q_offsets))
    return fail(PADOC_ERR_INVALID, "branch_decode: null branch arrays");
  if (b->n_pages == 0 && b->n_branches > 0) return fail(PADOC_ERR_INVALID, "branch_decode: branches without pages");
  if (b->n_pages > 0) {
    if (b->branch_offsets[0] != 0 || b->branch_offsets[b->n_pages] != b->n_branches)
      return fail(PADOC_ERR_INVALID, "branch_decode: branch_offsets must run from 0 to n_branches");
  }
  if (b->n_branches > 0 && b->q_offsets[0] != 0) return fail(PADOC_ERR_INVALID, "branch_decode: q_offsets[0] != 0");
  for (int32_t i = 0; i < b->n_branches; ++i) {
    const int32_t ql = b->q_offsets[i + 1] - b->q_offsets[i];
    if (ql < 1 || ql > 16) return fail(PADOC_ERR_INVALID, "branch_decode: branch %d has %d query rows (1..16)", i, ql);
  }
  const int32_t nq = b->n_branches ? b->q_offsets[b->n_branches] : 0;
  // One query token per branch gives G rows per (branch, kv head): the
  // CUDA-core own pass streams that at HBM speed.  Draft-tree verify stacks
  // up to 16 G rows, which needs the tensor cores.
  pl->tc_own = b->n_branches > 0 && static_cast<int64_t>(nq) * G >= 4 * static_cast<int64_t>(b->n_branches);
  // A verify step with G >= 2 fuses its own pass into the prefix pass when
  // every page's prefix fits one chunk.  A row tile then spans at most 64
  // query tokens, so the query blocks of the branches it touches (each at
  // most 16 tokens) lie within 15 + 64 + 15 < 128 tokens: one key tile.
  // PADOC_VERIFY_FUSED=0 keeps the two passes separate.
  static const bool fuse_allowed = !(std::getenv("PADOC_VERIFY_FUSED") &&
                                     std::string(std::getenv("PADOC_VERIFY_FUSED")) == "0");
  bool want_fused = pl->tc_own && G >= 2 && fuse_allowed;
  pl->q_plen.assign(nq, 0);
  pl->q_branch.assign(nq, 0);
  pl->branches.resize(b->n_branches);
  pl->pages.resize(b->n_pages);
  // chunk length from the total prefix work, so items fill the GPU
  int64_t work_tiles = 0;
  std::vector<int32_t> P(b->n_pages, 0);
  for (int32_t p = 0; p < b->n_pages; ++p) {
    const int32_t ps = b->page_seq[p];
    if (!pool->seq_ok(ps)) return fail(PADOC_ERR_INVALID, "branch_decode: page %d sequence %d not live", p, ps);
    const Seq& pseq = pool->seqs[ps];
    const int32_t b0 = b->branch_offsets[p], b1 = b->branch_offsets[p + 1];
    if (b1 < b0) return fail(PADOC_ERR_INVALID, "branch_decode: branch_offsets not ascending");
    for (int32_t i = b0; i < b1; ++i) {
      const int32_t s = b->branch_seq[i];
      if (!pool->seq_ok(s)) return fail(PADOC_ERR_INVALID, "branch_decode: branch %d sequence %d not live", i, s);
      const Seq& bs = pool->seqs[s];
      if (bs.fork_len > pseq.len)
        return fail(PADOC_ERR_INVALID, "branch_decode: branch %d sees %d prefix tokens, page has %d", i, bs.fork_len, pseq.len);
      if (bs.fork_len > pseq.fork_len && pseq.fork_len % pool->bs != 0)
        return fail(PADOC_ERR_UNSUPPORTED, "branch_decode: page %d prefix is not block aligned", p);
      // the branch's shared blocks are the page sequence's leading blocks
      // (one memcmp: a step checks some 10^4 branches of a few hundred blocks)
      if (bs.n_shared > static_cast<int32_t>(pseq.blocks.size()) ||
          (bs.n_shared > 0 &&
           std::memcmp(bs.blocks.data(), pseq.blocks.data(), static_cast<size_t>(bs.n_shared) * sizeof(int32_t)) != 0))
        return fail(PADOC_ERR_INVALID, "branch_decode: branch %d is not a fork of page %d's sequence", i, p);
      P[p] = std::max(P[p], bs.fork_len);
    }
    const int32_t nqp = (b1 > b0) ? b->q_offsets[b1] - b->q_offsets[b0] : 0;
    const int32_t rt = (nqp * G + kTileRows - 1) / kTileRows;
    work_tiles += static_cast<int64_t>(rt) * ((P[p] + kTileKeys - 1) / kTileKeys) * pool->Hkv;
  }
  int64_t ct = work_tiles / (2 * static_cast<int64_t>(n_sms));
  ct = std::max<int64_t>(8, std::min<int64_t>(kMaxChunkTiles, ct));
  if (want_fused) {
    int64_t max_tiles = 0;
    for (int32_t p = 0; p < b->n_pages; ++p) max_tiles = std::max<int64_t>(max_tiles, (P[p] + kTileKeys - 1) / kTileKeys);
    if (max_tiles <= kMaxChunkTiles)
      ct = std::max(ct, max_tiles);  // one chunk per page
    else
      want_fused = false;
  }
  int64_t rows = 0;
  for (int32_t p = 0; p < b->n_pages; ++p) {
    const int32_t b0 = b->branch_offsets[p], b1 = b->branch_offsets[p + 1];
    DecPage& pg = pl->pages[p];
    pg.seq = b->page_seq[p];
    pg.P = P[p];
    pg.q_first = (b1 > b0) ? b->q_offsets[b0] : 0;
    pg.nq = (b1 > b0) ? b->q_offsets[b1] - b->q_offsets[b0] : 0;
    pg.row_tiles = (pg.nq * G + kTileRows - 1) / kTileRows;
    const int32_t tiles = (pg.P + kTileKeys - 1) / kTileKeys;
    pg.n_chunks = (tiles == 0 || pg.nq == 0) ? 0 : static_cast<int32_t>((tiles + ct - 1) / ct);
    pg.chunk_tokens = pg.n_chunks ? ((tiles + pg.n_chunks - 1) / pg.n_chunks) * kTileKeys : 0;
    pg.n_chunks = pg.chunk_tokens ? (pg.P + pg.chunk_tokens - 1) / pg.chunk_tokens : 0;
    if (want_fused && pg.nq > 0 && pg.n_chunks == 0) pg.n_chunks = 1;  // no prefix: the unit walks own keys only
    pg.item_base = static_cast<int32_t>(pl->items.size());
    for (int32_t t = 0; t < pg.row_tiles && pg.n_chunks; ++t)
      for (int32_t c = 0; c < pg.n_chunks; ++c) {
        DecItem it{};
        it.page = p;
        it.tile = t;
        it.chunk = c;
        it.rows = std::min(kTileRows, pg.nq * G - t * kTileRows);
        it.row_base = static_cast<int32_t>(rows);
        const int32_t k0 = c * pg.chunk_tokens, k1 = std::min(pg.P, k0 + pg.chunk_tokens);
        it.n_tiles = k1 > k0 ? (k1 - k0 + kTileKeys - 1) / kTileKeys : 0;
        rows += static_cast<int64_t>(it.rows) * pool->Hkv;
        pl->items.push_back(it);
      }
    for (int32_t i = b0; i < b1; ++i) {
      const Seq& bs = pool->seqs[b->branch_seq[i]];
      DecBranch& br = pl->branches[i];
      br.page = p;
      br.seq = b->branch_seq[i];
      br.prefix_len = bs.fork_len;
      br.own_len = bs.len - bs.fork_len;
      br.n_shared = bs.n_shared;
      br.q_first = b->q_offsets[i];
      br.q_len = b->q_offsets[i + 1] - b->q_offsets[i];
      br.q_in_page = br.q_first - pg.q_first;
      for (int32_t r = br.q_first; r < br.q_first + br.q_len; ++r) {
        pl->q_plen[r] = br.prefix_len;
        pl->q_branch[r] = i;
      }
    }
    if (want_fused) {
      // the branches a row tile touches, and the first query token of the
      // first of them (the fused unit's query-block tile starts there)
      for (int32_t k = pg.item_base; k < static_cast<int32_t>(pl->items.size()); ++k) {
        DecItem& it = pl->items[k];
        const int32_t tok0 = pg.q_first + (it.tile * kTileRows) / G;
        const int32_t tok1 = pg.q_first + (it.tile * kTileRows + it.rows - 1) / G;
        const int32_t bf = pl->q_branch[tok0], bl = pl->q_branch[tok1];
        it.b_first = bf;
        it.b_count = bl - bf + 1;
        it.tok_lo = pl->branches[bf].q_first;
        for (int32_t b = bf; b <= bl; ++b) it.n_tiles += (pl->branches[b].own_len + kTileKeys - 1) / kTileKeys;
        it.n_tiles += 1;  // the query-block tile
        if (pl->branches[bl].q_first + pl->branches[bl].q_len - it.tok_lo > kTileKeys)
          return fail(PADOC_ERR_UNSUPPORTED, "branch_decode: query blocks of row tile %d span above %d tokens",
                      it.tile, kTileKeys);
      }
    }
  }
  if (rows >= (int64_t(1) << 31)) return fail(PADOC_ERR_UNSUPPORTED, "branch_decode: batch too large");
  pl->part_rows = rows;
  pl->fused = want_fused;
  size_t off = 0;
  pl->off_pages = off;
  off = align_up(off + pl->pages.size() * sizeof(DecPage), 256);
  pl->off_items = off;
  off = align_up(off + pl->items.size() * sizeof(DecItem), 256);
  pl->off_branches = off;
  off = align_up(off + pl->branches.size() * sizeof(DecBranch), 256);
  pl->off_qplen = off;
  off = align_up(off + pl->q_plen.size() * sizeof(int32_t), 256);
  pl->off_qbranch = off;
  off = align_up(off + pl->q_branch.size() * sizeof(int32_t), 256);
  pl->off_part_o = off;
  off = align_up(off + static_cast<size_t>(rows) * kHeadDim * sizeof(float), 256);
  pl->off_part_lse = off;
  off = align_up(off + static_cast<size_t>(rows) * sizeof(float), 256);
  pl->off_work = off;  // the unit counter of the tensor-core passes
  off = align_up(off + sizeof(int32_t), 256);
  pl->total = off;
  return PADOC_OK;
}

}  // namespace

extern "C" int padoc_branch_decode_ws_size(const padoc_kv_pool* pool, const padoc_decode_batch* batch, int32_t Hq,
                                           size_t* bytes) {
  if (!bytes) return fail(PADOC_ERR_INVALID, "branch_decode_ws_size: null bytes");
  DecodePlan pl;
  int rc;
  PADOC_TRY(rc = plan_decode(pool, batch, Hq, num_sms(), &pl));
  if (rc) return rc;
  *bytes = pl.total;
  return PADOC_OK;
}

struct padoc_decode_plan {
  padoc_kv_pool* pool = nullptr;
  int32_t Hq = 0;
  int32_t n_pages = 0, n_branches = 0;
  DecodePlan pl;
  std::vector<uint8_t> host;  // plan arrays as they are laid out in ws
};

extern "C" int padoc_decode_plan_create(padoc_kv_pool* pool, const padoc_decode_batch* batch, int32_t Hq,
                                        padoc_decode_plan** out) {
  if (!out) return fail(PADOC_ERR_INVALID, "decode_plan_create: null out");
  *out = nullptr;
  padoc_decode_plan* res = nullptr;
  PADOC_TRY({
    std::unique_ptr<padoc_decode_plan> p(new padoc_decode_plan());
    const int rc = plan_decode(pool, batch, Hq, num_sms(), &p->pl);
    if (rc) return rc;
    p->pool = pool;
    p->Hq = Hq;
    p->n_pages = batch->n_pages;
    p->n_branches = batch->n_branches;
    p->host.assign(p->pl.off_part_o, 0);
    std::memcpy(p->host.data() + p->pl.off_pages, p->pl.pages.data(), p->pl.pages.size() * sizeof(DecPage));
    std::memcpy(p->host.data() + p->pl.off_items, p->pl.items.data(), p->pl.items.size() * sizeof(DecItem));
    std::memcpy(p->host.data() + p->pl.off_branches, p->pl.branches.data(),
                p->pl.branches.size() * sizeof(DecBranch));
    std::memcpy(p->host.data() + p->pl.off_qplen, p->pl.q_plen.data(), p->pl.q_plen.size() * sizeof(int32_t));
    std::memcpy(p->host.data() + p->pl.off_qbranch, p->pl.q_branch.data(), p->pl.q_branch.size() * sizeof(int32_t));
    res = p.release();
  });
  *out = res;
  return PADOC_OK;
}

extern "C" int padoc_decode_plan_free(padoc_decode_plan* plan) {
  delete plan;
  return PADOC_OK;
}

extern "C" int padoc_decode_plan_ws_size(const padoc_decode_plan* plan, size_t* bytes) {
  if (!plan || !bytes) return fail(PADOC_ERR_INVALID, "decode_plan_ws_size: null argument");
  *bytes = plan->pl.total;
  return PADOC_OK;
}

extern "C" int padoc_decode_plan_fused(const padoc_decode_plan* plan, int32_t* fused) {
  if (!plan || !fused) return fail(PADOC_ERR_INVALID, "decode_plan_fused: null argument");
  *fused = plan->pl.fused ? 1 : 0;
  return PADOC_OK;
}

static int check_ws(const padoc_decode_plan* plan, const void* ws, size_t ws_bytes) {
  if (!ws) return fail(PADOC_ERR_INVALID, "decode: null workspace");
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return fail(PADOC_ERR_INVALID, "decode: ws must be 256-byte aligned");
  if (ws_bytes < plan->pl.total)
    return fail(PADOC_ERR_INVALID, "decode: workspace %zu bytes, need %zu", ws_bytes, plan->pl.total);
  return PADOC_OK;
}

extern "C" int padoc_decode_plan_upload(padoc_decode_plan* plan, void* ws, size_t ws_bytes, padoc_stream_t stream) {
  if (!plan) return fail(PADOC_ERR_INVALID, "decode_plan_upload: null plan");
  if (plan->n_branches == 0) return PADOC_OK;
  int rc = check_ws(plan, ws, ws_bytes);
  if (rc) return rc;
  if (!plan->pool->k || !plan->pool->v) return fail(PADOC_ERR_INVALID, "decode: pool has no storage");
  rc = padoc::pool_check_device(plan->pool, "decode_plan_upload");
  if (rc) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  rc = pool_sync(plan->pool, st);
  if (rc) return rc;
  cudaError_t e = cudaMemcpyAsync(ws, plan->host.data(), plan->host.size(), cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_fail(e, "decode: plan upload");
  return PADOC_OK;
}

static DecodeArgs decode_args(const padoc_decode_plan* plan, const void* q, const void* k_new, const void* v_new,
                              const uint16_t* tree_bits, void* o, float* lse, float scale, void* ws) {
  const DecodePlan& pl = plan->pl;
  const padoc_kv_pool* pool = plan->pool;
  uint8_t* w = static_cast<uint8_t*>(ws);
  DecodeArgs a;
  a.pages = reinterpret_cast<const DecPage*>(w + pl.off_pages);
  a.items = reinterpret_cast<const DecItem*>(w + pl.off_items);
  a.branches = reinterpret_cast<const DecBranch*>(w + pl.off_branches);
  a.q_plen = reinterpret_cast<const int32_t*>(w + pl.off_qplen);
  a.q_branch = reinterpret_cast<const int32_t*>(w + pl.off_qbranch);
  a.table = pool->d_table;
  a.max_bps = pool->max_bps;
  a.n_pages = plan->n_pages;
  a.n_items = static_cast<int32_t>(pl.items.size());
  a.n_branches = plan->n_branches;
  a.nq = static_cast<int32_t>(pl.q_plen.size());
  a.Hq = plan->Hq;
  a.Hkv = pool->Hkv;
  a.group = plan->Hq / pool->Hkv;
  a.d = pool->d;
  a.scale = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(pool->d));
  a.q = q;
  a.k_new = k_new;
  a.v_new = v_new;
  a.tree_bits = tree_bits;
  a.o = o;
  a.lse = lse;
  a.part_o = reinterpret_cast<float*>(w + pl.off_part_o);
  a.part_lse = reinterpret_cast<float*>(w + pl.off_part_lse);
  a.work = reinterpret_cast<int32_t*>(w + pl.off_work);
  a.k_pool = pool->k;
  a.v_pool = pool->v;
  a.num_blocks = pool->nb;
  return a;
}

extern "C" int padoc_decode_prefix_pass(const padoc_decode_plan* plan, const void* q, float scale, void* ws,
                                        padoc_stream_t stream) {
  if (!plan) return fail(PADOC_ERR_INVALID, "decode_prefix_pass: null plan");
  if (plan->n_branches == 0 || plan->pl.items.empty()) return PADOC_OK;
  if (plan->pl.fused) return PADOC_OK;  // the own pass walks the prefix too
  int rc = check_ws(plan, ws, SIZE_MAX);
  if (rc) return rc;
  if (!q || !aligned16(q)) return fail(PADOC_ERR_INVALID, "decode_prefix_pass: q must be a 16-byte aligned device pointer");
  if (!plan->pool->d_table) return fail(PADOC_ERR_INVALID, "decode_prefix_pass: plan was not uploaded");
  const DecodeArgs a = decode_args(plan, q, nullptr, nullptr, nullptr, nullptr, nullptr, scale, ws);
  std::string err;
  rc = launch_decode_prefix(a, reinterpret_cast<cudaStream_t>(stream), &err);
  if (rc) return fail(rc, "decode_prefix_pass: %s", err.c_str());
  return PADOC_OK;
}

extern "C" int padoc_decode_own_pass(const padoc_decode_plan* plan, const void* q, const void* k_new,
                                     const void* v_new, const uint16_t* tree_bits, void* o, float* lse, float scale,
                                     void* ws, padoc_stream_t stream) {
  if (!plan) return fail(PADOC_ERR_INVALID, "decode_own_pass: null plan");
  if (plan->n_branches == 0) return PADOC_OK;
  int rc = check_ws(plan, ws, SIZE_MAX);
  if (rc) return rc;
  if (!q || !k_new || !v_new || !o || !lse) return fail(PADOC_ERR_INVALID, "decode_own_pass: null tensor");
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(o) || !aligned16(lse))
    return fail(PADOC_ERR_INVALID, "decode_own_pass: tensors must be 16-byte aligned");
  if (!plan->pool->d_table) return fail(PADOC_ERR_INVALID, "decode_own_pass: plan was not uploaded");
  const DecodeArgs a = decode_args(plan, q, k_new, v_new, tree_bits, o, lse, scale, ws);
  std::string err;
  // Several query rows per (branch, kv head) (verify): tensor cores.  With
  // Hq / Hkv <= 2 a unit has at most 32 rows and the keys go on the MMA's M
  // side; PADOC_OWN_KERNEL=rows selects the rows-on-M engine instead (the
  // one used for larger groups).
  static const bool rows_major = std::getenv("PADOC_OWN_KERNEL") &&
                                 std::string(std::getenv("PADOC_OWN_KERNEL")) == "rows";
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (plan->pl.fused)
    rc = launch_decode_verify_fused(a, st, &err);
  else if (!plan->pl.tc_own)
    rc = launch_decode_own(a, st, &err);
  else if (a.group <= 2 && !rows_major)
    rc = launch_decode_own_kmajor(a, st, &err);
  else
    rc = launch_decode_own_tc(a, st, &err);
  if (rc) return fail(rc, "decode_own_pass: %s", err.c_str());
  return PADOC_OK;
}

extern "C" int padoc_branch_decode(padoc_kv_pool* pool, const padoc_decode_batch* batch, int32_t Hq, const void* q,
                                   const void* k_new, const void* v_new, const uint16_t* tree_bits, void* o,
                                   float* lse, float scale, void* ws, size_t ws_bytes, padoc_stream_t stream) {
  padoc_decode_plan* plan = nullptr;
  int rc = padoc_decode_plan_create(pool, batch, Hq, &plan);
  if (rc) return rc;
  std::unique_ptr<padoc_decode_plan> guard(plan);
  if (plan->n_branches == 0) return PADOC_OK;
  if (!q || !k_new || !v_new || !o || !lse) return fail(PADOC_ERR_INVALID, "branch_decode: null tensor");
  rc = padoc_decode_plan_upload(plan, ws, ws_bytes, stream);
  if (rc) return rc;
  rc = padoc_decode_prefix_pass(plan, q, scale, ws, stream);
  if (rc) return rc;
  return padoc_decode_own_pass(plan, q, k_new, v_new, tree_bits, o, lse, scale, ws, stream);
}

namespace padoc {
int set_error(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  return fail(code, "%s", buf);
}
bool pool_has_device_table(const padoc_kv_pool* pool) { return pool && pool->d_table; }
int pool_check_device(const padoc_kv_pool* pool, const char* what) {
  if (!pool || !pool->d_table) return PADOC_OK;
  int cur = -1;
  const cudaError_t e = cudaGetDevice(&cur);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (cur != pool->device)
    return fail(PADOC_ERR_INVALID, "%s: the pool's block table is on device %d but device %d is current", what,
                pool->device, cur);
  return PADOC_OK;
}
int32_t pool_num_blocks(const padoc_kv_pool* pool) { return pool ? pool->nb : 0; }
}  // namespace padoc

extern "C" int padoc_verify_accept(const void* logits, int32_t nq, int32_t vocab, const int32_t* tokens,
                                   const int32_t* parents, const int32_t* q_offsets, int32_t n_branches,
                                   int32_t max_nodes, float tau, int32_t* n_acc, int32_t* path, int32_t* free_token,
                                   padoc_stream_t stream) {
  if (n_branches < 0 || nq < 0 || vocab <= 0)
    return fail(PADOC_ERR_INVALID, "verify_accept: n_branches %d, nq %d, vocab %d", n_branches, nq, vocab);
  if (max_nodes < 1 || max_nodes > 16) return fail(PADOC_ERR_INVALID, "verify_accept: max_nodes %d outside [1, 16]", max_nodes);
  if (!(tau > 0.f) || !std::isfinite(tau)) return fail(PADOC_ERR_INVALID, "verify_accept: tau must be finite and > 0");
  if (n_branches == 0) return PADOC_OK;
  if (!q_offsets || !n_acc || !path || !free_token || (nq > 0 && (!logits || !tokens || !parents)))
    return fail(PADOC_ERR_INVALID, "verify_accept: null argument");
  std::string err;
  const int rc = launch_accept(logits, vocab, nq, tokens, parents, q_offsets, n_branches, max_nodes,
                               static_cast<float>(std::log(static_cast<double>(tau))), n_acc, path, free_token,
                               reinterpret_cast<cudaStream_t>(stream), &err);
  if (rc) return fail(rc, "verify_accept: %s", err.c_str());
  return PADOC_OK;
}

// ============================================================== small host helpers

extern "C" int padoc_tree_mask_build(const int32_t* parent, int32_t n, uint16_t* bits) {
  if (n < 0 || n > 16) return fail(PADOC_ERR_INVALID, "tree_mask_build: n=%d outside [0, 16]", n);
  if (n > 0 && (!parent || !bits)) return fail(PADOC_ERR_INVALID, "tree_mask_build: null argument");
  for (int32_t i = 0; i < n; ++i)
    if (parent[i] >= i || parent[i] < -1)
      return fail(PADOC_ERR_INVALID, "tree_mask_build: parent[%d]=%d must be -1 or an earlier node", i, parent[i]);
  for (int32_t i = 0; i < n; ++i) {
    const uint16_t up = parent[i] >= 0 ? bits[parent[i]] : 0;
    bits[i] = static_cast<uint16_t>(up | (1u << i));
  }
  return PADOC_OK;
}

extern "C" int padoc_depths(const int32_t* layout_len, const int32_t* content_len, int32_t n_regions,
                            int64_t* d_seq, int64_t* d_tree) {
  if (n_regions < 0) return fail(PADOC_ERR_INVALID, "depths: n_regions < 0");
  if (n_regions > 0 && (!layout_len || !content_len)) return fail(PADOC_ERR_INVALID, "depths: null arrays");
  int64_t seq = 0, tree = 0, acc = 0;
  for (int32_t k = 0; k < n_regions; ++k) {
    if (layout_len[k] < 0 || content_len[k] < 0) return fail(PADOC_ERR_INVALID, "depths: negative length");
    acc += layout_len[k];
    seq += layout_len[k] + content_len[k];
    tree = std::max(tree, acc + content_len[k]);
  }
  if (d_seq) *d_seq = seq;
  if (d_tree) *d_tree = tree;
  return PADOC_OK;
}

extern "C" int padoc_device_status(padoc_stream_t stream) {
  unsigned w = 0, wb = 0, wo = 0;
  int rc = read_and_clear_tc_error(reinterpret_cast<cudaStream_t>(stream), &w);
  if (!rc) rc = read_and_clear_bwd_error(reinterpret_cast<cudaStream_t>(stream), &wb);
  if (!rc) rc = read_and_clear_own_error(reinterpret_cast<cudaStream_t>(stream), &wo);
  if (rc) return fail(rc, "device_status: could not read the device error word");
  w |= wb | wo;
  if (w) return fail(PADOC_ERR_DEVICE_TIMEOUT, "a kernel gave up a bounded wait (site mask 0x%x)", w);
  return PADOC_OK;
}
