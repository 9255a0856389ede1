// Branch decode for callers that may not allocate device memory.
//
// The step's workspace (plan arrays and the prefix pass's partial results)
// comes from one file-scope device array instead of a caller buffer.  The
// kernels and host calls are the ones padoc_branch_decode uses; only the
// workspace address differs.
#include <mutex>
#include <string>

#include "../../include/padoc.h"
#include "padoc_internal.h"

namespace {

// Device memory reserved when the library's module is loaded on a GPU.
static __device__ __align__(256) unsigned char g_decode_scratch[PADOC_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// The array's device address on the current device, looked up once per
// device.  In host code the array's name only stands in for the symbol; the
// kernels must be given the address this returns.
int scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return padoc::set_error(PADOC_ERR_CUDA, "branch_decode_noalloc: cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices)
    return padoc::set_error(PADOC_ERR_UNSUPPORTED, "branch_decode_noalloc: device index above 63");
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || !p) {
      std::string m = std::string("branch_decode_noalloc: cudaGetSymbolAddress failed: ") + cudaGetErrorString(e);
      return padoc::set_error(PADOC_ERR_CUDA, m.c_str());
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return PADOC_OK;
}

}  // namespace

extern "C" int padoc_branch_decode_noalloc(padoc_kv_pool* pool, const padoc_decode_batch* batch, int32_t Hq,
                                           const void* q, const void* k_new, const void* v_new,
                                           const uint16_t* tree_bits, void* o, float* lse, float scale,
                                           padoc_stream_t stream) {
  padoc_decode_plan* plan = nullptr;
  int rc = padoc_decode_plan_create(pool, batch, Hq, &plan);
  if (rc) return rc;
  size_t need = 0;
  padoc_decode_plan_ws_size(plan, &need);
  if (batch->n_branches == 0) {
    padoc_decode_plan_free(plan);
    return PADOC_OK;
  }
  if (need > PADOC_NOALLOC_SCRATCH_BYTES) {
    padoc_decode_plan_free(plan);
    std::string m = "branch_decode_noalloc: this step needs " + std::to_string(need) +
                    " bytes of workspace, above the fixed " + std::to_string(PADOC_NOALLOC_SCRATCH_BYTES) +
                    "-byte scratch array; split the batch or use padoc_branch_decode";
    return padoc::set_error(PADOC_ERR_INVALID, m.c_str());
  }
  if (!padoc::pool_has_device_table(pool)) {
    padoc_decode_plan_free(plan);
    return padoc::set_error(PADOC_ERR_INVALID,
                            "branch_decode_noalloc: the pool's device table does not exist yet; call "
                            "padoc_kv_pool_sync once at set-up");
  }
  if (!q || !k_new || !v_new || !o || !lse) {
    padoc_decode_plan_free(plan);
    return padoc::set_error(PADOC_ERR_INVALID, "branch_decode_noalloc: null tensor");
  }
  // the scratch address is looked up for the current device: the pool's
  // table, the KV blocks and the caller's tensors must live there too
  rc = padoc::pool_check_device(pool, "branch_decode_noalloc");
  if (rc) {
    padoc_decode_plan_free(plan);
    return rc;
  }
  void* ws = nullptr;
  rc = scratch_address(&ws);
  if (!rc) rc = padoc_decode_plan_upload(plan, ws, PADOC_NOALLOC_SCRATCH_BYTES, stream);
  if (!rc) rc = padoc_decode_prefix_pass(plan, q, scale, ws, stream);
  if (!rc) rc = padoc_decode_own_pass(plan, q, k_new, v_new, tree_bits, o, lse, scale, ws, stream);
  padoc_decode_plan_free(plan);
  return rc;
}
