// pkv_paged_decode_static_workspace: the paged decode for callers that cannot
// allocate device memory themselves.  The decode's scratch comes from one
// static device array per GPU instead of a caller workspace; everything else
// is pkv_paged_decode unchanged.
#include <cstdio>
#include <mutex>

#include "pkv_internal.h"

namespace {

// Scratch of the decode (split-K partials, plan, work counter).  In host code
// this name is only a stand-in for the symbol, not a device address: the
// device address is looked up per device with cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_pkv_static_workspace[PKV_STATIC_WORKSPACE_MAX_BYTES];

constexpr int kMaxDevices = 64;
struct StaticWorkspace {
  void* ctx;   // the CUDA context the address belongs to
  void* addr;  // device address of this device's copy of the array
};
StaticWorkspace g_static_ws[kMaxDevices];
std::mutex g_static_ws_mutex;

// Device address of this device's copy of the array, looked up with the
// device current on first use and again whenever the device's context has
// changed since (cudaDeviceReset, or a released and re-created primary
// context, loads the module again, possibly at another address).
pkv_status static_workspace_address(void** addr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    pkv::set_last_error_message(cudaGetErrorString(e));
    return PKV_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    pkv::set_last_error_message("device ordinal outside the supported range");
    return PKV_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_static_ws_mutex);
  StaticWorkspace& w = g_static_ws[dev];
  void* ctx = pkv::current_context();
  if (w.addr == nullptr || ctx == nullptr || ctx != w.ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_pkv_static_workspace);  // makes the device's context current
    if (e != cudaSuccess || p == nullptr) {
      char msg[256];
      std::snprintf(msg, sizeof msg, "cudaGetSymbolAddress(static workspace): %s",
                    cudaGetErrorString(e));
      pkv::set_last_error_message(msg);
      return PKV_ERR_CUDA;
    }
    w.addr = p;
    w.ctx = pkv::current_context();
  }
  *addr = w.addr;
  return PKV_OK;
}

}  // namespace

extern "C" pkv_status pkv_paged_decode_static_workspace(
    const pkv_cache_desc* cache, const void* q, int32_t batch, int32_t num_q_heads,
    const void* k_cache, const void* v_cache, const float* k_scale, const float* v_scale,
    const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* context_lens,
    const int32_t* kv_group_ptr, int32_t num_layers, int32_t layer, float scale, void* out,
    const pkv_decode_opts* opts, void* stream) {
  const size_t need = pkv_decode_workspace_bytes(cache, batch, num_q_heads, max_blocks_per_seq, opts);
  if (need > PKV_STATIC_WORKSPACE_MAX_BYTES) {
    char msg[256];
    std::snprintf(msg, sizeof msg,
                  "decode needs %zu bytes of scratch but the built-in workspace holds %zu; "
                  "use a larger partition_blocks or pkv_paged_decode with a workspace",
                  need, static_cast<size_t>(PKV_STATIC_WORKSPACE_MAX_BYTES));
    pkv::set_last_error_message(msg);
    return PKV_ERR_WORKSPACE;
  }
  void* ws = nullptr;
  if (need != 0) {  // need == 0: bad arguments, reported by pkv_paged_decode below
    const pkv_status st = static_workspace_address(&ws);
    if (st != PKV_OK) return st;
  }
  return pkv_paged_decode(cache, q, batch, num_q_heads, k_cache, v_cache, k_scale, v_scale,
                          block_tables, max_blocks_per_seq, context_lens, kv_group_ptr,
                          num_layers, layer, scale, out, ws,
                          ws != nullptr ? static_cast<size_t>(PKV_STATIC_WORKSPACE_MAX_BYTES) : 0,
                          opts, stream);
}
