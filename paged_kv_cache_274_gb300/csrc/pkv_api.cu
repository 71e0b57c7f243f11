// C ABI of the library (see include/pkv.h): host-side validation, tensor-map
// encoding, launch configuration and the sticky device error word.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include <cudaTypedefs.h>

#include "pkv_internal.h"

namespace {

// Sticky device error word (PKV_DEVERR_* bits), one per device.
__device__ unsigned int g_pkv_device_error;

thread_local std::string t_last_error;

void set_error(const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
}

pkv_status fail(pkv_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return st;
}

pkv_status cuda_fail(cudaError_t e, const char* what) {
  return fail(PKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  void* ctx = nullptr;  // CUDA context the facts below belong to
  unsigned* err_word = nullptr;
  int num_sms = 0;
};
DeviceInfo g_devices[kMaxDevices];
std::mutex g_dev_mutex;

// Per-device facts, resolved with that device current and looked up again
// whenever the device's context changes (a cudaDeviceReset, or a released and
// re-created primary context, loads the module again, possibly at another
// address).
pkv_status device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(PKV_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceInfo& d = g_devices[dev];
  void* ctx = pkv::current_context();
  if (ctx == nullptr || ctx != d.ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_pkv_device_error);  // makes the device's context current
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(device error word)");
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
    d.err_word = static_cast<unsigned*>(p);
    d.num_sms = sms;
    d.ctx = pkv::current_context();
  }
  *out = d;
  return PKV_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

pkv_status tensor_map_encoder(PFN_cuTensorMapEncodeTiled_v12000* fn) {
  std::call_once(g_encode_once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  if (g_encode == nullptr) return fail(PKV_ERR_CUDA, "driver has no cuTensorMapEncodeTiled");
  *fn = g_encode;
  return PKV_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// page parameters: E4M3 scales are read as floats, INT8 (scale, zero) pairs as float2
bool scales_aligned(int dtype, const void* a, const void* b) {
  const uintptr_t m = dtype == PKV_KV_INT8 ? 7u : 3u;
  return ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b)) & m) == 0;
}

bool env_flag(const char* name) {
  const char* v = std::getenv(name);
  return v != nullptr && v[0] != '\0' && std::strcmp(v, "0") != 0;
}

int env_int(const char* name, int dflt) {
  const char* v = std::getenv(name);
  if (v == nullptr || v[0] == '\0') return dflt;
  return std::atoi(v);
}

pkv_status check_cache_desc(const pkv_cache_desc* c) {
  if (c == nullptr) return fail(PKV_ERR_INVALID_ARG, "cache descriptor is NULL");
  if (c->num_slots < 1 || c->num_blocks < 1 || c->num_kv_heads < 1)
    return fail(PKV_ERR_INVALID_ARG, "cache: slots, blocks and KV heads must be >= 1");
  if (c->dtype != PKV_KV_BF16 && c->dtype != PKV_KV_FP8_E4M3 && c->dtype != PKV_KV_INT8)
    return fail(PKV_ERR_INVALID_ARG, "cache: unknown dtype %d", c->dtype);
  if (c->block_size != 16 && c->block_size != 32)
    return fail(PKV_ERR_UNSUPPORTED, "cache: block_size %d (supported: 16, 32)", c->block_size);
  if (c->dtype == PKV_KV_BF16 && c->head_dim != 64 && c->head_dim != 128)
    return fail(PKV_ERR_UNSUPPORTED, "cache: head_dim %d (bf16 supports 64, 128)", c->head_dim);
  if (c->dtype != PKV_KV_BF16 && c->head_dim != 128)
    return fail(PKV_ERR_UNSUPPORTED, "cache: head_dim %d (E4M3 and INT8 support 128)", c->head_dim);
  const long long rows = static_cast<long long>(c->num_slots) * c->num_blocks * c->num_kv_heads *
                         c->block_size;
  if (rows >= (1LL << 31)) return fail(PKV_ERR_UNSUPPORTED, "cache has %lld rows (limit 2^31)", rows);
  return PKV_OK;
}

pkv_status encode_cache_map(CUtensorMap* map, const void* base, const pkv_cache_desc* c) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  pkv_status st = tensor_map_encoder(&enc);
  if (st != PKV_OK) return st;
  const bool fp8 = c->dtype != PKV_KV_BF16;  // one-byte elements
  const int elem = fp8 ? 1 : 2;
  const cuuint64_t rows = static_cast<cuuint64_t>(c->num_slots) * c->num_blocks * c->num_kv_heads *
                          c->block_size;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(c->head_dim), rows};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(c->head_dim) * elem};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / elem), static_cast<cuuint32_t>(c->block_size)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return PKV_OK;
}

// Store map of the split-K partial outputs part_o [B][T][Hq][pmax][D] fp32
// for the tcgen05 kernel: a box of 32 columns x one partition x the G heads of
// a KV head x the Tt query tokens of a row tile (128-byte rows, swizzled as
// the kernel stages them); the token dimension clips a ragged last tile.
pkv_status encode_partial_map(CUtensorMap* map, void* part_o, int B, int T, int Hq, int pmax, int D, int G,
                              int Tt) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  pkv_status st = tensor_map_encoder(&enc);
  if (st != PKV_OK) return st;
  const cuuint64_t row = static_cast<cuuint64_t>(D) * sizeof(float);
  cuuint64_t dims[5] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(pmax), static_cast<cuuint64_t>(Hq),
                        static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[4] = {row, row * pmax, row * pmax * Hq, row * pmax * Hq * T};
  cuuint32_t box[5] = {32, 1, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(Tt), 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, part_o, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled (partials) failed (%d)", static_cast<int>(r));
  return PKV_OK;
}

// Store map of the bf16 output out [B][T][Hq][D] for the tcgen05 kernel: a
// box of 64 columns x the G heads of a KV head x the Tt query tokens of a row
// tile (128-byte rows, swizzled as the kernel stages them).
pkv_status encode_output_map(CUtensorMap* map, void* out, int B, int T, int Hq, int D, int G, int Tt) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  pkv_status st = tensor_map_encoder(&enc);
  if (st != PKV_OK) return st;
  const cuuint64_t row = static_cast<cuuint64_t>(D) * 2;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hq), static_cast<cuuint64_t>(T),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {row, row * Hq, row * Hq * T};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(Tt), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, out, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled (output) failed (%d)", static_cast<int>(r));
  return PKV_OK;
}

// Load map of the queries q [B][T][Hq][D] bf16 for the tile-pair tcgen05
// kernel: a box of 64 columns x the G heads of a KV head x the Tt query
// tokens of a row tile (128-byte rows, 128-byte swizzle, the K-major layout
// of the MMA's A operand); tokens past T read as zeros.
pkv_status encode_query_map(CUtensorMap* map, const void* q, int B, int T, int Hq, int D, int G, int Tt) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  pkv_status st = tensor_map_encoder(&enc);
  if (st != PKV_OK) return st;
  const cuuint64_t row = static_cast<cuuint64_t>(D) * 2;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hq), static_cast<cuuint64_t>(T),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {row, row * Hq, row * Hq * T};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(Tt), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(q), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled (queries) failed (%d)", static_cast<int>(r));
  return PKV_OK;
}

// Host copies of device tables for PKV_VALIDATE.
template <typename T>
pkv_status fetch(std::vector<T>& dst, const T* src, size_t n, cudaStream_t stream) {
  dst.resize(n);
  if (n == 0) return PKV_OK;
  cudaError_t e = cudaMemcpyAsync(dst.data(), src, n * sizeof(T), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "PKV_VALIDATE copy");
  return PKV_OK;
}

}  // namespace

namespace pkv {
void set_last_error_message(const char* msg) { t_last_error = msg; }

void* current_context() {
  using GetCurrent = CUresult (*)(CUcontext*);
  static GetCurrent fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<GetCurrent>(p);
  }();
  CUcontext ctx = nullptr;
  if (fn == nullptr || fn(&ctx) != CUDA_SUCCESS) return nullptr;
  return ctx;
}
}  // namespace pkv

extern "C" {

int32_t pkv_abi_version(void) { return PKV_ABI_VERSION; }

const char* pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case PKV_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_DEVICE_INDEX: return "device reported an out-of-range index";
    case PKV_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

const char* pkv_last_error_message(void) { return t_last_error.c_str(); }

}  // extern "C"

// Validate a KV append into cache slot `slot` and resolve its launch
// arguments; *a is left untouched unless PKV_OK.  num_tokens >= 1.
static pkv_status prepare_append(const pkv_cache_desc* cache, int32_t slot, const void* k, const void* v,
                                 const int64_t* slot_mapping, int32_t num_tokens, void* k_cache,
                                 void* v_cache, const float* k_scale, const float* v_scale,
                                 cudaStream_t s, const DeviceInfo* dev, pkv::AppendArgs* a) {
  pkv_status st;
  if (slot < 0 || slot >= cache->num_slots)
    return fail(PKV_ERR_INVALID_ARG, "slot %d outside [0, %d)", slot, cache->num_slots);
  const bool fp8 = cache->dtype != PKV_KV_BF16;  // one-byte elements (E4M3 or INT8)
  if (!k || !v || !slot_mapping || !k_cache || !v_cache)
    return fail(PKV_ERR_INVALID_ARG, "NULL tensor pointer");
  if (fp8 && (!k_scale || !v_scale)) return fail(PKV_ERR_INVALID_ARG, "E4M3 and INT8 caches need k_scale and v_scale");
  if (fp8 && !scales_aligned(cache->dtype, k_scale, v_scale))
    return fail(PKV_ERR_ALIGNMENT, "k_scale and v_scale must be 4-byte (E4M3) or 8-byte (INT8) aligned");
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(PKV_ERR_ALIGNMENT, "k, v and caches must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(slot_mapping) & 7u) != 0)
    return fail(PKV_ERR_ALIGNMENT, "slot_mapping must be 8-byte aligned");
  const long long nslots = static_cast<long long>(cache->num_blocks) * cache->block_size;
  if (env_flag("PKV_VALIDATE")) {
    std::vector<int64_t> sm;
    if ((st = fetch(sm, slot_mapping, static_cast<size_t>(num_tokens), s)) != PKV_OK) return st;
    std::vector<int64_t> seen;
    for (int i = 0; i < num_tokens; ++i) {
      if (sm[i] < -1 || sm[i] >= nslots)
        return fail(PKV_ERR_INVALID_ARG, "slot_mapping[%d] = %lld outside [-1, %lld)", i,
                    static_cast<long long>(sm[i]), nslots);
      if (sm[i] >= 0) seen.push_back(sm[i]);
    }
    std::sort(seen.begin(), seen.end());
    if (std::adjacent_find(seen.begin(), seen.end()) != seen.end())
      return fail(PKV_ERR_INVALID_ARG, "slot_mapping has duplicate slots");
  }
  const size_t page_elems = static_cast<size_t>(cache->num_kv_heads) * cache->block_size * cache->head_dim;
  const size_t slot_elems = page_elems * cache->num_blocks;
  const size_t elem = fp8 ? 1 : 2;
  const size_t scale_off = static_cast<size_t>(slot) * cache->num_blocks * cache->num_kv_heads *
                           (cache->dtype == PKV_KV_INT8 ? 2 : 1);
  a->k = static_cast<const uint4*>(k);
  a->v = static_cast<const uint4*>(v);
  a->slot_mapping = slot_mapping;
  a->N = num_tokens;
  a->Hkv = cache->num_kv_heads;
  a->D = cache->head_dim;
  a->bs = cache->block_size;
  a->nslots = nslots;
  a->kc = static_cast<uint8_t*>(k_cache) + static_cast<size_t>(slot) * slot_elems * elem;
  a->vc = static_cast<uint8_t*>(v_cache) + static_cast<size_t>(slot) * slot_elems * elem;
  a->ks = fp8 ? k_scale + scale_off : nullptr;
  a->vs = fp8 ? v_scale + scale_off : nullptr;
  a->err = dev->err_word;
  return PKV_OK;
}

extern "C" {

pkv_status pkv_kv_append(const pkv_cache_desc* cache, int32_t slot, const void* k, const void* v,
                         const int64_t* slot_mapping, int32_t num_tokens, void* k_cache,
                         void* v_cache, const float* k_scale, const float* v_scale, void* stream) {
  pkv_status st = check_cache_desc(cache);
  if (st != PKV_OK) return st;
  if (slot < 0 || slot >= cache->num_slots)
    return fail(PKV_ERR_INVALID_ARG, "slot %d outside [0, %d)", slot, cache->num_slots);
  if (num_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "num_tokens %d < 0", num_tokens);
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache)
    return fail(PKV_ERR_INVALID_ARG, "NULL tensor pointer");
  const bool fp8 = cache->dtype != PKV_KV_BF16;
  if (fp8 && (!k_scale || !v_scale)) return fail(PKV_ERR_INVALID_ARG, "E4M3 and INT8 caches need k_scale and v_scale");
  if (fp8 && !scales_aligned(cache->dtype, k_scale, v_scale))
    return fail(PKV_ERR_ALIGNMENT, "k_scale and v_scale must be 4-byte (E4M3) or 8-byte (INT8) aligned");
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(PKV_ERR_ALIGNMENT, "k, v and caches must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(slot_mapping) & 7u) != 0)
    return fail(PKV_ERR_ALIGNMENT, "slot_mapping must be 8-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DeviceInfo dev_info;
  const DeviceInfo* dev = &dev_info;
  if ((st = device_info(&dev_info)) != PKV_OK) return st;
  pkv::AppendArgs a{};
  if ((st = prepare_append(cache, slot, k, v, slot_mapping, num_tokens, k_cache, v_cache, k_scale, v_scale, s,
                           dev, &a)) != PKV_OK)
    return st;
  cudaError_t e = pkv::launch_kv_append(cache->dtype, a, s);
  if (e != cudaSuccess) return cuda_fail(e, "kv_append launch");
  return PKV_OK;
}

// Resolve options into a full launch configuration (no device work).
static pkv_status resolve_decode(const pkv_cache_desc* c, int32_t batch, int32_t T, int32_t Hq,
                                 int32_t MB, const pkv_decode_opts* opts, int num_sms,
                                 pkv::DecodeLaunch* L) {
  pkv_status st = check_cache_desc(c);
  if (st != PKV_OK) return st;
  if (batch < 0) return fail(PKV_ERR_INVALID_ARG, "batch %d < 0", batch);
  if (T < 1 || T > PKV_MAX_QUERY_TOKENS)
    return fail(PKV_ERR_INVALID_ARG, "num_query_tokens %d outside 1..%d", T, PKV_MAX_QUERY_TOKENS);
  if (MB < 1) return fail(PKV_ERR_INVALID_ARG, "max_blocks_per_seq %d < 1", MB);
  if (Hq < 1 || Hq % c->num_kv_heads != 0)
    return fail(PKV_ERR_INVALID_ARG, "num_q_heads %d is not a multiple of num_kv_heads %d", Hq,
                c->num_kv_heads);
  if (static_cast<long long>(MB) * c->block_size >= (1LL << 31))
    return fail(PKV_ERR_UNSUPPORTED, "max_blocks_per_seq too large");
  const int G = Hq / c->num_kv_heads;
  pkv_decode_opts o{};
  if (opts) o = *opts;
  int math = o.math != 0 ? o.math : env_int("PKV_DECODE_MATH", PKV_MATH_AUTO);
  // tcgen05 tiles: multi-token calls with head_dim 128 (one-byte caches as
  // exact code values: E4M3 K pages as they are, the other pages widened to
  // f16 in shared memory)
  const bool tc_ok = c->head_dim == 128 && T > 1 && G <= 128;
  // measured on GB300 (Llama-8B layer, G 4): mma.sync tiles are faster up to
  // 16 rows per KV head (172 us at 4 tokens, one tile), tcgen05 tiles from 32
  // rows on (kernel 173 vs 234 us at 8 tokens, 173 vs 451 at 16, 183 vs 865
  // at 32, 583 vs 3402 at 128)
  if (math == PKV_MATH_AUTO) math = (tc_ok && static_cast<long long>(T) * G > 16) ? PKV_MATH_TC : PKV_MATH_MMA;
  if (math == PKV_MATH_TC && !tc_ok)
    return fail(PKV_ERR_UNSUPPORTED, "tcgen05 tiles need T > 1, head_dim 128 and G <= 128");
  if (math == PKV_MATH_MMA && G > 16)
    return fail(PKV_ERR_UNSUPPORTED, "G = %d query heads per KV head (mma supports <= 16)", G);
  if (math == PKV_MATH_FFMA && G != 1 && G != 2 && G != 4 && G != 8)
    return fail(PKV_ERR_UNSUPPORTED, "G = %d query heads per KV head (ffma supports 1, 2, 4, 8)", G);
  if (math != PKV_MATH_MMA && math != PKV_MATH_FFMA && math != PKV_MATH_TC)
    return fail(PKV_ERR_INVALID_ARG, "math %d", math);
  const bool tc = math == PKV_MATH_TC;
  if (math == PKV_MATH_FFMA && T > 1)
    return fail(PKV_ERR_UNSUPPORTED, "multi-token queries need the mma back-end");
  if (static_cast<long long>(batch) * T * Hq * c->head_dim >= (1LL << 31))
    return fail(PKV_ERR_UNSUPPORTED, "batch x query tokens x heads x head_dim too large");
  // row tiles of at most 16 (mma.sync) or 128 (tcgen05) (query token, head)
  // rows: whole query tokens per tile
  const int Tt = std::max(1, std::min(T, (tc ? 128 : 16) / G));
  const int NT = (T + Tt - 1) / Tt;
  const bool fp8 = c->dtype != PKV_KV_BF16;  // one-byte elements
  const size_t stage_bytes = static_cast<size_t>(2) * c->block_size * c->head_dim * (fp8 ? 1 : 2);
  // Defaults measured on GB300: 4 warps per CTA with shallow (2-stage)
  // rings give several CTAs, i.e. 8+ streaming warps, per SM; deeper rings
  // only cost occupancy.
  // (the tcgen05 kernels have fixed shapes: one 128-row tile per CTA with 4
  // compute warps, an MMA warp and two copy warps, a 4-stage K ring and a
  // 2-stage V ring of 64 tokens; or, with two or more row tiles per KV head,
  // a pair of tiles per CTA with 8 softmax warps, an MMA warp and two copy
  // warps, 2-stage K and V rings of 128 tokens -- PKV_TC_PAIR=0 keeps the
  // one-tile kernel there)
  const bool tc2 = tc && NT >= 2 && c->dtype == PKV_KV_BF16 && env_int("PKV_TC_PAIR", 1) != 0;
  int warps = tc2 ? pkv::kTcPairWarps
              : tc ? (c->dtype == PKV_KV_BF16 ? 7 : 8)  // + the converter warp of one-byte caches
                   : (o.warps_per_cta != 0 ? o.warps_per_cta : env_int("PKV_DECODE_WARPS", 4));
  int stages = tc2 ? 2 : tc ? 4 : (o.stages != 0 ? o.stages : env_int("PKV_DECODE_STAGES", 0));
  if (stages == 0) stages = stage_bytes >= (8u << 10) ? 2 : 3;
  if (!tc && (warps < 1 || warps > 8)) return fail(PKV_ERR_INVALID_ARG, "warps_per_cta %d outside 1..8", warps);
  if (stages < 2 || stages > 8) return fail(PKV_ERR_INVALID_ARG, "stages %d outside 2..8", stages);
  const size_t smem = pkv::decode_smem_bytes(fp8, c->head_dim, c->block_size, warps, stages, tc, tc2);
  if (smem > 227u * 1024u)
    return fail(PKV_ERR_INVALID_ARG, "warps x stages need %zu bytes of shared memory", smem);
  int ppu = o.partition_blocks != 0 ? o.partition_blocks : env_int("PKV_DECODE_PARTITION_BLOCKS", 0);
  // partitions of up to 64 blocks for the mma.sync kernels, up to a unit's
  // page table for the tcgen05 kernel
  const int ppu_max = tc ? pkv::kTcUnitMaxPages : 64;
  if (ppu < 0 || ppu > ppu_max) return fail(PKV_ERR_INVALID_ARG, "partition_blocks %d outside 1..%d", ppu, ppu_max);
  const bool auto_ppu = ppu == 0;
  if (ppu == 0) {
    // The decode is a persistent grid of W streaming warps pulling units of
    // work; its time follows how full the last round of units is.  Estimate
    // W from shared memory and about 200 registers a thread, count units for
    // the longest allowed context, take 64-block partitions when one round
    // holds every unit, else the size of {32, 16, 8} whose last round is
    // fullest (a larger size unless a smaller one is clearly better).
    const long long ctas_smem = std::max<long long>(1, (228LL * 1024) / static_cast<long long>(smem + 1024));
    const long long ctas_regs = std::max<long long>(1, 65536LL / (warps * 32LL * 200));
    // streams: warps of the mma.sync kernels; CTAs of the tcgen05 kernel
    // (two per SM: their accumulators fill the SM's tensor memory)
    const long long W = tc2 ? static_cast<long long>(num_sms)
                        : tc ? 2LL * num_sms
                             : static_cast<long long>(num_sms) * std::min(ctas_smem, ctas_regs) * warps;
    const int tiles_per_unit = tc2 ? 2 : 1;
    auto units = [&](int pp) {
      return static_cast<long long>(std::max(batch, 1)) * c->num_kv_heads * ((NT + tiles_per_unit - 1) / tiles_per_unit) *
             ((MB + pp - 1) / pp);
    };
    // Multi-token units carry T times the partials and load up to 16 query
    // rows each, so they stay at 32 or 64 blocks (measured on the 4- and
    // 8-token verify steps: 32 beats 16 by 4-10% in the kernel).
    const std::vector<int> sizes = T > 1 ? std::vector<int>{32, 64} : std::vector<int>{32, 16, 8};
    if (tc) {
      // tcgen05 units cost their 64-token steps plus a start-up and write-out
      // of about 6.5 steps (measured on GB300); rounds of 2 x SMs units:
      // the size of {64, 128, 256} blocks with the least modelled time
      // (long units also drop the split-K partials and the merge)
      // A sequence in several partitions also writes split-K partials that
      // the merge kernel reads back: (query rows) x (D + 2) fp32 per unit,
      // each way, at about 4 MB per modelled step (measured on GB300: the
      // 64-token verify step with 128-block units ran 393 us against 345
      // with whole-sequence units, whose kernel alone is 18 us slower).
      // The tile-pair kernel: steps of 128 tokens for two tiles, i.e. about
      // two 64-token steps of the one-tile kernel, and units twice as wide.
      const double partial_bytes = static_cast<double>(G) * Tt * (c->head_dim + 2) * 4.0 * tiles_per_unit;
      double best = 0.0;
      for (int pp : {64, 128, 256}) {
        const long long rounds = (units(pp) + W - 1) / W;
        const double merge = pp < MB ? static_cast<double>(units(pp)) * partial_bytes * 2.0 / 4.0e6 : 0.0;
        const double cost = static_cast<double>(rounds) *
                            (static_cast<double>(pp) * c->block_size / 64.0 + 6.5) + merge;
        if (best == 0.0 || cost < best) {
          best = cost;
          ppu = pp;
        }
        if (pp >= MB) break;  // one partition per sequence already
      }
    } else if (units(64) <= W) {
      // one round holds every unit: cut the sequences so that each SM gets
      // the same number of units, one per warp of a CTA per SM (measured on
      // GB300: 64-block units of the 70B-shaped 32K x 4 and 128K x 1 contexts
      // filled 128 CTAs of 4 warps on 152 SMs), in partitions of 16 to 64
      // blocks
      const long long seq_units = static_cast<long long>(std::max(batch, 1)) * c->num_kv_heads * NT;
      const long long parts = std::max<long long>((MB + 63) / 64, (static_cast<long long>(num_sms) * warps) / seq_units);
      ppu = static_cast<int>(std::min<long long>(64, std::max<long long>(16, (MB + parts - 1) / parts)));
    } else {
      double best = -1.0;
      for (int pp : sizes) {
        const double r = static_cast<double>(units(pp)) / static_cast<double>(W);
        const double eff = r / std::ceil(r);
        if (eff > best + 0.05) {
          best = eff;
          ppu = pp;
        }
      }
    }
  }
  ppu = std::min(ppu, MB);
  if ((MB + ppu - 1) / ppu > 65536)
    return fail(PKV_ERR_UNSUPPORTED, "more than 65536 partitions per sequence; raise partition_blocks");
  // The tile-pair kernel runs one unit per SM at a time, units of equal
  // length: when the last round of units would be at most half full, the
  // last sequences take partitions of half the length, so that the last
  // round's work spreads over twice as many units (with S sequences halved,
  // S >= r / u: the r units of the last round become at least 2r half
  // units).  Counted for sequences of the longest allowed context; with
  // shorter ones the split is still valid, only less useful.
  int half_from = batch, ppu_half = ppu;
  if (tc2 && auto_ppu && ppu >= 2 && env_int("PKV_TC_BALANCE", 1) != 0) {
    const long long u = static_cast<long long>((MB + ppu - 1) / ppu) * c->num_kv_heads * ((NT + 1) / 2);
    const long long n = static_cast<long long>(std::max(batch, 1)) * u;
    const long long r = n % num_sms;
    if (r > 0 && 2 * r <= num_sms) {
      half_from = batch - static_cast<int>(std::min<long long>(batch, (r + u - 1) / u));
      ppu_half = (ppu + 1) / 2;
    }
  }
  *L = pkv::DecodeLaunch{};
  L->B = batch;
  L->Hq = Hq;
  L->Hkv = c->num_kv_heads;
  L->G = G;
  L->T = T;
  L->Tt = Tt;
  L->NT = NT;
  L->tc = tc ? 1 : 0;
  L->tc2 = tc2 ? 1 : 0;
  L->MB = MB;
  L->NB = c->num_blocks;
  L->bs = c->block_size;
  L->D = c->head_dim;
  L->kv_fp8 = fp8;
  L->kv_dtype = c->dtype;
  L->ppu = ppu;
  L->half_from = half_from;
  L->ppu_half = ppu_half;
  L->pmax = (MB + ppu_half - 1) / ppu_half;  // ppu_half == ppu without half-length partitions
  L->math = math;
  L->warps = warps;
  L->stages = stages;
  L->num_sms = num_sms;
  return PKV_OK;
}

static pkv::WorkspaceLayout layout_of(const pkv::DecodeLaunch& L) {
  return pkv::workspace_layout(L.B, L.T, L.Hq, L.Hkv, L.NT, L.D, L.pmax);
}

size_t pkv_decode_multi_workspace_bytes(const pkv_cache_desc* cache, int32_t batch,
                                        int32_t num_query_tokens, int32_t num_q_heads,
                                        int32_t max_blocks_per_seq, const pkv_decode_opts* opts) {
  pkv::DecodeLaunch L;
  // The partition size (and so the workspace) must not depend on the device
  // the call later runs on: size with the largest SM count this build targets.
  if (resolve_decode(cache, batch, num_query_tokens, num_q_heads, max_blocks_per_seq, opts, 152, &L) !=
      PKV_OK)
    return 0;
  return layout_of(L).total;
}

size_t pkv_decode_workspace_bytes(const pkv_cache_desc* cache, int32_t batch, int32_t num_q_heads,
                                  int32_t max_blocks_per_seq, const pkv_decode_opts* opts) {
  return pkv_decode_multi_workspace_bytes(cache, batch, 1, num_q_heads, max_blocks_per_seq, opts);
}

pkv_status pkv_decode_multi_describe(const pkv_cache_desc* cache, int32_t batch,
                                     int32_t num_query_tokens, int32_t num_q_heads,
                                     int32_t max_blocks_per_seq, const pkv_decode_opts* opts,
                                     pkv_decode_plan* plan) {
  if (plan == nullptr) return fail(PKV_ERR_INVALID_ARG, "plan is NULL");
  pkv::DecodeLaunch L;
  pkv_status st = resolve_decode(cache, batch, num_query_tokens, num_q_heads, max_blocks_per_seq, opts,
                                 152, &L);
  if (st != PKV_OK) return st;
  plan->partition_blocks = L.ppu;
  plan->max_partitions = L.pmax;
  plan->math = L.math;
  plan->warps_per_cta = L.warps;
  plan->stages = L.stages;
  // the merge kernel runs above 4 partitions (tcgen05 kernel: above 1)
  plan->kernels_per_call = L.pmax > (L.tc ? 1 : 4) ? 3 : 2;
  plan->workspace_bytes = layout_of(L).total;
  plan->smem_bytes_per_cta = pkv::decode_smem_bytes(L.kv_fp8, L.D, L.bs, L.warps, L.stages, L.tc, L.tc2);
  plan->query_tokens_per_tile = L.Tt;
  plan->row_tiles = L.NT;
  return PKV_OK;
}

pkv_status pkv_decode_describe(const pkv_cache_desc* cache, int32_t batch, int32_t num_q_heads,
                               int32_t max_blocks_per_seq, const pkv_decode_opts* opts,
                               pkv_decode_plan* plan) {
  return pkv_decode_multi_describe(cache, batch, 1, num_q_heads, max_blocks_per_seq, opts, plan);
}

}  // extern "C"

// The new tokens of a fused append-and-decode call.
struct AppendRequest {
  const void* k;
  const void* v;
  const int64_t* slot_mapping;
  int32_t num_tokens;
};

static pkv_status decode_call(const pkv_cache_desc* cache, const void* q, int32_t batch,
                              int32_t num_query_tokens, int32_t num_q_heads, const void* k_cache,
                              const void* v_cache, const float* k_scale, const float* v_scale,
                              const int32_t* block_tables, int32_t max_blocks_per_seq,
                              const int32_t* context_lens, const int32_t* kv_group_ptr,
                              int32_t num_layers, int32_t layer, float scale, void* out,
                              void* workspace, size_t workspace_bytes,
                              const pkv_decode_opts* opts, void* stream, const AppendRequest* req) {
  pkv::DecodeLaunch L;
  pkv_status st = resolve_decode(cache, batch, num_query_tokens, num_q_heads, max_blocks_per_seq, opts,
                                 152, &L);
  if (st != PKV_OK) return st;
  if (kv_group_ptr == nullptr || num_layers < 1 || layer < 0 || layer >= num_layers)
    return fail(PKV_ERR_INVALID_ARG, "layer %d / num_layers %d / kv_group_ptr", layer, num_layers);
  const int32_t slot = kv_group_ptr[layer];
  if (slot < 0 || slot >= cache->num_slots)
    return fail(PKV_ERR_INVALID_ARG, "kv_group_ptr[%d] = %d outside [0, %d)", layer, slot, cache->num_slots);
  if (!std::isfinite(scale)) return fail(PKV_ERR_INVALID_ARG, "scale is not finite");
  if (batch == 0) {  // nothing to decode: only the append, if any
    if (req == nullptr || req->num_tokens == 0) return PKV_OK;
    return pkv_kv_append(cache, slot, req->k, req->v, req->slot_mapping, req->num_tokens,
                         const_cast<void*>(k_cache), const_cast<void*>(v_cache), k_scale, v_scale, stream);
  }
  const bool fp8 = cache->dtype != PKV_KV_BF16;  // one-byte elements (E4M3 or INT8)
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
    return fail(PKV_ERR_INVALID_ARG, "NULL tensor pointer");
  if (fp8 && (!k_scale || !v_scale)) return fail(PKV_ERR_INVALID_ARG, "E4M3 and INT8 caches need k_scale and v_scale");
  if (fp8 && !scales_aligned(cache->dtype, k_scale, v_scale))
    return fail(PKV_ERR_ALIGNMENT, "k_scale and v_scale must be 4-byte (E4M3) or 8-byte (INT8) aligned");
  if (!aligned16(q) || !aligned16(out) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(workspace))
    return fail(PKV_ERR_ALIGNMENT, "q, out, caches and workspace must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(context_lens) & 3u))
    return fail(PKV_ERR_ALIGNMENT, "block_tables and context_lens must be 4-byte aligned");
  const size_t qbytes = static_cast<size_t>(batch) * num_query_tokens * num_q_heads * cache->head_dim * 2;
  const uintptr_t qa = reinterpret_cast<uintptr_t>(q), oa = reinterpret_cast<uintptr_t>(out);
  if (qa < oa + qbytes && oa < qa + qbytes) return fail(PKV_ERR_INVALID_ARG, "out overlaps q");
  const pkv::WorkspaceLayout wl = layout_of(L);
  if (workspace == nullptr || workspace_bytes < wl.total)
    return fail(PKV_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu", wl.total, workspace_bytes);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DeviceInfo dev_info;
  const DeviceInfo* dev = &dev_info;
  if ((st = device_info(&dev_info)) != PKV_OK) return st;
  L.num_sms = dev->num_sms;

  if (env_flag("PKV_VALIDATE")) {
    std::vector<int32_t> ctx, bt;
    if ((st = fetch(ctx, context_lens, static_cast<size_t>(batch), s)) != PKV_OK) return st;
    if ((st = fetch(bt, block_tables, static_cast<size_t>(batch) * max_blocks_per_seq, s)) != PKV_OK) return st;
    for (int b = 0; b < batch; ++b) {
      if (ctx[b] < 0 || static_cast<long long>(ctx[b]) > static_cast<long long>(max_blocks_per_seq) * cache->block_size)
        return fail(PKV_ERR_INVALID_ARG, "context_lens[%d] = %d out of range", b, ctx[b]);
      for (int j = 0; j < (ctx[b] + cache->block_size - 1) / cache->block_size; ++j) {
        const int32_t blk = bt[static_cast<size_t>(b) * max_blocks_per_seq + j];
        if (blk < 0 || blk >= cache->num_blocks)
          return fail(PKV_ERR_INVALID_ARG, "block_tables[%d][%d] = %d outside [0, %d)", b, j, blk,
                      cache->num_blocks);
      }
    }
  }

  if ((st = encode_cache_map(&L.kmap, k_cache, cache)) != PKV_OK) return st;
  if ((st = encode_cache_map(&L.vmap, v_cache, cache)) != PKV_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  L.q = q;
  L.out = out;
  L.block_tables = block_tables;
  L.context_lens = context_lens;
  const size_t scale_off = static_cast<size_t>(slot) * cache->num_blocks * cache->num_kv_heads *
                           (cache->dtype == PKV_KV_INT8 ? 2 : 1);
  L.k_scale = fp8 ? k_scale + scale_off : nullptr;
  L.v_scale = fp8 ? v_scale + scale_off : nullptr;
  L.work_counter = reinterpret_cast<int32_t*>(ws + wl.counter);
  L.unit_start = reinterpret_cast<int32_t*>(ws + wl.unit_start);
  L.ctx_eff = reinterpret_cast<int32_t*>(ws + wl.ctx_eff);
  L.part_seq = reinterpret_cast<int32_t*>(ws + wl.part_seq);
  L.arrive = reinterpret_cast<int32_t*>(ws + wl.arrive);
  L.part_ml = reinterpret_cast<float*>(ws + wl.part_ml);
  L.part_o = reinterpret_cast<float*>(ws + wl.part_o);
  if (L.tc && !L.tc2 && L.pmax > 1 &&
      (st = encode_partial_map(&L.pmap, L.part_o, batch, L.T, L.Hq, L.pmax, L.D, L.G, L.Tt)) != PKV_OK)
    return st;
  if (L.tc && !L.tc2 && (st = encode_output_map(&L.omap, out, batch, L.T, L.Hq, L.D, L.G, L.Tt)) != PKV_OK)
    return st;
  if (L.tc2 && (st = encode_query_map(&L.qmap, q, batch, L.T, L.Hq, L.D, L.G, L.Tt)) != PKV_OK) return st;
  L.err = dev->err_word;
  L.row_base = static_cast<int>(static_cast<long long>(slot) * cache->num_blocks * cache->num_kv_heads *
                                cache->block_size);
  L.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  L.stream = s;
  if (opts != nullptr) {
    L.ev_start = static_cast<cudaEvent_t>(opts->event_decode_start);
    L.ev_end = static_cast<cudaEvent_t>(opts->event_decode_end);
  }
  pkv::AppendArgs app{};
  if (req != nullptr && req->num_tokens > 0) {
    if ((st = prepare_append(cache, slot, req->k, req->v, req->slot_mapping, req->num_tokens,
                             const_cast<void*>(k_cache), const_cast<void*>(v_cache), k_scale, v_scale, s,
                             dev, &app)) != PKV_OK)
      return st;
    L.append = &app;
    L.append_kind = cache->dtype;
  }
  int launched = 0;
  cudaError_t e = pkv::launch_decode(L, &launched);
  if (e != cudaSuccess) return cuda_fail(e, "paged_decode launch");
  return PKV_OK;
}

extern "C" {

pkv_status pkv_paged_decode_multi(const pkv_cache_desc* cache, const void* q, int32_t batch,
                                  int32_t num_query_tokens, int32_t num_q_heads, const void* k_cache,
                                  const void* v_cache, const float* k_scale, const float* v_scale,
                                  const int32_t* block_tables, int32_t max_blocks_per_seq,
                                  const int32_t* context_lens, const int32_t* kv_group_ptr,
                                  int32_t num_layers, int32_t layer, float scale, void* out,
                                  void* workspace, size_t workspace_bytes,
                                  const pkv_decode_opts* opts, void* stream) {
  return decode_call(cache, q, batch, num_query_tokens, num_q_heads, k_cache, v_cache, k_scale, v_scale,
                     block_tables, max_blocks_per_seq, context_lens, kv_group_ptr, num_layers, layer, scale,
                     out, workspace, workspace_bytes, opts, stream, nullptr);
}

pkv_status pkv_append_and_decode(const pkv_cache_desc* cache, const void* k_new, const void* v_new,
                                 const int64_t* slot_mapping, int32_t num_new_tokens, const void* q,
                                 int32_t batch, int32_t num_query_tokens, int32_t num_q_heads,
                                 void* k_cache, void* v_cache, const float* k_scale, const float* v_scale,
                                 const int32_t* block_tables, int32_t max_blocks_per_seq,
                                 const int32_t* context_lens, const int32_t* kv_group_ptr,
                                 int32_t num_layers, int32_t layer, float scale, void* out,
                                 void* workspace, size_t workspace_bytes, const pkv_decode_opts* opts,
                                 void* stream) {
  if (num_new_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "num_new_tokens %d < 0", num_new_tokens);
  const AppendRequest req{k_new, v_new, slot_mapping, num_new_tokens};
  return decode_call(cache, q, batch, num_query_tokens, num_q_heads, k_cache, v_cache, k_scale, v_scale,
                     block_tables, max_blocks_per_seq, context_lens, kv_group_ptr, num_layers, layer, scale,
                     out, workspace, workspace_bytes, opts, stream, &req);
}

pkv_status pkv_paged_decode(const pkv_cache_desc* cache, const void* q, int32_t batch,
                            int32_t num_q_heads, const void* k_cache, const void* v_cache,
                            const float* k_scale, const float* v_scale,
                            const int32_t* block_tables, int32_t max_blocks_per_seq,
                            const int32_t* context_lens, const int32_t* kv_group_ptr,
                            int32_t num_layers, int32_t layer, float scale, void* out,
                            void* workspace, size_t workspace_bytes, const pkv_decode_opts* opts,
                            void* stream) {
  return pkv_paged_decode_multi(cache, q, batch, 1, num_q_heads, k_cache, v_cache, k_scale, v_scale,
                                block_tables, max_blocks_per_seq, context_lens, kv_group_ptr,
                                num_layers, layer, scale, out, workspace, workspace_bytes, opts,
                                stream);
}

pkv_status pkv_copy_blocks(const pkv_cache_desc* cache, const void* src_k, const void* src_v,
                           const float* src_k_scale, const float* src_v_scale, int32_t src_num_blocks,
                           void* dst_k, void* dst_v, float* dst_k_scale, float* dst_v_scale,
                           int32_t dst_num_blocks, const int32_t* block_pairs, int32_t count,
                           void* stream) {
  pkv_status st = check_cache_desc(cache);
  if (st != PKV_OK) return st;
  if (count < 0 || src_num_blocks < 1 || dst_num_blocks < 1)
    return fail(PKV_ERR_INVALID_ARG, "count %d, src_num_blocks %d, dst_num_blocks %d", count,
                src_num_blocks, dst_num_blocks);
  if (count == 0) return PKV_OK;
  const bool fp8 = cache->dtype != PKV_KV_BF16;  // one-byte elements (E4M3 or INT8)
  if (!src_k || !src_v || !dst_k || !dst_v || !block_pairs)
    return fail(PKV_ERR_INVALID_ARG, "NULL pointer");
  if (fp8 && (!src_k_scale || !src_v_scale || !dst_k_scale || !dst_v_scale))
    return fail(PKV_ERR_INVALID_ARG, "E4M3 and INT8 pools need source and destination scales");
  if (fp8 && (!scales_aligned(cache->dtype, src_k_scale, src_v_scale) ||
              !scales_aligned(cache->dtype, dst_k_scale, dst_v_scale)))
    return fail(PKV_ERR_ALIGNMENT, "scales must be 4-byte (E4M3) or 8-byte (INT8) aligned");
  if (!aligned16(src_k) || !aligned16(src_v) || !aligned16(dst_k) || !aligned16(dst_v))
    return fail(PKV_ERR_ALIGNMENT, "pools must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(block_pairs) & 3u) != 0)
    return fail(PKV_ERR_ALIGNMENT, "block_pairs must be 4-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DeviceInfo dev_info;
  const DeviceInfo* dev = &dev_info;
  if ((st = device_info(&dev_info)) != PKV_OK) return st;
  if (env_flag("PKV_VALIDATE")) {
    std::vector<int32_t> pr;
    if ((st = fetch(pr, block_pairs, static_cast<size_t>(count) * 2, s)) != PKV_OK) return st;
    std::vector<int32_t> dsts;
    for (int i = 0; i < count; ++i) {
      if (pr[2 * i] < 0 || pr[2 * i] >= src_num_blocks || pr[2 * i + 1] < 0 || pr[2 * i + 1] >= dst_num_blocks)
        return fail(PKV_ERR_INVALID_ARG, "block_pairs[%d] = (%d, %d) out of range", i, pr[2 * i], pr[2 * i + 1]);
      dsts.push_back(pr[2 * i + 1]);
    }
    std::sort(dsts.begin(), dsts.end());
    if (std::adjacent_find(dsts.begin(), dsts.end()) != dsts.end())
      return fail(PKV_ERR_INVALID_ARG, "block_pairs has a repeated destination");
  }
  const int64_t block_bytes = static_cast<int64_t>(cache->num_kv_heads) * cache->block_size *
                              cache->head_dim * (fp8 ? 1 : 2);
  cudaError_t e = pkv::launch_copy_blocks(src_k, src_v, fp8 ? src_k_scale : nullptr,
                                          fp8 ? src_v_scale : nullptr, src_num_blocks, dst_k, dst_v,
                                          fp8 ? dst_k_scale : nullptr, fp8 ? dst_v_scale : nullptr,
                                          dst_num_blocks, block_pairs, count, block_bytes,
                                          cache->num_kv_heads * (cache->dtype == PKV_KV_INT8 ? 2 : 1),
                                          dev->num_sms, dev->err_word, s);
  if (e != cudaSuccess) return cuda_fail(e, "copy_blocks launch");
  return PKV_OK;
}

pkv_status pkv_read_probe(const void* data, size_t bytes, uint64_t* sum, void* stream) {
  if (bytes == 0) return PKV_OK;  // nothing to read, nothing launched
  if (data == nullptr || sum == nullptr) return fail(PKV_ERR_INVALID_ARG, "data or sum is NULL");
  if (bytes % 16 != 0) return fail(PKV_ERR_INVALID_ARG, "bytes %zu is not a multiple of 16", bytes);
  if (reinterpret_cast<uintptr_t>(data) % 16 != 0 || reinterpret_cast<uintptr_t>(sum) % 8 != 0)
    return fail(PKV_ERR_ALIGNMENT, "data must be 16-byte and sum 8-byte aligned");
  DeviceInfo dev_info;
  const DeviceInfo* dev = &dev_info;
  pkv_status st = device_info(&dev_info);
  if (st != PKV_OK) return st;
  cudaError_t e = pkv::launch_read_probe(data, bytes, reinterpret_cast<unsigned long long*>(sum), dev->num_sms,
                                         static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "read probe launch");
  return PKV_OK;
}

pkv_status pkv_read_device_error(uint32_t* flags, void* stream) {
  if (flags == nullptr) return fail(PKV_ERR_INVALID_ARG, "flags is NULL");
  DeviceInfo dev_info;
  const DeviceInfo* dev = &dev_info;
  pkv_status st = device_info(&dev_info);
  if (st != PKV_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned host = 0;
  cudaError_t e = cudaMemcpyAsync(&host, dev->err_word, sizeof host, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(dev->err_word, 0, sizeof host, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  *flags = host;
  if (host != 0) {
    set_error("device error word 0x%x", host);
    return PKV_ERR_DEVICE_INDEX;
  }
  return PKV_OK;
}

}  // extern "C"
