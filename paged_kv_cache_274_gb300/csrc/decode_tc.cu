// tcgen05 multi-token decode kernel instances (one 128-row tile per CTA),
// head_dim 128: bf16 caches, and E4M3 / INT8 caches widened in shared memory.
#include "paged_decode_tc.cuh"

namespace pkv {

template <int KV>
static const void* tc_instance(int bs, bool rot) {
  if (bs == 16) return rot ? reinterpret_cast<const void*>(&paged_decode_tc_kernel<16, true, KV>)
                           : reinterpret_cast<const void*>(&paged_decode_tc_kernel<16, false, KV>);
  if (bs == 32) return rot ? reinterpret_cast<const void*>(&paged_decode_tc_kernel<32, true, KV>)
                           : reinterpret_cast<const void*>(&paged_decode_tc_kernel<32, false, KV>);
  return nullptr;
}

// rot: tiles of at most 96 query rows, rotated into the highest TMEM lanes
const void* decode_kernel_tc(int bs, bool rot, int kv_dtype) {
  if (kv_dtype == PKV_KV_FP8_E4M3) return tc_instance<PKV_KV_FP8_E4M3>(bs, rot);
  if (kv_dtype == PKV_KV_INT8) return tc_instance<PKV_KV_INT8>(bs, rot);
  return tc_instance<PKV_KV_BF16>(bs, rot);
}

}  // namespace pkv
