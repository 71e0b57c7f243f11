// Multi-token decode kernel instances, one-byte caches (E4M3, INT8; head_dim 128).
#include "decode_instances.cuh"

namespace pkv {

const void* decode_kernel_mt_1byte(int kv_dtype, int bs, int gt) {
  if (kv_dtype == PKV_KV_FP8_E4M3) {
    if (bs == 16) return decode_kernel_mt_for<128, 16, true>(gt);
    if (bs == 32) return decode_kernel_mt_for<128, 32, true>(gt);
  } else if (kv_dtype == PKV_KV_INT8) {
    if (bs == 16) return decode_kernel_mt_for<128, 16, true, true>(gt);
    if (bs == 32) return decode_kernel_mt_for<128, 32, true, true>(gt);
  }
  return nullptr;
}

}  // namespace pkv
