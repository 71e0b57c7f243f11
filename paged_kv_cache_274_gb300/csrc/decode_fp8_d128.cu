// Decode kernel instances: head_dim 128, E4M3 cache.
#include "decode_instances.cuh"

namespace pkv {

const void* decode_kernel_fp8_d128(int bs, int math, int gt) {
  if (bs == 16) return decode_kernel_for<128, 16, true>(math, gt);
  if (bs == 32) return decode_kernel_for<128, 32, true>(math, gt);
  return nullptr;
}

}  // namespace pkv
