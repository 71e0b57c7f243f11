// Decode kernel instances: head_dim 128, INT8 cache.
#include "decode_instances.cuh"

namespace pkv {

const void* decode_kernel_int8_d128(int bs, int math, int gt) {
  if (bs == 16) return decode_kernel_for<128, 16, true, true>(math, gt);
  if (bs == 32) return decode_kernel_for<128, 32, true, true>(math, gt);
  return nullptr;
}

}  // namespace pkv
