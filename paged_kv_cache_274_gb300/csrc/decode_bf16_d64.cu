// Decode kernel instances: head_dim 64, bf16 cache.
#include "decode_instances.cuh"

namespace pkv {

const void* decode_kernel_bf16_d64(int bs, int math, int gt) {
  if (bs == 16) return decode_kernel_for<64, 16, false>(math, gt);
  if (bs == 32) return decode_kernel_for<64, 32, false>(math, gt);
  return nullptr;
}

}  // namespace pkv
