// Multi-token decode kernel instances, bf16 cache (head_dim 64 and 128).
#include "decode_instances.cuh"

namespace pkv {

const void* decode_kernel_mt_bf16(int D, int bs, int gt) {
  if (D == 64 && bs == 16) return decode_kernel_mt_for<64, 16, false>(gt);
  if (D == 64 && bs == 32) return decode_kernel_mt_for<64, 32, false>(gt);
  if (D == 128 && bs == 16) return decode_kernel_mt_for<128, 16, false>(gt);
  if (D == 128 && bs == 32) return decode_kernel_mt_for<128, 32, false>(gt);
  return nullptr;
}

}  // namespace pkv
