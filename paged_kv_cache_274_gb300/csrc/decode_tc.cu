// tcgen05 multi-token decode kernel instances: bf16 cache, head_dim 128.
#include "paged_decode_tc.cuh"

namespace pkv {

const void* decode_kernel_tc(int bs) {
  if (bs == 16) return reinterpret_cast<const void*>(&paged_decode_tc_kernel<16>);
  if (bs == 32) return reinterpret_cast<const void*>(&paged_decode_tc_kernel<32>);
  return nullptr;
}

}  // namespace pkv
