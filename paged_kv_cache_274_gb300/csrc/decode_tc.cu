// tcgen05 multi-token decode kernel instances: bf16 cache, head_dim 128.
#include "paged_decode_tc.cuh"

namespace pkv {

// rot: tiles of at most 96 query rows, rotated into the highest TMEM lanes
const void* decode_kernel_tc(int bs, bool rot) {
  if (bs == 16) return rot ? reinterpret_cast<const void*>(&paged_decode_tc_kernel<16, true>)
                           : reinterpret_cast<const void*>(&paged_decode_tc_kernel<16, false>);
  if (bs == 32) return rot ? reinterpret_cast<const void*>(&paged_decode_tc_kernel<32, true>)
                           : reinterpret_cast<const void*>(&paged_decode_tc_kernel<32, false>);
  return nullptr;
}

}  // namespace pkv
