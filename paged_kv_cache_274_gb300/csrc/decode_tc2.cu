// tcgen05 multi-token decode instances that serve a pair of row tiles per
// CTA (T x G > 128 query rows per KV head): bf16 cache, head_dim 128.
#include "paged_decode_tc2.cuh"

namespace pkv {

const void* decode_kernel_tc2(int bs) {
  if (bs == 16) return reinterpret_cast<const void*>(&paged_decode_tc2_kernel<16>);
  if (bs == 32) return reinterpret_cast<const void*>(&paged_decode_tc2_kernel<32>);
  return nullptr;
}

}  // namespace pkv
