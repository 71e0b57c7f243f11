// Block copy: whole physical blocks (all KV heads, K and V, and the
// page parameters of one-byte caches) from one block pool to another, by (source id, destination id)
// pairs.  Used for copy-on-write of a shared block before a sequence appends
// into it, and for moving a sequence's blocks between HBM and host memory.
//
// Source: "KV Cache Engineering: PagedAttention, Continuous Batching,
// Attention Variants, and the Bandwidth Wall" -- "PagedAttention" (block
// sharing); "KV-Cache Engineering: The Memory Wall of LLM Serving" --
// "Lever 5: Offloading", "When the cache fills" (swap to host memory).
//
// A CTA copies one slice of a pair: kCopySliceChunks 16-byte chunks of K and
// the same of V (4 KiB each), every load of a thread issued before its
// stores, coalesced on both sides.  Small slices keep the last wave of CTAs
// short.  Bandwidth-bound: 2 x block bytes moved per pair (read + write).
#include <algorithm>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

constexpr int kCopyThreads = 128;
constexpr int kCopySliceChunks = 256;                       // per tensor (K or V)
constexpr int kCopyPerThread = kCopySliceChunks / kCopyThreads;  // 2

__global__ void __launch_bounds__(kCopyThreads)
    copy_blocks_kernel(const uint4* __restrict__ src_k, const uint4* __restrict__ src_v,
                       const float* __restrict__ src_ks, const float* __restrict__ src_vs,
                       int src_nb, uint4* __restrict__ dst_k, uint4* __restrict__ dst_v,
                       float* __restrict__ dst_ks, float* __restrict__ dst_vs, int dst_nb,
                       const int32_t* __restrict__ pairs, int count, int64_t chunks_per_block,
                       int scales_per_block, unsigned* __restrict__ err) {
  pdl_trigger();
  pdl_wait();
  const int64_t slices = (chunks_per_block + kCopySliceChunks - 1) / kCopySliceChunks;
  const int64_t items = static_cast<int64_t>(count) * slices;
  for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
    const int i = static_cast<int>(it / slices);
    const int64_t slice = it - static_cast<int64_t>(i) * slices;
    const int s = pairs[2 * i], d = pairs[2 * i + 1];
    if (static_cast<unsigned>(s) >= static_cast<unsigned>(src_nb) ||
        static_cast<unsigned>(d) >= static_cast<unsigned>(dst_nb)) {
      if (threadIdx.x == 0 && slice == 0) atomicOr(err, PKV_DEVERR_BLOCK_ID);
      continue;
    }
    const int64_t base = slice * kCopySliceChunks;
    const uint4* sk = src_k + static_cast<int64_t>(s) * chunks_per_block + base;
    const uint4* sv = src_v + static_cast<int64_t>(s) * chunks_per_block + base;
    uint4* dk = dst_k + static_cast<int64_t>(d) * chunks_per_block + base;
    uint4* dv = dst_v + static_cast<int64_t>(d) * chunks_per_block + base;
    const int64_t rest = chunks_per_block - base;
    const int64_t n = rest < kCopySliceChunks ? rest : kCopySliceChunks;
    uint4 a[kCopyPerThread], b[kCopyPerThread];
#pragma unroll
    for (int u = 0; u < kCopyPerThread; ++u) {
      const int64_t c = threadIdx.x + u * kCopyThreads;
      if (c < n) {
        a[u] = sk[c];
        b[u] = sv[c];
      }
    }
#pragma unroll
    for (int u = 0; u < kCopyPerThread; ++u) {
      const int64_t c = threadIdx.x + u * kCopyThreads;
      if (c < n) {
        dk[c] = a[u];
        dv[c] = b[u];
      }
    }
    if (src_ks != nullptr && slice == 0) {
      for (int h = threadIdx.x; h < scales_per_block; h += kCopyThreads) {
        dst_ks[static_cast<int64_t>(d) * scales_per_block + h] = src_ks[static_cast<int64_t>(s) * scales_per_block + h];
        dst_vs[static_cast<int64_t>(d) * scales_per_block + h] = src_vs[static_cast<int64_t>(s) * scales_per_block + h];
      }
    }
  }
}

cudaError_t launch_copy_blocks(const void* src_k, const void* src_v, const float* src_ks,
                               const float* src_vs, int src_nb, void* dst_k, void* dst_v,
                               float* dst_ks, float* dst_vs, int dst_nb, const int32_t* pairs,
                               int count, int64_t block_bytes, int scales_per_block,
                               int num_sms, unsigned* err, cudaStream_t stream) {
  // one CTA per slice of a pair (the hardware scheduler balances the tail); a
  // grid-stride loop covers counts beyond the grid limit
  const int64_t chunks = block_bytes / 16;
  const int64_t items = static_cast<int64_t>(count) * ((chunks + kCopySliceChunks - 1) / kCopySliceChunks);
  const int grid = static_cast<int>(std::min<int64_t>(items, 1 << 30));
  (void)num_sms;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(std::max(grid, 1)));
  cfg.blockDim = dim3(kCopyThreads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, copy_blocks_kernel, static_cast<const uint4*>(src_k),
                            static_cast<const uint4*>(src_v), src_ks, src_vs, src_nb,
                            static_cast<uint4*>(dst_k), static_cast<uint4*>(dst_v), dst_ks, dst_vs,
                            dst_nb, pairs, count, block_bytes / 16, scales_per_block, err);
}

}  // namespace pkv
