// Kernel table for one (head_dim, KV dtype) family of the decode kernel.
#pragma once

#include "paged_decode.cuh"

namespace pkv {

// gt: query rows per tile (heads of the group x query tokens per tile).
template <int D, int BS, bool FP8, bool I8 = false>
const void* decode_kernel_for(int math, int gt) {
  if (math == PKV_MATH_MMA) {
    // GT = 8: at most 8 rows per tile (half tiles); 16: up to 16
    if (gt <= 8) return reinterpret_cast<const void*>(&paged_decode_kernel<D, BS, FP8, PKV_MATH_MMA, 8, I8>);
    if (gt <= 16) return reinterpret_cast<const void*>(&paged_decode_kernel<D, BS, FP8, PKV_MATH_MMA, 16, I8>);
    return nullptr;
  }
  if (math != PKV_MATH_FFMA) return nullptr;
  switch (gt) {
    case 1: return reinterpret_cast<const void*>(&paged_decode_kernel<D, BS, FP8, PKV_MATH_FFMA, 1, I8>);
    case 2: return reinterpret_cast<const void*>(&paged_decode_kernel<D, BS, FP8, PKV_MATH_FFMA, 2, I8>);
    case 4: return reinterpret_cast<const void*>(&paged_decode_kernel<D, BS, FP8, PKV_MATH_FFMA, 4, I8>);
    case 8: return reinterpret_cast<const void*>(&paged_decode_kernel<D, BS, FP8, PKV_MATH_FFMA, 8, I8>);
    default: return nullptr;
  }
}

// Multi-token kernels (tensor-core back-end only).
template <int D, int BS, bool FP8, bool I8 = false>
const void* decode_kernel_mt_for(int gt) {
  if (gt <= 8) return reinterpret_cast<const void*>(&paged_decode_kernel<D, BS, FP8, PKV_MATH_MMA, 8, I8, true>);
  if (gt <= 16) return reinterpret_cast<const void*>(&paged_decode_kernel<D, BS, FP8, PKV_MATH_MMA, 16, I8, true>);
  return nullptr;
}

}  // namespace pkv
