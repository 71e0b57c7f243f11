// KV append: write each new token's K and V rows into their physical slots.
//
// Source: "KV Cache Engineering: PagedAttention, Continuous Batching,
// Attention Variants, and the Bandwidth Wall" -- "What the KV Cache Stores
// and Why" (a step computes K,V for the new token only and stores them for
// later steps) and "Continuous Batching" (a growing sequence takes a free
// block when it needs one; the caller's slot mapping says which).
//
// One thread moves one 16-byte chunk: 8 bf16 values, or 8 values quantised
// to 8 bytes with the page's parameters, the division in IEEE binary32:
//   E4M3: e4m3_rn_satfinite(float(x) / scale)
//   INT8: clamp(rne(float(x) / scale) + zero, lo, 127), lo = -127 for a
//         symmetric page (zero == 0) else -128; NaN stores the zero point
//         ([BW] "INT8 KV cache").
// The chunk loop is a device function so that the decode's planner launch
// can run it on extra CTAs (append and plan in one launch).
#pragma once

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {


__device__ __forceinline__ uint32_t int8_code(float x, float scale, float zero) {
  const float t = __fdiv_rn(x, scale);
  if (isnan(t)) return static_cast<uint32_t>(static_cast<int>(zero)) & 0xffu;
  const float lo = (zero == 0.f) ? -127.f : -128.f;
  const float q = fminf(fmaxf(rintf(t) + zero, lo), 127.f);
  return static_cast<uint32_t>(static_cast<int>(q)) & 0xffu;
}

// Chunks first, first + stride, ... of the 2 * N * Hkv * D / 8 chunks (K then V).
template <int KV>  // pkv_kv_dtype
__device__ __forceinline__ void append_chunks(const AppendArgs& a, int64_t first, int64_t stride) {
  const int chunks_per_row = a.D / 8;
  const int64_t per_tensor = static_cast<int64_t>(a.N) * a.Hkv * chunks_per_row;
  const int64_t total = 2 * per_tensor;
  for (int64_t idx = first; idx < total; idx += stride) {
    const bool is_v = idx >= per_tensor;
    const int64_t r = is_v ? idx - per_tensor : idx;
    const int c = static_cast<int>(r % chunks_per_row);
    const int64_t th = r / chunks_per_row;  // token * Hkv + head
    const int h = static_cast<int>(th % a.Hkv);
    const int64_t i = th / a.Hkv;
    const int64_t s = __ldg(a.slot_mapping + i);
    if (s == -1) continue;
    if (s < -1 || s >= a.nslots) {
      if (!is_v && h == 0 && c == 0) atomicOr(a.err, PKV_DEVERR_SLOT);
      continue;
    }
    const int64_t blk = s / a.bs, off = s % a.bs;
    const int64_t page = blk * a.Hkv + h;
    const int64_t dst_elem = (page * a.bs + off) * a.D + 8 * c;
    const uint4 w = __ldg((is_v ? a.v : a.k) + th * chunks_per_row + c);
    if constexpr (KV == PKV_KV_BF16) {
      *reinterpret_cast<uint4*>((is_v ? a.vc : a.kc) + 2 * dst_elem) = w;
    } else if constexpr (KV == PKV_KV_INT8) {
      const float2 sz = __ldg(reinterpret_cast<const float2*>(is_v ? a.vs : a.ks) + page);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
      uint32_t outw[2] = {0u, 0u};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t lo = int8_code(bf16lo_to_f32(ws[j]), sz.x, sz.y);
        const uint32_t hi = int8_code(bf16hi_to_f32(ws[j]), sz.x, sz.y);
        outw[j >> 1] |= (lo | (hi << 8)) << (16 * (j & 1));
      }
      *reinterpret_cast<uint2*>((is_v ? a.vc : a.kc) + dst_elem) = make_uint2(outw[0], outw[1]);
    } else {
      const float scale = __ldg((is_v ? a.vs : a.ks) + page);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
      uint32_t outw[2];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t packed = 0;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const uint32_t word = ws[2 * half + j];
          const float2 x = make_float2(__fdiv_rn(bf16lo_to_f32(word), scale),
                                       __fdiv_rn(bf16hi_to_f32(word), scale));
          const __nv_fp8x2_storage_t q = __nv_cvt_float2_to_fp8x2(x, __NV_SATFINITE, __NV_E4M3);
          packed |= static_cast<uint32_t>(q) << (16 * j);
        }
        outw[half] = packed;
      }
      *reinterpret_cast<uint2*>((is_v ? a.vc : a.kc) + dst_elem) = make_uint2(outw[0], outw[1]);
    }
  }
}

}  // namespace pkv
