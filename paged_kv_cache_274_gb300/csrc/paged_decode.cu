// Planner and split-K merge kernels, and the host-side launch sequence of a
// paged decode (planner -> decode -> merge).
//
// Split-K ("flash-decoding"): a long sequence is cut into partitions of
// `ppu` blocks that different warps process at the same time; each writes
// its running max m_p (log2 domain), sum l_p and unnormalised output O_p.
// The merge takes M = max_p m_p and returns
//   out = sum_p 2^(m_p - M) O_p / sum_p 2^(m_p - M) l_p,
// which is the softmax over the union of the partitions' tokens.
#include <algorithm>

#include "paged_decode.cuh"
#include "pkv_internal.h"

namespace pkv {

// Kernel tables of the instantiation units.
const void* decode_kernel_bf16_d64(int bs, int math, int gt);
const void* decode_kernel_bf16_d128(int bs, int math, int gt);
const void* decode_kernel_fp8_d128(int bs, int math, int gt);

// ---------------------------------------------------------------------------
// planner: one CTA validates context lengths, counts each sequence's
// partitions, prefix-sums them into unit_start, resets the work queue and
// writes zeros for sequences that attend to nothing.
// ---------------------------------------------------------------------------
constexpr int kPlanThreads = 1024;

__global__ void __launch_bounds__(kPlanThreads)
    plan_kernel(const int32_t* __restrict__ context_lens, int B, int max_ctx, int tokens_per_part,
                int32_t* work_counter, int32_t* unit_start, int32_t* ctx_eff,
                __nv_bfloat16* out, int row_elems /* Hq * D */, unsigned* err) {
  __shared__ int warp_tot[kPlanThreads / 32];
  __shared__ int carry_s;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) carry_s = 0;
  __syncthreads();
  bool bad_any = false;
  for (int base = 0; base < B; base += kPlanThreads) {
    const int b = base + tid;
    int parts = 0;
    if (b < B) {
      int c = context_lens[b];
      if (c < 0 || c > max_ctx) {
        bad_any = true;
        c = 0;
      }
      ctx_eff[b] = c;
      parts = (c + tokens_per_part - 1) / tokens_per_part;
    }
    // inclusive scan within the warp, then across warps
    int x = parts;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = warp_tot[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, w, o);
        if (lane >= o) w += y;
      }
      warp_tot[lane] = w;  // inclusive prefix of warp totals
    }
    __syncthreads();
    const int before = (warp > 0 ? warp_tot[warp - 1] : 0) + x - parts;
    if (b < B) unit_start[b] = carry_s + before;
    __syncthreads();
    if (tid == kPlanThreads - 1) carry_s += warp_tot[31];
    __syncthreads();
  }
  if (tid == 0) {
    unit_start[B] = carry_s;
    *work_counter = 0;
  }
  if (__syncthreads_or(bad_any) && tid == 0) atomicOr(err, PKV_DEVERR_CONTEXT_LEN);
  // zeros for inactive sequences (one warp per sequence)
  for (int b = warp; b < B; b += kPlanThreads / 32) {
    if (ctx_eff[b] != 0) continue;
    uint4* o = reinterpret_cast<uint4*>(out + static_cast<size_t>(b) * row_elems);
    for (int i = lane; i < row_elems / 8; i += 32) o[i] = make_uint4(0, 0, 0, 0);
  }
}

// ---------------------------------------------------------------------------
// merge: one warp per (sequence, query head) with more than one partition
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256)
    merge_kernel(const float* __restrict__ part_ml, const float* __restrict__ part_o,
                 const int32_t* __restrict__ unit_start, int B, int Hq, int pmax,
                 __nv_bfloat16* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (gw >= B * Hq) return;
  const int b = gw / Hq;
  const int P = unit_start[b + 1] - unit_start[b];
  if (P < 2) return;
  const size_t base = static_cast<size_t>(gw) * pmax;
  float M = -INFINITY;
  for (int i = lane; i < P; i += 32) M = fmaxf(M, part_ml[2 * (base + i)]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
  constexpr int kPer = D / 32;
  float acc[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) acc[j] = 0.f;
  float L = 0.f;
  if (M != -INFINITY) {
    for (int i = 0; i < P; ++i) {
      const float2 ml = *reinterpret_cast<const float2*>(part_ml + 2 * (base + i));
      const float w = exp2f(ml.x - M);  // 0 for an empty partition (m = -inf)
      L = fmaf(w, ml.y, L);
      const float* src = part_o + (base + i) * D + lane * kPer;
      if constexpr (kPer == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        acc[0] = fmaf(w, v.x, acc[0]);
        acc[1] = fmaf(w, v.y, acc[1]);
        acc[2] = fmaf(w, v.z, acc[2]);
        acc[3] = fmaf(w, v.w, acc[3]);
      } else {
        const float2 v = *reinterpret_cast<const float2*>(src);
        acc[0] = fmaf(w, v.x, acc[0]);
        acc[1] = fmaf(w, v.y, acc[1]);
      }
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  __nv_bfloat16* o = out + static_cast<size_t>(gw) * D + lane * kPer;
#pragma unroll
  for (int j = 0; j < kPer; j += 2)
    *reinterpret_cast<__nv_bfloat162*>(o + j) = __floats2bfloat162_rn(acc[j] * inv, acc[j + 1] * inv);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

WorkspaceLayout workspace_layout(int B, int Hq, int D, int pmax) {
  WorkspaceLayout w{};
  size_t off = 0;
  w.counter = off;
  off += 256;
  w.unit_start = off;
  off = align_up(off + sizeof(int32_t) * (static_cast<size_t>(B) + 1), 256);
  w.ctx_eff = off;
  off = align_up(off + sizeof(int32_t) * static_cast<size_t>(B), 256);
  const size_t parts = pmax > 1 ? static_cast<size_t>(B) * Hq * pmax : 0;
  w.part_ml = off;
  off = align_up(off + sizeof(float) * 2 * parts, 256);
  w.part_o = off;
  off = align_up(off + sizeof(float) * D * parts, 256);
  w.total = off;
  return w;
}

size_t decode_smem_bytes(int kv_fp8, int D, int bs, int warps, int stages) {
  if (kv_fp8) {
    return bs == 16 ? decode_smem_layout_bytes<128, 16, true>(warps, stages)
                    : decode_smem_layout_bytes<128, 32, true>(warps, stages);
  }
  if (D == 64)
    return bs == 16 ? decode_smem_layout_bytes<64, 16, false>(warps, stages)
                    : decode_smem_layout_bytes<64, 32, false>(warps, stages);
  return bs == 16 ? decode_smem_layout_bytes<128, 16, false>(warps, stages)
                  : decode_smem_layout_bytes<128, 32, false>(warps, stages);
}

static const void* pick_kernel(const DecodeLaunch& L) {
  const int gt = (L.math == PKV_MATH_FFMA) ? L.G : 0;
  if (L.kv_fp8) return decode_kernel_fp8_d128(L.bs, L.math, gt);
  if (L.D == 64) return decode_kernel_bf16_d64(L.bs, L.math, gt);
  return decode_kernel_bf16_d128(L.bs, L.math, gt);
}

int decode_ctas_per_sm(const DecodeLaunch& L, size_t smem) {
  const void* fn = pick_kernel(L);
  if (fn == nullptr) return 0;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, L.warps * 32, smem) != cudaSuccess) return 0;
  return n;
}

cudaError_t launch_decode(const DecodeLaunch& L, int* launched) {
  *launched = 0;
  const void* fn = pick_kernel(L);
  if (fn == nullptr) return cudaErrorInvalidDeviceFunction;
  const size_t smem = decode_smem_bytes(L.kv_fp8, L.D, L.bs, L.warps, L.stages);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;

  // 1. planner
  plan_kernel<<<1, kPlanThreads, 0, L.stream>>>(L.context_lens, L.B, L.MB * L.bs, L.ppu * L.bs,
                                                L.work_counter, L.unit_start, L.ctx_eff,
                                                static_cast<__nv_bfloat16*>(L.out), L.Hq * L.D, L.err);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  *launched += 1;

  // 2. decode: persistent grid, at most one warp per possible unit
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, L.warps * 32, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const long long max_units = static_cast<long long>(L.B) * L.Hkv * L.pmax;
  long long grid = static_cast<long long>(L.num_sms) * per_sm;
  grid = std::min(grid, (max_units + L.warps - 1) / L.warps);
  grid = std::max(grid, 1LL);

  DecodeParams p{};
  p.q = static_cast<const __nv_bfloat16*>(L.q);
  p.out = static_cast<__nv_bfloat16*>(L.out);
  p.block_tables = L.block_tables;
  p.k_scale = L.k_scale;
  p.v_scale = L.v_scale;
  p.work_counter = L.work_counter;
  p.unit_start = L.unit_start;
  p.ctx_eff = L.ctx_eff;
  p.part_ml = L.part_ml;
  p.part_o = L.part_o;
  p.err = L.err;
  p.B = L.B;
  p.Hq = L.Hq;
  p.Hkv = L.Hkv;
  p.G = L.G;
  p.MB = L.MB;
  p.NB = L.NB;
  p.pmax = L.pmax;
  p.ppu = L.ppu;
  p.stages = L.stages;
  p.row_base = L.row_base;
  p.scale_log2 = L.scale_log2;
  CUtensorMap kmap = L.kmap, vmap = L.vmap;
  void* args[] = {&kmap, &vmap, &p};
  if (L.ev_start != nullptr && (e = cudaEventRecord(L.ev_start, L.stream)) != cudaSuccess) return e;
  e = cudaLaunchKernel(fn, dim3(static_cast<unsigned>(grid)), dim3(L.warps * 32), args, smem, L.stream);
  if (e != cudaSuccess) return e;
  if (L.ev_end != nullptr && (e = cudaEventRecord(L.ev_end, L.stream)) != cudaSuccess) return e;
  *launched += 1;

  // 3. merge (only when some sequence can span more than one partition)
  if (L.pmax > 1) {
    const int warps_total = L.B * L.Hq;
    const int blocks = (warps_total + 7) / 8;
    if (L.D == 64)
      merge_kernel<64><<<blocks, 256, 0, L.stream>>>(L.part_ml, L.part_o, L.unit_start, L.B, L.Hq,
                                                     L.pmax, static_cast<__nv_bfloat16*>(L.out));
    else
      merge_kernel<128><<<blocks, 256, 0, L.stream>>>(L.part_ml, L.part_o, L.unit_start, L.B, L.Hq,
                                                      L.pmax, static_cast<__nv_bfloat16*>(L.out));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    *launched += 1;
  }
  return cudaSuccess;
}

}  // namespace pkv
