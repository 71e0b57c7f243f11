// Planner and merge kernels and the host-side launch sequence of a paged
// decode (planner -> decode [-> merge when sequences span many partitions]).
//
// Split-K ("flash-decoding"): a long sequence is cut into partitions of
// `ppu` blocks that different warps process at the same time; each writes
// its running max m_p (log2 domain), sum l_p and unnormalised output O_p,
// and the warp that finishes a (sequence, KV head) last combines them.
//
// Both kernels are launched with programmatic dependent launch, so each can
// be scheduled while its predecessor on the stream drains; each waits for
// that predecessor (griddepcontrol.wait) before reading any global memory.
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <tuple>
#include <vector>

#include "kv_append.cuh"
#include "paged_decode.cuh"
#include "paged_decode_tc.cuh"
#include "paged_decode_tc2.cuh"
#include "pkv_internal.h"

namespace pkv {

static_assert(kTcMaxPages == kTcUnitMaxPages, "the tcgen05 unit's page table");
static_assert(kT2Threads == 32 * kTcPairWarps, "the tile-pair kernel's warps");

// Kernel tables of the instantiation units.
const void* decode_kernel_bf16_d64(int bs, int math, int gt);
const void* decode_kernel_bf16_d128(int bs, int math, int gt);
const void* decode_kernel_fp8_d128(int bs, int math, int gt);
const void* decode_kernel_int8_d128(int bs, int math, int gt);
const void* decode_kernel_mt_bf16(int D, int bs, int gt);
const void* decode_kernel_mt_1byte(int kv_dtype, int bs, int gt);
const void* decode_kernel_tc(int bs, bool rot, int kv_dtype);
const void* decode_kernel_tc2(int bs);

// ---------------------------------------------------------------------------
// planner: one CTA validates context lengths, counts each sequence's
// partitions, prefix-sums them into unit_start, resets the work queue and
// the split-K arrival counters, and writes zeros for sequences that attend
// to nothing.
// ---------------------------------------------------------------------------
constexpr int kPlanThreads = 1024;

// Sequences of at most this many partitions are merged inside the decode
// kernel by the warp that finishes last; longer ones by merge_kernel (the
// in-kernel merge is serial per (sequence, KV head) and lands in the tail).
constexpr int kFusedMergeMaxParts = 4;

// KV >= 0: CTAs 1.. of the same launch first run a KV append of that kind
// (pkv_kv_dtype), so that a decode step's append and plan cost one launch.
template <int KV>
__global__ void __launch_bounds__(kPlanThreads)
    plan_kernel(const int32_t* __restrict__ context_lens, int B, int num_arrive /* B * Hkv * NT */,
                int max_ctx, int tokens_per_part, int half_from /* sequences from here: */,
                int tokens_per_part_half /* partitions of this many tokens */, int32_t* work_counter, int32_t* unit_start,
                int32_t* ctx_eff, int32_t* part_seq, int32_t* arrive, __nv_bfloat16* out,
                int row_elems /* T * Hq * D */, unsigned* err, const AppendArgs app) {
  __shared__ int warp_tot[kPlanThreads / 32];
  __shared__ int carry_s;
  pdl_trigger();
  pdl_wait();
  if constexpr (KV >= 0) {
    if (blockIdx.x > 0) {  // block-uniform: these CTAs never reach the planner's barriers
      append_chunks<KV>(app, (blockIdx.x - 1) * static_cast<int64_t>(blockDim.x) + threadIdx.x,
                        static_cast<int64_t>(gridDim.x - 1) * blockDim.x);
      return;
    }
  }
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
      const int tpp = b >= half_from ? tokens_per_part_half : tokens_per_part;
      parts = (c + tpp - 1) / tpp;
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
  for (int i = tid; i < num_arrive; i += kPlanThreads) arrive[i] = 0;
  if (__syncthreads_or(bad_any) && tid == 0) atomicOr(err, PKV_DEVERR_CONTEXT_LEN);
  // the sequence of every global partition (one warp per sequence), so that
  // a decode unit finds its sequence with one load
  for (int b = warp; b < B; b += kPlanThreads / 32)
    for (int q = unit_start[b] + lane; q < unit_start[b + 1]; q += 32) part_seq[q] = b;
  // zeros for inactive sequences (one warp per sequence)
  for (int b = warp; b < B; b += kPlanThreads / 32) {
    if (ctx_eff[b] != 0) continue;
    uint4* o = reinterpret_cast<uint4*>(out + static_cast<size_t>(b) * row_elems);
    for (int i = lane; i < row_elems / 8; i += 32) o[i] = make_uint4(0, 0, 0, 0);
  }
}

// ---------------------------------------------------------------------------
// merge kernel (many partitions): one CTA per (sequence, query token, query
// head) row, in two phases so that no load waits on another:
//   1. M = max_p m_p over the row's partitions (all threads, strided);
//   2. thread (pg, dg) owns 4 columns of head_dim and partitions pg, pg + kPG,
//      ...; with M known every weight 2^(m_p - M) is final, so its loads are
//      independent and are issued four partitions at a time;
// then the kPG partial sums are added through shared memory:
//   out = sum_p 2^(m_p - M) O_p / sum_p 2^(m_p - M) l_p.
// Empty partitions (m = -inf) have weight 0; a row whose partitions are all
// empty gets zeros.
// ---------------------------------------------------------------------------
constexpr int kMergeThreads = 256;

template <int D>
__global__ void __launch_bounds__(kMergeThreads)
    merge_kernel(const float* __restrict__ part_ml, const float* __restrict__ part_o,
                 const int32_t* __restrict__ unit_start, int rows_per_seq /* T * Hq */,
                 int pmax, int row0, __nv_bfloat16* __restrict__ out) {
  constexpr int kDG = D / 4;                  // threads along head_dim
  constexpr int kPG = kMergeThreads / kDG;    // partition groups
  constexpr int kBatch = 4;                   // partitions in flight per thread
  __shared__ float4 s_acc[kPG][kDG];
  __shared__ float s_l[kPG][kDG];
  __shared__ float s_max[kMergeThreads / 32];
  pdl_trigger();
  pdl_wait();
  const int bh = row0 + blockIdx.x;  // row (b * T + t) * Hq + h
  const int b = bh / rows_per_seq;
  const int P = unit_start[b + 1] - unit_start[b];
  if (P < 2) return;  // written by the decode kernel (or zero-filled by the planner)
  const int tid = threadIdx.x;
  const size_t base = static_cast<size_t>(bh) * pmax;
  const float2* ml = reinterpret_cast<const float2*>(part_ml) + base;

  // 1. row maximum
  float M = -INFINITY;
  for (int i = tid; i < P; i += kMergeThreads) M = fmaxf(M, ml[i].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
  if ((tid & 31) == 0) s_max[tid >> 5] = M;
  __syncthreads();
  M = s_max[0];
#pragma unroll
  for (int w = 1; w < kMergeThreads / 32; ++w) M = fmaxf(M, s_max[w]);

  // 2. weighted sums, four independent partitions at a time
  const int dg = tid % kDG, pg = tid / kDG;
  float L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -INFINITY) {
    const float* ob = part_o + base * D + 4 * dg;
    for (int i0 = pg; i0 < P; i0 += kPG * kBatch) {
      float2 m[kBatch];
      float4 v[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int i = i0 + k * kPG;
        if (i < P) {
          m[k] = ml[i];
          v[k] = *reinterpret_cast<const float4*>(ob + static_cast<size_t>(i) * D);
        } else {
          m[k] = make_float2(-INFINITY, 0.f);
          v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const float w = exp2f(m[k].x - M);  // 0 for an empty partition or a missing one
        L = fmaf(w, m[k].y, L);
        acc.x = fmaf(w, v[k].x, acc.x);
        acc.y = fmaf(w, v[k].y, acc.y);
        acc.z = fmaf(w, v[k].z, acc.z);
        acc.w = fmaf(w, v[k].w, acc.w);
      }
    }
  }
  s_acc[pg][dg] = acc;
  s_l[pg][dg] = L;
  __syncthreads();
  if (pg != 0) return;
#pragma unroll
  for (int g = 1; g < kPG; ++g) {
    const float4 a = s_acc[g][dg];
    acc.x += a.x;
    acc.y += a.y;
    acc.z += a.z;
    acc.w += a.w;
    L += s_l[g][dg];
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  __nv_bfloat16* o = out + static_cast<size_t>(bh) * D + 4 * dg;
  *reinterpret_cast<__nv_bfloat162*>(o) = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  *reinterpret_cast<__nv_bfloat162*>(o + 2) = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
}

// ---------------------------------------------------------------------------
// merge for rows of at most 32 partitions: one warp per row, 2 rows per CTA.
// Lane p loads partition p's (m, l); the warp reduces M and L; then every
// lane loads its D/32 columns of all partitions at once (independent loads)
// and weights them with 2^(m_p - M) taken from lane p.
// ---------------------------------------------------------------------------
constexpr int kMergeRowsPerCta = 2;
constexpr int kMergeWarpMaxParts = 32;

template <int D>
__global__ void __launch_bounds__(kMergeRowsPerCta * 32)
    merge_rows_kernel(const float* __restrict__ part_ml, const float* __restrict__ part_o,
                      const int32_t* __restrict__ unit_start, int rows_per_seq /* T * Hq */,
                      int pmax, int row0, int num_rows, __nv_bfloat16* __restrict__ out) {
  constexpr int kPer = D / 32;  // columns per lane
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int row = row0 + blockIdx.x * kMergeRowsPerCta + (threadIdx.x >> 5);  // (b * T + t) * Hq + h
  if (row >= num_rows) return;
  const int b = row / rows_per_seq;
  const int P = unit_start[b + 1] - unit_start[b];
  if (P < 2) return;  // written by the decode kernel (or zero-filled by the planner)
  const size_t base = static_cast<size_t>(row) * pmax;
  const float2 mine = lane < P ? reinterpret_cast<const float2*>(part_ml)[base + lane]
                               : make_float2(-INFINITY, 0.f);
  float M = mine.x;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
  const float w = (M == -INFINITY) ? 0.f : exp2f(mine.x - M);  // 0 past P and for empty partitions
  float L = w * mine.y;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(kFull, L, o);
  float acc[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) acc[j] = 0.f;
  const float* ob = part_o + base * D + lane * kPer;
#pragma unroll 16
  for (int p = 0; p < P; ++p) {
    const float wp = __shfl_sync(kFull, w, p);
    if constexpr (kPer == 4) {
      const float4 v = *reinterpret_cast<const float4*>(ob + static_cast<size_t>(p) * D);
      acc[0] = fmaf(wp, v.x, acc[0]);
      acc[1] = fmaf(wp, v.y, acc[1]);
      acc[2] = fmaf(wp, v.z, acc[2]);
      acc[3] = fmaf(wp, v.w, acc[3]);
    } else {
      const float2 v = *reinterpret_cast<const float2*>(ob + static_cast<size_t>(p) * D);
      acc[0] = fmaf(wp, v.x, acc[0]);
      acc[1] = fmaf(wp, v.y, acc[1]);
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  __nv_bfloat16* o = out + static_cast<size_t>(row) * D + lane * kPer;
#pragma unroll
  for (int j = 0; j < kPer; j += 2)
    *reinterpret_cast<__nv_bfloat162*>(o + j) = __floats2bfloat162_rn(acc[j] * inv, acc[j + 1] * inv);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

WorkspaceLayout workspace_layout(int B, int T, int Hq, int Hkv, int NT, int D, int pmax) {
  WorkspaceLayout w{};
  size_t off = 0;
  w.counter = off;
  off += 256;
  w.unit_start = off;
  off = align_up(off + sizeof(int32_t) * (static_cast<size_t>(B) + 1), 256);
  w.ctx_eff = off;
  off = align_up(off + sizeof(int32_t) * static_cast<size_t>(B), 256);
  w.part_seq = off;
  off = align_up(off + sizeof(int32_t) * static_cast<size_t>(B) * pmax, 256);
  w.arrive = off;
  off = align_up(off + sizeof(int32_t) * static_cast<size_t>(B) * Hkv * NT, 256);
  const size_t parts = pmax > 1 ? static_cast<size_t>(B) * T * Hq * pmax : 0;
  w.part_ml = off;
  off = align_up(off + sizeof(float) * 2 * parts, 256);
  w.part_o = off;
  off = align_up(off + sizeof(float) * D * parts, 256);
  w.total = off;
  return w;
}

size_t decode_smem_bytes(int kv_fp8, int D, int bs, int warps, int stages, int tc, int tc2) {
  if (tc2) return tc2_smem_layout_bytes();
  if (tc) return tc_smem_layout_bytes(kv_fp8 != 0);
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

// gt: query rows per tile; mt: multi-token kernel (T > 1); tc2: the
// tcgen05 kernel for pairs of row tiles.
static const void* pick_kernel(int kv_dtype, int D, int bs, int math, int gt, bool mt, bool tc2 = false) {
  if (math == PKV_MATH_TC && tc2) return (kv_dtype == PKV_KV_BF16 && D == 128) ? decode_kernel_tc2(bs) : nullptr;
  if (math == PKV_MATH_TC) return D == 128 ? decode_kernel_tc(bs, gt <= kTcRotMaxRows, kv_dtype) : nullptr;
  if (mt) {
    if (math != PKV_MATH_MMA) return nullptr;
    return kv_dtype == PKV_KV_BF16 ? decode_kernel_mt_bf16(D, bs, gt) : decode_kernel_mt_1byte(kv_dtype, bs, gt);
  }
  if (kv_dtype == PKV_KV_INT8) return decode_kernel_int8_d128(bs, math, gt);
  if (kv_dtype == PKV_KV_FP8_E4M3) return decode_kernel_fp8_d128(bs, math, gt);
  if (D == 64) return decode_kernel_bf16_d64(bs, math, gt);
  return decode_kernel_bf16_d128(bs, math, gt);
}

bool pdl_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("PKV_PDL");
    return v == nullptr || std::strcmp(v, "0") != 0;
  }();
  return on;
}

// CTAs of the decode kernel that fit on one SM, per (device, kernel, shape);
// also raises the kernel's dynamic shared memory limit the first time.
static cudaError_t ctas_per_sm(const void* fn, int threads, size_t smem, int* out) {
  struct Entry {
    int dev;
    void* ctx;  // the kernel attribute set below belongs to this context
    const void* fn;
    int threads;
    size_t smem;
    int n;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  void* ctx = current_context();
  {
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry& x : cache)
      if (x.dev == dev && x.ctx == ctx && ctx != nullptr && x.fn == fn && x.threads == threads && x.smem == smem) {
        *out = x.n;
        return cudaSuccess;
      }
  }
  // Raise the kernel's limit to the device's opt-in maximum (not to this
  // request), so a cached entry never leaves a smaller limit behind.
  int optin = 0;
  e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  if (smem > static_cast<size_t>(optin)) return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  if (e != cudaSuccess) return e;
  int n = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  cache.push_back(Entry{dev, current_context(), fn, threads, smem, n});
  *out = n;
  return cudaSuccess;
}

int decode_ctas_per_sm(const DecodeLaunch& L, size_t smem) {
  const void* fn = pick_kernel(L.kv_dtype, L.D, L.bs, L.math, L.G * L.Tt, L.T > 1, L.tc2 != 0);
  int n = 0;
  if (fn == nullptr || ctas_per_sm(fn, L.warps * 32, smem, &n) != cudaSuccess) return 0;
  return n;
}

cudaError_t launch_decode(const DecodeLaunch& L, int* launched) {
  *launched = 0;
  const void* fn = pick_kernel(L.kv_dtype, L.D, L.bs, L.math, L.G * L.Tt, L.T > 1, L.tc2 != 0);
  if (fn == nullptr) return cudaErrorInvalidDeviceFunction;
  const size_t smem = decode_smem_bytes(L.kv_fp8, L.D, L.bs, L.warps, L.stages, L.tc, L.tc2);
  int per_sm = 0;
  cudaError_t e = ctas_per_sm(fn, L.warps * 32, smem, &per_sm);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;

  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;

  // 1. planner (with the step's KV append on extra CTAs when one is given)
  {
    cudaLaunchConfig_t cfg{};
    long long append_blocks = 0;
    if (L.append != nullptr) {
      const long long total = 2LL * L.append->N * L.append->Hkv * (L.append->D / 8);
      append_blocks = std::min<long long>((total + kPlanThreads - 1) / kPlanThreads, 1 << 16);
    }
    cfg.gridDim = dim3(static_cast<unsigned>(1 + append_blocks));
    cfg.blockDim = dim3(kPlanThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = L.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const AppendArgs none{};
    const AppendArgs& app = L.append != nullptr ? *L.append : none;
    auto plan = L.append == nullptr                ? plan_kernel<-1>
                : L.append_kind == PKV_KV_INT8      ? plan_kernel<PKV_KV_INT8>
                : L.append_kind == PKV_KV_FP8_E4M3  ? plan_kernel<PKV_KV_FP8_E4M3>
                                                    : plan_kernel<PKV_KV_BF16>;
    e = cudaLaunchKernelEx(&cfg, plan, L.context_lens, L.B, L.B * L.Hkv * L.NT, L.MB * L.bs,
                           L.ppu * L.bs, L.half_from, L.ppu_half * L.bs, L.work_counter, L.unit_start, L.ctx_eff, L.part_seq, L.arrive,
                           static_cast<__nv_bfloat16*>(L.out), L.T * L.Hq * L.D, L.err, app);
    if (e != cudaSuccess) return e;
    *launched += 1;
  }

  // 2. decode: persistent grid, at most one warp per possible unit
  // (the tile-pair kernel: one unit per pair of row tiles)
  const long long max_units =
      static_cast<long long>(L.B) * L.Hkv * (L.tc2 ? (L.NT + 1) / 2 : L.NT) * L.pmax;
  // The tcgen05 kernel holds 256 of an SM's 512 TMEM columns: two CTAs per SM
  // (the occupancy query does not see the tensor memory and may say one);
  // the tile-pair kernel holds all 512: one CTA per SM.
  if (L.tc) per_sm = L.tc2 ? 1 : 2;
  long long grid = static_cast<long long>(L.num_sms) * per_sm;
  // a warp of the mma.sync kernels, a CTA of the tcgen05 kernel, per unit
  grid = std::min(grid, L.tc ? max_units : (max_units + L.warps - 1) / L.warps);
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
  p.part_seq = L.part_seq;
  p.part_ml = L.part_ml;
  p.part_o = L.part_o;
  p.arrive = L.arrive;
  p.err = L.err;
  p.B = L.B;
  p.Hq = L.Hq;
  p.Hkv = L.Hkv;
  p.G = L.G;
  p.T = L.T;
  p.Tt = L.Tt;
  p.NT = L.NT;
  p.MB = L.MB;
  p.NB = L.NB;
  p.pmax = L.pmax;
  p.ppu = L.ppu;
  p.half_from = L.half_from;
  p.ppu_half = L.ppu_half;
  p.stages = L.stages;
  // the tcgen05 kernel leaves every split-K merge to the merge kernels
  p.fused_merge = (!L.tc && L.pmax <= kFusedMergeMaxParts) ? 1 : 0;
  p.row_base = L.row_base;
  p.scale_log2 = L.scale_log2;
  CUtensorMap kmap = L.kmap, vmap = L.vmap, pmap = L.pmap, omap = L.omap, qmap = L.qmap;
  void* args_mma[] = {&kmap, &vmap, &p};
  void* args_tc[] = {&kmap, &vmap, &pmap, &omap, &p};  // + the partial and output store maps
  void* args_tc2[] = {&kmap, &vmap, &qmap, &p};        // + the query load map
  void** args = L.tc2 ? args_tc2 : L.tc ? args_tc : args_mma;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(L.warps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = L.stream;
  // An event recorded between the planner and the decode would sit between
  // them on the stream; launch without the overlap attribute then.
  cfg.attrs = attr;
  cfg.numAttrs = (L.ev_start == nullptr) ? 1 : 0;
  if (L.ev_start != nullptr && (e = cudaEventRecord(L.ev_start, L.stream)) != cudaSuccess) return e;
  e = cudaLaunchKernelExC(&cfg, fn, args);
  if (e != cudaSuccess) return e;
  if (L.ev_end != nullptr && (e = cudaEventRecord(L.ev_end, L.stream)) != cudaSuccess) return e;
  *launched += 1;

  // 3. merge kernel when sequences may span many partitions: a warp per row
  //    up to 32 partitions, a CTA per row beyond
  if (!p.fused_merge && L.pmax > 1) {
    const int rows = L.B * L.T * L.Hq;
    // with one partition of ppu >= MB blocks per sequence, only the
    // half-length sequences (half_from ..) have partials: merge their rows
    const int row0 = (L.ppu >= L.MB && L.half_from < L.B) ? L.half_from * L.T * L.Hq : 0;
    const int merge_rows = rows - row0;
    const bool by_warp = L.pmax <= kMergeWarpMaxParts;
    cudaLaunchConfig_t mc{};
    mc.gridDim =
        dim3(static_cast<unsigned>(by_warp ? (merge_rows + kMergeRowsPerCta - 1) / kMergeRowsPerCta : merge_rows));
    mc.blockDim = dim3(by_warp ? kMergeRowsPerCta * 32 : kMergeThreads);
    mc.dynamicSmemBytes = 0;
    mc.stream = L.stream;
    mc.attrs = attr;
    mc.numAttrs = (L.ev_end == nullptr) ? 1 : 0;
    const float* pml = static_cast<const float*>(L.part_ml);
    const float* po = static_cast<const float*>(L.part_o);
    const int32_t* us = static_cast<const int32_t*>(L.unit_start);
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(L.out);
    const int rps = L.T * L.Hq;
    if (by_warp)
      e = L.D == 64 ? cudaLaunchKernelEx(&mc, merge_rows_kernel<64>, pml, po, us, rps, L.pmax, row0, rows, o)
                    : cudaLaunchKernelEx(&mc, merge_rows_kernel<128>, pml, po, us, rps, L.pmax, row0, rows, o);
    else
      e = L.D == 64 ? cudaLaunchKernelEx(&mc, merge_kernel<64>, pml, po, us, rps, L.pmax, row0, o)
                    : cudaLaunchKernelEx(&mc, merge_kernel<128>, pml, po, us, rps, L.pmax, row0, o);
    if (e != cudaSuccess) return e;
    *launched += 1;
  }
  return cudaSuccess;
}

}  // namespace pkv
