// Multi-token decode on the 5th-generation tensor cores (tcgen05 + TMEM),
// bf16 cache, head_dim 128.
//
// A query of T new tokens per sequence has T x G (query token, head) rows per
// KV head ("KV-Cache Engineering: Paged Attention, Prefix Cache,
// Disaggregation (2026)": speculative decoding scores the draft's T tokens in
// one pass over the shared cache; "KV Cache Engineering: PagedAttention,
// Continuous Batching, Attention Variants, and the Bandwidth Wall",
// "Continuous Batching": chunked prefill).  With more than 16 rows the page
// work is a real matrix product, so here one CTA takes a tile of 128 rows
// (M of the MMA) and steps through its pages 64 tokens at a time (a
// tcgen05.mma of M 128 and K 16 costs the same up to N 128, so S = Q . K^T
// wants wide steps):
//
//   * Warp-specialised, with no CTA-wide barrier between units: a K copy
//     warp takes units from the planner's counter, writes each unit's
//     descriptor and page ids (one-byte caches: and the pages' scales and
//     zero points) into a 2-slot ring, and issues the tensor-map
//     copies (TMA, 128-byte swizzle) of each step's K pages into a 4-stage
//     ring; a V copy warp fills a 2-stage V ring; an MMA warp issues
//     S = Q . K^T (M 128, N 64, K 128; the query tile is the A operand in
//     TMEM) one step ahead of the softmax and O += P . V (M 128, N 128,
//     K 64; V read MN-major straight from the page) when the compute warps
//     have P ready; four compute warps own the 128 rows.  The roles hand work
//     over only through mbarriers, so copies, products and softmax of
//     neighbouring steps and units overlap.
//   * Each compute thread owns one row of the tile (thread r row r in full
//     tiles; see partial tiles below): it loads its 64 scores from TMEM (and
//     tells the MMA warp that the S slot is free), masks them (sequence end,
//     bad pages, the causal limit of its query token), and keeps the online
//     softmax state in registers.  The running maximum is lazy: the output is
//     rescaled only when a row's maximum grows by more than 2^8, so P stays
//     below 256 and the rescale of O in TMEM is rare; it runs after the
//     step's P is written, when the scores no longer hold registers.  P goes as bf16 (K-major, no swizzle)
//     into the step's K stage, which is dead once S is done.  V rows of
//     tokens outside the sequence (or of a bad page) are cleared in the stage,
//     as P is 0 there but the stale rows may hold NaN.
//   * When a unit's last S is done, the compute warps put the next unit's
//     query rows into TMEM; at the end of the unit each thread reads its row
//     of O and writes the bf16 output or the split-K partials (m, l, O) of
//     the merge kernels.
//   * Tiles with at most 96 query rows (kRot) place their rows in the
//     highest TMEM lanes: thread tid owns tile row (tid - rot) mod 128 with
//     rot = 128 - (rows rounded up to 32).  A warp all of whose rows are
//     empty then skips the scores, the softmax and P (its rows of P and O are
//     never stored): at T x G = 32, say, only warp 3 works, and warp 0, which
//     shares its sub-partition with the MMA warp, stays idle.
//
// One-byte caches (E4M3, INT8) take the same path ("KV Cache Engineering:
// PagedAttention, Continuous Batching, Attention Variants, and the
// Bandwidth Wall", "Quantized KV Cache": dequantise on read).  The copy
// warps land a step's codes in the upper half of a stage.  V pages, and
// INT8 K pages, are rewritten there by a converter warp as f16 code values
// (E4M3 value; INT8 code - zero for V, 1152 + code for K), which are exact
// in f16, and feed kind::f16 products; E4M3 K pages are an operand of the
// tensor cores as they are (kind::f8f6f4), against a query tile held as two
// E4M3 parts (high and residual) whose sum is the scaled query.  The page
// scales are applied where they cost nothing per element of the cache: a
// row's scores of page q are S' x c x k_scale[q] (one multiply per score,
// folded into the softmax; INT8 adds the bias and zero-point term), and P
// carries v_scale[q] / v_max (v_max: the unit's largest |v_scale|, so P
// stays below 256), the output v_max.  The query rows are scaled by a power
// of two per row, which the row's softmax coefficient takes back.  With one
// page, P = 1 and the output is bf16(code value x scale) exactly as the
// widened value.
//
// Units are (sequence, KV head, row tile, partition) from the planner's
// counter; the merge kernel combines partitions.  Every wait is bounded; a
// CTA that gives up records PKV_DEVERR_TIMEOUT, lets the copies and products
// it issued finish (bounded) and frees its tensor memory.
#pragma once

#include "paged_decode.cuh"

namespace pkv {

constexpr int kTcRows = 128;        // query rows per tile (MMA M)
constexpr int kTcTokens = 64;       // tokens per step (N of S)
constexpr int kTcKStages = 4;       // K ring; a stage holds K(g), then P(g)
constexpr int kTcVStages = 2;       // V ring
constexpr int kTcMaxPages = 256;    // pages of a unit (the planner's partition length for this kernel)
constexpr int kTcComputeWarps = 4;  // one row of the tile per thread
constexpr int kTcThreads = 32 * (kTcComputeWarps + 3);  // + MMA warp + K copy warp + V copy warp
// one-byte caches add a converter warp (two CTAs of 8 warps x 128 registers
// fill an SM's register file)
constexpr int kTcThreads1B = kTcThreads + 32;
__host__ __device__ constexpr int tc_threads(int kv) { return kv == PKV_KV_BF16 ? kTcThreads : kTcThreads1B; }
constexpr uint32_t kTcCols = 256;   // TMEM columns: S at 0, Q at 64, O at 128
constexpr uint32_t kTcSCol = 0;     // S(g): 64 fp32 columns
constexpr uint32_t kTcQCol = 64;    // query tile: 128 d as 64 columns of bf16 pairs
constexpr uint32_t kTcOCol = 128;   // O: 128 fp32 columns
constexpr int kTcRotMaxRows = 96;   // tiles of at most this many rows use the rotated-row instance

struct TcLayout {  // byte offsets from the 1024-aligned shared-memory base
  static constexpr uint32_t kRegion = kTcTokens * 128;       // half (64 of 128 d) of a step's tile: 8 KiB
  static constexpr uint32_t kTile = 2 * kRegion;             // a step's K (or P) or V tile: 16 KiB
  static constexpr uint32_t kK = 0;                          // K ring
  static constexpr uint32_t kV = kK + kTcKStages * kTile;    // V ring
  static constexpr uint32_t kBars = kV + kTcVStages * kTile;
  // full_k[4], kp_free[4], full_v[2], v_free[2], s_done, s_free, p_ready[4],
  // q_ready, slot_full[2], slot_free[2], stg_full, stg_free, o_ready,
  // mma_drain, then for one-byte caches tma_k[4], tma_v[2] (codes landed)
  static constexpr int kNumBars = 3 * kTcKStages + 2 * kTcVStages + 3 + 4 + 4 + kTcKStages + kTcVStages;
  static constexpr uint32_t kMisc = kBars + 8 * kNumBars;    // TMEM base
  static constexpr uint32_t kSlots = kMisc + 16;             // 2 unit slots
  static constexpr uint32_t kSlotPages = 32;                 // after 8 int32 of descriptor
  static constexpr uint32_t kSlotBad = kSlotPages + 4 * kTcMaxPages;
  static constexpr uint32_t kSlot = kSlotBad + kTcMaxPages;  // 1312 bytes
  static constexpr uint32_t kEnd = kSlots + 2 * kSlot;
  // one-byte caches: each slot's page parameters (k scale, k zero, v scale,
  // v zero) as a float4 per page, read by the compute and converter warps
  static constexpr uint32_t kPar = (kEnd + 15) & ~15u;
  static constexpr uint32_t kParSlot = 16 * kTcMaxPages;  // 4 KiB
  static constexpr uint32_t kEnd1B = kPar + 2 * kParSlot;
};

__host__ __device__ constexpr size_t tc_smem_layout_bytes(bool one_byte) {
  return 1024 + (one_byte ? TcLayout::kEnd1B : TcLayout::kEnd);
}

// K-major, no-swizzle core-matrix layout of a [128 rows x 64 tokens] bf16 P
// tile: core matrix (r/8, k/8) of 8 rows x 16 bytes at (r/8) * 1024 + (k/8) * 128.
__device__ __forceinline__ uint32_t tc_p_off(int r, int k8) {
  return static_cast<uint32_t>((r >> 3) * 1024 + k8 * 128 + (r & 7) * 16);
}

// Three-input maximum and minimum (one instruction each on sm_103a).
__device__ __forceinline__ float fmax3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float fmin3f(float a, float b, float c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Maximum (kMax) or minimum of 64 scores (bit patterns of floats) as a tree
// of three-input operations: 32 instructions, depth 5.
template <bool kMax>
__device__ __forceinline__ float tree_ext64(const uint32_t (&v)[kTcTokens]) {
  auto op3 = [](float a, float b, float c) { return kMax ? fmax3f(a, b, c) : fmin3f(a, b, c); };
  float t[22];
#pragma unroll
  for (int i = 0; i < 21; ++i)
    t[i] = op3(__uint_as_float(v[3 * i]), __uint_as_float(v[3 * i + 1]), __uint_as_float(v[3 * i + 2]));
  t[21] = __uint_as_float(v[63]);
#pragma unroll
  for (int i = 0; i < 7; ++i) t[i] = op3(t[3 * i], t[3 * i + 1], t[3 * i + 2]);  // 22 -> 8
  t[7] = t[21];
  const float u0 = op3(t[0], t[1], t[2]), u1 = op3(t[3], t[4], t[5]);  // 8 -> 4
  const float w = op3(u0, u1, t[6]);
  return kMax ? fmaxf(w, t[7]) : fminf(w, t[7]);
}

// A unit as the descriptor slot holds it.
struct TcUnit {
  int u, b, pidx, nparts, ctx, kvh, tile, t0, t1, npages, nsteps;
};

// Widen 16 one-byte codes (a 16-byte chunk, element i in byte i) to their
// f16 code values (E4M3 value, INT8 code - zero; both exact in f16) as two
// 16-byte chunks.
// kBiased (INT8 K pages): 1152 + code instead, two instructions fewer per
// four codes; the compute warps take (1152 + zero) x sum(q) off the scores.
template <int KV, bool kBiased = false>
__device__ __forceinline__ void widen16(const uint4 c, uint32_t zc, uint4& o0, uint4& o1) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
  uint32_t r[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if constexpr (KV == PKV_KV_INT8 && kBiased)
      int8x4_to_f16x2x2_biased(w[q], r[2 * q], r[2 * q + 1]);
    else if constexpr (KV == PKV_KV_INT8)
      int8x4_to_f16x2x2(w[q], zc, r[2 * q], r[2 * q + 1]);
    else
      e4m3x4_to_f16x2x2(w[q], r[2 * q], r[2 * q + 1]);
  }
  o0 = make_uint4(r[0], r[1], r[2], r[3]);
  o1 = make_uint4(r[4], r[5], r[6], r[7]);
}

// Rewrite a stage of `rows` token rows (64-d halves kRegion apart, 128-byte
// rows, 16-byte chunks XOR-swizzled by row % 8) whose one-byte codes a
// tensor-map copy put in the upper half (row r's 128 codes at
// kRegion + 128 r) as f16 code values; the caller gives row r's INT8 zero
// constant.  One warp; lane l takes rows l, l + 32, ...: all of a row's
// codes are read before any of its 16 widened chunks is written (a row's
// codes occupy only the bytes of its own upper half), so the eight loads
// issue back to back.
template <int KV, int ROWS, bool kBiased = false>
__device__ __forceinline__ void widen_stage(uint8_t* stage, uint32_t region, int lane, const uint32_t (&zc)[ROWS / 32],
                                            int valid_rows) {
#pragma unroll
  for (int rr = 0; rr < ROWS / 32; ++rr) {
    const int r = lane + 32 * rr;
    if (r >= valid_rows) continue;
    const int sw = r & 7;
    uint8_t* hi = stage + region + r * 128;  // codes; then d 64 .. 127
    uint8_t* lo = stage + r * 128;           // d 0 .. 63
    uint4 codes[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) codes[c] = *reinterpret_cast<const uint4*>(hi + ((c ^ sw) << 4));
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint4 o0, o1;
      widen16<KV, kBiased>(codes[c], zc[rr], o0, o1);
      uint8_t* dst = c < 4 ? lo : hi;
      *reinterpret_cast<uint4*>(dst + (((2 * (c & 3)) ^ sw) << 4)) = o0;
      *reinterpret_cast<uint4*>(dst + (((2 * (c & 3) + 1) ^ sw) << 4)) = o1;
    }
  }
}

template <int BS, bool kRot, int KV = PKV_KV_BF16>
// Two CTAs per SM: a sub-partition's 16384 registers hold four of the 14
// (16 with a converter warp) warps at 128 registers a thread.
__global__ void __launch_bounds__(tc_threads(KV), 2)
    paged_decode_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                           const __grid_constant__ CUtensorMap vmap,
                           const __grid_constant__ CUtensorMap pmap,  // split-K partials (pmax > 1)
                           const __grid_constant__ CUtensorMap omap,  // bf16 output
                           const DecodeParams p) {
  constexpr int D = 128;
  constexpr int PPI = kTcTokens / BS;  // pages per step
  constexpr bool kOneByte = KV != PKV_KV_BF16;
  // E4M3 K pages are an operand of the tensor cores as they are (kind::f8f6f4)
  constexpr bool kF8K = KV == PKV_KV_FP8_E4M3;
  static_assert(kTcMaxPages % PPI == 0, "");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  // Barrier phases are counted over the CTA's lifetime: by the global step
  // index g (K stage and full_k[] / kp_free[] / p_ready[] by g % 4, V stage
  // and full_v[] / v_free[] by g % 2, s_done / s_free once per step) or by
  // the unit index i (slot_full[] / slot_free[] by i % 2, q_ready and o_ready
  // once per unit) or by the output chunks (stg_full once per chunk, stg_free
  // twice per split-K unit).
  // Every barrier completes one phase per use, and a waiter is never two
  // phases away from the phase it waits for (a parity wait cannot tell them
  // apart): each next use of a barrier depends on the wait.  p_ready has one
  // barrier per K stage for this reason: its next use, step g + 4, needs
  // K(g + 4) in the stage, i.e. P . V(g) done.
  uint64_t* full_k = reinterpret_cast<uint64_t*>(sm + TcLayout::kBars);  // [4] K(g) landed
  uint64_t* kp_free = full_k + kTcKStages;    // [4] P . V(g) done: K stage (holding P(g)) free
  uint64_t* full_v = kp_free + kTcKStages;    // [2] V(g) landed
  uint64_t* v_free = full_v + kTcVStages;     // [2] P . V(g) done: V stage free, O quiescent
  uint64_t* s_done = v_free + kTcVStages;     // S(g) in TMEM
  uint64_t* s_free = s_done + 1;              // S(g) read by the compute warps
  uint64_t* p_ready = s_free + 1;             // [4] P(g) in shared memory (its K stage)
  uint64_t* q_ready = p_ready + kTcKStages;   // the unit's query tile in TMEM
  uint64_t* slot_full = q_ready + 1;          // [2] unit slot written
  uint64_t* slot_free = slot_full + 2;        // [2] unit slot released by every reader
  uint64_t* stg_full = slot_free + 2;         // a chunk of the unit's output staged by every compute warp
  uint64_t* stg_free = stg_full + 1;          // split-K partials: a store has read its staging buffer
  uint64_t* o_ready = stg_free + 1;           // a unit's last P . V done: O final, its K and V stages idle
  uint64_t* mma_drain = o_ready + 1;          // after a timeout: every product issued is done
  uint64_t* tma_k = mma_drain + 1;            // [4] one-byte caches: K(g)'s codes landed (then full_k: widened)
  uint64_t* tma_v = tma_k + kTcKStages;       // [2] one-byte caches: V(g)'s codes landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + TcLayout::kMisc);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const bool mma_warp = warp == kTcComputeWarps;
  const bool kcopy = warp == kTcComputeWarps + 1;
  const bool vcopy = warp == kTcComputeWarps + 2;
  const bool widen = kOneByte && warp == kTcComputeWarps + 3;  // converter warp (one-byte caches)

  if (tid == 0) {
    for (int s = 0; s < kTcKStages; ++s) {
      mbar_init(&full_k[s], 1);
      mbar_init(&kp_free[s], 1);
    }
    for (int s = 0; s < kTcVStages; ++s) {
      mbar_init(&full_v[s], 1);
      mbar_init(&v_free[s], 1);
    }
    mbar_init(s_done, 1);
    mbar_init(s_free, kTcComputeWarps);  // one lane per compute warp
    for (int s = 0; s < kTcKStages; ++s) mbar_init(&p_ready[s], 32 * kTcComputeWarps);
    mbar_init(q_ready, kTcComputeWarps);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&slot_full[s], 1);
      // compute warps, MMA warp, V copy warp (and the converter warp)
      mbar_init(&slot_free[s], kTcComputeWarps + 2 + (kOneByte ? 1 : 0));
    }
    if (kOneByte) {
      for (int s = 0; s < kTcKStages; ++s) mbar_init(&tma_k[s], 1);
      for (int s = 0; s < kTcVStages; ++s) mbar_init(&tma_v[s], 1);
    }
    mbar_init(stg_full, kTcComputeWarps);
    mbar_init(stg_free, 1);
    mbar_init(o_ready, 1);
    mbar_init(mma_drain, 1);
    fence_mbar_init();
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
    if (p.pmax > 1) prefetch_tensormap(&pmap);
    prefetch_tensormap(&omap);
  }
  if (warp == 0) tc_alloc(tmem_slot, kTcCols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_lane = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);  // compute warp's 32 lanes
  const uint64_t policy = p.NT > 1 ? l2_policy_evict_normal() : l2_policy_evict_first();
  // one-byte caches: f16 query, code values and P
  constexpr uint32_t kIdescS = kF8K       ? tc_idesc_e4m3_f32(kTcRows, kTcTokens)
                               : kOneByte ? tc_idesc_f16_f32(kTcRows, kTcTokens)
                                          : tc_idesc_bf16_f32(kTcRows, kTcTokens);
  constexpr uint32_t kIdescO = kOneByte ? tc_idesc_f16_f32(kTcRows, D, /*b_mn_major=*/true)
                                        : tc_idesc_bf16_f32(kTcRows, D, /*b_mn_major=*/true);
  pdl_trigger();
  pdl_wait();

  const int units_per_part = p.Hkv * p.NT;
  const int total_units = p.unit_start[p.B] * units_per_part;
  const int ppu_tokens = p.ppu * BS;
  bool timed_out = false;
  // end (global step) of this thread's own asynchronous work, for the drain
  // after a timeout: copies issued (copy warps), products committed (MMA warp)
  uint32_t copies_end = 0, s_end = 0, pv_end = 0;

  auto slot_desc = [&](int k) { return reinterpret_cast<volatile int*>(sm + TcLayout::kSlots + k * TcLayout::kSlot); };
  auto slot_pages = [&](int k) {
    return reinterpret_cast<const volatile int*>(sm + TcLayout::kSlots + k * TcLayout::kSlot + TcLayout::kSlotPages);
  };
  auto slot_bad = [&](int k) {
    return reinterpret_cast<const volatile uint8_t*>(sm + TcLayout::kSlots + k * TcLayout::kSlot + TcLayout::kSlotBad);
  };
  // one-byte caches: the slot's page parameters (k scale, k zero, v scale, v zero)
  auto slot_par = [&](int k) { return reinterpret_cast<float4*>(sm + TcLayout::kPar + k * TcLayout::kParSlot); };
  auto read_unit = [&](int k) {
    const volatile int* d = slot_desc(k);
    TcUnit U;
    U.u = d[0];
    U.b = d[1];
    U.pidx = d[2];
    U.nparts = d[3];
    U.ctx = d[4];
    const int part = U.u / units_per_part;
    const int rem = U.u - part * units_per_part;
    U.kvh = rem / p.NT;
    U.tile = rem - U.kvh * p.NT;
    U.t0 = U.pidx * ppu_tokens;
    U.t1 = min(U.ctx, U.t0 + ppu_tokens);
    U.npages = (U.t1 - U.t0 + BS - 1) / BS;  // 1 .. kTcMaxPages
    U.nsteps = (U.npages + PPI - 1) / PPI;
    return U;
  };
  // this warp waits (lane 0, bounded) for phase `parity` of `bar`; false on timeout
  auto warp_wait = [&](uint64_t* bar, uint32_t parity, bool suspend) {
    int ok = 1;
    if (lane == 0)
      ok = (suspend ? mbar_wait_bounded(bar, parity, kWaitLimitNs) : mbar_wait_spin(bar, parity, kWaitLimitNs)) ? 1 : 0;
    return __shfl_sync(kFull, ok, 0) != 0;
  };

  // One-byte caches: wait until step g's K (is_k) or V codes have landed,
  // widen them in the stage to f16 code values (INT8: with each row's page
  // zero point), publish with full_k / full_v.  Rows of pages past the unit's end are left as
  // they are (their scores are masked and their V rows cleared).  Whole
  // warp; false on timeout.
  auto widen_pages = [&](bool is_k, const TcUnit& U, const float4* par, int j, uint32_t g) -> bool {
    if constexpr (!kOneByte) {
      return true;
    } else {
      uint64_t* landed = is_k ? &tma_k[g % kTcKStages] : &tma_v[g % kTcVStages];
      const uint32_t parity = is_k ? (g / kTcKStages) & 1u : (g / kTcVStages) & 1u;
      if (!warp_wait(landed, parity, true)) return false;
      uint8_t* st = sm + (is_k ? TcLayout::kK + (g % kTcKStages) * TcLayout::kTile
                               : TcLayout::kV + (g % kTcVStages) * TcLayout::kTile);
      const int np = min(PPI, U.npages - j * PPI);
      uint32_t zc[2] = {0u, 0u};
      if constexpr (KV == PKV_KV_INT8) {
        if (is_k) {  // K: biased code values, no zero points
          widen_stage<KV, kTcTokens, true>(st, TcLayout::kRegion, lane, zc, np * BS);
        } else {
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const int q = (lane + 32 * rr) / BS;
            if (q < np) zc[rr] = int8_zero_const(par[j * PPI + q].w);
          }
          widen_stage<KV, kTcTokens>(st, TcLayout::kRegion, lane, zc, np * BS);
        }
      } else {
        widen_stage<KV, kTcTokens>(st, TcLayout::kRegion, lane, zc, np * BS);
      }
      fence_proxy_async_smem();  // the widened rows are read by the tensor cores
      __syncwarp();
      if (lane == 0) mbar_arrive(is_k ? &full_k[g % kTcKStages] : &full_v[g % kTcVStages]);
      return true;
    }
  };

  if (kcopy) {
    // Units: take the next unit from the counter once its slot is free, look
    // up its sequence, partition and pages, publish the slot.  Then the K
    // pages of its steps: K(g) into stage g % 4 once P . V(g - 4) is done;
    // lane 2q + h copies half h (64 of 128 d) of the step's page q.
    uint32_t g = 0;
    for (int i = 0;; ++i) {
      const int k = i & 1;
      if (i >= 2 && !warp_wait(&slot_free[k], ((i - 2) >> 1) & 1u, true)) {
        timed_out = true;
        break;
      }
      volatile int* d = slot_desc(k);
      int u = 0, b = 0, pidx = 0, ctx = 0;
      if (lane == 0) {
        u = atomicAdd(p.work_counter, 1);
        d[0] = u;
        if (u < total_units) {
          const int part = u / units_per_part;
          b = __ldg(p.part_seq + part);
          const int us = __ldg(p.unit_start + b);
          pidx = part - us;
          ctx = __ldg(p.ctx_eff + b);
          d[1] = b;
          d[2] = pidx;
          d[3] = __ldg(p.unit_start + b + 1) - us;
          d[4] = ctx;
        }
      }
      u = __shfl_sync(kFull, u, 0);
      int nsteps = 0, kvh = 0;
      if (u < total_units) {
        b = __shfl_sync(kFull, b, 0);
        pidx = __shfl_sync(kFull, pidx, 0);
        ctx = __shfl_sync(kFull, ctx, 0);
        const int rem = u - (u / units_per_part) * units_per_part;
        kvh = rem / p.NT;
        const int t0 = pidx * ppu_tokens;
        const int npages = (min(ctx, t0 + ppu_tokens) - t0 + BS - 1) / BS;  // 1 .. kTcMaxPages
        nsteps = (npages + PPI - 1) / PPI;
        const int* trow = p.block_tables + static_cast<size_t>(b) * p.MB + t0 / BS;
        volatile int* pg = reinterpret_cast<volatile int*>(sm + TcLayout::kSlots + k * TcLayout::kSlot + TcLayout::kSlotPages);
        volatile uint8_t* bd = sm + TcLayout::kSlots + k * TcLayout::kSlot + TcLayout::kSlotBad;
        float vmax = 0.f;
        for (int q = lane; q < npages; q += 32) {
          int e = __ldg(trow + q);
          const bool isbad = static_cast<unsigned>(e) >= static_cast<unsigned>(p.NB);
          if (isbad) {
            e = 0;
            atomicOr(p.err, PKV_DEVERR_BLOCK_ID);
          }
          pg[q] = e;
          bd[q] = isbad ? 1 : 0;
          if constexpr (kOneByte) {  // the page's parameters (0 for a bad page: its tokens are masked)
            float4 par = make_float4(0.f, 0.f, 0.f, 0.f);
            if (!isbad) {
              const size_t pi = static_cast<size_t>(e) * p.Hkv + kvh;
              if constexpr (KV == PKV_KV_INT8) {
                const float2 kp = __ldg(reinterpret_cast<const float2*>(p.k_scale) + pi);
                const float2 vp = __ldg(reinterpret_cast<const float2*>(p.v_scale) + pi);
                par = make_float4(kp.x, kp.y, vp.x, vp.y);
              } else {
                par = make_float4(__ldg(p.k_scale + pi), 0.f, __ldg(p.v_scale + pi), 0.f);
              }
              vmax = fmaxf(vmax, fabsf(par.z));
            }
            slot_par(k)[q] = par;
          }
        }
        if constexpr (kOneByte) {  // the unit's largest |v_scale| (1 if none): P carries v_scale / it
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(kFull, vmax, o));
          if (lane == 0) d[5] = __float_as_int(vmax > 0.f ? vmax : 1.f);
        }
        __threadfence_block();
        // the unit's query rows into L2, for the compute warps' TMEM fill
        const int tile = rem - kvh * p.NT;
        for (int r = lane; r < kTcRows; r += 32) {
          int t = 0, h = 0;
          if (tile_row<true>(p, kvh, tile, r, t, h)) {
            const __nv_bfloat16* qa = p.q + (static_cast<size_t>(b * p.T + t) * p.Hq + h) * D;
            asm volatile("prefetch.global.L2 [%0];" ::"l"(qa));
            asm volatile("prefetch.global.L2 [%0];" ::"l"(qa + 64));
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&slot_full[k]);  // release: the slot's writes by this warp
      if (u >= total_units) break;
      const volatile int* pages = slot_pages(k);
      const int npages_total = (min(ctx, pidx * ppu_tokens + ppu_tokens) - pidx * ppu_tokens + BS - 1) / BS;
      for (int j = 0; j < nsteps; ++j, ++g) {
        if (g >= kTcKStages && !warp_wait(&kp_free[g % kTcKStages], ((g - kTcKStages) / kTcKStages) & 1u, true)) {
          timed_out = true;
          break;
        }
        uint8_t* st = sm + TcLayout::kK + (g % kTcKStages) * TcLayout::kTile;
        uint64_t* bar = (kOneByte && !kF8K) ? &tma_k[g % kTcKStages] : &full_k[g % kTcKStages];
        const int np = min(PPI, npages_total - j * PPI);
        if (lane == 0) {
          fence_proxy_async_smem();  // the stage held P (generic writes) before
          mbar_arrive_expect_tx(bar, static_cast<uint32_t>(np) * (kOneByte ? 128u : 2u * 64u * 2u) * BS);
        }
        __syncwarp();
        if (kOneByte) {  // one box of 128 codes per page, into the upper half (the converter's input; E4M3: S's operand)
          if (lane < np) {
            const int row = p.row_base + (pages[j * PPI + lane] * p.Hkv + kvh) * BS;
            tma_load_2d(st + TcLayout::kRegion + lane * BS * 128, &kmap, bar, 0, row, policy);
          }
        } else if (lane < 2 * np) {
          const int q = lane >> 1, half = lane & 1;
          const int row = p.row_base + (pages[j * PPI + q] * p.Hkv + kvh) * BS;
          tma_load_2d(st + half * TcLayout::kRegion + q * BS * 128, &kmap, bar, half * 64, row, policy);
        }
        copies_end = g + 1;
      }
      if (timed_out) break;
    }
  } else if (vcopy) {
    // V(g) into stage g % 2 once P . V(g - 2) is done; releases each unit's
    // slot after its last copy.
    uint32_t g = 0;
    for (int i = 0;; ++i) {
      const int k = i & 1;
      if (!warp_wait(&slot_full[k], (i >> 1) & 1u, true)) {
        timed_out = true;
        break;
      }
      const TcUnit U = read_unit(k);
      if (U.u >= total_units) break;
      const volatile int* pages = slot_pages(k);
      for (int j = 0; j < U.nsteps; ++j, ++g) {
        if (g >= kTcVStages && !warp_wait(&v_free[g % kTcVStages], ((g - kTcVStages) / kTcVStages) & 1u, true)) {
          timed_out = true;
          break;
        }
        uint8_t* st = sm + TcLayout::kV + (g % kTcVStages) * TcLayout::kTile;
        uint64_t* bar = kOneByte ? &tma_v[g % kTcVStages] : &full_v[g % kTcVStages];
        const int np = min(PPI, U.npages - j * PPI);
        if (lane == 0) {
          fence_proxy_async_smem();  // after the compute warps' clearing of stale V rows
          mbar_arrive_expect_tx(bar, static_cast<uint32_t>(np) * (kOneByte ? 128u : 2u * 64u * 2u) * BS);
        }
        __syncwarp();
        if (kOneByte) {
          if (lane < np) {
            const int row = p.row_base + (pages[j * PPI + lane] * p.Hkv + U.kvh) * BS;
            tma_load_2d(st + TcLayout::kRegion + lane * BS * 128, &vmap, bar, 0, row, policy);
          }
        } else if (lane < 2 * np) {
          const int q = lane >> 1, half = lane & 1;
          const int row = p.row_base + (pages[j * PPI + q] * p.Hkv + U.kvh) * BS;
          tma_load_2d(st + half * TcLayout::kRegion + q * BS * 128, &vmap, bar, half * 64, row, policy);
        }
        copies_end = g + 1;
      }
      if (timed_out) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&slot_free[k]);
    }
  } else if (widen) {
    // Converter (one-byte caches): per unit, K of its first step, then per
    // step j the K codes of step j + 1 and the V codes of step j (the order
    // the MMA warp needs them: S runs one step ahead of P . V), each once its
    // codes have landed; E4M3 caches only V (their K pages feed the
    // products as they are).  (Widening V in the V copy warp instead,
    // between its copies, delayed the next copy: 780 against 573 us for the
    // 32-token verify step on an E4M3 cache, with the earlier f32 widening.)
    uint32_t gk = 0, gv = 0;
    for (int i = 0;; ++i) {
      const int k = i & 1;
      if (!warp_wait(&slot_full[k], (i >> 1) & 1u, true)) {
        timed_out = true;
        break;
      }
      const TcUnit U = read_unit(k);
      if (U.u >= total_units) break;
      const float4* par = slot_par(k);
      bool ok = kF8K || widen_pages(true, U, par, 0, gk++);
      for (int j = 0; ok && j < U.nsteps; ++j) {
        if (!kF8K && j + 1 < U.nsteps) ok = widen_pages(true, U, par, j + 1, gk++);
        if (ok) ok = widen_pages(false, U, par, j, gv++);
      }
      if (!ok) {
        timed_out = true;
        break;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&slot_free[k]);
    }
  } else if (mma_warp) {
    if (lane == 0) {
      // S(g) into the S slot once the compute warps have read S(g - 1) and
      // K(g) has landed
      auto issue_s = [&](uint32_t g) -> bool {
        if (g >= 1 && !mbar_wait_spin(s_free, (g - 1) & 1u, kWaitLimitNs)) return false;
        if (!mbar_wait_bounded(&full_k[g % kTcKStages], (g / kTcKStages) & 1u, kWaitLimitNs)) return false;
        const uint32_t k_addr = smem_addr(sm + TcLayout::kK + (g % kTcKStages) * TcLayout::kTile);
        tc_fence_after_sync();
        if constexpr (kF8K) {
          // E4M3: the codes' 128-byte rows in the upper half, 32 d per
          // product, once with each part of the query (columns 0-31: the
          // high part, 32-63: the low part)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t koff = static_cast<uint32_t>((kk & 3) * 32);  // 32 d = 32 bytes along the row
            const uint64_t bdesc = tc_smem_desc(k_addr + TcLayout::kRegion + koff, 16, 1024, 2);
            tc_mma_e4m3_ts(tmem + kTcSCol, tmem + kTcQCol + 32 * (kk >> 2) + 8 * (kk & 3), bdesc, kIdescS, kk > 0);
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = static_cast<uint32_t>((kk & 3) * 32);  // 16 d = 32 bytes along the row
            const uint64_t bdesc = tc_smem_desc(k_addr + (kk >> 2) * TcLayout::kRegion + koff, 16, 1024, 2);
            tc_mma_bf16_ts(tmem + kTcSCol, tmem + kTcQCol + 8 * kk, bdesc, kIdescS, kk > 0);
          }
        }
        tc_commit(s_done);
        s_end = g + 1;
        return true;
      };
      // O (+)= P(g) . V(g): P K-major in the K stage, V MN-major as the page
      // holds it (64-d halves kRegion apart, 8-token groups 1024 B apart);
      // the commits release the stages (and let the compute warps read O)
      auto issue_pv = [&](uint32_t g, bool first, bool last) -> bool {
        if (!mbar_wait_spin(&p_ready[g % kTcKStages], (g / kTcKStages) & 1u, kWaitLimitNs)) return false;
        if (!mbar_wait_bounded(&full_v[g % kTcVStages], (g / kTcVStages) & 1u, kWaitLimitNs)) return false;
        const uint32_t pa = smem_addr(sm + TcLayout::kK + (g % kTcKStages) * TcLayout::kTile);
        const uint32_t v_addr = smem_addr(sm + TcLayout::kV + (g % kTcVStages) * TcLayout::kTile);
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < kTcTokens / 16; ++kk) {
          const uint64_t a = tc_smem_desc(pa + kk * 256, 128, 1024, 0);
          const uint64_t bdesc = tc_smem_desc(v_addr + kk * 2048, TcLayout::kRegion, 1024, 2);
          tc_mma_bf16(tmem + kTcOCol, a, bdesc, kIdescO, !first || kk > 0);
        }
        // the K and V stages of a unit's last step are released by the
        // compute warps, who stage the unit's output there
        if (last) {
          tc_commit(o_ready);
        } else {
          tc_commit(&kp_free[g % kTcKStages]);
          tc_commit(&v_free[g % kTcVStages]);
        }
        pv_end = g + 1;
        return true;
      };
      bool ok = mbar_wait_bounded(&slot_full[0], 0, kWaitLimitNs);
      bool more = ok && slot_desc(0)[0] < total_units;
      int nsteps = more ? read_unit(0).nsteps : 0;
      if (more) ok = mbar_wait_spin(q_ready, 0, kWaitLimitNs) && issue_s(0);
      uint32_t g0 = 0;
      for (int i = 0; ok && more; ++i) {
        int next_steps = 0;
        for (int j = 0; ok && j < nsteps; ++j) {
          const uint32_t g = g0 + j;
          if (j + 1 < nsteps) {  // S one step ahead, then P . V
            ok = issue_s(g + 1) && issue_pv(g, j == 0, false);
          } else {  // the unit's last P . V, then the next unit's first S once its query tile is in TMEM
            ok = issue_pv(g, j == 0, true) &&
                 mbar_wait_bounded(&slot_full[(i + 1) & 1], ((i + 1) >> 1) & 1u, kWaitLimitNs);
            more = ok && slot_desc((i + 1) & 1)[0] < total_units;
            if (more) {
              next_steps = read_unit((i + 1) & 1).nsteps;
              ok = mbar_wait_spin(q_ready, (i + 1) & 1u, kWaitLimitNs) && issue_s(g + 1);
            }
          }
        }
        if (!ok) break;
        mbar_arrive(&slot_free[i & 1]);
        g0 += static_cast<uint32_t>(nsteps);
        nsteps = next_steps;
      }
      if (!ok) timed_out = true;
    }
    __syncwarp();
  } else {
    // compute warps: thread tid owns row vrow of the tile (tid itself unless
    // the rows are rotated into the highest lanes); a warp without rows
    // (warp_dead) only keeps the barriers' counts and clears stale V rows
    const int rot = kRot ? 128 - ((p.G * p.Tt + 31) & ~31) : 0;
    const int vrow = kRot ? ((tid - rot) & 127) : tid;
    const bool warp_dead = kRot && (32 * warp + 31) < rot;
    // this row of unit U's query tile: loads (in flight until used), then
    // into its TMEM lane, then q_ready
    auto load_query = [&](const TcUnit& U, int half, uint4 (&qv)[8]) {  // d 64 half .. +63
      int t = 0, h = 0;
      const bool ok = tile_row<true>(p, U.kvh, U.tile, vrow, t, h);
      const uint4* src = reinterpret_cast<const uint4*>(p.q + (static_cast<size_t>(U.b * p.T + t) * p.Hq + h) * D) + 8 * half;
#pragma unroll
      for (int c = 0; c < 8; ++c) qv[c] = ok ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
    };
    auto store_query = [&](int half, const uint4 (&qv)[8]) {
      uint32_t w[32];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        w[4 * c] = qv[c].x;
        w[4 * c + 1] = qv[c].y;
        w[4 * c + 2] = qv[c].z;
        w[4 * c + 3] = qv[c].w;
      }
      tc_st32(t_lane + kTcQCol + 32 * half, w);
    };
    // one-byte caches: the row scaled by 2^-kq, in the type of S's other
    // operand; returns kq, which the row's softmax coefficient takes back.
    // INT8 (f16 K code values): the largest |q| in [2^14, 2^15), exact for
    // every bf16 value within 2^-10 of it.  E4M3 (K codes as they are): the
    // largest |q'| in [2^7, 2^8), as two E4M3 parts qh = e4m3(q'),
    // ql = e4m3(q' - qh); q' has 8 significant bits, qh holds the first 4
    // and the residual the rest, so qh + ql = q' exactly wherever the
    // residual is no finer than E4M3's 2^-9 (|q'| >= 2^-2), within 2^-10
    // below
    float qsum_next = 0.f;  // INT8 caches: sum of the row's stored f16 query values (next unit)
    auto put_query = [&](const TcUnit& U) -> int {
      if constexpr (!kOneByte) {
        for (int half = 0; half < 2; ++half) {
          uint4 qv[8];
          load_query(U, half, qv);
          store_query(half, qv);
        }
        return 0;
      } else {
        uint4 qv[2][8];
        load_query(U, 0, qv[0]);
        load_query(U, 1, qv[1]);
        uint32_t mx = 0;  // largest |q| as bf16 bits
#pragma unroll
        for (int half = 0; half < 2; ++half)
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const uint32_t w4[4] = {qv[half][c4].x, qv[half][c4].y, qv[half][c4].z, qv[half][c4].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) mx = max(mx, max(w4[e] & 0x7fffu, (w4[e] >> 16) & 0x7fffu));
          }
        const int kq = mx == 0 ? 0 : max(-100, min(100, static_cast<int>(mx >> 7) - 127 - (kF8K ? 7 : 14)));
        const float sc = __uint_as_float(static_cast<uint32_t>(127 - kq) << 23);  // 2^-kq
        if constexpr (kF8K) {
          // per d half: 16 columns of each part (four E4M3 values a column:
          // d 4c .. 4c + 3), high part at column 16 half, low at 32 + 16 half
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t wh[16], wl[16];
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
              const uint32_t w4[4] = {qv[half][c4].x, qv[half][c4].y, qv[half][c4].z, qv[half][c4].w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {  // d = 64 half + 8 c4 + 2 e, + 1
                const float2 v = make_float2(bf16lo_to_f32(w4[e]) * sc, bf16hi_to_f32(w4[e]) * sc);
                const __nv_fp8x2_storage_t h = __nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, __NV_E4M3);
                const float2 hv = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(h, __NV_E4M3)));
                const __nv_fp8x2_storage_t lo =
                    __nv_cvt_float2_to_fp8x2(make_float2(v.x - hv.x, v.y - hv.y), __NV_SATFINITE, __NV_E4M3);
                const int col = 2 * c4 + (e >> 1);
                if (e & 1) {
                  wh[col] |= static_cast<uint32_t>(h) << 16;
                  wl[col] |= static_cast<uint32_t>(lo) << 16;
                } else {
                  wh[col] = static_cast<uint32_t>(h);
                  wl[col] = static_cast<uint32_t>(lo);
                }
              }
            }
            tc_st16(t_lane + kTcQCol + 16 * half, wh);
            tc_st16(t_lane + kTcQCol + 32 + 16 * half, wl);
          }
        } else {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t w[32];
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
              const uint32_t w4[4] = {qv[half][c4].x, qv[half][c4].y, qv[half][c4].z, qv[half][c4].w};
#pragma unroll
              for (int e = 0; e < 4; ++e) w[4 * c4 + e] = pack_f16x2(bf16lo_to_f32(w4[e]) * sc, bf16hi_to_f32(w4[e]) * sc);
            }
            if constexpr (KV == PKV_KV_INT8) {  // exact f16 values, summed in fp32
              float s0 = 0.f, s1 = 0.f;
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
                s0 += f.x;
                s1 += f.y;
              }
              qsum_next = (half == 0 ? 0.f : qsum_next) + (s0 + s1);
            }
            tc_st32(t_lane + kTcQCol + 32 * half, w);
          }
        }
        return kq;
      }
    };
    const float c = p.scale_log2;
    uint32_t nchunk = 0, nfree = 0;  // phases of stg_full, stg_free
    // The unit stays in its slot until these warps release it, so only what
    // the steps need is kept in registers; the rest is read again for the
    // output.
    bool ok = warp_wait(&slot_full[0], 0, true);
    bool more = ok && slot_desc(0)[0] < total_units;
    int kq_next = 0;  // one-byte caches: the next unit's query exponent of this row
    if (more) {
      const TcUnit U = read_unit(0);
      kq_next = put_query(U);
      tc_wait_st();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_ready);
    }
    uint32_t g0 = 0;
    for (int i = 0; more; ++i) {
      const int k = i & 1;
      int nsteps, t0, t1, lim;  // steps, token range, keys of this row: positions < lim
      bool row_ok;
      {
        const TcUnit U = read_unit(k);
        int t = 0, h = 0;
        row_ok = tile_row<true>(p, U.kvh, U.tile, vrow, t, h);
        nsteps = U.nsteps;
        t0 = U.t0;
        t1 = U.t1;
        lim = U.ctx - p.T + 1 + t;
      }
      const volatile uint8_t* bad = slot_bad(k);
      bool has_next = false;
      float m = -INFINITY, l = 0.f;  // log2-domain running max (lazy) and sum of this row
      // one-byte caches: the scores arrive as S' x 2^-kq per row and code
      // value per key; cq = c 2^kq scales them back (with k_scale per page),
      // and the softmax works on the scaled scores with coefficient 1
      const float cq = kOneByte ? c * __uint_as_float(static_cast<uint32_t>(127 + kq_next) << 23) : c;
      const float qsum = qsum_next;  // INT8: this unit's (the next put_query overwrites qsum_next)
      const float cs = kOneByte ? 1.f : c;
      const float inv_vmax = kOneByte ? 1.f / __int_as_float(slot_desc(k)[5]) : 1.f;
      const int npages_u = (t1 - t0 + BS - 1) / BS;

      // tokens of step j that belong to the sequence (and to a valid page),
      // then those this row attends to (its causal limit)
      auto step_masks = [&](int j, uint64_t& vmask, uint64_t& rmask) {
        const int pos0 = t0 + j * kTcTokens;
        const int nvalid = t1 - pos0;
        vmask = nvalid >= kTcTokens ? ~0ull : ((1ull << nvalid) - 1ull);
#pragma unroll
        for (int q = 0; q < PPI; ++q)
          if (bad[j * PPI + q]) vmask &= ~(((1ull << BS) - 1ull) << (q * BS));
        const int nrow = lim - pos0;
        rmask = row_ok ? (vmask & (nrow >= kTcTokens ? ~0ull : (nrow <= 0 ? 0ull : ((1ull << nrow) - 1ull)))) : 0ull;
      };
      // the step's masked extremum of the raw scores -> running maximum; a
      // row whose maximum grew by more than 2^8 (grow) rescales l here and
      // its O by the returned factor once P is written (rescale_o)
      auto update_max = [&](float ext, uint64_t rmask, bool& grow) -> float {
        const float smax = rmask != 0ull ? ext * cs : -INFINITY;
        const float mnew = fmaxf(m, smax);
        grow = (m == -INFINITY) ? (mnew != -INFINITY) : (mnew > m + 8.f);
        float factor = 1.f;
        if (grow) {
          factor = (m == -INFINITY) ? 0.f : ex2_approx(m - mnew);
          l *= factor;
          m = mnew;
        }
        return factor;
      };
      // O *= factor in TMEM once P . V(g - 1) is done; after the step's P is
      // written, so that the scores no longer hold registers.  False on
      // timeout.
      auto rescale_o = [&](float factor, uint32_t g) -> bool {
        if (!mbar_wait_spin(&v_free[(g - 1) % kTcVStages], ((g - 1) / kTcVStages) & 1u, kWaitLimitNs))
          timed_out = true;
        tc_fence_after_sync();
#pragma unroll 1
        for (int cc = 0; cc < D; cc += 32) {
          uint32_t ov[32];
          tc_ld32(t_lane + kTcOCol + cc, ov);
          tc_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * factor);
          tc_st32(t_lane + kTcOCol + cc, ov);
        }
        tc_wait_st();
        return !__any_sync(kFull, timed_out);  // the only wait here
      };
      // V rows of tokens outside the sequence (or of a bad page) may hold
      // anything (even NaN) and P is 0 there: once V(g) has landed, thread
      // (warp w, lane l) clears 16-byte d-chunks 4w .. 4w+3 of token rows l
      // and l + 32.  False on timeout.
      auto clear_stale_v = [&](uint64_t vmask, uint32_t g) -> bool {
        if (vmask == ~0ull) return true;
        if (!mbar_wait_bounded(&full_v[g % kTcVStages], (g / kTcVStages) & 1u, kWaitLimitNs)) timed_out = true;
        if (__any_sync(kFull, timed_out)) return false;
        uint8_t* vb = sm + TcLayout::kV + (g % kTcVStages) * TcLayout::kTile;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int tk = lane + 32 * r;  // token row
#pragma unroll
          for (int i4 = 0; i4 < 4; ++i4) {
            const int dc = 4 * warp + i4;  // 16-byte d-chunk
            if (!((vmask >> tk) & 1ull))
              *reinterpret_cast<uint4*>(vb + (dc >> 3) * TcLayout::kRegion + tk * 128 +
                                        (((dc & 7) ^ (tk & 7)) << 4)) = make_uint4(0, 0, 0, 0);
          }
        }
        return true;
      };
      // 32 scores (bit patterns) -> P (bf16, 8 tokens per 16-byte store) at
      // token columns 32 half .. +31 of the step's K stage; returns their sum
      // (one-byte caches: P in f16 times v_scale / v_max of the token's page;
      // va for tokens 0-15 of the 32, vb for 16-31)
      auto write_p = [&](const uint32_t (&sc)[32], uint32_t hm, bool all32, uint8_t* pbuf, int half, float va,
                         float vb) -> float {
        const float neg_m = (m == -INFINITY) ? 0.f : -m;
        float psum = 0.f;
        // the common all-valid case without per-element mask tests (kept out
        // of the unrolled loop: they cost ALU issue slots on every score)
        if (all32) {
          // arguments, sums (and the one-byte P factors) by packed pair
          // instructions: one issue slot for two scores
          float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
          for (int k8 = 0; k8 < 4; ++k8) {
            uint32_t pw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int kk = 8 * k8 + 2 * e;
              float a0, a1;
              ffma2(a0, a1, __uint_as_float(sc[kk]), __uint_as_float(sc[kk + 1]), cs, cs, neg_m, neg_m);
              const float p0 = ex2_approx(a0);
              const float p1 = ex2_approx(a1);
              fadd2(ps0, ps1, ps0, ps1, p0, p1);
              if constexpr (kOneByte) {
                const float vq = kk < 16 ? va : vb;
                float q0, q1;
                fmul2(q0, q1, p0, p1, vq, vq);
                pw[e] = pack_f16x2(q0, q1);
              } else {
                pw[e] = pack_bf16x2(p0, p1);
              }
            }
            *reinterpret_cast<uint4*>(pbuf + tc_p_off(tid, 4 * half + k8)) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
          }
          return ps0 + ps1;
        }
#pragma unroll
        for (int k8 = 0; k8 < 4; ++k8) {
          uint32_t pw[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int kk = 8 * k8 + 2 * e;
            float p0 = ex2_approx(fmaf(__uint_as_float(sc[kk]), cs, neg_m));
            float p1 = ex2_approx(fmaf(__uint_as_float(sc[kk + 1]), cs, neg_m));
            p0 = ((hm >> kk) & 1u) ? p0 : 0.f;
            p1 = ((hm >> (kk + 1)) & 1u) ? p1 : 0.f;
            psum += p0 + p1;
            const float vq = kk < 16 ? va : vb;
            pw[e] = kOneByte ? pack_f16x2(p0 * vq, p1 * vq) : pack_bf16x2(p0, p1);
          }
          *reinterpret_cast<uint4*>(pbuf + tc_p_off(tid, 4 * half + k8)) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
        }
        return psum;
      };
      auto finish_step = [&](uint32_t g) {
        fence_proxy_async_smem();  // P and the cleared V rows are read by the tensor cores
        tc_fence_before_sync();
        mbar_arrive(&p_ready[g % kTcKStages]);
      };

      for (int j = 0; j < nsteps; ++j) {
        const uint32_t g = g0 + j;
        uint64_t vmask, rmask;
        step_masks(j, vmask, rmask);  // independent of S: computed while it is on its way
        // one-byte caches: the step's pages' score coefficients and P factors
        // (pages past the unit's end: 0, their tokens are masked)
        float ckq[PPI], vrq[PPI], cadd[PPI];
#pragma unroll
        for (int q = 0; q < PPI; ++q) {
          ckq[q] = 0.f;
          cadd[q] = 0.f;
          vrq[q] = 0.f;
          if constexpr (kOneByte) {
            if (j * PPI + q < npages_u) {
              const float4 pr = slot_par(k)[j * PPI + q];
              ckq[q] = cq * pr.x;
              // the biased INT8 K code values add (1152 + zero) x sum(q) to S'
              if constexpr (KV == PKV_KV_INT8) cadd[q] = -(kInt8Bias + pr.y) * qsum * ckq[q];
              vrq[q] = inv_vmax * pr.z;
            }
          }
        }
        if (!mbar_wait_bounded(s_done, g & 1u, kWaitLimitNs)) timed_out = true;
        if (__any_sync(kFull, timed_out)) {  // warp-uniform exit (the loads below are collective)
          ok = false;
          break;
        }
        tc_fence_after_sync();
        if (j + 1 == nsteps) {
          // the unit's last S is done, so the next unit's query tile can take
          // its TMEM columns (before this step's scores occupy the registers)
          if (!warp_wait(&slot_full[k ^ 1], ((i + 1) >> 1) & 1u, true)) {
            ok = false;
            break;
          }
          has_next = slot_desc(k ^ 1)[0] < total_units;
          if (has_next) {
            const TcUnit U = read_unit(k ^ 1);
            kq_next = put_query(U);
            tc_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(q_ready);
          }
        }
        if (warp_dead) {  // no scores to read: S(g + 1) may come at once
          __syncwarp();
          if (lane == 0) mbar_arrive(s_free);
          if (!clear_stale_v(vmask, g)) {
            ok = false;
            break;
          }
          finish_step(g);
          continue;
        }
        uint32_t sv[kTcTokens];
        tc_ld32(t_lane + kTcSCol, *reinterpret_cast<uint32_t(*)[32]>(sv));
        tc_ld32(t_lane + kTcSCol + 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
        tc_wait_ld();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_free);  // the slot may take S(g + 1)
        if constexpr (kOneByte) {  // the scaled scores, in log2 units (two per packed instruction)
#pragma unroll
          for (int t = 0; t < kTcTokens; t += 2) {
            const float kq = ckq[t / BS];
            float a0, a1;
            if constexpr (KV == PKV_KV_INT8)
              ffma2(a0, a1, __uint_as_float(sv[t]), __uint_as_float(sv[t + 1]), kq, kq, cadd[t / BS], cadd[t / BS]);
            else
              fmul2(a0, a1, __uint_as_float(sv[t]), __uint_as_float(sv[t + 1]), kq, kq);
            sv[t] = __float_as_uint(a0);
            sv[t + 1] = __float_as_uint(a1);
          }
        }
        // masked extremum of the raw scores (maximum for a non-negative
        // scale); a step whose tokens are all this row's takes branch-free code
        const bool all = rmask == ~0ull;
        const bool cpos = kOneByte || c >= 0.f;
        float ext;
        if (all) {
          if (cpos)
            ext = tree_ext64<true>(sv);
          else
            ext = tree_ext64<false>(sv);
        } else if (cpos) {
          ext = -INFINITY;
#pragma unroll
          for (int kk = 0; kk < kTcTokens; ++kk)
            if ((rmask >> kk) & 1ull) ext = fmaxf(ext, __uint_as_float(sv[kk]));
        } else {
          ext = INFINITY;
#pragma unroll
          for (int kk = 0; kk < kTcTokens; ++kk)
            if ((rmask >> kk) & 1ull) ext = fminf(ext, __uint_as_float(sv[kk]));
        }
        bool grow;
        const float factor = update_max(ext, rmask, grow);
        if (!clear_stale_v(vmask, g)) {
          ok = false;
          break;
        }
        uint8_t* pbuf = sm + TcLayout::kK + (g % kTcKStages) * TcLayout::kTile;
        l += write_p(*reinterpret_cast<const uint32_t(*)[32]>(sv), static_cast<uint32_t>(rmask), all, pbuf, 0, vrq[0],
                     vrq[16 / BS]) +
             write_p(*reinterpret_cast<const uint32_t(*)[32]>(sv + 32), static_cast<uint32_t>(rmask >> 32), all, pbuf, 1,
                     vrq[32 / BS], vrq[48 / BS]);
        if (j > 0 && __any_sync(kFull, grow) && !rescale_o(factor, g)) {
          ok = false;
          break;
        }
        finish_step(g);
      }
      if (!ok || __any_sync(kFull, timed_out)) {
        ok = false;
        break;
      }
      // the unit's last P . V, then the output, staged in the last step's K
      // and V stages (P . V is done with them) and written by tensor-map
      // stores; every lane loads (tcgen05.ld is warp-collective), and the
      // store box holds only the tile's query rows (tokens past T clipped)
      const uint32_t gl = g0 + nsteps - 1;
      if (!mbar_wait_bounded(o_ready, i & 1u, kWaitLimitNs)) timed_out = true;
      if (__any_sync(kFull, timed_out)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const TcUnit U = read_unit(k);
      size_t qrow;
      {
        int t = 0, h = 0;
        tile_row<true>(p, U.kvh, U.tile, vrow, t, h);
        qrow = static_cast<size_t>(U.b * p.T + t) * p.Hq + h;
      }
      const bool direct = U.nparts == 1;
      uint8_t* stg_base = sm + TcLayout::kK + (gl % kTcKStages) * TcLayout::kTile;  // [128 rows][128 B]
      if (direct) {
        // bf16 output (O / l): two chunks of 64 columns as 128-byte rows of
        // bf16, staged in the last step's K and V stages (16-byte chunks
        // XOR-swizzled by row, as the output map's 128-byte swizzle reads
        // them) and written by thread 0 with one tensor-map store each
        const float osc = l > 0.f ? (kOneByte ? __int_as_float(slot_desc(k)[5]) : 1.f) / l : 0.f;
        uint8_t* vbuf = sm + TcLayout::kV + (gl % kTcVStages) * TcLayout::kTile;
#pragma unroll 1
        for (int k2 = 0; k2 < 2; ++k2, ++nchunk) {
          uint8_t* buf = k2 ? vbuf : stg_base;
#pragma unroll 1
          for (int hh = 0; hh < 2; ++hh) {  // 32 columns at a time
            uint32_t ov[32];
            tc_ld32(t_lane + kTcOCol + 64 * k2 + 32 * hh, ov);
            tc_wait_ld();
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
              const float* f = reinterpret_cast<const float*>(ov + 8 * c4);
              *reinterpret_cast<uint4*>(buf + vrow * 128 + (((4 * hh + c4) ^ (vrow & 7)) << 4)) =
                  make_uint4(pack_bf16x2(f[0] * osc, f[1] * osc), pack_bf16x2(f[2] * osc, f[3] * osc),
                             pack_bf16x2(f[4] * osc, f[5] * osc), pack_bf16x2(f[6] * osc, f[7] * osc));
            }
          }
          fence_proxy_async_smem();  // read by the tensor-map store
          __syncwarp();
          if (lane == 0) mbar_arrive(stg_full);
          if (tid == 0) {
            if (mbar_wait_spin(stg_full, nchunk & 1u, kWaitLimitNs)) {
              tma_store_4d(&omap, buf, 64 * k2, U.kvh * p.G, U.tile * p.Tt, U.b);
              bulk_commit();
            } else {
              timed_out = true;
            }
          }
        }
        // both stages go back to the copy warps once the stores have read them
        if (tid == 0 && !timed_out) {
          bulk_wait_read_all();
          mbar_arrive(&kp_free[gl % kTcKStages]);
          mbar_arrive(&v_free[gl % kTcVStages]);
        }
      } else {
        // split-K partials (m, l, unnormalised O): the tile's rows are staged
        // 32 columns at a time (row r at r * 128 bytes, 16-byte chunks
        // XOR-swizzled by r % 8, as the store map's 128-byte swizzle reads
        // them), alternately in the last step's K and V stages, and thread 0
        // stores each chunk with one tensor-map store; a buffer is restaged
        // once the store before has read it
        uint8_t* vbuf = sm + TcLayout::kV + (gl % kTcVStages) * TcLayout::kTile;
#pragma unroll 1
        for (int k = 0; k < D / 32; ++k, ++nchunk) {
          const int cc = 32 * k;
          uint32_t ov[32];
          tc_ld32(t_lane + kTcOCol + cc, ov);
          tc_wait_ld();
          if constexpr (kOneByte) {  // O in value units
            const float vmx = __int_as_float(slot_desc(i & 1)[5]);
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * vmx);
          }
          if (k >= 2 && !warp_wait(stg_free, (nfree + k - 2) & 1u, false)) {
            timed_out = true;
            break;
          }
          uint8_t* buf = (k & 1) ? vbuf : stg_base;
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4)
            *reinterpret_cast<uint4*>(buf + vrow * 128 + ((c4 ^ (vrow & 7)) << 4)) =
                make_uint4(ov[4 * c4], ov[4 * c4 + 1], ov[4 * c4 + 2], ov[4 * c4 + 3]);
          fence_proxy_async_smem();  // read by the tensor-map store
          __syncwarp();
          if (lane == 0) mbar_arrive(stg_full);
          if (tid == 0) {
            if (mbar_wait_spin(stg_full, nchunk & 1u, kWaitLimitNs)) {
              tma_store_5d(&pmap, buf, cc, U.pidx, U.kvh * p.G, U.tile * p.Tt, U.b);
              bulk_commit();
              if (k == 1 || k == 2) {  // the store of chunk k - 1 has read its buffer
                bulk_wait_read_but1();
                mbar_arrive(stg_free);
              }
            } else {
              timed_out = true;
            }
          }
        }
        nfree += 2;
        if (row_ok) *reinterpret_cast<float2*>(p.part_ml + 2 * (qrow * p.pmax + U.pidx)) = make_float2(m, l);
        // both stages go back to the copy warps once the last stores have read them
        if (tid == 0 && !timed_out) {
          bulk_wait_read_all();
          mbar_arrive(&kp_free[gl % kTcKStages]);
          mbar_arrive(&v_free[gl % kTcVStages]);
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&slot_free[i & 1]);
      g0 += static_cast<uint32_t>(nsteps);
      more = ok && has_next;
    }
    if (!ok) timed_out = true;
  }

  timed_out = __syncthreads_or(timed_out) != 0;  // every role has left its loop
  if (timed_out) {
    if (tid == 0) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
    // each role lets its own copies and products still in flight finish
    // (bounded) before the shared and tensor memory are released: the last
    // steps' copies (one per stage, so one phase per barrier) and the MMA
    // warp's last commits (each covers every earlier product)
    if (kcopy && lane == 0)
      for (uint32_t g = copies_end > kTcKStages ? copies_end - kTcKStages : 0; g < copies_end; ++g)
        mbar_wait_bounded((kOneByte && !kF8K) ? &tma_k[g % kTcKStages] : &full_k[g % kTcKStages], (g / kTcKStages) & 1u,
                          kWaitLimitNs / 16);
    if (vcopy && lane == 0)
      for (uint32_t g = copies_end > kTcVStages ? copies_end - kTcVStages : 0; g < copies_end; ++g)
        mbar_wait_bounded(kOneByte ? &tma_v[g % kTcVStages] : &full_v[g % kTcVStages], (g / kTcVStages) & 1u,
                          kWaitLimitNs / 16);
    if (mma_warp && lane == 0 && (s_end > 0 || pv_end > 0)) {  // one commit covers every product issued
      tc_commit(mma_drain);
      mbar_wait_bounded(mma_drain, 0, kWaitLimitNs / 16);
    }
  }
  if (tid == 0) bulk_wait_all();  // the partials' stores are written before the CTA retires
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tc_dealloc(tmem, kTcCols);
}

}  // namespace pkv
