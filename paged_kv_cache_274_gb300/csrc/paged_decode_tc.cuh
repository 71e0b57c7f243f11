// Multi-token decode on the 5th-generation tensor cores (tcgen05 + TMEM),
// bf16 cache, head_dim 128.
//
// A query of T new tokens per sequence has T x G (query token, head) rows per
// KV head ("KV-Cache Engineering: Paged Attention, Prefix Cache,
// Disaggregation (2026)": speculative decoding scores the draft's T tokens in
// one pass over the shared cache; "KV Cache Engineering: PagedAttention,
// Continuous Batching, Attention Variants, and the Bandwidth Wall",
// "Continuous Batching": chunked prefill).  With more than 16 rows the page
// work is a real matrix product, so here one CTA of 4 warps takes a tile of
// 128 rows (M of the MMA) and steps through its pages 32 tokens at a time:
//
//   * Warp-specialised: two copy warps issue the tensor-map copies (TMA,
//     128-byte swizzle) of each step's K and V pages into 3-stage rings, K
//     into a stage as soon as the product that read its last K is done, V
//     once P . V of its last V is done; an MMA warp issues S = Q . K^T
//     (M 128, N 32, K 128; the query tile is the A operand in TMEM, so a
//     step reads only K from shared memory) into a double-buffered TMEM slot
//     two steps ahead of the softmax, and O += P . V (M 128, N 128, K 32, V read MN-major
//     straight from the page) when the compute warps have P ready; four
//     compute warps own the 128 rows.  The roles hand work over only through
//     mbarriers, so copies, products and softmax of neighbouring steps
//     overlap.
//   * Thread r owns row r: it loads its 32 scores from TMEM (and tells the MMA
//     warp that the slot is free), masks them (sequence end, causal limit of
//     its query token), and keeps the online softmax state in registers.  The
//     running maximum is lazy: the output is rescaled only when a row's
//     maximum grows by more than 2^8, so P stays below 256 and the rescale of
//     O in TMEM is rare.  P goes to shared memory as bf16 (K-major, no
//     swizzle).  V rows of tokens outside the sequence (or of a bad page) are
//     cleared in the stage, as P is 0 there but the stale rows may hold NaN.
//   * At the end of the unit each thread reads its row of O and writes the
//     bf16 output or the split-K partials (m, l, O) of the other kernels.
//
// Units are (sequence, KV head, row tile, partition) from the planner's
// counter; the merge kernel combines partitions.  Every wait is bounded; a
// CTA that gives up records PKV_DEVERR_TIMEOUT, lets its copies and products
// finish (bounded) and frees its tensor memory.
#pragma once

#include "paged_decode.cuh"

namespace pkv {

constexpr int kTcRows = 128;      // query rows per tile (MMA M)
constexpr int kTcTokens = 32;     // tokens per step
constexpr int kTcStages = 3;
constexpr int kTcComputeWarps = 4;  // one row of the tile per thread
constexpr int kTcThreads = 32 * (kTcComputeWarps + 3);  // + MMA warp + K copy warp + V copy warp
constexpr uint32_t kTcCols = 256;  // TMEM columns: S at 0 and 32 (double buffer), Q at 64, O at 128
constexpr uint32_t kTcSCol = 0;
constexpr uint32_t kTcQCol = 64;   // query tile: 128 d as 64 columns of bf16 pairs
constexpr uint32_t kTcOCol = 128;

struct TcLayout {  // byte offsets from the 1024-aligned shared-memory base
  static constexpr uint32_t kRegion = kTcTokens * 128;       // half (64 of 128 d) of a 32-token tile: 4 KiB
  static constexpr uint32_t kTile = 2 * kRegion;             // a K or V tile: 8 KiB
  static constexpr uint32_t kStage = 2 * kTile;              // K then V: 16 KiB
  static constexpr uint32_t kStages = 0;
  static constexpr uint32_t kP = kStages + kTcStages * kStage;  // 2 x [128 x 32] bf16 core-matrix layout
  static constexpr uint32_t kPBuf = kTcRows * kTcTokens * 2;      // 8 KiB
  static constexpr uint32_t kBars = kP + 2 * kPBuf;
  // full_k[3], full_v[3], k_free[3], o_done[3], s_done[2], s_free[2], p_ready[2]
  static constexpr int kNumBars = 4 * kTcStages + 3 * 2;
  static constexpr uint32_t kMisc = kBars + 8 * kNumBars;     // TMEM base
  static constexpr uint32_t kDesc = kMisc + 16;               // 2 x 8 int32: unit descriptors
  static constexpr uint32_t kPages = kDesc + 64;              // int32 physical ids of the unit's pages
  static constexpr uint32_t kBad = kPages + 64 * 4;           // uint8 bad-id flags
  static constexpr uint32_t kEnd = kBad + 64;
};

__host__ __device__ constexpr size_t tc_smem_layout_bytes() { return 1024 + TcLayout::kEnd; }

// K-major, no-swizzle core-matrix layout of a [rows x 32] bf16 tile: core
// matrix (r/8, k/8) of 8 rows x 16 bytes at (r/8) * 512 + (k/8) * 128.
__device__ __forceinline__ uint32_t tc_core_off(int r, int k8) {
  return static_cast<uint32_t>((r >> 3) * 512 + k8 * 128 + (r & 7) * 16);
}

template <int BS>
__global__ void __launch_bounds__(kTcThreads, 2)
    paged_decode_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                           const __grid_constant__ CUtensorMap vmap, const DecodeParams p) {
  constexpr int D = 128;
  constexpr int PPI = kTcTokens / BS;  // pages per step
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  // Barrier phases are counted over the CTA's lifetime with the global step
  // index g: stages and full_k[] / full_v[] / k_free[] / o_done[] by g % 3,
  // S slot and s_done[] / s_free[] / p_ready[] by g % 2.  Every barrier
  // completes one phase per step that uses it, and no waiter can fall two
  // phases behind (each next use of a barrier depends on the wait).
  uint64_t* full_k = reinterpret_cast<uint64_t*>(sm + TcLayout::kBars);  // [3] K(g) landed
  uint64_t* full_v = full_k + kTcStages;                                 // [3] V(g) landed
  uint64_t* k_free = full_v + kTcStages;                                 // [3] S(g) done: K stage free
  uint64_t* o_done = k_free + kTcStages;                                 // [3] P . V(g) done
  uint64_t* s_done = o_done + kTcStages;                                 // [2] S(g) in TMEM
  uint64_t* s_free = s_done + 2;                                         // [2] S(g) read by the compute warps
  uint64_t* p_ready = s_free + 2;                                        // [2] P(g) in shared memory
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + TcLayout::kMisc);
  volatile int* desc = reinterpret_cast<volatile int*>(sm + TcLayout::kDesc);  // [2][8]
  int* pages = reinterpret_cast<int*>(sm + TcLayout::kPages);
  uint8_t* bad = sm + TcLayout::kBad;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const bool compute = warp < kTcComputeWarps;
  const bool mma_warp = warp == kTcComputeWarps;
  const bool kcopy = warp == kTcComputeWarps + 1;
  const bool vcopy = warp == kTcComputeWarps + 2;

  if (tid == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&full_k[s], 1);
      mbar_init(&full_v[s], 1);
      mbar_init(&k_free[s], 1);
      mbar_init(&o_done[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_done[s], 1);
      mbar_init(&s_free[s], kTcComputeWarps);  // one lane per compute warp
      mbar_init(&p_ready[s], 32 * kTcComputeWarps);
    }
    fence_mbar_init();
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
  }
  if (warp == 0) tc_alloc(tmem_slot, kTcCols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_lane = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);  // compute warp's 32 lanes
  const uint64_t policy = p.NT > 1 ? l2_policy_evict_normal() : l2_policy_evict_first();
  constexpr uint32_t kIdescS = tc_idesc_bf16_f32(kTcRows, kTcTokens);
  constexpr uint32_t kIdescO = tc_idesc_bf16_f32(kTcRows, D, /*b_mn_major=*/true);
  pdl_trigger();
  pdl_wait();

  const int units_per_part = p.Hkv * p.NT;
  const int total_units = p.unit_start[p.B] * units_per_part;
  const int ppu_tokens = p.ppu * BS;
  uint32_t g0 = 0;  // global index of the current unit's first step
  bool timed_out = false;
  // end (global step) of this thread's own asynchronous work, for the drain
  // after a timeout: copies issued (copy warps), products committed (MMA warp)
  uint32_t copies_end = 0, s_end = 0, pv_end = 0;

  // One thread takes the next unit from the counter and looks up its
  // sequence, partition index, partition count and length into descriptor
  // slot `k` (u >= total_units: no more work); done one unit ahead, so that
  // these dependent loads overlap the current unit.
  auto fetch_unit = [&](int k) {
    volatile int* d = desc + 8 * k;
    const int u = atomicAdd(p.work_counter, 1);
    d[0] = u;
    if (u < total_units) {
      const int part = u / units_per_part;
      const int b = __ldg(p.part_seq + part);
      const int us = __ldg(p.unit_start + b);
      d[1] = b;
      d[2] = part - us;
      d[3] = __ldg(p.unit_start + b + 1) - us;
      d[4] = __ldg(p.ctx_eff + b);
    }
  };
  if (tid == 0) fetch_unit(0);
  int cur = 0;

  for (;;) {
    __syncthreads();  // descriptor `cur` is in place
    const volatile int* d = desc + 8 * cur;
    const int u = d[0];
    if (u >= total_units) break;
    const int part = u / units_per_part;
    const int rem = u - part * units_per_part;
    const int kvh = rem / p.NT;
    const int tile = rem - kvh * p.NT;
    const int b = d[1];
    const int pidx = d[2];
    const int nparts = d[3];
    const int ctx = d[4];
    const int t0 = pidx * ppu_tokens;
    const int t1 = min(ctx, t0 + ppu_tokens);
    const int npages = (t1 - t0 + BS - 1) / BS;  // 1 .. 64
    const int nsteps = (npages + PPI - 1) / PPI;
    const int* trow = p.block_tables + static_cast<size_t>(b) * p.MB + t0 / BS;
    if (tid < npages) {
      int e = __ldg(trow + tid);
      const bool isbad = static_cast<unsigned>(e) >= static_cast<unsigned>(p.NB);
      if (isbad) {
        e = 0;
        atomicOr(p.err, PKV_DEVERR_BLOCK_ID);
      }
      pages[tid] = e;
      bad[tid] = isbad ? 1 : 0;
    }
    // compute thread tid: query row tid of the tile (token t, head h)
    int t = 0, h = 0;
    const bool row_ok = compute && tile_row<true>(p, kvh, tile, tid, t, h);
    const size_t qrow = static_cast<size_t>(b * p.T + t) * p.Hq + h;
    if (compute) {  // this row of the query tile -> its TMEM lane (the unit's products are all done)
      const uint4* src = reinterpret_cast<const uint4*>(p.q + qrow * D);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t qv[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 w = row_ok ? __ldg(src + 8 * half + c) : make_uint4(0, 0, 0, 0);
          qv[4 * c] = w.x;
          qv[4 * c + 1] = w.y;
          qv[4 * c + 2] = w.z;
          qv[4 * c + 3] = w.w;
        }
        tc_st32(t_lane + kTcQCol + 32 * half, qv);
      }
      tc_wait_st();
    }
    const int lim = ctx - p.T + 1 + t;  // keys of this row: positions < lim
    tc_fence_before_sync();
    __syncthreads();  // page ids and the query tile are in place
    tc_fence_after_sync();

    if (kcopy || vcopy) {
      // K(g) into its stage once S(g - 3) is done, V(g) once P . V(g - 3) is
      // done; lane 2q + h issues the copy of half h (64 of 128 d) of the
      // step's page q.  The K warp also fetches the next unit, after its
      // first copies are on their way.
      uint64_t* fbar = kcopy ? full_k : full_v;
      uint64_t* free_bar = kcopy ? k_free : o_done;
      const CUtensorMap* map = kcopy ? &kmap : &vmap;
      const uint32_t part_off = kcopy ? 0u : TcLayout::kTile;
      for (int j = 0; j < nsteps; ++j) {
        if (kcopy && j == kTcStages && lane == 0) fetch_unit(cur ^ 1);
        const uint32_t g = g0 + j;
        int ok = 1;
        if (lane == 0 && g >= kTcStages)  // a suspending wait: the copies run ahead, the issue slots are the softmax's
          ok = mbar_wait_bounded(&free_bar[g % kTcStages], ((g - kTcStages) / kTcStages) & 1u, kWaitLimitNs) ? 1 : 0;
        if (!__shfl_sync(kFull, ok, 0)) {
          timed_out = true;
          break;
        }
        uint8_t* st = sm + TcLayout::kStages + (g % kTcStages) * TcLayout::kStage + part_off;
        uint64_t* bar = &fbar[g % kTcStages];
        const int np = min(PPI, npages - j * PPI);
        if (lane == 0) {
          if (vcopy) fence_proxy_async_smem();  // after the compute warps' clearing of stale V rows
          mbar_arrive_expect_tx(bar, static_cast<uint32_t>(np) * 2u * 64u * BS * 2u);
        }
        __syncwarp();
        if (lane < 2 * np) {
          const int q = lane >> 1, half = lane & 1;
          const int row = p.row_base + (pages[j * PPI + q] * p.Hkv + kvh) * BS;
          tma_load_2d(st + half * TcLayout::kRegion + q * BS * 128, map, bar, half * 64, row, policy);
        }
        copies_end = g + 1;
      }
      if (kcopy && nsteps <= kTcStages && lane == 0 && !timed_out) fetch_unit(cur ^ 1);
      __syncwarp();
    } else if (mma_warp) {
      if (lane == 0) {
        // S(g) into TMEM slot g % 2, once the compute warps have read S(g - 2)
        // from it and K(g) has landed
        auto issue_s = [&](uint32_t g) -> bool {
          if (g >= 2 && !mbar_wait_spin(&s_free[g & 1u], ((g - 2) >> 1) & 1u, kWaitLimitNs)) return false;
          if (!mbar_wait_bounded(&full_k[g % kTcStages], (g / kTcStages) & 1u, kWaitLimitNs)) return false;
          const uint32_t k_addr = smem_addr(sm + TcLayout::kStages + (g % kTcStages) * TcLayout::kStage);
          tc_fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = static_cast<uint32_t>((kk & 3) * 32);  // 16 d = 32 bytes along the row
            const uint64_t bdesc = tc_smem_desc(k_addr + (kk >> 2) * TcLayout::kRegion + koff, 16, 1024, 2);
            tc_mma_bf16_ts(tmem + kTcSCol + 32 * (g & 1u), tmem + kTcQCol + 8 * kk, bdesc, kIdescS, kk > 0);
          }
          tc_commit(&s_done[g & 1u]);
          tc_commit(&k_free[g % kTcStages]);
          s_end = g + 1;
          return true;
        };
        // O += P(g) . V(g): P K-major in shared memory, V MN-major as the page
        // holds it (64-d halves kRegion apart, 8-token groups 1024 B apart)
        auto issue_pv = [&](uint32_t g) -> bool {
          if (!mbar_wait_spin(&p_ready[g & 1u], (g >> 1) & 1u, kWaitLimitNs)) return false;
          if (!mbar_wait_bounded(&full_v[g % kTcStages], (g / kTcStages) & 1u, kWaitLimitNs)) return false;
          const uint32_t v_addr =
              smem_addr(sm + TcLayout::kStages + (g % kTcStages) * TcLayout::kStage + TcLayout::kTile);
          const uint32_t pa = smem_addr(sm + TcLayout::kP + (g & 1u) * TcLayout::kPBuf);
          tc_fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < kTcTokens / 16; ++kk) {
            const uint64_t a = tc_smem_desc(pa + kk * 256, 128, 512, 0);
            const uint64_t bdesc = tc_smem_desc(v_addr + kk * 2048, TcLayout::kRegion, 1024, 2);
            tc_mma_bf16(tmem + kTcOCol, a, bdesc, kIdescO, g > g0 || kk > 0);
          }
          tc_commit(&o_done[g % kTcStages]);
          pv_end = g + 1;
          return true;
        };
        bool ok = issue_s(g0) && (nsteps < 2 || issue_s(g0 + 1));
        for (int j = 0; ok && j < nsteps; ++j) {
          const uint32_t g = g0 + j;
          if (j + 2 < nsteps) ok = issue_s(g + 2);
          if (ok) ok = issue_pv(g);
        }
        if (!ok) timed_out = true;
      }
      __syncwarp();
    } else {
      // compute warps: one row each
      float m = -INFINITY, l = 0.f;  // log2-domain running max (lazy) and sum of this row
      for (int j = 0; j < nsteps; ++j) {
        const uint32_t g = g0 + j;
        uint8_t* st = sm + TcLayout::kStages + (g % kTcStages) * TcLayout::kStage;
        if (!mbar_wait_spin(&s_done[g & 1u], (g >> 1) & 1u, kWaitLimitNs)) timed_out = true;
        if (__any_sync(kFull, timed_out)) {  // warp-uniform exit (the loads below are collective)
          timed_out = true;
          break;
        }
        tc_fence_after_sync();
        uint32_t sv[32];
        tc_ld32(t_lane + kTcSCol + 32 * (g & 1u), sv);
        tc_wait_ld();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[g & 1u]);  // the slot may take S(g + 2)

        // tokens of this step that belong to the sequence (and to a valid
        // page), then those this row attends to (its causal limit)
        const int pos0 = t0 + j * kTcTokens;
        const int nvalid = t1 - pos0;
        uint32_t vmask = nvalid >= kTcTokens ? ~0u : ((1u << nvalid) - 1u);
#pragma unroll
        for (int q = 0; q < PPI; ++q)
          if (bad[j * PPI + q]) vmask &= ~((BS == 32 ? ~0u : ((1u << BS) - 1u)) << (q * BS));
        const int nrow = lim - pos0;
        const uint32_t rmask =
            row_ok ? (vmask & (nrow >= kTcTokens ? ~0u : (nrow <= 0 ? 0u : ((1u << nrow) - 1u)))) : 0u;
        // masked maximum of the scaled scores, then p = 2^(s * scale - m)
        float smax = -INFINITY;
#pragma unroll
        for (int k = 0; k < kTcTokens; ++k)
          if ((rmask >> k) & 1u) smax = fmaxf(smax, __uint_as_float(sv[k]) * p.scale_log2);
        const float mnew = fmaxf(m, smax);
        const bool grow = (m == -INFINITY) ? (mnew != -INFINITY) : (mnew > m + 8.f);
        float factor = 1.f;
        if (grow) {
          factor = (m == -INFINITY) ? 0.f : ex2_approx(m - mnew);
          l *= factor;
          m = mnew;
        }
        const float neg_m = (m == -INFINITY) ? 0.f : -m;
        uint32_t pw[kTcTokens / 2];
        float psum = 0.f;
#pragma unroll
        for (int k = 0; k < kTcTokens; k += 2) {
          const float p0 = ((rmask >> k) & 1u) ? ex2_approx(fmaf(__uint_as_float(sv[k]), p.scale_log2, neg_m)) : 0.f;
          const float p1 =
              ((rmask >> (k + 1)) & 1u) ? ex2_approx(fmaf(__uint_as_float(sv[k + 1]), p.scale_log2, neg_m)) : 0.f;
          psum += p0 + p1;
          pw[k / 2] = pack_bf16x2(p0, p1);
        }
        l += psum;
        // a row whose maximum grew: scale its O (TMEM) once P . V(g - 1) is done
        if (j > 0 && __any_sync(kFull, grow)) {
          if (!mbar_wait_spin(&o_done[(g - 1) % kTcStages], ((g - 1) / kTcStages) & 1u, kWaitLimitNs))
            timed_out = true;
          tc_fence_after_sync();
#pragma unroll 1
          for (int c = 0; c < D; c += 32) {
            uint32_t ov[32];
            tc_ld32(t_lane + kTcOCol + c, ov);
            tc_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * factor);
            tc_st32(t_lane + kTcOCol + c, ov);
          }
          tc_wait_st();
        }
        // V rows of tokens outside the sequence (or of a bad page) may hold
        // anything (even NaN) and P is 0 there: once V(g) has landed, warp w
        // clears 16-byte d-chunks 4w .. 4w+3 of those rows (lane = token).
        if (vmask != ~0u) {
          if (!mbar_wait_bounded(&full_v[g % kTcStages], (g / kTcStages) & 1u, kWaitLimitNs)) timed_out = true;
          if (__any_sync(kFull, timed_out)) {
            timed_out = true;
            break;
          }
          uint8_t* vb = st + TcLayout::kTile;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int k = lane;           // token row
            const int dc = 4 * warp + i;  // 16-byte d-chunk
            if (!((vmask >> k) & 1u))
              *reinterpret_cast<uint4*>(vb + (dc >> 3) * TcLayout::kRegion + k * 128 +
                                        (((dc & 7) ^ (k & 7)) << 4)) = make_uint4(0, 0, 0, 0);
          }
        }
        // P row -> buffer g % 2 (K-major core matrices), free once P . V(g - 2) is done
        if (j >= 2 && !mbar_wait_spin(&o_done[(g - 2) % kTcStages], ((g - 2) / kTcStages) & 1u, kWaitLimitNs))
          timed_out = true;
        uint8_t* pbuf = sm + TcLayout::kP + (g & 1u) * TcLayout::kPBuf;
#pragma unroll
        for (int k8 = 0; k8 < kTcTokens / 8; ++k8)
          *reinterpret_cast<uint4*>(pbuf + tc_core_off(tid, k8)) =
              make_uint4(pw[4 * k8], pw[4 * k8 + 1], pw[4 * k8 + 2], pw[4 * k8 + 3]);
        fence_proxy_async_smem();  // P and the cleared V rows are read by the tensor cores
        tc_fence_before_sync();
        mbar_arrive(&p_ready[g & 1u]);
      }
      // the unit's last P . V, then this row's output; every lane loads
      // (tcgen05.ld is warp-collective), rows without a query token write nothing
      const uint32_t gl = g0 + nsteps - 1;
      if (!timed_out && !mbar_wait_spin(&o_done[gl % kTcStages], (gl / kTcStages) & 1u, kWaitLimitNs))
        timed_out = true;
      tc_fence_after_sync();
      const bool direct = nparts == 1;
      if (!__any_sync(kFull, timed_out)) {
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const size_t slot = qrow * p.pmax + pidx;
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t ov[32];
        tc_ld32(t_lane + kTcOCol + c, ov);
        tc_wait_ld();
        if (row_ok && direct) {
          __nv_bfloat16* o = p.out + qrow * D + c;
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(ov[e]) * inv, __uint_as_float(ov[e + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(ov[e + 2]) * inv, __uint_as_float(ov[e + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(ov[e + 4]) * inv, __uint_as_float(ov[e + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(ov[e + 6]) * inv, __uint_as_float(ov[e + 7]) * inv);
            *reinterpret_cast<uint4*>(o + e) = w;
          }
        } else if (row_ok) {
          float* o = p.part_o + slot * D + c;
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(o + e) = make_float4(__uint_as_float(ov[e]), __uint_as_float(ov[e + 1]),
                                                            __uint_as_float(ov[e + 2]), __uint_as_float(ov[e + 3]));
        }
      }
      if (row_ok && !direct) *reinterpret_cast<float2*>(p.part_ml + 2 * slot) = make_float2(m, l);
      } else {
        timed_out = true;
      }
    }
    g0 += static_cast<uint32_t>(nsteps);
    cur ^= 1;
    tc_fence_before_sync();
    if (__syncthreads_or(timed_out)) {  // the unit is done in every role
      timed_out = true;
      break;
    }
    tc_fence_after_sync();
  }

  if (timed_out) {
    if (tid == 0) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
    // each role lets its own copies and products still in flight finish
    // (bounded) before the shared and tensor memory are released: the last
    // three steps' copies (one per stage, so one phase per barrier) and the
    // MMA warp's last commits (each covers every earlier product)
    if ((kcopy || vcopy) && lane == 0) {
      uint64_t* fbar = kcopy ? full_k : full_v;
      for (uint32_t g = copies_end > kTcStages ? copies_end - kTcStages : 0; g < copies_end; ++g)
        mbar_wait_bounded(&fbar[g % kTcStages], (g / kTcStages) & 1u, kWaitLimitNs / 16);
    }
    if (mma_warp && lane == 0) {
      if (s_end > 0)
        mbar_wait_bounded(&k_free[(s_end - 1) % kTcStages], ((s_end - 1) / kTcStages) & 1u, kWaitLimitNs / 16);
      if (pv_end > 0)
        mbar_wait_bounded(&o_done[(pv_end - 1) % kTcStages], ((pv_end - 1) / kTcStages) & 1u, kWaitLimitNs / 16);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tc_dealloc(tmem, kTcCols);
}

}  // namespace pkv
