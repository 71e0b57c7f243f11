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
//   * Warp-specialised: a producer warp issues the tensor-map copies (TMA,
//     128-byte swizzle) of each step's K and V pages into a 3-stage ring; an
//     MMA warp issues S = Q . K^T (M 128, N 32, K 128) into TMEM as soon as a
//     step's pages land (the query tile sits in shared memory, 128-byte
//     swizzle, K-major) and O += P . V when the compute warps have P ready;
//     four compute warps own the 128 rows.  The roles hand work over only
//     through mbarriers, so copies, products and softmax of neighbouring
//     steps overlap.
//   * Thread r owns row r: it loads its 32 scores from TMEM, masks them
//     (sequence end, causal limit of its query token), and keeps the online
//     softmax state in registers.  The running maximum is lazy: the output is
//     rescaled only when a row's maximum grows by more than 2^8, so P stays
//     below 256 and the rescale of O in TMEM is rare.  P goes to shared memory
//     as bf16 (K-major, no swizzle).
//   * The page's V is transposed by the threads into the K area of its stage
//     (K-major for the B operand; K is dead once S is done), with rows past
//     the sequence end written as zeros, and one thread issues
//     O += P . V (M 128, N 128, K 32) into TMEM.
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
constexpr int kTcThreads = 32 * (kTcComputeWarps + 2);  // + MMA warp + producer warp
constexpr uint32_t kTcCols = 256;  // TMEM columns: S at 0 and 32 (double buffer), O at 128 (128)
constexpr uint32_t kTcSCol = 0;
constexpr uint32_t kTcOCol = 128;

struct TcLayout {  // byte offsets from the 1024-aligned shared-memory base
  static constexpr uint32_t kQ = 0;                          // 2 x [128 rows x 128 B], 128B swizzle
  static constexpr uint32_t kQRegion = kTcRows * 128;        // 16 KiB
  static constexpr uint32_t kRegion = kTcTokens * 128;       // half (64 of 128 d) of a 32-token tile: 4 KiB
  static constexpr uint32_t kTile = 2 * kRegion;             // a K or V tile: 8 KiB
  static constexpr uint32_t kStage = 2 * kTile;              // K then V: 16 KiB
  static constexpr uint32_t kStages = kQ + 2 * kQRegion;
  static constexpr uint32_t kP = kStages + kTcStages * kStage;  // 2 x [128 x 32] bf16 core-matrix layout
  static constexpr uint32_t kPBuf = kTcRows * kTcTokens * 2;      // 8 KiB
  static constexpr uint32_t kBars = kP + 2 * kPBuf;
  // full[3], s_done[2], p_ready[2], o_done[3]
  static constexpr uint32_t kMisc = kBars + 8 * (kTcStages + 2 + 2 + 3);  // TMEM base, unit
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
__global__ void __launch_bounds__(kTcThreads, 1)
    paged_decode_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                           const __grid_constant__ CUtensorMap vmap, const DecodeParams p) {
  constexpr int D = 128;
  constexpr int PPI = kTcTokens / BS;  // pages per step
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  // Barrier phases are counted over the CTA's lifetime with the global step
  // index g: stage and full[] by g % 3, S buffer and s_done[] / p_ready[] by
  // g % 2, o_done[] by g % 3.  Every barrier completes one phase per use and
  // no waiter can fall two phases behind (each next use depends on the wait).
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + TcLayout::kBars);  // [3] copies landed
  uint64_t* s_done = full + kTcStages;                                  // [2] S(g) in TMEM
  uint64_t* p_ready = s_done + 2;                                       // [2] P(g), V^T(g) in smem
  uint64_t* o_done = p_ready + 2;                                       // [3] P . V(g) done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + TcLayout::kMisc);
  volatile int* desc = reinterpret_cast<volatile int*>(sm + TcLayout::kDesc);  // [2][8]
  int* pages = reinterpret_cast<int*>(sm + TcLayout::kPages);
  uint8_t* bad = sm + TcLayout::kBad;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const bool compute = warp < kTcComputeWarps;
  const bool mma_warp = warp == kTcComputeWarps;
  const bool producer = warp == kTcComputeWarps + 1;

  if (tid == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&o_done[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_done[s], 1);
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
  const uint32_t q_addr = smem_addr(sm + TcLayout::kQ);
  constexpr uint32_t kIdescS = tc_idesc_bf16_f32(kTcRows, kTcTokens);
  constexpr uint32_t kIdescO = tc_idesc_bf16_f32(kTcRows, D);
  pdl_trigger();
  pdl_wait();

  const int units_per_part = p.Hkv * p.NT;
  const int total_units = p.unit_start[p.B] * units_per_part;
  const int ppu_tokens = p.ppu * BS;
  uint32_t g0 = 0;  // global index of the current unit's first step
  bool timed_out = false;

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
    if (compute) {
      const uint4* src = reinterpret_cast<const uint4*>(p.q + qrow * D);
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const uint4 w = row_ok ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
        const uint32_t off = TcLayout::kQ + (c >> 3) * TcLayout::kQRegion +
                             static_cast<uint32_t>(tid * 128 + (((c & 7) ^ (tid & 7)) << 4));
        *reinterpret_cast<uint4*>(sm + off) = w;
      }
      fence_proxy_async_smem();  // the query tile is read by the tensor cores
    }
    const int lim = ctx - p.T + 1 + t;  // keys of this row: positions < lim
    tc_fence_before_sync();
    __syncthreads();  // page ids and the query tile are in place
    tc_fence_after_sync();

    if (producer) {
      // step j's K and V pages into stage (g0 + j) % 3, once P . V of the step
      // that last used the stage (g0 + j - 3) is done; lane 4q + 2h + kv issues
      // the copy of half h of K (kv 0) or V (kv 1) of the step's page q.
      // After the first copies are on their way, lane 0 fetches the next unit.
      for (int j = 0; j < nsteps; ++j) {
        if (j == kTcStages && lane == 0) fetch_unit(cur ^ 1);
        const uint32_t g = g0 + j;
        int ok = 1;
        if (lane == 0 && g >= kTcStages)
          ok = mbar_wait_spin(&o_done[g % kTcStages], ((g - kTcStages) / kTcStages) & 1u, kWaitLimitNs) ? 1 : 0;
        if (!__shfl_sync(kFull, ok, 0)) {
          timed_out = true;
          break;
        }
        uint8_t* st = sm + TcLayout::kStages + (g % kTcStages) * TcLayout::kStage;
        uint64_t* bar = &full[g % kTcStages];
        const int np = min(PPI, npages - j * PPI);
        if (lane == 0) {
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(bar, static_cast<uint32_t>(np) * 4u * 64u * BS * 2u);
        }
        __syncwarp();
        if (lane < 4 * np) {
          const int q = lane >> 2, half = (lane >> 1) & 1, kv = lane & 1;
          const int row = p.row_base + (pages[j * PPI + q] * p.Hkv + kvh) * BS;
          tma_load_2d(st + kv * TcLayout::kTile + half * TcLayout::kRegion + q * BS * 128, kv ? &vmap : &kmap, bar,
                      half * 64, row, policy);
        }
      }
      if (nsteps <= kTcStages && lane == 0 && !timed_out) fetch_unit(cur ^ 1);
      __syncwarp();
    } else if (mma_warp) {
      if (lane == 0) {
        auto issue_pv = [&](uint32_t g) {  // O += P(g) . V(g)
          const uint32_t k_addr = smem_addr(sm + TcLayout::kStages + (g % kTcStages) * TcLayout::kStage);
          const uint32_t pa = smem_addr(sm + TcLayout::kP + (g & 1u) * TcLayout::kPBuf);
          tc_fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < kTcTokens / 16; ++kk) {
            const uint64_t a = tc_smem_desc(pa + kk * 256, 128, 512, 0);
            const uint64_t bdesc = tc_smem_desc(k_addr + kk * 256, 128, 512, 0);
            tc_mma_bf16(tmem + kTcOCol, a, bdesc, kIdescO, g > g0 || kk > 0);
          }
          tc_commit(&o_done[g % kTcStages]);
        };
        for (int j = 0; j <= nsteps && !timed_out; ++j) {
          const uint32_t g = g0 + j;
          if (j < nsteps) {
            // S(g): its pages have landed; its TMEM buffer was read by the
            // compute warps before they signalled P(g - 2) (waited below)
            if (!mbar_wait_bounded(&full[g % kTcStages], (g / kTcStages) & 1u, kWaitLimitNs)) {
              timed_out = true;
              break;
            }
            const uint32_t k_addr = smem_addr(sm + TcLayout::kStages + (g % kTcStages) * TcLayout::kStage);
            tc_fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t koff = static_cast<uint32_t>((kk & 3) * 32);  // 16 d = 32 bytes along the row
              const uint64_t a = tc_smem_desc(q_addr + (kk >> 2) * TcLayout::kQRegion + koff, 16, 1024, 2);
              const uint64_t bdesc = tc_smem_desc(k_addr + (kk >> 2) * TcLayout::kRegion + koff, 16, 1024, 2);
              tc_mma_bf16(tmem + kTcSCol + 32 * (g & 1u), a, bdesc, kIdescS, kk > 0);
            }
            tc_commit(&s_done[g & 1u]);
          }
          if (j > 0) {  // P . V of the previous step once its P and V^T are in place
            const uint32_t gp = g - 1;
            if (!mbar_wait_spin(&p_ready[gp & 1u], (gp >> 1) & 1u, kWaitLimitNs)) {
              timed_out = true;
              break;
            }
            issue_pv(gp);
          }
        }
      }
      __syncwarp();
    } else {
      // compute warps: one row each
      float m = -INFINITY, l = 0.f;  // log2-domain running max (lazy) and sum of this row
      for (int j = 0; j < nsteps; ++j) {
        const uint32_t g = g0 + j;
        uint8_t* st = sm + TcLayout::kStages + (g % kTcStages) * TcLayout::kStage;
        const uint32_t k_addr = smem_addr(st);
        if (!mbar_wait_spin(&s_done[g & 1u], (g >> 1) & 1u, kWaitLimitNs)) timed_out = true;
        if (__any_sync(kFull, timed_out)) {  // warp-uniform exit (the loads below are collective)
          timed_out = true;
          break;
        }
        tc_fence_after_sync();
        uint32_t sv[32];
        tc_ld32(t_lane + kTcSCol + 32 * (g & 1u), sv);
        tc_wait_ld();

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
        // V^T -> the stage's K area (K is spent once S is done): warp w moves
        // the 8x8 blocks of d-chunks 4w .. 4w+3 with ldmatrix from the swizzled
        // page and a transposing stmatrix.  Rows of tokens outside the
        // sequence (or of a bad page) may hold anything (even NaN) and P is 0
        // there, so this warp's chunks of them are cleared first.
        if (!mbar_wait_bounded(&full[g % kTcStages], (g / kTcStages) & 1u, kWaitLimitNs)) timed_out = true;
        if (__any_sync(kFull, timed_out)) {
          timed_out = true;
          break;
        }
        {
          const uint32_t v_base = k_addr + TcLayout::kTile;
          if (vmask != ~0u) {
            uint8_t* vb = st + TcLayout::kTile;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int k = lane;           // token row
              const int dc = 4 * warp + i;  // 16-byte d-chunk
              if (!((vmask >> k) & 1u))
                *reinterpret_cast<uint4*>(vb + (dc >> 3) * TcLayout::kRegion + k * 128 +
                                          (((dc & 7) ^ (k & 7)) << 4)) = make_uint4(0, 0, 0, 0);
            }
            __syncwarp();
          }
          const int dc = 4 * warp + (lane >> 3);
#pragma unroll
          for (int q = 0; q < kTcTokens / 8; ++q) {
            const int k = 8 * q + (lane & 7);
            uint32_t r0, r1, r2, r3;
            ldsm_x4(v_base + (dc >> 3) * TcLayout::kRegion + k * 128 + (((dc & 7) ^ (k & 7)) << 4), r0, r1, r2, r3);
            stsm_x4_t(k_addr + tc_core_off(8 * dc + (lane & 7), q), r0, r1, r2, r3);
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
        fence_proxy_async_smem();  // P and V^T are read by the tensor cores
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
    // copies and products still in flight finish (bounded) before the shared
    // and tensor memory are released
    if (tid == 0) {
      for (int k = 0; k < kTcStages; ++k) {
        if (g0 + k < kTcStages) continue;
        const uint32_t g = g0 + k - kTcStages;  // the last use of each stage
        mbar_wait_bounded(&full[g % kTcStages], (g / kTcStages) & 1u, kWaitLimitNs / 16);
        mbar_wait_bounded(&o_done[g % kTcStages], (g / kTcStages) & 1u, kWaitLimitNs / 16);
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tc_dealloc(tmem, kTcCols);
}

}  // namespace pkv
