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
//   * K and V pages arrive by tensor-map copies (TMA, 128-byte swizzle) in a
//     3-stage ring; one thread issues S = Q . K^T (M 128, N 32, K 128) into
//     TMEM with the query tile in shared memory (128-byte swizzle, K-major).
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
constexpr int kTcThreads = 128;
constexpr uint32_t kTcCols = 256;  // TMEM columns: S at 0 (32), O at 128 (128)
constexpr uint32_t kTcSCol = 0;
constexpr uint32_t kTcOCol = 128;

struct TcLayout {  // byte offsets from the 1024-aligned shared-memory base
  static constexpr uint32_t kQ = 0;                          // 2 x [128 rows x 128 B], 128B swizzle
  static constexpr uint32_t kQRegion = kTcRows * 128;        // 16 KiB
  static constexpr uint32_t kRegion = kTcTokens * 128;       // half (64 of 128 d) of a 32-token tile: 4 KiB
  static constexpr uint32_t kTile = 2 * kRegion;             // a K or V tile: 8 KiB
  static constexpr uint32_t kStage = 2 * kTile;              // K then V: 16 KiB
  static constexpr uint32_t kStages = kQ + 2 * kQRegion;
  static constexpr uint32_t kP = kStages + kTcStages * kStage;  // [128 x 32] bf16 core-matrix layout
  static constexpr uint32_t kBars = kP + kTcRows * kTcTokens * 2;
  static constexpr uint32_t kMisc = kBars + 8 * (kTcStages + 2);  // TMEM base, unit, abort
  static constexpr uint32_t kPages = kMisc + 16;              // int32 physical ids of the unit's pages
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
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + TcLayout::kBars);
  uint64_t* s_done = full + kTcStages;
  uint64_t* o_done = s_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + TcLayout::kMisc);
  volatile int* unit_slot = reinterpret_cast<volatile int*>(sm + TcLayout::kMisc + 4);
  int* pages = reinterpret_cast<int*>(sm + TcLayout::kPages);
  uint8_t* bad = sm + TcLayout::kBad;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;

  if (tid == 0) {
    for (int s = 0; s < kTcStages; ++s) mbar_init(&full[s], 1);
    mbar_init(s_done, 1);
    mbar_init(o_done, 1);
    fence_mbar_init();
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
  }
  if (warp == 0) tc_alloc(tmem_slot, kTcCols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_lane = tmem + (static_cast<uint32_t>(warp * 32) << 16);  // this warp's 32 lanes
  const uint64_t policy = p.NT > 1 ? l2_policy_evict_normal() : l2_policy_evict_first();
  const uint32_t q_addr = smem_addr(sm + TcLayout::kQ);
  const uint32_t p_addr = smem_addr(sm + TcLayout::kP);
  constexpr uint32_t kIdescS = tc_idesc_bf16_f32(kTcRows, kTcTokens);
  constexpr uint32_t kIdescO = tc_idesc_bf16_f32(kTcRows, D);
  pdl_trigger();
  pdl_wait();

  const int units_per_part = p.Hkv * p.NT;
  const int total_units = p.unit_start[p.B] * units_per_part;
  const int ppu_tokens = p.ppu * BS;
  uint32_t git = 0;    // steps this CTA has started (ring stage git % 3)
  uint32_t sdone = 0;  // S products completed so far
  uint32_t odone = 0;  // P.V products committed so far
  bool timed_out = false;
  int outstanding = 0;  // thread 0: copies issued and not yet consumed

  for (;;) {
    if (tid == 0) *unit_slot = atomicAdd(p.work_counter, 1);
    __syncthreads();
    const int u = *unit_slot;
    __syncthreads();
    if (u >= total_units) break;
    const int part = u / units_per_part;
    const int rem = u - part * units_per_part;
    const int kvh = rem / p.NT;
    const int tile = rem - kvh * p.NT;
    int lo = 0, hi = p.B;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(p.unit_start + mid) <= part) lo = mid; else hi = mid;
    }
    const int b = lo;
    const int pidx = part - __ldg(p.unit_start + b);
    const int nparts = __ldg(p.unit_start + b + 1) - __ldg(p.unit_start + b);
    const int ctx = __ldg(p.ctx_eff + b);
    const int t0 = pidx * ppu_tokens;
    const int t1 = min(ctx, t0 + ppu_tokens);
    const int npages = (t1 - t0 + BS - 1) / BS;  // <= 64
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
    // this thread's query row: token t of the tile, head h
    int t, h;
    const bool row_ok = tile_row<true>(p, kvh, tile, tid, t, h);
    const size_t qrow = static_cast<size_t>(b * p.T + (row_ok ? t : 0)) * p.Hq + (row_ok ? h : 0);
    {
      const uint4* src = reinterpret_cast<const uint4*>(p.q + qrow * D);
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const uint4 w = row_ok ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
        const uint32_t off = TcLayout::kQ + (c >> 3) * TcLayout::kQRegion +
                             static_cast<uint32_t>(tid * 128 + (((c & 7) ^ (tid & 7)) << 4));
        *reinterpret_cast<uint4*>(sm + off) = w;
      }
    }
    const int lim = ctx - p.T + 1 + (row_ok ? t : 0);  // keys of this row: positions < lim
    fence_proxy_async_smem();  // the query tile is read by the tensor cores
    __syncthreads();           // page ids and the query tile are in place

    auto issue_step = [&](int step, uint32_t g) {  // thread 0: the step's K and V pages into stage g % 3
      uint8_t* st = sm + TcLayout::kStages + (g % kTcStages) * TcLayout::kStage;
      uint64_t* bar = &full[g % kTcStages];
      const int np = min(PPI, npages - step * PPI);
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(np) * 4u * 64u * BS * 2u);
      for (int q = 0; q < np; ++q) {
        const int row = p.row_base + (pages[step * PPI + q] * p.Hkv + kvh) * BS;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          tma_load_2d(st + half * TcLayout::kRegion + q * BS * 128, &kmap, bar, half * 64, row, policy);
          tma_load_2d(st + TcLayout::kTile + half * TcLayout::kRegion + q * BS * 128, &vmap, bar, half * 64, row,
                      policy);
        }
      }
    };
    if (tid == 0) {
      for (int k = 0; k < min(kTcStages, nsteps); ++k) issue_step(k, git + k);
      outstanding = min(kTcStages, nsteps);
    }

    float m = -INFINITY, l = 0.f;  // log2-domain running max (lazy) and sum of this row
    for (int step = 0; step < nsteps; ++step, ++git) {
      const uint32_t sidx = git % kTcStages;
      uint8_t* st = sm + TcLayout::kStages + sidx * TcLayout::kStage;
      const uint32_t k_addr = smem_addr(st);
      if (!mbar_wait_bounded(&full[sidx], (git / kTcStages) & 1u, kWaitLimitNs)) timed_out = true;
      if (tid == 0) {
        --outstanding;
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = static_cast<uint32_t>((kk & 3) * 32);  // 16 d = 32 bytes along the row
          const uint64_t a = tc_smem_desc(q_addr + (kk >> 2) * TcLayout::kQRegion + koff, 16, 1024, 2);
          const uint64_t bdesc = tc_smem_desc(k_addr + (kk >> 2) * TcLayout::kRegion + koff, 16, 1024, 2);
          tc_mma_bf16(tmem + kTcSCol, a, bdesc, kIdescS, kk > 0);
        }
        tc_commit(s_done);
      }
      if (!mbar_wait_bounded(s_done, sdone & 1u, kWaitLimitNs)) timed_out = true;
      ++sdone;
      tc_fence_after_sync();
      uint32_t sv[32];
      tc_ld32(t_lane + kTcSCol, sv);
      tc_wait_ld();

      // scores of this row: masked, log2 domain
      const int pos0 = t0 + step * kTcTokens;
      float sc[kTcTokens];
      float smax = -INFINITY;
#pragma unroll
      for (int k = 0; k < kTcTokens; ++k) {
        const int pos = pos0 + k;
        const bool ok = row_ok && pos < t1 && pos < lim && !bad[step * PPI + k / BS];
        sc[k] = ok ? __uint_as_float(sv[k]) * p.scale_log2 : -INFINITY;
        smax = fmaxf(smax, sc[k]);
      }
      const float mnew = fmaxf(m, smax);
      const bool grow = (m == -INFINITY) ? (mnew != -INFINITY) : (mnew > m + 8.f);
      float factor = 1.f;
      if (grow) {
        factor = (m == -INFINITY) ? 0.f : ex2_approx(m - mnew);
        l *= factor;
        m = mnew;
      }
      uint32_t pw[kTcTokens / 2];
      float psum = 0.f;
#pragma unroll
      for (int k = 0; k < kTcTokens; k += 2) {
        const float p0 = (m == -INFINITY) ? 0.f : ex2_approx(sc[k] - m);
        const float p1 = (m == -INFINITY) ? 0.f : ex2_approx(sc[k + 1] - m);
        psum += p0 + p1;
        pw[k / 2] = pack_bf16x2(p0, p1);
      }
      l += psum;

      // the previous step's P . V is done: P, O and that step's stage are free
      if (step > 0) {
        if (!mbar_wait_bounded(o_done, (odone - 1) & 1u, kWaitLimitNs)) timed_out = true;
        tc_fence_after_sync();
        if (tid == 0 && step + 2 < nsteps) {
          issue_step(step + 2, git + 2);
          ++outstanding;
        }
        if (__any_sync(kFull, grow)) {  // rescale this warp's rows of O (lanes that did not grow: x1)
#pragma unroll 1
          for (int c = 0; c < D; c += 32) {
            uint32_t ov[32];
            tc_ld32(t_lane + kTcOCol + c, ov);
            tc_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * factor);
            tc_st32(t_lane + kTcOCol + c, ov);
          }
          tc_wait_st();
        }
      }
      // P row -> shared memory (K-major core matrices)
#pragma unroll
      for (int k8 = 0; k8 < kTcTokens / 8; ++k8)
        *reinterpret_cast<uint4*>(sm + TcLayout::kP + tc_core_off(tid, k8)) =
            make_uint4(pw[4 * k8], pw[4 * k8 + 1], pw[4 * k8 + 2], pw[4 * k8 + 3]);
      // V^T (row d = tid, 32 tokens) -> the stage's K area; tokens past the
      // sequence end, or of a bad page, are zeros
      {
        const uint8_t* vb = st + TcLayout::kTile + (tid >> 6) * TcLayout::kRegion;
        const int dc = (tid & 63) >> 3, de = tid & 7;
#pragma unroll
        for (int k8 = 0; k8 < kTcTokens / 8; ++k8) {
          uint32_t w[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t pair = 0;
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
              const int k = 8 * k8 + 2 * j + e2;
              const bool ok = pos0 + k < t1 && !bad[step * PPI + k / BS];
              const uint16_t v = ok ? *reinterpret_cast<const uint16_t*>(vb + k * 128 + ((dc ^ (k & 7)) << 4) + de * 2)
                                    : static_cast<uint16_t>(0);
              pair |= static_cast<uint32_t>(v) << (16 * e2);
            }
            w[j] = pair;
          }
          *reinterpret_cast<uint4*>(st + tc_core_off(tid, k8)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      fence_proxy_async_smem();  // P and V^T are read by the tensor cores
      tc_fence_before_sync();
      if (__syncthreads_or(timed_out)) {
        timed_out = true;
        break;
      }
      tc_fence_after_sync();
      if (tid == 0) {
#pragma unroll
        for (int kk = 0; kk < kTcTokens / 16; ++kk) {
          const uint64_t a = tc_smem_desc(p_addr + kk * 256, 128, 512, 0);
          const uint64_t bdesc = tc_smem_desc(k_addr + kk * 256, 128, 512, 0);
          tc_mma_bf16(tmem + kTcOCol, a, bdesc, kIdescO, step > 0 || kk > 0);
        }
        tc_commit(o_done);
      }
      ++odone;
    }
    if (timed_out) break;

    // the unit's last P . V (a unit has at least one page), then this row's output
    if (!mbar_wait_bounded(o_done, (odone - 1) & 1u, kWaitLimitNs)) timed_out = true;
    tc_fence_after_sync();
    if (__syncthreads_or(timed_out)) {
      timed_out = true;
      break;
    }
    // every lane of a warp loads (tcgen05.ld is warp-collective); rows
    // without a query token write nothing
    {
      const bool direct = nparts == 1;
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
          for (int j = 0; j < 32; j += 8) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(ov[j]) * inv, __uint_as_float(ov[j + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(ov[j + 2]) * inv, __uint_as_float(ov[j + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(ov[j + 4]) * inv, __uint_as_float(ov[j + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(ov[j + 6]) * inv, __uint_as_float(ov[j + 7]) * inv);
            *reinterpret_cast<uint4*>(o + j) = w;
          }
        } else if (row_ok) {
          float* o = p.part_o + slot * D + c;
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(o + j) = make_float4(__uint_as_float(ov[j]), __uint_as_float(ov[j + 1]),
                                                            __uint_as_float(ov[j + 2]), __uint_as_float(ov[j + 3]));
        }
      }
      if (row_ok && !direct) *reinterpret_cast<float2*>(p.part_ml + 2 * slot) = make_float2(m, l);
    }
    tc_fence_before_sync();
    __syncthreads();  // every row's O is read before the next unit's products
    tc_fence_after_sync();
  }

  if (timed_out) {
    if (tid == 0) {
      atomicOr(p.err, PKV_DEVERR_TIMEOUT);
      // copies still in flight land before the shared memory is released
      for (int k = 0; k < outstanding; ++k) {
        const uint32_t g = git + 1 + static_cast<uint32_t>(k);
        mbar_wait_bounded(&full[g % kTcStages], (g / kTcStages) & 1u, kWaitLimitNs / 16);
      }
      // and the last products issued finish before the tensor memory is freed
      if (sdone > 0) mbar_wait_bounded(s_done, (sdone - 1) & 1u, kWaitLimitNs / 16);
      if (odone > 0) mbar_wait_bounded(o_done, (odone - 1) & 1u, kWaitLimitNs / 16);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tc_dealloc(tmem, kTcCols);
}

}  // namespace pkv
