// Multi-token decode for long query windows on the 5th-generation tensor
// cores: one CTA serves TWO row tiles of the same KV head and reads each K/V
// page once for both (bf16 cache, head_dim 128).
//
// With T x G > 128 (query token, head) rows per KV head -- verification of
// long draft windows ("KV-Cache Engineering: Paged Attention, Prefix Cache,
// Disaggregation (2026)": speculative decoding checks the draft's tokens in
// one pass over the shared cache) and chunked prefill ("KV Cache
// Engineering: PagedAttention, Continuous Batching, Attention Variants, and
// the Bandwidth Wall", "Continuous Batching") -- the rows of a KV head form
// several 128-row tiles.  Streaming each tile separately re-reads the pages
// once per tile and leaves the tensor pipe idle while a tile's softmax runs.
// Here one CTA per SM holds a pair of tiles:
//
//   * tensor memory (all 512 columns): S0, S1 (128 fp32 columns each: the
//     scores of 128 tokens) and O0, O1 (128 fp32 columns each); the query
//     tiles Q0, Q1 sit in shared memory (tensor-map copies, 128-byte
//     swizzle), and each tile's softmax weights P (bf16) are written back
//     into the first 64 columns of its own S, where the P . V product reads
//     them as its A operand;
//   * 128-token steps, so that S = Q . K^T is one N = 128 product per k
//     slice (a tcgen05.mma of M 128 costs the same up to N 128);
//   * one MMA thread issues, per step g, PV0(g-1) S0(g) PV1(g-1) S1(g): the
//     tensor pipe works on one tile while the other tile's softmax runs
//     (ping-pong), and tcgen05 operations of one thread execute in issue
//     order, so S_i(g) overwrites P_i(g-1) only after PV_i(g-1) has read it;
//   * eight softmax warps, four per tile, one row per thread.  A tile's
//     softmax, not the tensor pipe, sets the pace (each round trip to tensor
//     memory, a tcgen05.ld and its wait, costs ~250-300 cycles under load:
//     measured with clock stamps), so a thread loads its row's 128 scores
//     with one round trip and keeps them in registers; its P (bf16 pairs)
//     goes over the first 64 columns of S;
//   * a K copy warp (unit descriptors and K pages) and a V copy warp (query
//     tiles and V pages) fill two-stage rings of 32 KiB; each softmax thread
//     writes its row of the output (or of the split-K partials) straight
//     from registers.
//
// The softmax keeps a lazy running maximum per row (the output is rescaled
// only when a row's maximum grows by more than 2^8, so P < 256), masks the
// sequence end, bad pages and the row's causal limit, and clears the V rows
// of tokens outside the sequence (they may hold anything, even NaN, while P
// is 0 there).  Units are (sequence, KV head, tile pair, partition) from the
// planner's counter; the merge kernels combine partitions.  Every wait is
// bounded; a CTA that gives up records PKV_DEVERR_TIMEOUT, lets its own
// copies and products finish (bounded) and frees its tensor memory.
#pragma once

#include "paged_decode_tc.cuh"

namespace pkv {

constexpr int kT2Rows = 128;     // query rows per tile (MMA M)
constexpr int kT2Tokens = 128;   // tokens per step (N of S, K of P . V)
constexpr int kT2Stages = 2;     // K ring and V ring
constexpr int kT2SoftWarps = 8;  // four per tile, one per 32-row quarter
constexpr int kT2Threads = 32 * (kT2SoftWarps + 3);  // + MMA warp + K copy warp + V copy warp
constexpr uint32_t kT2Cols = 512;  // S0 0, S1 128, O0 256, O1 384

struct T2Layout {  // byte offsets from the 1024-aligned shared-memory base
  static constexpr uint32_t kRegion = kT2Tokens * 128;     // 64 of 128 d of 128 rows: 16 KiB
  static constexpr uint32_t kTile = 2 * kRegion;           // a query tile, or a step's K or V: 32 KiB
  static constexpr uint32_t kQ = 0;                        // Q0, Q1
  static constexpr uint32_t kK = kQ + 2 * kTile;           // K ring
  static constexpr uint32_t kV = kK + kT2Stages * kTile;   // V ring
  static constexpr uint32_t kBars = kV + kT2Stages * kTile;
  // k_full[2] k_free[2] v_full[2] v_free[2] s_full[2] p_full[2] o_free[2]
  // o_full[2] slot_full[2] slot_free[2] q_full q_free mma_drain
  static constexpr int kNumBars = 10 * 2 + 3;
  static constexpr uint32_t kMisc = kBars + 8 * kNumBars;  // TMEM base
  static constexpr uint32_t kSlots = kMisc + 16;           // 2 unit slots
  static constexpr uint32_t kSlotPages = 32;               // after 8 int32 of descriptor
  static constexpr uint32_t kSlotBad = kSlotPages + 4 * kTcMaxPages;
  static constexpr uint32_t kSlot = kSlotBad + kTcMaxPages;
  static constexpr uint32_t kEnd = kSlots + 2 * kSlot;
};

__host__ __device__ constexpr size_t tc2_smem_layout_bytes() { return 1024 + T2Layout::kEnd; }

// L2 prefetch of a tensor-map box (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_4d(const CUtensorMap* map, int32_t c0, int32_t c1, int32_t c2,
                                                int32_t c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}

// 4-D tiled copy global -> shared (the query tiles).
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar, int32_t c0,
                                            int32_t c1, int32_t c2, int32_t c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_addr(bar))
      : "memory");
}

// Maximum (kMax) or minimum of 32 scores (bit patterns of floats): a tree
// of three-input operations.
template <bool kMax>
__device__ __forceinline__ float tree_ext32(const uint32_t (&v)[32]) {
  auto op3 = [](float a, float b, float c) { return kMax ? fmax3f(a, b, c) : fmin3f(a, b, c); };
  float t[11];
#pragma unroll
  for (int i = 0; i < 10; ++i)
    t[i] = op3(__uint_as_float(v[3 * i]), __uint_as_float(v[3 * i + 1]), __uint_as_float(v[3 * i + 2]));
  t[10] = kMax ? fmaxf(__uint_as_float(v[30]), __uint_as_float(v[31]))
               : fminf(__uint_as_float(v[30]), __uint_as_float(v[31]));
  const float u0 = op3(t[0], t[1], t[2]), u1 = op3(t[3], t[4], t[5]), u2 = op3(t[6], t[7], t[8]);
  const float w = op3(u0, u1, u2);
  return op3(w, t[9], t[10]);
}

// tcgen05.wait::ld that also names the loaded registers, so that the
// compiler cannot move their uses above the wait.
__device__ __forceinline__ void tc_wait_ld_regs(uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]), "+r"(v[7]),
        "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]), "+r"(v[14]), "+r"(v[15]),
        "+r"(v[16]), "+r"(v[17]), "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]), "+r"(v[22]), "+r"(v[23]),
        "+r"(v[24]), "+r"(v[25]), "+r"(v[26]), "+r"(v[27]), "+r"(v[28]), "+r"(v[29]), "+r"(v[30]), "+r"(v[31])
      :
      : "memory");
}
// After a tcgen05.wait::ld (which covers every earlier tcgen05.ld of the
// thread): ties more loaded registers to that point without another wait.
__device__ __forceinline__ void tc_regs_loaded(uint32_t (&v)[32]) {
  asm volatile(""
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]), "+r"(v[7]),
                 "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]), "+r"(v[14]),
                 "+r"(v[15]), "+r"(v[16]), "+r"(v[17]), "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]),
                 "+r"(v[22]), "+r"(v[23]), "+r"(v[24]), "+r"(v[25]), "+r"(v[26]), "+r"(v[27]), "+r"(v[28]),
                 "+r"(v[29]), "+r"(v[30]), "+r"(v[31])
               :
               : "memory");
}
__device__ __forceinline__ void tc_wait_ld_regs16(uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]), "+r"(v[7]),
        "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]), "+r"(v[14]), "+r"(v[15])
      :
      : "memory");
}

template <int BS>
__global__ void __launch_bounds__(kT2Threads, 1)
    paged_decode_tc2_kernel(const __grid_constant__ CUtensorMap kmap,
                            const __grid_constant__ CUtensorMap vmap,
                            const __grid_constant__ CUtensorMap qmap,  // q [B][T][Hq][D], box 64 x G x Tt
                            const DecodeParams p) {
  constexpr int D = 128;
  constexpr int PPI = kT2Tokens / BS;  // pages per step
  static_assert(kTcMaxPages % PPI == 0, "");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  // Barrier phases: k/v rings by the global step g (stage g % 2, phase
  // (g / 2) & 1); s_full[] / p_full[] once per step; q_full, q_free,
  // o_full, o_free[] once per unit; the slot ring by the unit index.  Each
  // next use of a barrier depends on the wait for its previous phase, so no
  // waiter is ever two phases behind.
  uint64_t* k_full = reinterpret_cast<uint64_t*>(sm + T2Layout::kBars);
  uint64_t* k_free = k_full + 2;     // S0(g), S1(g) done: K stage free
  uint64_t* v_full = k_free + 2;
  uint64_t* v_free = v_full + 2;     // PV0(g), PV1(g) done: V stage free
  uint64_t* s_full = v_free + 2;     // [tile] S_i(g) (and everything issued before) done
  uint64_t* p_full = s_full + 2;     // [tile] P_i(g) in TMEM, V(g) stale rows cleared
  uint64_t* o_free = p_full + 2;     // [tile] the unit's O_i read out by its softmax warps
  uint64_t* o_full = o_free + 2;     // [tile] the unit's last PV_i done
  uint64_t* slot_full = o_full + 2;
  uint64_t* slot_free = slot_full + 2;
  uint64_t* q_full = slot_free + 2;  // both query tiles landed
  uint64_t* q_free = q_full + 1;     // the unit's last S0 and S1 done: Q may be replaced
  uint64_t* mma_drain = q_free + 1;  // after a timeout: every product issued is done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + T2Layout::kMisc);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const bool mma_warp = warp == kT2SoftWarps;
  const bool kcopy = warp == kT2SoftWarps + 1;
  const bool vcopy = warp == kT2SoftWarps + 2;

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_free[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_free[s], 1);
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], kT2Rows);
      mbar_init(&o_free[s], 4);                        // one lane per softmax warp of the tile
      mbar_init(&o_full[s], 1);
      mbar_init(&slot_full[s], 1);
      mbar_init(&slot_free[s], kT2SoftWarps + 2);      // softmax warps, MMA warp, V copy warp
    }
    mbar_init(q_full, 1);
    mbar_init(q_free, 1);
    mbar_init(mma_drain, 1);
    fence_mbar_init();
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
    prefetch_tensormap(&qmap);
  }
  if (warp == 0) tc_alloc(tmem_slot, kT2Cols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint64_t policy = l2_policy_evict_normal();  // the pairs of a KV head read the same pages
  constexpr uint32_t kIdescS = tc_idesc_bf16_f32(kT2Rows, kT2Tokens);
  constexpr uint32_t kIdescO = tc_idesc_bf16_f32(kT2Rows, D, /*b_mn_major=*/true);
  pdl_trigger();
  pdl_wait();

  const int NP = (p.NT + 1) >> 1;  // tile pairs per KV head
  const int units_per_part = p.Hkv * NP;
  const int total_units = p.unit_start[p.B] * units_per_part;
  // partition length of sequence b in tokens (the planner's half-length
  // partitions for the last sequences balance the last round of units)
  auto ppu_tokens_of = [&](int b) { return (b >= p.half_from ? p.ppu_half : p.ppu) * BS; };
  const uint32_t q_tile_bytes = 2u * 128u * static_cast<uint32_t>(p.G * p.Tt);  // both d halves
  bool timed_out = false;
  uint32_t copies_end = 0, mma_issued = 0, q_loads = 0;  // for the drain after a timeout

  auto slot_desc = [&](int k) { return reinterpret_cast<volatile int*>(sm + T2Layout::kSlots + k * T2Layout::kSlot); };
  auto slot_pages = [&](int k) {
    return reinterpret_cast<volatile int*>(sm + T2Layout::kSlots + k * T2Layout::kSlot + T2Layout::kSlotPages);
  };
  auto slot_bad = [&](int k) {
    return reinterpret_cast<volatile uint8_t*>(sm + T2Layout::kSlots + k * T2Layout::kSlot + T2Layout::kSlotBad);
  };
  // the unit in slot k: kvh and the pair from the unit index, the rest from
  // the descriptor the K copy warp wrote
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
    U.kvh = rem / NP;
    U.tile = 2 * (rem - U.kvh * NP);  // first tile of the pair
    const int ppu_tokens = ppu_tokens_of(U.b);
    U.t0 = U.pidx * ppu_tokens;
    U.t1 = min(U.ctx, U.t0 + ppu_tokens);
    U.npages = (U.t1 - U.t0 + BS - 1) / BS;
    U.nsteps = (U.npages + PPI - 1) / PPI;
    return U;
  };
  auto warp_wait = [&](uint64_t* bar, uint32_t parity) {
    int ok = 1;
    if (lane == 0) ok = mbar_wait_bounded(bar, parity, kWaitLimitNs) ? 1 : 0;
    return __shfl_sync(kFull, ok, 0) != 0;
  };

  if (kcopy) {
    // unit descriptors and page ids into the slot ring; K pages of each
    // step into stage g % 2 once S0 and S1 of step g - 2 are done
    uint32_t g = 0;
    for (int iu = 0;; ++iu) {
      const int k = iu & 1;
      if (iu >= 2 && !warp_wait(&slot_free[k], ((iu - 2) >> 1) & 1u)) {
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
      int nsteps = 0, npages = 0, kvh = 0;
      if (u < total_units) {
        b = __shfl_sync(kFull, b, 0);
        pidx = __shfl_sync(kFull, pidx, 0);
        ctx = __shfl_sync(kFull, ctx, 0);
        const int rem = u - (u / units_per_part) * units_per_part;
        kvh = rem / NP;
        const int tile0 = 2 * (rem - kvh * NP);
        const int ppu_tokens = ppu_tokens_of(b);
        const int t0 = pidx * ppu_tokens;
        npages = (min(ctx, t0 + ppu_tokens) - t0 + BS - 1) / BS;  // 1 .. kTcMaxPages
        nsteps = (npages + PPI - 1) / PPI;
        const int* trow = p.block_tables + static_cast<size_t>(b) * p.MB + t0 / BS;
        volatile int* pg = slot_pages(k);
        volatile uint8_t* bd = slot_bad(k);
        for (int q = lane; q < npages; q += 32) {
          int e = __ldg(trow + q);
          const bool isbad = static_cast<unsigned>(e) >= static_cast<unsigned>(p.NB);
          if (isbad) {
            e = 0;
            atomicOr(p.err, PKV_DEVERR_BLOCK_ID);
          }
          pg[q] = e;
          bd[q] = isbad ? 1 : 0;
        }
        __threadfence_block();
        // the unit's query tiles into L2 for the V copy warp's copies
        if (lane < 4) {
          const int tile = tile0 + (lane >> 1);
          if (tile < p.NT) tma_prefetch_4d(&qmap, 64 * (lane & 1), kvh * p.G, tile * p.Tt, b);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&slot_full[k]);  // release: the slot's writes by this warp
      if (u >= total_units) break;
      const volatile int* pages = slot_pages(k);
      for (int j = 0; j < nsteps; ++j, ++g) {
        if (g >= kT2Stages && !warp_wait(&k_free[g % kT2Stages], ((g - kT2Stages) / kT2Stages) & 1u)) {
          timed_out = true;
          break;
        }
        uint8_t* st = sm + T2Layout::kK + (g % kT2Stages) * T2Layout::kTile;
        uint64_t* bar = &k_full[g % kT2Stages];
        const int np = min(PPI, npages - j * PPI);
        if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(np) * 2u * BS * 128u);
        __syncwarp();
        if (lane < 2 * np) {
          const int q = lane >> 1, half = lane & 1;
          const int row = p.row_base + (pages[j * PPI + q] * p.Hkv + kvh) * BS;
          tma_load_2d(st + half * T2Layout::kRegion + q * BS * 128, &kmap, bar, half * 64, row, policy);
        }
        copies_end = g + 1;
      }
      if (timed_out) break;
    }
  } else if (vcopy) {
    // per unit: the two query tiles (once the previous unit's S products
    // are done), then the V pages of each step into stage g % 2 once PV0
    // and PV1 of step g - 2 are done
    uint32_t g = 0;
    for (int iu = 0;; ++iu) {
      const int k = iu & 1;
      if (!warp_wait(&slot_full[k], (iu >> 1) & 1u)) {
        timed_out = true;
        break;
      }
      const TcUnit U = read_unit(k);
      if (U.u >= total_units) break;
      if (iu > 0 && !warp_wait(q_free, (iu - 1) & 1u)) {
        timed_out = true;
        break;
      }
      if (lane == 0) mbar_arrive_expect_tx(q_full, 2u * q_tile_bytes);
      __syncwarp();
      if (lane < 4) {  // tile lane / 2, d half lane % 2; rows past T are zero-filled
        const int i = lane >> 1, half = lane & 1;
        tma_load_4d(sm + T2Layout::kQ + i * T2Layout::kTile + half * T2Layout::kRegion, &qmap, q_full, 64 * half,
                    U.kvh * p.G, (U.tile + i) * p.Tt, U.b);
      }
      ++q_loads;
      const volatile int* pages = slot_pages(k);
      for (int j = 0; j < U.nsteps; ++j, ++g) {
        if (g >= kT2Stages && !warp_wait(&v_free[g % kT2Stages], ((g - kT2Stages) / kT2Stages) & 1u)) {
          timed_out = true;
          break;
        }
        uint8_t* st = sm + T2Layout::kV + (g % kT2Stages) * T2Layout::kTile;
        uint64_t* bar = &v_full[g % kT2Stages];
        const int np = min(PPI, U.npages - j * PPI);
        if (lane == 0) {
          fence_proxy_async_smem();  // after the softmax warps' clearing of stale V rows
          mbar_arrive_expect_tx(bar, static_cast<uint32_t>(np) * 2u * BS * 128u);
        }
        __syncwarp();
        if (lane < 2 * np) {
          const int q = lane >> 1, half = lane & 1;
          const int row = p.row_base + (pages[j * PPI + q] * p.Hkv + U.kvh) * BS;
          tma_load_2d(st + half * T2Layout::kRegion + q * BS * 128, &vmap, bar, half * 64, row, policy);
        }
        copies_end = g + 1;
      }
      if (timed_out) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&slot_free[k]);
    }
  } else if (mma_warp) {
    if (lane == 0) {
      // descriptors of the operands' first k slices; a slice further along
      // adds its byte offset / 16 to the start-address field
      const uint64_t q_desc0 = tc_smem_desc(smem_addr(sm + T2Layout::kQ), 16, 1024, 2);
      const uint64_t q_desc1 = tc_smem_desc(smem_addr(sm + T2Layout::kQ + T2Layout::kTile), 16, 1024, 2);
      static_assert(kT2Stages == 2, "stage descriptors are selected, not indexed");
      const uint64_t k_desc0 = tc_smem_desc(smem_addr(sm + T2Layout::kK), 16, 1024, 2);
      const uint64_t k_desc1 = tc_smem_desc(smem_addr(sm + T2Layout::kK + T2Layout::kTile), 16, 1024, 2);
      const uint64_t v_desc0 = tc_smem_desc(smem_addr(sm + T2Layout::kV), T2Layout::kRegion, 1024, 2);
      const uint64_t v_desc1 = tc_smem_desc(smem_addr(sm + T2Layout::kV + T2Layout::kTile), T2Layout::kRegion, 1024, 2);
      // S_i(g) = Q_i . K(g)^T: 8 products of K 16 (d), A and B K-major with
      // the 128-byte swizzle
      auto issue_s = [&](int i, uint32_t g) {
        const uint64_t qd = i ? q_desc1 : q_desc0;
        const uint64_t kd = (g & 1u) ? k_desc1 : k_desc0;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = static_cast<uint64_t>(((kk >> 2) * T2Layout::kRegion + (kk & 3) * 32) >> 4);
          tc_mma_bf16(tmem + 128u * i, qd + off, kd + off, kIdescS, kk > 0);
        }
        ++mma_issued;
      };
      // O_i (+)= P_i(g) . V(g): P of tokens 16kk .. 16kk + 15 in columns
      // 8kk .. 8kk + 7 of S_i (A from TMEM), V MN-major as the pages hold it
      // (64-d halves kRegion apart, 8-token groups 1024 B apart); 8
      // products of K 16 (tokens)
      auto issue_pv = [&](int i, uint32_t g, bool acc) {
        const uint64_t vd = (g & 1u) ? v_desc1 : v_desc0;
#pragma unroll
        for (int kk = 0; kk < kT2Tokens / 16; ++kk)
          tc_mma_bf16_ts(tmem + 256u + 128u * i, tmem + 128u * i + 8u * kk,
                         vd + static_cast<uint64_t>(kk * 2048 >> 4), kIdescO, acc || kk > 0);
        ++mma_issued;
      };
      auto wait_pv_inputs = [&](int i, uint32_t g, bool first_pv, int iu) -> bool {
        if (!mbar_wait_fast(&p_full[i], g & 1u, kWaitLimitNs)) return false;
        if (i == 0 && !mbar_wait_fast(&v_full[g % kT2Stages], (g / kT2Stages) & 1u, kWaitLimitNs)) return false;
        if (first_pv && iu > 0 && !mbar_wait_fast(&o_free[i], (iu - 1) & 1u, kWaitLimitNs)) return false;
        tc_fence_after_sync();
        return true;
      };
      bool ok = mbar_wait_fast(&slot_full[0], 0, kWaitLimitNs);
      bool more = ok && slot_desc(0)[0] < total_units;
      uint32_t g0 = 0;
      for (int iu = 0; ok && more; ++iu) {
        const int k = iu & 1;
        const int n = read_unit(k).nsteps;
        ok = mbar_wait_fast(q_full, iu & 1u, kWaitLimitNs);
        for (int j = 0; ok && j < n; ++j) {
          const uint32_t g = g0 + j;
          ok = mbar_wait_fast(&k_full[g % kT2Stages], (g / kT2Stages) & 1u, kWaitLimitNs);
          if (!ok) break;
          tc_fence_after_sync();
          if (j > 0) {
            if (!(ok = wait_pv_inputs(0, g - 1, j == 1, iu))) break;
            issue_pv(0, g - 1, j > 1);
          }
          issue_s(0, g);
          tc_commit(&s_full[0]);
          if (j > 0) {
            if (!(ok = wait_pv_inputs(1, g - 1, j == 1, iu))) break;
            issue_pv(1, g - 1, j > 1);
            tc_commit(&v_free[(g - 1) % kT2Stages]);
          }
          issue_s(1, g);
          tc_commit(&s_full[1]);
          tc_commit(&k_free[g % kT2Stages]);
          if (j + 1 == n) tc_commit(q_free);
        }
        if (!ok) break;
        const uint32_t gl = g0 + n - 1;  // the unit's last P . V products
        if (!(ok = wait_pv_inputs(0, gl, n == 1, iu))) break;
        issue_pv(0, gl, n > 1);
        tc_commit(&o_full[0]);
        if (!(ok = wait_pv_inputs(1, gl, n == 1, iu))) break;
        issue_pv(1, gl, n > 1);
        tc_commit(&v_free[gl % kT2Stages]);
        tc_commit(&o_full[1]);
        mbar_arrive(&slot_free[k]);
        g0 += static_cast<uint32_t>(n);
        ok = mbar_wait_fast(&slot_full[(iu + 1) & 1], ((iu + 1) >> 1) & 1u, kWaitLimitNs);
        more = ok && slot_desc((iu + 1) & 1)[0] < total_units;
      }
      if (!ok) timed_out = true;
    }
    __syncwarp();
  } else {
    // softmax warps: tile i = warp / 4, row r = 32 (warp % 4) + lane, in
    // TMEM lane r
    const int i = warp >> 2;
    const int r = tid & 127;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + lane_base + 128u * i;
    const uint32_t t_o = tmem + lane_base + 256u + 128u * i;
    const float c = p.scale_log2;
    uint32_t g0 = 0;
    bool ok = true;
    for (int iu = 0; ok; ++iu) {
      const int k = iu & 1;
      if (!warp_wait(&slot_full[k], (iu >> 1) & 1u)) {
        ok = false;
        break;
      }
      // only what the steps need stays in registers; the output re-reads the
      // unit from its slot (the slot is released after the output)
      int lim, nsteps, t0, t1;  // lim: keys of this row are positions < lim
      {
        const TcUnit U = read_unit(k);
        if (U.u >= total_units) break;
        int t = 0, h = 0;
        lim = tile_row<true>(p, U.kvh, U.tile + i, r, t, h) ? U.ctx - p.T + 1 + t : INT_MIN / 2;
        nsteps = U.nsteps;
        t0 = U.t0;
        t1 = U.t1;
      }
      const volatile uint8_t* bad = slot_bad(k);
      float m = -INFINITY, l = 0.f;  // log2-domain lazy running maximum and sum of this row
      for (int j = 0; j < nsteps; ++j) {
        const uint32_t g = g0 + j;
        const int pos0 = t0 + j * kT2Tokens;
        const int nvs = t1 - pos0;  // tokens of the step in the sequence
        // the step's pages' bad-page flags, one byte each (PPI of them)
        const uint64_t badw = PPI == 8 ? *reinterpret_cast<const volatile uint64_t*>(bad + j * PPI)
                                       : *reinterpret_cast<const volatile uint32_t*>(bad + j * PPI);
        const bool full = nvs >= kT2Tokens && lim - pos0 >= kT2Tokens && badw == 0;
        if (!mbar_wait_bounded(&s_full[i], g & 1u, kWaitLimitNs)) timed_out = true;
        if (__any_sync(kFull, timed_out)) {  // warp-uniform exit (the TMEM accesses are collective)
          ok = false;
          break;
        }
        tc_fence_after_sync();
        float factor = 1.f;
        bool grow = false;
        if (__all_sync(kFull, full)) {
          // every token of the step is every row's (the common case): the
          // row's 128 scores in one round trip, kept in registers
          uint32_t x0[32], x1[32], x2[32], x3[32];
          tc_ld32(t_s, x0);
          tc_ld32(t_s + 32, x1);
          tc_ld32(t_s + 64, x2);
          tc_ld32(t_s + 96, x3);
          tc_wait_ld_regs(x0);  // one wait for the four loads
          tc_regs_loaded(x1);
          tc_regs_loaded(x2);
          tc_regs_loaded(x3);
          const float ext = c >= 0.f ? fmaxf(fmaxf(tree_ext32<true>(x0), tree_ext32<true>(x1)),
                                             fmaxf(tree_ext32<true>(x2), tree_ext32<true>(x3)))
                                     : fminf(fminf(tree_ext32<false>(x0), tree_ext32<false>(x1)),
                                             fminf(tree_ext32<false>(x2), tree_ext32<false>(x3)));
          // lazy maximum: move it (and rescale l here, O below) only when
          // the step's maximum exceeds it by more than 2^8
          const float smax = ext * c;
          grow = (m == -INFINITY) ? (smax != -INFINITY) : (smax > m + 8.f);
          if (grow) {
            factor = (m == -INFINITY) ? 0.f : ex2_approx(m - smax);
            l *= factor;
            m = smax;
          }
          // P = 2^(s c - m) as bf16 pairs over columns 0 .. 63 of S; the
          // arguments and the two running sums by packed pair instructions
          // (one issue slot for two scores: the exponential phase is bound
          // by issue, measured 7% faster at T = 64 and 128)
          const float neg_m = (m == -INFINITY) ? 0.f : -m;
          float ps[2] = {0.f, 0.f};  // two partial sums: shorter dependency chains
          auto write_p = [&](const uint32_t (&x)[32], int col) {
            uint32_t pw[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              float a0, a1;
              ffma2(a0, a1, __uint_as_float(x[2 * e]), __uint_as_float(x[2 * e + 1]), c, c, neg_m, neg_m);
              const float p0 = ex2_approx(a0);
              const float p1 = ex2_approx(a1);
              fadd2(ps[0], ps[1], ps[0], ps[1], p0, p1);
              pw[e] = pack_bf16x2(p0, p1);
            }
            tc_st16(t_s + col, pw);
          };
          write_p(x0, 0);
          write_p(x1, 16);
          write_p(x2, 32);
          write_p(x3, 48);
          l += ps[0] + ps[1];
        } else {
          // a step with masked tokens (the sequence end, the causal limit,
          // bad pages): the tokens of the step in the sequence and in a
          // valid page, then those this row attends to; 32 scores at a time,
          // the masked maximum first, then P (a chunk's P goes over columns
          // whose scores are already read)
          uint64_t rm0 = nvs >= 64 ? ~0ull : (nvs <= 0 ? 0ull : ((1ull << nvs) - 1ull));
          uint64_t rm1 = nvs >= 128 ? ~0ull : (nvs <= 64 ? 0ull : ((1ull << (nvs - 64)) - 1ull));
#pragma unroll
          for (int q = 0; q < PPI; ++q)
            if ((badw >> (8 * q)) & 0xffu) {
              const uint64_t pm = ((1ull << BS) - 1ull) << ((q * BS) & 63);
              if (q * BS < 64) rm0 &= ~pm; else rm1 &= ~pm;
            }
          const int nr = lim - pos0;
          rm0 &= nr >= 64 ? ~0ull : (nr <= 0 ? 0ull : ((1ull << nr) - 1ull));
          rm1 &= nr >= 128 ? ~0ull : (nr <= 64 ? 0ull : ((1ull << (nr - 64)) - 1ull));
          const float ext_init = c >= 0.f ? -INFINITY : INFINITY;
          float ext = ext_init;
#pragma unroll 1
          for (int cq = 0; cq < 4; ++cq) {
            uint32_t x[32];
            tc_ld32(t_s + 32 * cq, x);
            const uint64_t r64 = cq < 2 ? rm0 : rm1;
            const uint32_t mk = (cq & 1) ? static_cast<uint32_t>(r64 >> 32) : static_cast<uint32_t>(r64);
            tc_wait_ld_regs(x);
#pragma unroll
            for (int kk = 0; kk < 32; ++kk) {
              const float v = ((mk >> kk) & 1u) ? __uint_as_float(x[kk]) : ext_init;
              ext = c >= 0.f ? fmaxf(ext, v) : fminf(ext, v);
            }
          }
          const float smax = (rm0 | rm1) != 0ull ? ext * c : -INFINITY;
          grow = (m == -INFINITY) ? (smax != -INFINITY) : (smax > m + 8.f);
          if (grow) {
            factor = (m == -INFINITY) ? 0.f : ex2_approx(m - smax);
            l *= factor;
            m = smax;
          }
          const float neg_m = (m == -INFINITY) ? 0.f : -m;
          float ps0 = 0.f, ps1 = 0.f;
#pragma unroll 1
          for (int cq = 0; cq < 4; ++cq) {
            uint32_t x[32];
            tc_ld32(t_s + 32 * cq, x);
            const uint64_t r64 = cq < 2 ? rm0 : rm1;
            const uint32_t mk = (cq & 1) ? static_cast<uint32_t>(r64 >> 32) : static_cast<uint32_t>(r64);
            tc_wait_ld_regs(x);
            uint32_t pw[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              float a0, a1;
              ffma2(a0, a1, __uint_as_float(x[2 * e]), __uint_as_float(x[2 * e + 1]), c, c, neg_m, neg_m);
              float p0 = ex2_approx(a0);
              float p1 = ex2_approx(a1);
              p0 = ((mk >> (2 * e)) & 1u) ? p0 : 0.f;
              p1 = ((mk >> (2 * e + 1)) & 1u) ? p1 : 0.f;
              fadd2(ps0, ps1, ps0, ps1, p0, p1);
              pw[e] = pack_bf16x2(p0, p1);
            }
            tc_st16(t_s + 16 * cq, pw);
          }
          l += ps0 + ps1;
        }
        // O of the earlier steps, rarely (quiescent: PV_i(g - 1) finished
        // before S_i(g), and PV_i(g) waits for this step's p_full)
        if (j > 0 && __any_sync(kFull, grow)) {
#pragma unroll 1
          for (int oc = 0; oc < D; oc += 32) {
            uint32_t ov[32];
            tc_ld32(t_o + oc, ov);
            tc_wait_ld_regs(ov);
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              float a, b;
              fmul2(a, b, __uint_as_float(ov[e]), __uint_as_float(ov[e + 1]), factor, factor);
              ov[e] = __float_as_uint(a);
              ov[e + 1] = __float_as_uint(b);
            }
            tc_st32(t_o + oc, ov);
          }
        }
        // V rows of tokens outside the sequence (or of a bad page) may hold
        // anything and P is 0 there: once V(g) has landed, thread r of each
        // tile clears token row r (each tile's P . V waits only for its own
        // softmax warps; both tiles write the same zeros)
        const bool stale = nvs < kT2Tokens || badw != 0;
        if (stale) {
          if (!mbar_wait_bounded(&v_full[g % kT2Stages], (g / kT2Stages) & 1u, kWaitLimitNs)) timed_out = true;
          if (!timed_out && (r >= nvs || ((badw >> (8 * (r / BS))) & 0xffu))) {
            uint8_t* vb = sm + T2Layout::kV + (g % kT2Stages) * T2Layout::kTile + r * 128;
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
              *reinterpret_cast<uint4*>(vb + 16 * cc) = make_uint4(0, 0, 0, 0);
              *reinterpret_cast<uint4*>(vb + T2Layout::kRegion + 16 * cc) = make_uint4(0, 0, 0, 0);
            }
          }
        }
        tc_wait_st();
        if (stale) fence_proxy_async_smem();  // the cleared rows are read by the tensor cores
        tc_fence_before_sync();
        mbar_arrive(&p_full[i]);
        if (__any_sync(kFull, timed_out)) {
          ok = false;
          break;
        }
      }
      if (!ok) break;
      // the unit's output: O_i / l as bf16 rows, or the split-K partials
      // (m, l, unnormalised O); each thread writes its own row
      if (!mbar_wait_bounded(&o_full[i], iu & 1u, kWaitLimitNs)) timed_out = true;
      if (__any_sync(kFull, timed_out)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const TcUnit U = read_unit(k);
      int t = 0, h = 0;
      const bool row_ok = tile_row<true>(p, U.kvh, U.tile + i, r, t, h);
      const size_t qrow = static_cast<size_t>(U.b * p.T + t) * p.Hq + h;
      const bool direct = U.nparts == 1;
      const float osc = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
      for (int cc = 0; cc < D; cc += 32) {
        uint32_t ov[32];
        tc_ld32(t_o + cc, ov);
        tc_wait_ld_regs(ov);
        if (row_ok) {
          if (direct) {
            uint4* dst = reinterpret_cast<uint4*>(p.out + qrow * D + cc);
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
              uint32_t w4[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                float a, b;
                fmul2(a, b, __uint_as_float(ov[8 * c8 + 2 * e]), __uint_as_float(ov[8 * c8 + 2 * e + 1]), osc, osc);
                w4[e] = pack_bf16x2(a, b);
              }
              dst[c8] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
          } else {
            uint4* dst = reinterpret_cast<uint4*>(p.part_o + (qrow * p.pmax + U.pidx) * D + cc);
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) dst[c4] = make_uint4(ov[4 * c4], ov[4 * c4 + 1], ov[4 * c4 + 2], ov[4 * c4 + 3]);
          }
        }
      }
      if (row_ok && !direct) *reinterpret_cast<float2*>(p.part_ml + 2 * (qrow * p.pmax + U.pidx)) = make_float2(m, l);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&o_free[i]);
        mbar_arrive(&slot_free[k]);
      }
      g0 += static_cast<uint32_t>(nsteps);
    }
    if (!ok) timed_out = true;
  }

  timed_out = __syncthreads_or(timed_out) != 0;  // every role has left its loop
  if (timed_out) {
    if (tid == 0) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
    // each role lets its own copies and products still in flight finish
    // (bounded) before the shared and tensor memory are released
    if (kcopy && lane == 0)
      for (uint32_t g = copies_end > kT2Stages ? copies_end - kT2Stages : 0; g < copies_end; ++g)
        mbar_wait_bounded(&k_full[g % kT2Stages], (g / kT2Stages) & 1u, kWaitLimitNs / 16);
    if (vcopy && lane == 0) {
      for (uint32_t g = copies_end > kT2Stages ? copies_end - kT2Stages : 0; g < copies_end; ++g)
        mbar_wait_bounded(&v_full[g % kT2Stages], (g / kT2Stages) & 1u, kWaitLimitNs / 16);
      if (q_loads > 0) mbar_wait_bounded(q_full, (q_loads - 1) & 1u, kWaitLimitNs / 16);
    }
    if (mma_warp && lane == 0 && mma_issued > 0) {  // one commit covers every product issued
      tc_commit(mma_drain);
      mbar_wait_bounded(mma_drain, 0, kWaitLimitNs / 16);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tc_dealloc(tmem, kT2Cols);
}

}  // namespace pkv
