// Paged single-token decode attention, sm_103a.
//
// Sources ("KV Cache Engineering: PagedAttention, Continuous Batching,
// Attention Variants, and the Bandwidth Wall"): "What the KV Cache Stores
// and Why" (the new query attends over every cached K,V), "PagedAttention"
// (the kernel reaches physical blocks through the per-sequence block table;
// only the last block is partly filled), "Attention Variants" (GQA: a group
// of query heads shares one K/V head), "FP8 KV cache" and "INT8 KV cache"
// (dequantise on read),
// "Two Costs: Capacity and Bandwidth" (every step streams the whole cache,
// so the kernel is bound by HBM bandwidth).
//
// Multi-token queries: T >= 1 new query tokens per sequence (speculative
// decoding's verification step, "KV-Cache Engineering: Paged Attention,
// Prefix Cache, Disaggregation (2026)"), already appended as the last T
// cached tokens; query token t attends to positions 0 .. ctx - T + t.
//
// Structure
//   * Work unit = (sequence b, KV head, row tile, partition p): a run of up
//     to `ppu` consecutive logical blocks.  A row tile is up to 16 query
//     rows (query token, head of the group); T = 1 has one tile of G rows.  Units are handed out one at a time from a
//     global counter to warps of a persistent grid (each warp is an
//     independent streamer: no cross-warp synchronisation).
//   * Each warp owns a ring of `stages` shared-memory stages.  Lane 0 reads
//     the physical block id from the block table and issues two tensor-map
//     bulk copies (TMA) per K and V page into a stage, with 128-byte
//     swizzling; completion is tracked by one mbarrier per stage.  The warp
//     consumes stages in logical order and refills each one as soon as it
//     is done with it, so `stages - 1` pages are in flight per warp.
//   * All G query heads of the unit's KV group are computed from the one
//     K/V page read (GQA reuse).  Online softmax in the log2 domain with
//     fp32 state; the reduction order depends only on logical positions.
//   * A unit that covers its whole sequence writes the bf16 output; other
//     units write (max, sum, unnormalised output) partials (flash-decoding
//     split-K).  With few partitions per sequence the warp that completes
//     the last partition of a (sequence, KV head) merges them in place; with
//     many, a separate merge kernel spreads that work over the GPU.
//   * Two math back-ends share the pipeline: MMA (mma.sync m16n8k16 with the
//     group's heads on M, tokens on N for q.K^T, and head_dim on N, tokens
//     on K for P.V) and FFMA (fp32 CUDA-core dot products).
#pragma once

#include "pkv_device.cuh"

namespace pkv {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: a copy that has not landed by then never will

struct DecodeParams {
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  const int32_t* block_tables;
  const float* k_scale;
  const float* v_scale;
  int32_t* work_counter;
  const int32_t* unit_start;
  const int32_t* ctx_eff;
  const int32_t* part_seq;  // sequence of each global partition (written by the planner)
  float* part_ml;
  float* part_o;
  int32_t* arrive;  // [B][Hkv] partitions finished so far (zeroed by the planner)
  unsigned* err;
  int B, Hq, Hkv, G, MB, NB, pmax, ppu, stages;
  int half_from, ppu_half;  // sequences b >= half_from: partitions of ppu_half blocks
  int T, Tt, NT;  // query tokens per sequence, per row tile; row tiles
  int fused_merge;  // 1: the last warp of a (sequence, KV head) merges; 0: the merge kernel does
  int row_base;
  float scale_log2;
};

// Query row `row` (0..15) of row tile `tile` of KV head `kvh`: query token
// t = tile * Tt + row / G, query head h = kvh * G + row % G.  False for rows
// past the tile's tokens.  The row's offset in q, out and the partials is
// (b * T + t) * Hq + h.  MT = false: single-token kernels (T = 1, one tile).
template <bool MT>
__device__ __forceinline__ bool tile_row(const DecodeParams& p, int kvh, int tile, int row, int& t,
                                         int& h) {
  if constexpr (!MT) {
    t = 0;
    h = kvh * p.G + row;
    return row < p.G;
  }
  const int tl = row / p.G;
  t = tile * p.Tt + tl;
  h = kvh * p.G + (row - tl * p.G);
  return tl < p.Tt && t < p.T;
}

template <int D, int BS, bool FP8>
struct PageGeom {
  static constexpr int kElem = FP8 ? 1 : 2;
  static constexpr int kRowBytes = D * kElem;          // bytes of one token row
  static constexpr int kRegions = kRowBytes / 128;      // 128-byte wide tensor-map boxes
  static constexpr int kBoxInner = 128 / kElem;         // elements per box row
  static constexpr int kRegionBytes = BS * 128;
  static constexpr int kTensorBytes = kRegions * kRegionBytes;  // one K (or V) page
  static constexpr int kStageBytes = 2 * kTensorBytes;
  static_assert(kRowBytes % 128 == 0, "rows must be whole 128-byte boxes");
};

// Shared memory layout per CTA: [warps][stages] stage buffers (1024-aligned),
// then [warps][8] mbarriers, then [warps][BS * 16] floats of P scratch.
template <int D, int BS, bool FP8>
__host__ __device__ constexpr size_t decode_smem_layout_bytes(int warps, int stages) {
  return 1024 /* alignment slack */ +
         static_cast<size_t>(warps) * stages * PageGeom<D, BS, FP8>::kStageBytes +
         static_cast<size_t>(warps) * 8 * sizeof(uint64_t) +
         static_cast<size_t>(warps) * BS * 16 * sizeof(float);
}

// ---------------------------------------------------------------------------
// MMA back-end state and page step
// ---------------------------------------------------------------------------
// m16n8k16 tiles with the group's heads on M.  HI = false: at most 8 heads,
// rows 8..15 of every tile are zero and only rows 0..7 are carried (half the
// registers); HI = true: up to 16 heads, both row halves carried.
// Fragment arrays hold {row g k-lo, row g k-hi, row g+8 k-lo, row g+8 k-hi}
// (A operands) and {row g c0, c1, row g+8 c0, c1} (C/D).
template <int D, int BS, bool FP8, bool HI>
struct MmaState {
  static constexpr int kR = HI ? 2 : 1;
  uint32_t qa[D / 16][2 * kR];  // q as A fragments, one entry per k-step of 16 d
  float o[D / 8][2 * kR];       // output accumulators, one entry per 8 columns of d
  float m[kR];                  // running max of rows g (and g+8), log2 domain
  float l[kR];                  // this lane's share of the running sums
  // INT8 pages enter the products as 1152 + code (see int8x4_to_f16x2x2_biased):
  float qs[kR];    // sum over d of the f16 query row, for removing the K bias
  float corr[kR];  // V bias carried by every column of o (same rescaling as o)
};

constexpr uint32_t kOnesF16x2 = 0x3C003C00u;  // f16x2 (1, 1)

template <bool FP8, bool HI, int N>
__device__ __forceinline__ void mma_rows(float (&d)[N], const uint32_t (&a)[N], uint32_t b0,
                                         uint32_t b1) {
  if constexpr (HI) {
    const uint32_t full[4] = {a[0], a[2], a[1], a[3]};
    if constexpr (FP8) mma_f16(d, full, b0, b1); else mma_bf16(d, full, b0, b1);
  } else {
    if constexpr (FP8) mma_f16_lo(d, a[0], a[1], b0, b1); else mma_bf16_lo(d, a[0], a[1], b0, b1);
  }
}

template <int D, int BS, bool FP8, bool HI, bool MT>
__device__ __forceinline__ void mma_load_q(MmaState<D, BS, FP8, HI>& st, const DecodeParams& p,
                                           int b, int kvh, int tile, int lane) {
  constexpr int kR = HI ? 2 : 1;
  const int g = lane >> 2, tig = lane & 3;
  const __nv_bfloat16* qrow[kR];
#pragma unroll
  for (int half = 0; half < kR; ++half) {
    int t, h;
    qrow[half] = tile_row<MT>(p, kvh, tile, g + 8 * half, t, h)
                     ? p.q + (static_cast<size_t>(b * p.T + t) * p.Hq + h) * D
                     : nullptr;
  }
#pragma unroll
  for (int s = 0; s < D / 16; ++s) {
#pragma unroll
    for (int half = 0; half < kR; ++half) {
      uint32_t lo = 0, hi = 0;
      if (qrow[half] != nullptr) {
        const __nv_bfloat16* qr = qrow[half];
        if constexpr (!FP8) {
          // k = 2tig, 2tig+1 -> d = 16s + 2tig (+1); k + 8 -> d + 8
          lo = *reinterpret_cast<const uint32_t*>(qr + 16 * s + 2 * tig);
          hi = *reinterpret_cast<const uint32_t*>(qr + 16 * s + 8 + 2 * tig);
        } else {
          // E4M3 pages are read 4 bytes per lane per chunk: k = 2tig, 2tig+1
          // -> d = 16s + 4tig (+1); k + 8 -> d = 16s + 4tig + 2 (+1)
          const uint32_t w0 = *reinterpret_cast<const uint32_t*>(qr + 16 * s + 4 * tig);
          const uint32_t w1 = *reinterpret_cast<const uint32_t*>(qr + 16 * s + 4 * tig + 2);
          lo = pack_f16x2(bf16lo_to_f32(w0), bf16hi_to_f32(w0));
          hi = pack_f16x2(bf16lo_to_f32(w1), bf16hi_to_f32(w1));
        }
      }
      st.qa[s][2 * half] = lo;
      st.qa[s][2 * half + 1] = hi;
    }
  }
#pragma unroll
  for (int n = 0; n < D / 8; ++n)
#pragma unroll
    for (int e = 0; e < 2 * kR; ++e) st.o[n][e] = 0.f;
#pragma unroll
  for (int r = 0; r < kR; ++r) {
    st.m[r] = -INFINITY;
    st.l[r] = 0.f;
  }
}

// Token held in column `r` (0..7) of q.K^T n-tile `nt`.  bf16 pages use the
// natural order.  E4M3 pages permute tokens inside each 16-token k-step so
// that P's k-slots (2t, 2t+1) and (2t+8, 2t+9) are tokens 4t, 4t+1 and
// 4t+2, 4t+3: the token quads that the byte-transposing ldmatrix hands each
// lane of the V operand.
template <bool FP8>
__device__ __forceinline__ int qk_token(int nt, int r) {
  if constexpr (!FP8) return nt * 8 + r;
  return 16 * (nt >> 1) + 4 * (r >> 1) + 2 * (nt & 1) + (r & 1);
}

// Four one-byte codes -> two f16x2 words (exact): E4M3 by hardware
// conversion, INT8 as code - zero (zc from int8_zero_const).
template <bool I8>
__device__ __forceinline__ void bytes4_to_f16x2x2(uint32_t x, uint32_t zc, uint32_t& lo, uint32_t& hi) {
  if constexpr (I8) int8x4_to_f16x2x2(x, zc, lo, hi); else e4m3x4_to_f16x2x2(x, lo, hi);
}

// Tensor-core back-end form: INT8 codes stay biased by 1152 + zero and the
// bias is removed per row after the products (one subtraction per score and
// per output column instead of one per cache element).
template <bool I8>
__device__ __forceinline__ void bytes4_to_f16x2x2_mma(uint32_t x, uint32_t& lo, uint32_t& hi) {
  if constexpr (I8) int8x4_to_f16x2x2_biased(x, lo, hi); else e4m3x4_to_f16x2x2(x, lo, hi);
}

// INT8: qs = sum over d of each head's f16 query row (q . 1 on the tensor
// cores, fp32 accumulation), and the V bias accumulator cleared.
template <int D, int BS, bool FP8, bool HI>
__device__ __forceinline__ void mma_int8_prepare(MmaState<D, BS, FP8, HI>& st) {
  constexpr int kR = HI ? 2 : 1;
  float acc[2 * kR];
#pragma unroll
  for (int e = 0; e < 2 * kR; ++e) acc[e] = 0.f;
#pragma unroll
  for (int s = 0; s < D / 16; ++s) mma_rows<FP8, HI>(acc, st.qa[s], kOnesF16x2, kOnesF16x2);
#pragma unroll
  for (int r = 0; r < kR; ++r) {
    st.qs[r] = acc[2 * r];
    st.corr[r] = 0.f;
  }
}

// INT8: remove the V bias from every output column (once per work unit).
template <int D, int BS, bool FP8, bool HI>
__device__ __forceinline__ void mma_int8_unbias(MmaState<D, BS, FP8, HI>& st) {
  constexpr int kR = HI ? 2 : 1;
#pragma unroll
  for (int n = 0; n < D / 8; ++n)
#pragma unroll
    for (int e = 0; e < 2 * kR; ++e) st.o[n][e] -= st.corr[e >> 1];
}

// One page (BS tokens) of the online softmax with tensor-core tiles.
// `valid` = tokens of the page that belong to the sequence (0..BS); `rv[r]`
// = tokens of the page that query row g + 8r attends to (<= valid; below it
// for the earlier tokens of a multi-token query); `partial` = some row of
// the tile attends to fewer than BS tokens of the page (warp-uniform); `sl` =
// softmax scale * log2(e) (* the page's K scale for one-byte pages);
// `vscale` = the page's V scale (one-byte pages); `kc`, `vc` = the page's
// INT8 biases 1152 + zero of K and V.
template <int D, int BS, bool FP8, bool HI, bool I8>
__device__ __forceinline__ void mma_page(MmaState<D, BS, FP8, HI>& st, uint8_t* stage, int valid,
                                         const int (&rv)[HI ? 2 : 1], bool partial, float sl,
                                         float vscale, float kc, float vc, int lane) {
  using Geo = PageGeom<D, BS, FP8>;
  constexpr int kR = HI ? 2 : 1;
  constexpr int kC = 2 * kR;
  const int tig = lane & 3;
  const uint32_t kbase = smem_addr(stage);
  const uint32_t vbase = kbase + Geo::kTensorBytes;

  // ---- S = q . K^T  (rows = heads, cols = tokens) ----
  float s[BS / 8][kC];
#pragma unroll
  for (int nt = 0; nt < BS / 8; ++nt) {
#pragma unroll
    for (int e = 0; e < kC; ++e) s[nt][e] = 0.f;
    const int row = qk_token<FP8>(nt, lane & 7);
    if constexpr (!FP8) {
#pragma unroll
      for (int kk = 0; kk < D / 32; ++kk) {
        const int region = kk >> 1;
        const int chunk = (kk & 1) * 4 + (lane >> 3);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kbase + region * Geo::kRegionBytes + swz128(row, chunk), b0, b1, b2, b3);
        mma_rows<FP8, HI>(s[nt], st.qa[2 * kk], b0, b1);
        mma_rows<FP8, HI>(s[nt], st.qa[2 * kk + 1], b2, b3);
      }
    } else {
#pragma unroll
      for (int c4 = 0; c4 < D / 64; ++c4) {
        uint32_t r[4];
        ldsm_x4(kbase + swz128(row, c4 * 4 + (lane >> 3)), r[0], r[1], r[2], r[3]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint32_t b0, b1;
          bytes4_to_f16x2x2_mma<I8>(r[i], b0, b1);
          mma_rows<FP8, HI>(s[nt], st.qa[c4 * 4 + i], b0, b1);
        }
      }
    }
  }

  // ---- online softmax (log2 domain) ----
  // INT8: q . (K' - kc) = q . K' - kc * qs, folded into the scaling
  float kb[kR];
#pragma unroll
  for (int r = 0; r < kR; ++r) kb[r] = I8 ? -kc * st.qs[r] * sl : 0.f;
  float mx[kR];
#pragma unroll
  for (int r = 0; r < kR; ++r) mx[r] = -INFINITY;
  if (partial) {
#pragma unroll
    for (int nt = 0; nt < BS / 8; ++nt)
#pragma unroll
      for (int e = 0; e < kC; ++e) {
        const int tok = qk_token<FP8>(nt, 2 * tig + (e & 1));
        const float v = (tok < rv[e >> 1]) ? fmaf(s[nt][e], sl, kb[e >> 1]) : -INFINITY;
        s[nt][e] = v;
        mx[e >> 1] = fmaxf(mx[e >> 1], v);
      }
  } else {
#pragma unroll
    for (int nt = 0; nt < BS / 8; ++nt)
#pragma unroll
      for (int e = 0; e < kC; ++e) {
        const float v = fmaf(s[nt][e], sl, kb[e >> 1]);
        s[nt][e] = v;
        mx[e >> 1] = fmaxf(mx[e >> 1], v);
      }
  }
  float alpha[kR], muse[kR];
  bool changed = false;
#pragma unroll
  for (int r = 0; r < kR; ++r) {
    mx[r] = fmaxf(mx[r], __shfl_xor_sync(kFull, mx[r], 1));
    mx[r] = fmaxf(mx[r], __shfl_xor_sync(kFull, mx[r], 2));
    const float mnew = fmaxf(st.m[r], mx[r]);
    muse[r] = (mnew == -INFINITY) ? 0.f : mnew;
    alpha[r] = ex2_approx(st.m[r] - muse[r]);
    changed |= (mnew != st.m[r]);
    st.m[r] = mnew;
  }
  float psum[kR];
#pragma unroll
  for (int r = 0; r < kR; ++r) psum[r] = 0.f;
#pragma unroll
  for (int nt = 0; nt < BS / 8; ++nt)
#pragma unroll
    for (int e = 0; e < kC; ++e) {
      const float pv = ex2_approx(s[nt][e] - muse[e >> 1]);
      s[nt][e] = pv;
      psum[e >> 1] += pv;
    }
#pragma unroll
  for (int r = 0; r < kR; ++r) st.l[r] = fmaf(st.l[r], alpha[r], psum[r]);
  // Rescale O only when some row's running max moved (rare after the first
  // pages); alpha is exactly 1 for rows whose max did not move.
  if (__any_sync(kFull, changed)) {
#pragma unroll
    for (int n = 0; n < D / 8; ++n)
#pragma unroll
      for (int e = 0; e < kC; ++e) st.o[n][e] *= alpha[e >> 1];
    if constexpr (I8) {
#pragma unroll
      for (int r = 0; r < kR; ++r) st.corr[r] *= alpha[r];
    }
  }

  // P as A fragments: k-step ks covers tokens 16ks .. 16ks+15 (n-tiles 2ks, 2ks+1)
  uint32_t pa[BS / 16][kC];
#pragma unroll
  for (int ks = 0; ks < BS / 16; ++ks)
#pragma unroll
    for (int r = 0; r < kR; ++r)
#pragma unroll
      for (int kh = 0; kh < 2; ++kh) {
        const float* src = s[2 * ks + kh];
        if constexpr (!FP8)
          pa[ks][2 * r + kh] = pack_bf16x2(src[2 * r], src[2 * r + 1]);
        else
          pa[ks][2 * r + kh] = pack_f16x2(src[2 * r], src[2 * r + 1]);
      }

  // INT8: P . (V' - vc) = P . V' - vc * sum(P), with sum(P) taken over the
  // same f16 P (P . 1 on the tensor cores) and applied to o at the end
  if constexpr (I8) {
    float ps[kC];
#pragma unroll
    for (int e = 0; e < kC; ++e) ps[e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < BS / 16; ++ks) mma_rows<FP8, HI>(ps, pa[ks], kOnesF16x2, kOnesF16x2);
#pragma unroll
    for (int r = 0; r < kR; ++r) st.corr[r] = fmaf(vscale * vc, ps[2 * r], st.corr[r]);
  }

  // Rows of V past the sequence end may hold anything (E4M3 and bf16: even
  // NaN); P is 0 there but 0 * NaN is NaN, so clear them before the product.
  // Every INT8 byte is a finite value.
  if (!I8 && valid < BS) {
    uint8_t* vp = stage + Geo::kTensorBytes;
    for (int idx = lane; idx < Geo::kTensorBytes / 16; idx += 32) {
      const int row = (idx % (Geo::kRegionBytes / 16)) / 8;
      if (row >= valid) reinterpret_cast<uint4*>(vp)[idx] = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
    __syncwarp();
  }

  // ---- O += P . V ----
  if constexpr (!FP8) {
#pragma unroll
    for (int ks = 0; ks < BS / 16; ++ks) {
      const int mi = lane >> 3;
      const int row = ks * 16 + (mi & 1) * 8 + (lane & 7);
#pragma unroll
      for (int np = 0; np < D / 16; ++np) {
        const int region = (np * 16) / 64;
        const int chunk = ((np * 16) % 64) / 8 + (mi >> 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vbase + region * Geo::kRegionBytes + swz128(row, chunk), b0, b1, b2, b3);
        mma_rows<FP8, HI>(st.o[2 * np], pa[ks], b0, b1);
        mma_rows<FP8, HI>(st.o[2 * np + 1], pa[ks], b2, b3);
      }
    }
  } else {
    // E4M3 V: a byte-transposing ldmatrix gives each lane four consecutive
    // tokens of one column (the quads P's k-slots were arranged for), which
    // convert to two f16x2 B registers; two 16-column chunks per load.
#pragma unroll
    for (int cp = 0; cp < D / 32; ++cp) {
      float t[4][kC];  // this page's P . V8 for n-tiles 4*cp .. 4*cp+3
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < kC; ++e) t[j][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < BS / 16; ++ks) {
        uint32_t q[4];
        ldsm_x2_t_b8(vbase + swz128(ks * 16 + (lane & 15), 2 * cp + (lane >> 4)), q[0], q[1], q[2], q[3]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t b0, b1;
          bytes4_to_f16x2x2_mma<I8>(q[j], b0, b1);
          mma_rows<FP8, HI>(t[j], pa[ks], b0, b1);
        }
      }
      // the page's V scale applies to its whole product, in fp32
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < kC; ++e) st.o[4 * cp + j][e] = fmaf(vscale, t[j][e], st.o[4 * cp + j][e]);
    }
  }
}

template <int D, int BS, bool FP8, bool HI, bool MT>
__device__ __forceinline__ void mma_finish(MmaState<D, BS, FP8, HI>& st, const DecodeParams& p,
                                           int b, int kvh, int tile, int pidx, int nparts, int lane) {
  constexpr int kR = HI ? 2 : 1;
  const int g = lane >> 2, tig = lane & 3;
#pragma unroll
  for (int r = 0; r < kR; ++r) {
    st.l[r] += __shfl_xor_sync(kFull, st.l[r], 1);
    st.l[r] += __shfl_xor_sync(kFull, st.l[r], 2);
  }
#pragma unroll
  for (int r = 0; r < kR; ++r) {
    int t, h;
    if (!tile_row<MT>(p, kvh, tile, g + 8 * r, t, h)) continue;
    const size_t qrow = static_cast<size_t>(b * p.T + t) * p.Hq + h;
    if (nparts == 1) {
      const float inv = st.l[r] > 0.f ? 1.f / st.l[r] : 0.f;
      __nv_bfloat16* o = p.out + qrow * D;
#pragma unroll
      for (int n = 0; n < D / 8; ++n)
        *reinterpret_cast<__nv_bfloat162*>(o + 8 * n + 2 * tig) =
            __floats2bfloat162_rn(st.o[n][2 * r] * inv, st.o[n][2 * r + 1] * inv);
    } else {
      const size_t slot = qrow * p.pmax + pidx;
      float* o = p.part_o + slot * D;
#pragma unroll
      for (int n = 0; n < D / 8; ++n)
        *reinterpret_cast<float2*>(o + 8 * n + 2 * tig) = make_float2(st.o[n][2 * r], st.o[n][2 * r + 1]);
      if (tig == 0) *reinterpret_cast<float2*>(p.part_ml + 2 * slot) = make_float2(st.m[r], st.l[r]);
    }
  }
}

// ---------------------------------------------------------------------------
// FFMA back-end (fp32 CUDA cores); GT = heads per KV group (compile time)
// ---------------------------------------------------------------------------
// QK lane layout: lane = 8 * tl + dl; token rows 4i + tl, head_dim slice
// [dl * D/8, (dl+1) * D/8).  PV lane layout: lane owns D/32 consecutive d.
template <int D, int BS, bool FP8, int GT>
struct FfmaState {
  float q[GT][D / 8];
  float o[GT][D / 32];
  float m[GT];
  float l[GT];
};

template <int D, int BS, bool FP8, int GT>
__device__ __forceinline__ void ffma_load_q(FfmaState<D, BS, FP8, GT>& st,
                                            const __nv_bfloat16* qg, int lane) {
  const int dl = lane & 7;
#pragma unroll
  for (int h = 0; h < GT; ++h) {
    const uint4* src = reinterpret_cast<const uint4*>(qg + static_cast<size_t>(h) * D + dl * (D / 8));
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
      const uint4 w = src[c];
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        st.q[h][8 * c + 2 * i] = bf16lo_to_f32(ws[i]);
        st.q[h][8 * c + 2 * i + 1] = bf16hi_to_f32(ws[i]);
      }
    }
#pragma unroll
    for (int j = 0; j < D / 32; ++j) st.o[h][j] = 0.f;
    st.m[h] = -INFINITY;
    st.l[h] = 0.f;
  }
}

// D/8 consecutive K values of token row `row`, starting at d = dl * D/8.
template <int D, int BS, bool FP8, bool I8>
__device__ __forceinline__ void ffma_load_k(const uint8_t* kp, int row, int dl, uint32_t zc,
                                            float (&kf)[D / 8]) {
  using Geo = PageGeom<D, BS, FP8>;
  if constexpr (!FP8) {
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
      const int d0 = dl * (D / 8) + 8 * c;
      const int region = d0 / 64, chunk = (d0 % 64) / 8;
      const uint4 w = *reinterpret_cast<const uint4*>(kp + region * Geo::kRegionBytes + swz128(row, chunk));
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        kf[8 * c + 2 * i] = bf16lo_to_f32(ws[i]);
        kf[8 * c + 2 * i + 1] = bf16hi_to_f32(ws[i]);
      }
    }
  } else {
    static_assert(D == 128, "E4M3 pages need head_dim 128");
    // D/8 = 16 bytes = one chunk
    const uint4 w = *reinterpret_cast<const uint4*>(kp + swz128(row, dl));
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t h01, h23;
      bytes4_to_f16x2x2<I8>(ws[i], zc, h01, h23);
      const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
      const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
      kf[4 * i] = f01.x;
      kf[4 * i + 1] = f01.y;
      kf[4 * i + 2] = f23.x;
      kf[4 * i + 3] = f23.y;
    }
  }
}

// D/32 consecutive V values of token row `row`, starting at d = lane * D/32.
template <int D, int BS, bool FP8, bool I8>
__device__ __forceinline__ void ffma_load_v(const uint8_t* vp, int row, int lane, uint32_t zc,
                                            float (&vf)[D / 32]) {
  using Geo = PageGeom<D, BS, FP8>;
  const int d0 = lane * (D / 32);
  if constexpr (!FP8) {
    const int region = d0 / 64, chunk = (d0 % 64) / 8, within = (d0 % 8) * 2;
    const uint8_t* src = vp + region * Geo::kRegionBytes + swz128(row, chunk) + within;
    if constexpr (D / 32 == 4) {
      const uint2 w = *reinterpret_cast<const uint2*>(src);
      vf[0] = bf16lo_to_f32(w.x);
      vf[1] = bf16hi_to_f32(w.x);
      vf[2] = bf16lo_to_f32(w.y);
      vf[3] = bf16hi_to_f32(w.y);
    } else {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(src);
      vf[0] = bf16lo_to_f32(w);
      vf[1] = bf16hi_to_f32(w);
    }
  } else {
    static_assert(D / 32 == 4, "E4M3 pages need head_dim 128");
    const uint32_t w = *reinterpret_cast<const uint32_t*>(vp + swz128(row, d0 >> 4) + (d0 & 15));
    uint32_t h01, h23;
    bytes4_to_f16x2x2<I8>(w, zc, h01, h23);
    const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
    const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
    vf[0] = f01.x;
    vf[1] = f01.y;
    vf[2] = f23.x;
    vf[3] = f23.y;
  }
}

template <int D, int BS, bool FP8, int GT, bool I8>
__device__ __forceinline__ void ffma_page(FfmaState<D, BS, FP8, GT>& st, uint8_t* stage, int valid,
                                          float sl, float vscale, uint32_t kzc, uint32_t vzc,
                                          float* pbuf, int lane) {
  using Geo = PageGeom<D, BS, FP8>;
  const int tl = lane >> 3, dl = lane & 7;
  const uint8_t* kp = stage;
  const uint8_t* vp = stage + Geo::kTensorBytes;
  float s[BS / 4][GT];
#pragma unroll
  for (int i = 0; i < BS / 4; ++i) {
    const int row = 4 * i + tl;
    float kf[D / 8];
    ffma_load_k<D, BS, FP8, I8>(kp, row, dl, kzc, kf);
#pragma unroll
    for (int h = 0; h < GT; ++h) {
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < D / 8; ++j) acc = fmaf(st.q[h][j], kf[j], acc);
      acc += __shfl_xor_sync(kFull, acc, 1);
      acc += __shfl_xor_sync(kFull, acc, 2);
      acc += __shfl_xor_sync(kFull, acc, 4);
      s[i][h] = (row < valid) ? acc * sl : -INFINITY;
    }
  }
  float alpha[GT];
#pragma unroll
  for (int h = 0; h < GT; ++h) {
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < BS / 4; ++i) mx = fmaxf(mx, s[i][h]);
    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
    const float mnew = fmaxf(st.m[h], mx);
    const float muse = (mnew == -INFINITY) ? 0.f : mnew;
    alpha[h] = exp2f(st.m[h] - muse);
    st.m[h] = mnew;
    float ps = 0.f;
#pragma unroll
    for (int i = 0; i < BS / 4; ++i) {
      const float pv = exp2f(s[i][h] - muse);
      s[i][h] = pv;
      ps += pv;
    }
    st.l[h] = st.l[h] * alpha[h] + ps;
  }
  if (dl == 0) {
#pragma unroll
    for (int i = 0; i < BS / 4; ++i)
#pragma unroll
      for (int h = 0; h < GT; ++h) pbuf[(4 * i + tl) * GT + h] = s[i][h] * vscale;
  }
  __syncwarp();
#pragma unroll
  for (int h = 0; h < GT; ++h)
#pragma unroll
    for (int j = 0; j < D / 32; ++j) st.o[h][j] *= alpha[h];
#pragma unroll 4
  for (int t = 0; t < valid; ++t) {
    float vf[D / 32];
    ffma_load_v<D, BS, FP8, I8>(vp, t, lane, vzc, vf);
    float pv[GT];
#pragma unroll
    for (int h = 0; h < GT; ++h) pv[h] = pbuf[t * GT + h];
#pragma unroll
    for (int h = 0; h < GT; ++h)
#pragma unroll
      for (int j = 0; j < D / 32; ++j) st.o[h][j] = fmaf(pv[h], vf[j], st.o[h][j]);
  }
}

template <int D, int BS, bool FP8, int GT>
__device__ __forceinline__ void ffma_finish(FfmaState<D, BS, FP8, GT>& st, const DecodeParams& p,
                                            int b, int kvh, int pidx, int nparts, int lane) {
#pragma unroll
  for (int h = 0; h < GT; ++h) {
    float lt = st.l[h];
    lt += __shfl_xor_sync(kFull, lt, 8);
    lt += __shfl_xor_sync(kFull, lt, 16);
    const int hq = kvh * GT + h;
    if (nparts == 1) {
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      __nv_bfloat16* o = p.out + (static_cast<size_t>(b) * p.Hq + hq) * D + lane * (D / 32);
#pragma unroll
      for (int j = 0; j < D / 32; j += 2)
        *reinterpret_cast<__nv_bfloat162*>(o + j) = __floats2bfloat162_rn(st.o[h][j] * inv, st.o[h][j + 1] * inv);
    } else {
      const size_t slot = (static_cast<size_t>(b) * p.Hq + hq) * p.pmax + pidx;
      float* o = p.part_o + slot * D + lane * (D / 32);
#pragma unroll
      for (int j = 0; j < D / 32; j += 2) *reinterpret_cast<float2*>(o + j) = make_float2(st.o[h][j], st.o[h][j + 1]);
      if (lane == 0) *reinterpret_cast<float2*>(p.part_ml + 2 * slot) = make_float2(st.m[h], lt);
    }
  }
}

// ---------------------------------------------------------------------------
// split-K merge, done by the warp that finishes a (sequence, KV head) last
// ---------------------------------------------------------------------------
// With partials (m_p, l_p, O_p) of partitions p of one head, M = max_p m_p:
//   out = sum_p 2^(m_p - M) O_p / sum_p 2^(m_p - M) l_p,
// the softmax over the union of the partitions' tokens.  An empty partition
// (m = -inf) has weight 0.
template <int D, bool MT>
__device__ __forceinline__ void arrive_and_merge(const DecodeParams& p, int b, int kvh, int tile,
                                                 int nparts, int lane) {
  // publish this warp's partials, then count the partition as done
  __threadfence();
  __syncwarp();
  int* counter = p.arrive + (MT ? (b * p.Hkv + kvh) * p.NT + tile : b * p.Hkv + kvh);
  int prev = 0;
  if (lane == 0) prev = atomicAdd(counter, 1);
  prev = __shfl_sync(kFull, prev, 0);
  if (prev != nparts - 1) return;
  __threadfence();  // the other partitions' partials are visible from here on
  constexpr int kPer = D / 32;
  for (int r = 0; r < (MT ? p.G * p.Tt : p.G); ++r) {
    int t, h;
    if (!tile_row<MT>(p, kvh, tile, r, t, h)) break;
    const size_t qrow = static_cast<size_t>(b * p.T + t) * p.Hq + h;
    const size_t base = qrow * p.pmax;
    float M = -INFINITY;
    for (int i = lane; i < nparts; i += 32) M = fmaxf(M, __ldcg(p.part_ml + 2 * (base + i)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
    float acc[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) acc[j] = 0.f;
    float L = 0.f;
    if (M != -INFINITY) {
#pragma unroll 4
      for (int i = 0; i < nparts; ++i) {
        const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.part_ml + 2 * (base + i)));
        const float w = exp2f(ml.x - M);
        L = fmaf(w, ml.y, L);
        const float* src = p.part_o + (base + i) * D + lane * kPer;
        if constexpr (kPer == 4) {
          const float4 v = __ldcg(reinterpret_cast<const float4*>(src));
          acc[0] = fmaf(w, v.x, acc[0]);
          acc[1] = fmaf(w, v.y, acc[1]);
          acc[2] = fmaf(w, v.z, acc[2]);
          acc[3] = fmaf(w, v.w, acc[3]);
        } else {
          const float2 v = __ldcg(reinterpret_cast<const float2*>(src));
          acc[0] = fmaf(w, v.x, acc[0]);
          acc[1] = fmaf(w, v.y, acc[1]);
        }
      }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    __nv_bfloat16* o = p.out + qrow * D + lane * kPer;
#pragma unroll
    for (int j = 0; j < kPer; j += 2)
      *reinterpret_cast<__nv_bfloat162*>(o + j) = __floats2bfloat162_rn(acc[j] * inv, acc[j + 1] * inv);
  }
  if (lane == 0) *counter = 0;  // ready for the next call on this workspace
}

// ---------------------------------------------------------------------------
// a unit's pages: physical ids, bad-id masks and dequantisation parameters;
// lane i holds pages i and i + 32 (a unit has at most 64 pages)
// ---------------------------------------------------------------------------
struct UnitPages {
  int e0, e1;
  uint32_t badm0, badm1;
  float ks0, ks1, vs0, vs1;  // E4M3 / INT8 scales (1 for bf16)
  float kz0, kz1, vz0, vz1;  // INT8 zero points (0 otherwise)
};

template <bool FP8, bool I8>
__device__ __forceinline__ UnitPages load_unit_pages(const DecodeParams& p, int kvh, const int* trow,
                                                     int npages, int lane) {
  UnitPages u;
  u.e0 = 0;
  u.e1 = 0;
  bool bad0 = false, bad1 = false;
  if (lane < npages) {
    u.e0 = __ldg(trow + lane);
    if (static_cast<unsigned>(u.e0) >= static_cast<unsigned>(p.NB)) { bad0 = true; u.e0 = 0; }
  }
  if (lane + 32 < npages) {
    u.e1 = __ldg(trow + lane + 32);
    if (static_cast<unsigned>(u.e1) >= static_cast<unsigned>(p.NB)) { bad1 = true; u.e1 = 0; }
  }
  u.badm0 = __ballot_sync(kFull, bad0);
  u.badm1 = __ballot_sync(kFull, bad1);
  u.ks0 = u.ks1 = u.vs0 = u.vs1 = 1.f;
  u.kz0 = u.kz1 = u.vz0 = u.vz1 = 0.f;
  if (FP8 && !I8) {
    if (lane < npages) {
      u.ks0 = __ldg(p.k_scale + static_cast<size_t>(u.e0) * p.Hkv + kvh);
      u.vs0 = __ldg(p.v_scale + static_cast<size_t>(u.e0) * p.Hkv + kvh);
    }
    if (lane + 32 < npages) {
      u.ks1 = __ldg(p.k_scale + static_cast<size_t>(u.e1) * p.Hkv + kvh);
      u.vs1 = __ldg(p.v_scale + static_cast<size_t>(u.e1) * p.Hkv + kvh);
    }
  } else if (I8) {
    const float2* kp2 = reinterpret_cast<const float2*>(p.k_scale);
    const float2* vp2 = reinterpret_cast<const float2*>(p.v_scale);
    if (lane < npages) {
      const float2 a = __ldg(kp2 + static_cast<size_t>(u.e0) * p.Hkv + kvh);
      const float2 c = __ldg(vp2 + static_cast<size_t>(u.e0) * p.Hkv + kvh);
      u.ks0 = a.x; u.kz0 = a.y; u.vs0 = c.x; u.vz0 = c.y;
    }
    if (lane + 32 < npages) {
      const float2 a = __ldg(kp2 + static_cast<size_t>(u.e1) * p.Hkv + kvh);
      const float2 c = __ldg(vp2 + static_cast<size_t>(u.e1) * p.Hkv + kvh);
      u.ks1 = a.x; u.kz1 = a.y; u.vs1 = c.x; u.vz1 = c.y;
    }
  }
  return u;
}

// Page j's value of a per-lane pair (lane j holds pages j, j + 32); warp-wide.
__device__ __forceinline__ float unit_pick(float v0, float v1, int j) {
  return (j < 32) ? __shfl_sync(kFull, v0, j & 31) : __shfl_sync(kFull, v1, j & 31);
}
__device__ __forceinline__ int unit_pick(int v0, int v1, int j) {
  return (j < 32) ? __shfl_sync(kFull, v0, j & 31) : __shfl_sync(kFull, v1, j & 31);
}
__device__ __forceinline__ bool unit_bad(const UnitPages& u, int j) {
  return (j < 32) ? ((u.badm0 >> (j & 31)) & 1u) : ((u.badm1 >> (j & 31)) & 1u);
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
// MT: multi-token queries (T >= 1, row tiles, per-row causal limits);
// false: single-token kernels, T = 1 only.
template <int D, int BS, bool FP8, int MATH, int GT, bool I8 = false, bool MT = false>
__global__ void __launch_bounds__(256, 1)
    paged_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const DecodeParams p) {
  using Geo = PageGeom<D, BS, FP8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const int R = p.stages;
  uint8_t* ring = smem + static_cast<size_t>(warp) * R * Geo::kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(nwarps) * R * Geo::kStageBytes) + warp * 8;
  float* pbuf = reinterpret_cast<float*>(smem + static_cast<size_t>(nwarps) * R * Geo::kStageBytes +
                                         nwarps * 8 * sizeof(uint64_t)) + warp * BS * 16;

  if (lane == 0) {
    for (int s = 0; s < R; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
    if (warp == 0) {
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
    }
  }
  __syncwarp();
  // Pages are read once, except by the row tiles of one (sequence, KV head,
  // partition), which are adjacent units: keep those lines in L2 then.
  const uint64_t policy = (MT && p.NT > 1) ? l2_policy_evict_normal() : l2_policy_evict_first();
  pdl_trigger();
  pdl_wait();  // the planner's output and every input are complete from here on

  const int units_per_part = MT ? p.Hkv * p.NT : p.Hkv;
  const int total_units = p.unit_start[p.B] * units_per_part;
  uint32_t it = 0;  // pages this warp has consumed (stage = it % R, phase = (it / R) & 1)
  const int ppu_tokens = p.ppu * BS;

  for (;;) {
    int u = 0;
    if (lane == 0) u = atomicAdd(p.work_counter, 1);
    u = __shfl_sync(kFull, u, 0);
    if (u >= total_units) break;
    const int part = u / units_per_part;
    const int rem = u - part * units_per_part;
    const int kvh = MT ? rem / p.NT : rem;
    const int tile = MT ? rem - kvh * p.NT : 0;
    const int b = __ldg(p.part_seq + part);  // the sequence owning global partition `part`
    const int pidx = part - __ldg(p.unit_start + b);
    const int nparts = __ldg(p.unit_start + b + 1) - __ldg(p.unit_start + b);
    const int ctx = __ldg(p.ctx_eff + b);
    const int t0 = pidx * ppu_tokens;
    const int t1 = min(ctx, t0 + ppu_tokens);
    const int npages = (t1 - t0 + BS - 1) / BS;
    const int* trow = p.block_tables + static_cast<size_t>(b) * p.MB + t0 / BS;

    const UnitPages up = load_unit_pages<FP8, I8>(p, kvh, trow, npages, lane);
    if (lane == 0 && (up.badm0 | up.badm1)) atomicOr(p.err, PKV_DEVERR_BLOCK_ID);

    auto issue = [&](int j, uint32_t slot_it) {
      const int phys = unit_pick(up.e0, up.e1, j);
      if (lane == 0) {
        const int s = static_cast<int>(slot_it % static_cast<uint32_t>(R));
        uint8_t* st = ring + static_cast<size_t>(s) * Geo::kStageBytes;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&bars[s], Geo::kStageBytes);
        const int row = p.row_base + (phys * p.Hkv + kvh) * BS;
#pragma unroll
        for (int r = 0; r < Geo::kRegions; ++r)
          tma_load_2d(st + r * Geo::kRegionBytes, &kmap, &bars[s], r * Geo::kBoxInner, row, policy);
#pragma unroll
        for (int r = 0; r < Geo::kRegions; ++r)
          tma_load_2d(st + Geo::kTensorBytes + r * Geo::kRegionBytes, &vmap, &bars[s],
                      r * Geo::kBoxInner, row, policy);
      }
    };

    const int pre = min(R, npages);
    for (int j = 0; j < pre; ++j) issue(j, it + j);
    int issued = pre;  // pages of this unit handed to the copy engine
    int consumed = 0;

    bool timed_out = false;
    if (MATH == PKV_MATH_MMA) {
      constexpr bool kHi = GT > 8;
      constexpr int kR = kHi ? 2 : 1;
      MmaState<D, BS, FP8, kHi> st;
      mma_load_q<D, BS, FP8, kHi, MT>(st, p, b, kvh, tile, lane);
      if constexpr (I8) mma_int8_prepare(st);
      // causal limits: query row g + 8r attends to positions < lim[r];
      // lim_min is the smallest over the tile (T = 1: both are ctx)
      int lim[kR];
#pragma unroll
      for (int r = 0; r < kR; ++r) {
        int t, h;
        tile_row<MT>(p, kvh, tile, (lane >> 2) + 8 * r, t, h);
        lim[r] = MT ? ctx - p.T + 1 + min(t, p.T - 1) : ctx;
      }
      const int lim_min = MT ? ctx - p.T + 1 + tile * p.Tt : ctx;
      for (int j = 0; j < npages; ++j) {
        const uint32_t s = it % static_cast<uint32_t>(R);
        const bool landed = mbar_wait_bounded(&bars[s], (it / R) & 1u, kWaitLimitNs);
        if (!__all_sync(kFull, landed)) { timed_out = true; break; }
        const int valid = unit_bad(up, j) ? 0 : min(BS, t1 - (t0 + j * BS));
        float ksc = 1.f, vsc = 1.f, kc = 0.f, vc = 0.f;
        if (FP8) {
          ksc = unit_pick(up.ks0, up.ks1, j);
          vsc = unit_pick(up.vs0, up.vs1, j);
        }
        if (I8) {
          kc = kInt8Bias + unit_pick(up.kz0, up.kz1, j);
          vc = kInt8Bias + unit_pick(up.vz0, up.vz1, j);
        }
        const int pos0 = t0 + j * BS;
        int rv[kR];
#pragma unroll
        for (int r = 0; r < kR; ++r) rv[r] = MT ? min(valid, lim[r] - pos0) : valid;
        const bool partial = MT ? (valid < BS || lim_min - pos0 < BS) : valid < BS;
        mma_page<D, BS, FP8, kHi, I8>(st, ring + static_cast<size_t>(s) * Geo::kStageBytes, valid, rv,
                                      partial, p.scale_log2 * ksc, vsc, kc, vc, lane);
        fence_proxy_async_smem();  // this lane's reads of the stage precede the refill
        __syncwarp();
        if (j + R < npages) { issue(j + R, it + R); ++issued; }
        ++it;
        ++consumed;
      }
      if (!timed_out) {
        if constexpr (I8) mma_int8_unbias(st);
        mma_finish<D, BS, FP8, kHi, MT>(st, p, b, kvh, tile, pidx, nparts, lane);
        if (nparts > 1 && p.fused_merge) arrive_and_merge<D, MT>(p, b, kvh, tile, nparts, lane);
      }
    } else {
      // single-token queries only (the host rejects T > 1 here)
      const __nv_bfloat16* qg = p.q + (static_cast<size_t>(b) * p.Hq + kvh * p.G) * D;
      FfmaState<D, BS, FP8, (GT > 0 ? GT : 1)> st;
      ffma_load_q<D, BS, FP8, (GT > 0 ? GT : 1)>(st, qg, lane);
      for (int j = 0; j < npages; ++j) {
        const uint32_t s = it % static_cast<uint32_t>(R);
        const bool landed = mbar_wait_bounded(&bars[s], (it / R) & 1u, kWaitLimitNs);
        if (!__all_sync(kFull, landed)) { timed_out = true; break; }
        const int valid = unit_bad(up, j) ? 0 : min(BS, t1 - (t0 + j * BS));
        float ksc = 1.f, vsc = 1.f;
        uint32_t kzc = 0u, vzc = 0u;
        if (FP8) {
          ksc = unit_pick(up.ks0, up.ks1, j);
          vsc = unit_pick(up.vs0, up.vs1, j);
        }
        if (I8) {
          kzc = int8_zero_const(unit_pick(up.kz0, up.kz1, j));
          vzc = int8_zero_const(unit_pick(up.vz0, up.vz1, j));
        }
        ffma_page<D, BS, FP8, (GT > 0 ? GT : 1), I8>(st, ring + static_cast<size_t>(s) * Geo::kStageBytes,
                                                     valid, p.scale_log2 * ksc, vsc, kzc, vzc, pbuf, lane);
        fence_proxy_async_smem();  // this lane's reads of the stage precede the refill
        __syncwarp();
        if (j + R < npages) { issue(j + R, it + R); ++issued; }
        ++it;
        ++consumed;
      }
      if (!timed_out) {
        ffma_finish<D, BS, FP8, (GT > 0 ? GT : 1)>(st, p, b, kvh, pidx, nparts, lane);
        if (nparts > 1 && p.fused_merge) arrive_and_merge<D, false>(p, b, kvh, 0, nparts, lane);
      }
    }
    if (timed_out) {
      // Record the failure, give copies still in flight a bounded chance to
      // land (the stage memory stays owned by this CTA meanwhile), and stop.
      if (lane == 0) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
      for (int k = 1; k < issued - consumed; ++k) {
        const uint32_t q = it + static_cast<uint32_t>(k);
        mbar_wait_bounded(&bars[q % static_cast<uint32_t>(R)], (q / R) & 1u, kWaitLimitNs / 16);
      }
      return;
    }
  }
}

}  // namespace pkv
