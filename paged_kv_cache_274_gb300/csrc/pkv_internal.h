// Host-side plumbing shared by the library's translation units (not part of
// the public ABI).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "pkv.h"

namespace pkv {

// One KV append, resolved and validated by the API layer: rows of N tokens
// [N][Hkv][D] bf16 into the selected cache slot's pages.
struct AppendArgs {
  const uint4* k;
  const uint4* v;
  const int64_t* slot_mapping;
  int N, Hkv, D, bs;
  int64_t nslots;
  uint8_t* kc;  // the slot's K pages
  uint8_t* vc;
  const float* ks;  // the slot's page parameters (one-byte caches)
  const float* vs;
  unsigned* err;
};

// Everything one decode launch needs, resolved and validated by the API layer.
struct DecodeLaunch {
  const void* q;
  void* out;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const float* k_scale;  // already offset to the selected slot (E4M3 only)
  const float* v_scale;
  int32_t* work_counter;  // workspace: dynamic work queue head
  int32_t* unit_start;    // workspace: [B+1] prefix of partitions per sequence
  int32_t* ctx_eff;       // workspace: [B] validated context lengths
  int32_t* part_seq;      // workspace: [B * pmax] sequence of each global partition
  int32_t* arrive;        // workspace: [B][Hkv][NT] split-K partitions finished
  float* part_ml;         // workspace: [B][T][Hq][pmax][2] (running max, sum)
  float* part_o;          // workspace: [B][T][Hq][pmax][D]
  unsigned* err;          // device error word
  int B, Hq, Hkv, G, MB, NB, bs, D;
  int T;   // query tokens per sequence (1: single-token decode)
  int Tt;  // query tokens per row tile (G * Tt <= 16 rows)
  int NT;  // row tiles per (sequence, KV head): ceil(T / Tt)
  int tc;  // 1: tcgen05 kernel (128-row tiles, math PKV_MATH_TC)
  int tc2; // 1: the tcgen05 kernel that serves a pair of row tiles per CTA (NT >= 2)
  int kv_fp8;    // one-byte elements (E4M3 or INT8)
  int kv_dtype;  // pkv_kv_dtype
  int pmax;  // max partitions of a sequence (ceil(MB / ppu), or ceil(MB / ppu_half))
  int ppu;   // pages (blocks) per partition
  // sequences half_from .. B - 1 take partitions of ppu_half blocks (the
  // tile-pair kernel's balancing of the last round of units; B: none)
  int half_from, ppu_half;
  int row_base;  // first tensor-map row of the selected slot
  float scale_log2;
  int math;    // PKV_MATH_FFMA or PKV_MATH_MMA (resolved)
  int warps;   // per CTA
  int stages;  // per warp
  CUtensorMap kmap, vmap;
  CUtensorMap pmap;  // tcgen05 kernel with split-K: store map of part_o ([B][T][Hq][pmax][D] fp32)
  CUtensorMap omap;  // tcgen05 kernel: store map of out ([B][T][Hq][D] bf16)
  CUtensorMap qmap;  // tile-pair kernel: load map of q ([B][T][Hq][D] bf16, box 64 x G x Tt)
  cudaStream_t stream;
  int num_sms;
  cudaEvent_t ev_start, ev_end;  // optional, recorded around the decode kernel
  const AppendArgs* append;  // optional: append run by the planner launch (the decode sees it)
  int append_kind;           // pkv_kv_dtype of that append
};

// Workspace layout for one decode call.
struct WorkspaceLayout {
  size_t counter, unit_start, ctx_eff, part_seq, arrive, part_ml, part_o, total;
};
WorkspaceLayout workspace_layout(int B, int T, int Hq, int Hkv, int NT, int D, int pmax);

// Programmatic dependent launch on (default) or off (PKV_PDL=0).
bool pdl_enabled();

// Shared memory per CTA of the decode kernel.
// pages a tcgen05 work unit may span (its descriptor slot's page table)
constexpr int kTcUnitMaxPages = 256;
// warps per CTA of the tile-pair tcgen05 kernel (8 softmax, MMA, 2 copy)
constexpr int kTcPairWarps = 11;
size_t decode_smem_bytes(int kv_fp8, int D, int bs, int warps, int stages, int tc, int tc2 = 0);

// Launch planner + decode (the decode merges split-K partials itself).  Returns cudaSuccess or
// the first launch error.
cudaError_t launch_decode(const DecodeLaunch& L, int* launched_kernels);

// Decode kernel occupancy (CTAs per SM) for a configuration.
int decode_ctas_per_sm(const DecodeLaunch& L, size_t smem);

// Replace the calling thread's pkv_last_error_message() text.
void set_last_error_message(const char* msg);

// The calling thread's current CUDA context (a CUcontext), or NULL when none
// is current.  Device addresses of the library's __device__ variables and
// kernel attributes belong to one context; a cache of them is valid only
// while the context it was filled in stays current.
void* current_context();

// KV append.
cudaError_t launch_kv_append(int kv_dtype, const AppendArgs& a, cudaStream_t stream);

// Block copy between two pools of the same page shape.
cudaError_t launch_copy_blocks(const void* src_k, const void* src_v, const float* src_ks,
                               const float* src_vs, int src_nb, void* dst_k, void* dst_v,
                               float* dst_ks, float* dst_vs, int dst_nb, const int32_t* pairs,
                               int count, int64_t block_bytes, int scales_per_block,
                               int num_sms, unsigned* err, cudaStream_t stream);

// Read-only probe: sums the 32-bit words of `bytes` bytes (a multiple of 16,
// 16-byte aligned) into *sum; one launch of up to 8 CTAs per SM.
cudaError_t launch_read_probe(const void* data, size_t bytes, unsigned long long* sum, int num_sms,
                              cudaStream_t stream);

}  // namespace pkv
