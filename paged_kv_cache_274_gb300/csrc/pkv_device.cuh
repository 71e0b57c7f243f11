// Device-side building blocks for the sm_103a kernels: mbarriers, tensor-map
// bulk copies (TMA), ldmatrix, mma.sync and small conversions.  Inline PTX,
// no library code.
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "pkv.h"

namespace pkv {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// programmatic dependent launch: a kernel launched with the programmatic
// stream-serialisation attribute may start before the previous kernel on the
// stream has finished; it must call pdl_wait() before touching memory that
// kernel writes.  pdl_trigger() lets the next such kernel start launching.
// Both are no-ops for kernels launched without the attribute.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Makes barrier initialisation visible to the asynchronous (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later asynchronous-proxy (TMA) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// One arrival without transaction bytes (release at CTA scope).
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for phase `parity` of `bar` to complete; gives up after `limit_ns`
// nanoseconds of wall time and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// Bounded wait for threads on the critical path of a pipeline (the tcgen05
// issuing thread): the phase is first tested without suspending -- a
// try_wait on a completed phase still costs on the order of a hundred
// cycles -- then waited for with suspending try_waits.
__device__ __forceinline__ bool mbar_test_wait_fwd(uint64_t* bar, uint32_t parity);
__device__ __forceinline__ bool mbar_wait_fast(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_test_wait_fwd(bar, parity)) return true;
  return mbar_wait_bounded(bar, parity, limit_ns);
}

// Non-blocking test of phase `parity`.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_test_wait_fwd(uint64_t* bar, uint32_t parity) { return mbar_test_wait(bar, parity); }

// Same as mbar_wait_bounded, spinning on the non-blocking test instead of the
// potentially suspending try_wait: for phases that complete within a
// microsecond, where a suspended thread could wake up late.  A spinning warp
// takes issue slots from the other warps of its sub-partition, so whole warps
// that wait while others compute on the same sub-partition (the tcgen05
// kernel's compute warps waiting for S) use mbar_wait_bounded.  The clock is
// read only once the phase is found open, so a phase that has already
// completed costs one test.
__device__ __forceinline__ bool mbar_wait_spin(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_test_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// ---------------------------------------------------------------------------
// tensor-map bulk copies
// ---------------------------------------------------------------------------
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled copy global -> shared; completion is signalled on `bar` as
// transaction bytes.  x must be a multiple of 16 bytes worth of elements.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// 5-D tiled copy shared -> global (a tensor-map store); completion is
// tracked with bulk async-groups of the issuing thread.
__device__ __forceinline__ void tma_store_5d(const CUtensorMap* map, const void* src, int32_t c0, int32_t c1,
                                             int32_t c2, int32_t c3, int32_t c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5, %6}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_addr(src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, const void* src, int32_t c0, int32_t c1,
                                             int32_t c2, int32_t c3) {
  asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_addr(src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// This thread's bulk stores have finished reading their shared-memory sources.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// All but this thread's most recent bulk store have read their sources.
__device__ __forceinline__ void bulk_wait_read_but1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// This thread's bulk stores are complete (written to global memory).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// L2 policy for data read exactly once per step (the KV stream).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// ---------------------------------------------------------------------------
// ldmatrix / mma.sync
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Two 16x16-byte tiles, transposed: lanes 0-15 give the row addresses of
// tile 0, lanes 16-31 those of tile 1.  Lane 4g + t receives, per tile, the
// bytes of rows 4t..4t+3 in column g (first register) and in column g + 8
// (second register).
__device__ __forceinline__ void ldsm_x2_t_b8(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                             uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m16n16.x2.trans.shared.b8 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D = A(16x16, row) * B(16x8, col) + D, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Same with f16 inputs.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Variants for tiles whose rows 8..15 of A are zero (at most 8 heads in the
// group): only the lower half of C/D is carried; the upper half is fed zeros
// and its results are discarded.  a0 = A(row g, k 2t..2t+1), a2 = A(row g,
// k 2t+8..2t+9).
__device__ __forceinline__ void mma_bf16_lo(float (&d)[2], uint32_t a0, uint32_t a2, uint32_t b0,
                                            uint32_t b1) {
  float u0, u1;  // rows 8..15 of D: zeros, discarded
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%5}, "
      "{%7,%8}, {%0,%1,%9,%9};"
      : "+f"(d[0]), "+f"(d[1]), "=f"(u0), "=f"(u1)
      : "r"(a0), "r"(0u), "r"(a2), "r"(b0), "r"(b1), "f"(0.f));
  asm volatile("" ::"f"(u0), "f"(u1));  // consumed here; emits nothing
}

__device__ __forceinline__ void mma_f16_lo(float (&d)[2], uint32_t a0, uint32_t a2, uint32_t b0,
                                           uint32_t b1) {
  float u0, u1;
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%5}, "
      "{%7,%8}, {%0,%1,%9,%9};"
      : "+f"(d[0]), "+f"(d[1]), "=f"(u0), "=f"(u1)
      : "r"(a0), "r"(0u), "r"(a2), "r"(b0), "r"(b1), "f"(0.f));
  asm volatile("" ::"f"(u0), "f"(u1));  // consumed here; emits nothing
}

// 2^x with the SFU's approximate exponential (relative error about 2^-22;
// results below 2^-126 flush to zero, -inf gives 0).
// Packed pairs of fp32 operations (one instruction for two lanes of work on
// sm_100 and later): d = a * b + c and d = a + b, element-wise, round to
// nearest even, as two separate fmaf / multiplications / additions would
// round them.
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b0, float b1, float c0,
                                      float c1) {
  uint64_t d;
  asm("{\n .reg .b64 ra, rb, rc;\n mov.b64 ra, {%1, %2};\n mov.b64 rb, {%3, %4};\n mov.b64 rc, {%5, %6};\n"
      " fma.rn.f32x2 %0, ra, rb, rc;\n}\n"
      : "=l"(d)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
  d0 = __uint_as_float(static_cast<uint32_t>(d));
  d1 = __uint_as_float(static_cast<uint32_t>(d >> 32));
}
__device__ __forceinline__ void fmul2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  uint64_t d;
  asm("{\n .reg .b64 ra, rb;\n mov.b64 ra, {%1, %2};\n mov.b64 rb, {%3, %4};\n mul.rn.f32x2 %0, ra, rb;\n}\n"
      : "=l"(d)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
  d0 = __uint_as_float(static_cast<uint32_t>(d));
  d1 = __uint_as_float(static_cast<uint32_t>(d >> 32));
}
__device__ __forceinline__ void fadd2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  uint64_t d;
  asm("{\n .reg .b64 ra, rb;\n mov.b64 ra, {%1, %2};\n mov.b64 rb, {%3, %4};\n add.rn.f32x2 %0, ra, rb;\n}\n"
      : "=l"(d)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
  d0 = __uint_as_float(static_cast<uint32_t>(d));
  d1 = __uint_as_float(static_cast<uint32_t>(d >> 32));
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// conversions
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Four E4M3 codes (byte i = element i) -> two f16x2 words: lo = elements
// (0, 1), hi = elements (2, 3).  The 32-bit word is split into its 16-bit
// halves and each half converted by the hardware (exact).
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t x, uint32_t& lo, uint32_t& hi) {
  asm("{\n"
      " .reg .b16 l, h;\n"
      " mov.b32 {l, h}, %2;\n"
      " cvt.rn.f16x2.e4m3x2 %0, l;\n"
      " cvt.rn.f16x2.e4m3x2 %1, h;\n"
      "}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(x));
}

// Four INT8 codes (byte i = element i) -> two f16x2 words holding
// (code - zero): lo = elements (0, 1), hi = elements (2, 3).  Flipping the
// sign bit gives code + 128 in 0..255; that byte placed under the f16
// exponent of 1024 (high byte 0x64) is the f16 value 1024 + code + 128, and
// subtracting zc = f16x2(1152 + zero) leaves code - zero.  Every value here
// is an integer of magnitude <= 2048, so all of it is exact in f16.
__device__ __forceinline__ void int8x4_to_f16x2x2(uint32_t x, uint32_t zc, uint32_t& lo, uint32_t& hi) {
  const uint32_t y = x ^ 0x80808080u;
  const uint32_t l = __byte_perm(y, 0x64646464u, 0x4140);
  const uint32_t h = __byte_perm(y, 0x64646464u, 0x4342);
  const __half2 z = *reinterpret_cast<const __half2*>(&zc);
  const __half2 lh = __hsub2(*reinterpret_cast<const __half2*>(&l), z);
  const __half2 hh = __hsub2(*reinterpret_cast<const __half2*>(&h), z);
  lo = *reinterpret_cast<const uint32_t*>(&lh);
  hi = *reinterpret_cast<const uint32_t*>(&hh);
}

// Four INT8 codes -> two f16x2 words holding 1152 + code (exact): the same
// sign flip and exponent placement as int8x4_to_f16x2x2 without the
// subtraction, for callers that remove the constant 1152 + zero after the
// product (it is the same for every element of a page).
__device__ __forceinline__ void int8x4_to_f16x2x2_biased(uint32_t x, uint32_t& lo, uint32_t& hi) {
  const uint32_t y = x ^ 0x80808080u;
  lo = __byte_perm(y, 0x64646464u, 0x4140);
  hi = __byte_perm(y, 0x64646464u, 0x4342);
}

// Bias of int8x4_to_f16x2x2_biased: the f16 value of code 0 before the flip.
constexpr float kInt8Bias = 1152.f;

// f16x2 constant (1152 + zero, 1152 + zero) for int8x4_to_f16x2x2.
__device__ __forceinline__ uint32_t int8_zero_const(float zero) {
  const __half h = __float2half_rn(1152.f + zero);
  const uint16_t b = *reinterpret_cast<const uint16_t*>(&h);
  return static_cast<uint32_t>(b) | (static_cast<uint32_t>(b) << 16);
}

// bf16 pair in a 32-bit word -> two floats (exact).
__device__ __forceinline__ float bf16lo_to_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// ---------------------------------------------------------------------------
// tcgen05 (5th-generation tensor cores): TMEM allocation, MMA from shared
// memory descriptors, commit to an mbarrier, TMEM loads and stores
// ---------------------------------------------------------------------------
// Shared-memory matrix descriptor: start address, leading-dimension byte
// offset (K-major: between core matrices adjacent along K), stride byte
// offset (between 8-row groups along M/N), version 1, layout
// (0 = no swizzle, 2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t tc_smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(layout & 7u) << 61;
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, f32 D, M x N; A K-major,
// B K-major or (b_mn_major, bit 16) MN-major.
__host__ __device__ constexpr uint32_t tc_idesc_bf16_f32(int M, int N, bool b_mn_major = false) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn_major ? (1u << 16) : 0u) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
// The same with f16 A and B (both operands of a kind::f16 product have one
// type).
__host__ __device__ constexpr uint32_t tc_idesc_f16_f32(int M, int N, bool b_mn_major = false) {
  return (1u << 4) | (b_mn_major ? (1u << 16) : 0u) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
// kind::f8f6f4 with E4M3 A and B (format code 0 in both fields), fp32 D,
// both K-major.
__host__ __device__ constexpr uint32_t tc_idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] . B[smem]^T; issued by one thread.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u));
}

// D[tmem] (+)= A[tmem] . B[smem]^T: A read from tensor memory (row i of A in
// lane i, two bf16 per 32-bit column, K along the columns); one thread.
__device__ __forceinline__ void tc_mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                               bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u));
}

// D[tmem] (+)= A[tmem] . B[smem]^T with E4M3 A and B (kind::f8f6f4, fp32
// accumulate): row i of A in lane i, four E4M3 values per 32-bit column
// (byte j = element 4c + j), so a product of K 32 reads 8 columns; B K-major
// in shared memory (32 bytes of each row per product).  One thread.
__device__ __forceinline__ void tc_mma_e4m3_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                               bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u));
}

// The MMAs this thread issued so far arrive on `bar` when complete.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Whole warp: allocate / free `ncols` TMEM columns (power of 2, >= 32); the
// base address is written to *slot (shared memory).
__device__ __forceinline__ void tc_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(slot)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Whole warp: registers to 16 consecutive 32-bit TMEM columns of this
// thread's lane.
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// Whole warp: 32 consecutive 32-bit columns of this thread's TMEM lane
// (warp w of the CTA reads lanes 32w .. 32w + 31).
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
      "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Byte offset of 16-byte chunk `chunk` of 128-byte row `row` inside a region
// written by a tensor-map copy with 128-byte swizzling (region base aligned
// to 1024 bytes): chunk index XOR (row mod 8).
__device__ __forceinline__ uint32_t swz128(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

}  // namespace pkv
