// Read-only HBM probe: streams a buffer once and sums its 32-bit words.
//
// A measurement aid beside the decode, not part of it.  The decode reads its
// cache and writes almost nothing, while the copy rate the roofline uses
// moves read and write traffic; this probe gives the read-only rate of the
// same device ("KV Cache Engineering: PagedAttention, Continuous Batching,
// Attention Variants, and the Bandwidth Wall", "Two Costs: Capacity and
// Bandwidth": a decode step is bound by how fast the cache streams from HBM).
// The sum keeps every load live and lets a test check that every byte was
// read.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

constexpr int kProbeThreads = 256;
constexpr int kProbeCtasPerSm = 8;   // 2048 threads per SM
constexpr int kProbeUnroll = 4;      // 16-byte loads in flight per thread

__global__ void __launch_bounds__(kProbeThreads)
    read_probe_kernel(const uint4* __restrict__ src, size_t n16, unsigned long long* __restrict__ sum) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  unsigned long long acc = 0;
  auto add = [&](const uint4& v) {
    acc += static_cast<unsigned long long>(v.x) + v.y + static_cast<unsigned long long>(v.z) + v.w;
  };
  for (; i + (kProbeUnroll - 1) * stride < n16; i += kProbeUnroll * stride) {
    uint4 v[kProbeUnroll];
#pragma unroll
    for (int u = 0; u < kProbeUnroll; ++u) v[u] = __ldcs(src + i + u * stride);
#pragma unroll
    for (int u = 0; u < kProbeUnroll; ++u) add(v[u]);
  }
  for (; i < n16; i += stride) add(__ldcs(src + i));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0 && acc != 0) atomicAdd(sum, acc);
}

cudaError_t launch_read_probe(const void* data, size_t bytes, unsigned long long* sum, int num_sms,
                              cudaStream_t stream) {
  const size_t n16 = bytes / 16;
  if (n16 == 0) return cudaSuccess;
  const size_t want = (n16 + kProbeThreads - 1) / kProbeThreads;
  const size_t cap = static_cast<size_t>(num_sms) * kProbeCtasPerSm;
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  read_probe_kernel<<<grid, kProbeThreads, 0, stream>>>(static_cast<const uint4*>(data), n16, sum);
  return cudaGetLastError();
}

}  // namespace pkv
