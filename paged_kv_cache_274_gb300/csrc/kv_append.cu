// The standalone KV append launch (the chunk loop is in kv_append.cuh).
#include <algorithm>

#include "kv_append.cuh"
#include "pkv_internal.h"

namespace pkv {

template <int KV>  // pkv_kv_dtype
__global__ void __launch_bounds__(256) kv_append_kernel(const AppendArgs a) {
  pdl_trigger();
  pdl_wait();  // inputs may come from the previous kernel on the stream
  append_chunks<KV>(a, blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x,
                    static_cast<int64_t>(gridDim.x) * blockDim.x);
}

cudaError_t launch_kv_append(int kv_dtype, const AppendArgs& a, cudaStream_t stream) {
  const int64_t total = 2LL * a.N * a.Hkv * (a.D / 8);
  const int threads = 256;
  const int64_t blocks = std::min<int64_t>((total + threads - 1) / threads, 1 << 16);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(threads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  auto kernel = kv_dtype == PKV_KV_INT8        ? kv_append_kernel<PKV_KV_INT8>
                : kv_dtype == PKV_KV_FP8_E4M3 ? kv_append_kernel<PKV_KV_FP8_E4M3>
                                              : kv_append_kernel<PKV_KV_BF16>;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

}  // namespace pkv
