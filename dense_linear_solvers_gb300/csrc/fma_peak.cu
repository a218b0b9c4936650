// Arithmetic-throughput probe: independent fused multiply-add chains in FP32 or
// FP64, used to measure the plain-ALU peak that the FP64-bound solvers are judged
// against. Each thread runs CHAINS independent chains so that the FMA pipe, not
// the dependency latency, limits the rate. flops per launch =
// 2 * CHAINS * UNROLL * iters * blocks * threads.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

constexpr int CHAINS = 8;
constexpr int UNROLL = 8;

template <typename T>
__global__ void fma_chains_kernel(T* __restrict__ sink, int iters, T a, T b) {
  T x[CHAINS];
#pragma unroll
  for (int c = 0; c < CHAINS; ++c) x[c] = T(threadIdx.x + c) * T(1e-3);
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
#pragma unroll
      for (int c = 0; c < CHAINS; ++c) x[c] = fma(x[c], a, b);
    }
  }
  T s = T(0);
#pragma unroll
  for (int c = 0; c < CHAINS; ++c) s += x[c];
  // The store keeps the chains alive; every thread writes its own slot.
  sink[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

}  // namespace

#define BS_PROBE_API extern "C" __attribute__((visibility("default")))

BS_PROBE_API int bs_probe_fma_launch(int dtype, int blocks, int threads, int iters, void* sink,
                                     void* stream) {
  if (blocks <= 0 || threads <= 0 || threads > 1024 || iters <= 0 || sink == nullptr)
    return 1;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == 0) {
    fma_chains_kernel<float><<<blocks, threads, 0, s>>>(static_cast<float*>(sink), iters,
                                                        0.999999f, 1e-6f);
  } else if (dtype == 1) {
    fma_chains_kernel<double><<<blocks, threads, 0, s>>>(static_cast<double*>(sink), iters,
                                                         0.999999999, 1e-9);
  } else {
    return 1;
  }
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

BS_PROBE_API int64_t bs_probe_fma_flops_per_thread_iter(void) { return 2LL * CHAINS * UNROLL; }
