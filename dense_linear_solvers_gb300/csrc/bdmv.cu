// Block-tridiagonal matrix-vector product y = A x (GLASS API reference, "Block-tridiagonal
// Ops", section "Block-tridiagonal matrix-vector product (glass::bdmv)"): block-row br of a
// system is a BS x 3BS row-major strip [L | D | R]; it reads the padded window
// x[br*BS, br*BS + 3BS) and writes y[(br+1)*BS + row]. The pads of y are not written.
//
// The work is one pass over the strips (24 reads per 2 flops at BS = 8): HBM bound. One
// thread per output row reads its contiguous strip row with 16-byte loads (consecutive
// threads take consecutive rows, so a warp streams one contiguous stretch of the strip
// array) and its window of x through the read-only cache (each x entry serves the BS
// rows of a block-row and the neighbouring block-rows). Each entry is one dot product in
// increasing column order, one fused multiply-add per term from zero: the CPU oracle's
// order, so results are bit-identical.
//
// Grid: blockIdx.x covers the rows of one system, blockIdx.y strides over the systems, so
// no thread divides by the system size.
#include "common.cuh"
#include "kernels.h"

namespace bsolve {
namespace {

// DUAL: the page's second form, the same product stored into a second padded output too
template <typename T, int BS, bool DUAL>
__global__ void __launch_bounds__(256)
bdmv_kernel(int nbr, int64_t batch, const T* __restrict__ strips, const T* __restrict__ xpad,
            T* __restrict__ ypad, T* __restrict__ ypad2) {
  constexpr int W = 3 * BS;
  constexpr bool kVec = (W * sizeof(T)) % 16 == 0;
  constexpr int V = 16 / sizeof(T);
  const int per = nbr * BS;                       // rows per system
  const int within = blockIdx.x * blockDim.x + threadIdx.x;
  if (within >= per) return;
  const int br = within / BS;
  const int r = within - br * BS;
  const int64_t vstride = static_cast<int64_t>(nbr + 2) * BS;
  for (int64_t s = blockIdx.y; s < batch; s += gridDim.y) {
    const T* srow = strips + (s * per + within) * W;
    const T* xw = xpad + s * vstride + static_cast<int64_t>(br) * BS;
    T v[W];
    if constexpr (kVec) {
#pragma unroll
      for (int c = 0; c < W; c += V) {
        if constexpr (sizeof(T) == 8) {
          const double2 q = __ldg(reinterpret_cast<const double2*>(srow + c));
          v[c] = q.x;
          v[c + 1] = q.y;
        } else {
          const float4 q = __ldg(reinterpret_cast<const float4*>(srow + c));
          v[c] = q.x;
          v[c + 1] = q.y;
          v[c + 2] = q.z;
          v[c + 3] = q.w;
        }
      }
    } else {
#pragma unroll
      for (int c = 0; c < W; ++c) v[c] = __ldg(srow + c);
    }
    T acc = T(0);
#pragma unroll
    for (int c = 0; c < W; ++c) acc = fma_rn<T>(v[c], __ldg(xw + c), acc);
    const int64_t at = s * vstride + static_cast<int64_t>(br + 1) * BS + r;
    ypad[at] = acc;
    if constexpr (DUAL) ypad2[at] = acc;
  }
}

template <typename T, int BS>
cudaError_t launch_bs(int nbr, int64_t batch, const T* strips, const T* xpad, T* ypad,
                      T* ypad2, cudaStream_t stream) {
  const int per = nbr * BS;
  const int threads = per >= 256 ? 256 : (per + 31) / 32 * 32;
  const int64_t bx = (per + threads - 1) / threads;
  if (bx > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  const unsigned by = static_cast<unsigned>(batch < 65535 ? batch : 65535);
  const dim3 grid(static_cast<unsigned>(bx), by);
  if (ypad2 != nullptr)
    bdmv_kernel<T, BS, true><<<grid, threads, 0, stream>>>(nbr, batch, strips, xpad, ypad, ypad2);
  else
    bdmv_kernel<T, BS, false><<<grid, threads, 0, stream>>>(nbr, batch, strips, xpad, ypad,
                                                            nullptr);
  return cudaGetLastError();
}

}  // namespace

template <typename T>
cudaError_t launch_bdmv(int nbr, int bs, int64_t batch, const T* strips, const T* xpad, T* ypad,
                        T* ypad2, cudaStream_t stream) {
  switch (bs) {
    case 1: return launch_bs<T, 1>(nbr, batch, strips, xpad, ypad, ypad2, stream);
    case 2: return launch_bs<T, 2>(nbr, batch, strips, xpad, ypad, ypad2, stream);
    case 3: return launch_bs<T, 3>(nbr, batch, strips, xpad, ypad, ypad2, stream);
    case 4: return launch_bs<T, 4>(nbr, batch, strips, xpad, ypad, ypad2, stream);
    case 5: return launch_bs<T, 5>(nbr, batch, strips, xpad, ypad, ypad2, stream);
    case 6: return launch_bs<T, 6>(nbr, batch, strips, xpad, ypad, ypad2, stream);
    case 7: return launch_bs<T, 7>(nbr, batch, strips, xpad, ypad, ypad2, stream);
    case 8: return launch_bs<T, 8>(nbr, batch, strips, xpad, ypad, ypad2, stream);
    default: return cudaErrorInvalidValue;
  }
}

template cudaError_t launch_bdmv<float>(int, int, int64_t, const float*, const float*, float*,
                                        float*, cudaStream_t);
template cudaError_t launch_bdmv<double>(int, int, int64_t, const double*, const double*,
                                         double*, double*, cudaStream_t);

}  // namespace bsolve
