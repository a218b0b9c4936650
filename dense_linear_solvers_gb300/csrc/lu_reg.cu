// Dispatch of the register-resident LU kernels (n <= 32) by layout: FP32 orders 9..16 take
// the two-rows-per-lane kernel (lu_rows2.cu); the others the one-row-per-lane kernel and its
// tiers in lu_reg.cuh, instantiated per dtype and layout in lu_reg_*.cu.
#include "common.cuh"
#include "kernels.h"

namespace bsolve {
namespace lu_reg_detail {
template <typename T, int LAYOUT>
cudaError_t launch_layout(int n, int nrhs, int64_t batch, T* A, T* B, int32_t* ipiv,
                          int32_t* info, cudaStream_t stream);
template <typename T, int LAYOUT>
cudaError_t launch_layout_il(int n, int nrhs, int64_t batch, int64_t ilv, T* A, T* B,
                             int32_t* ipiv, int32_t* info, cudaStream_t stream);
}  // namespace lu_reg_detail

template <typename T>
cudaError_t launch_lu_reg_il(int layout, int n, int nrhs, int64_t batch, int64_t ilv, T* A, T* B,
                             int32_t* ipiv, int32_t* info, cudaStream_t stream) {
  if constexpr (sizeof(T) == 4) {
    if (n > 8 && n <= 16)
      return launch_lu_rows2(layout, n, nrhs, batch, A, B, ipiv, info, stream, ilv);
  }
  if (layout == kRowMajor)
    return lu_reg_detail::launch_layout_il<T, kRowMajor>(n, nrhs, batch, ilv, A, B, ipiv, info,
                                                         stream);
  return lu_reg_detail::launch_layout_il<T, kColMajor>(n, nrhs, batch, ilv, A, B, ipiv, info,
                                                       stream);
}

template <typename T>
cudaError_t launch_lu_reg(int layout, int n, int nrhs, int64_t batch, T* A, T* B,
                          int32_t* ipiv, int32_t* info, cudaStream_t stream) {
  if constexpr (sizeof(T) == 4) {
    // FP32 orders 9..16: two rows per lane (four systems per warp)
    if (n > 8 && n <= 16) return launch_lu_rows2(layout, n, nrhs, batch, A, B, ipiv, info, stream);
  }
  if (layout == kRowMajor)
    return lu_reg_detail::launch_layout<T, kRowMajor>(n, nrhs, batch, A, B, ipiv, info, stream);
  return lu_reg_detail::launch_layout<T, kColMajor>(n, nrhs, batch, A, B, ipiv, info, stream);
}

template cudaError_t launch_lu_reg<float>(int, int, int, int64_t, float*, float*, int32_t*,
                                          int32_t*, cudaStream_t);
template cudaError_t launch_lu_reg_il<float>(int, int, int, int64_t, int64_t, float*, float*,
                                             int32_t*, int32_t*, cudaStream_t);
template cudaError_t launch_lu_reg_il<double>(int, int, int, int64_t, int64_t, double*, double*,
                                              int32_t*, int32_t*, cudaStream_t);
template cudaError_t launch_lu_reg<double>(int, int, int, int64_t, double*, double*, int32_t*,
                                           int32_t*, cudaStream_t);

}  // namespace bsolve
