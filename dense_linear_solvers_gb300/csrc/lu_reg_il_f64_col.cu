// Instances of the register-resident LU kernel on the interleaved batched layout, one
// dtype and storage order per translation unit (so that they compile in parallel).
#include "lu_reg.cuh"

namespace bsolve {
namespace lu_reg_detail {
template cudaError_t launch_layout_il<double, kColMajor>(int, int, int64_t, int64_t, double*, double*,
                                                    int32_t*, int32_t*, cudaStream_t);
}  // namespace lu_reg_detail
}  // namespace bsolve
