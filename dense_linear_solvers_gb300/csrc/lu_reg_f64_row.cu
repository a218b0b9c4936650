// Instances of the register-resident LU kernel for one dtype and one layout (split into
// several translation units so that they compile in parallel).
#include "lu_reg.cuh"

namespace bsolve {
namespace lu_reg_detail {
template cudaError_t launch_layout<double, kRowMajor>(int, int, int64_t, double*, double*, int32_t*,
                                                int32_t*, cudaStream_t);
}  // namespace lu_reg_detail
}  // namespace bsolve
