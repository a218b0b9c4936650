// potrs for FP64, n <= 32, one right-hand side: one system per lane.
//
// On this part the FP64 pipe charges a warp instruction whatever its active lanes, and the
// substitution sweeps of one small system have a scalar step per column (the reciprocal of
// the diagonal and the scaling of y_k) that a row-per-lane layout runs with one useful
// lane per system. Here lane l of a warp owns system s0 + l whole, y in registers, so every
// FP64 instruction of the warp does the work of 32 systems. The factor is streamed column
// by column through shared memory (cp.async), one odd-pitch row per system so that the 32
// lanes reading entry i of their own column hit distinct banks. Occupancy sets the speed
// (the FP64 pipe is fed by many warps, none of which has much independent work): one
// warp per block, one column buffer per warp, and the diagonal reciprocals of the forward
// sweep parked in the system's own slots of B (dead between the load of b and the store
// of x) instead of registers, so that 20 warps fit on an SM (FP64 n=32: 0.79 ms with
// double-buffered columns and the reciprocals in registers at 12 warps per SM, 0.70 ms
// here).
//
// Arithmetic (the CPU oracle's, operation by operation): forward, for k = 0..n-1:
// y_k = b_k * (1/l_kk), then b_i -= l_ik y_k for i > k (column k of L); backward, for
// i = n-1..0: b_i -= l_ki x_k for k = n-1 down to i+1 (column i of L, the same updates of
// b_i in the same decreasing-k order as the column sweep of L^T x = y), then
// x_i = b_i * (1/l_ii). Every update one fused multiply-add.
#include "common.cuh"
#include "kernels.h"

namespace bsolve {
namespace {

constexpr int kLaneWarps = 1;

// 20 blocks per SM when n is the tier's order; the guarded instances (runtime n) keep
// more values live and get a looser bound, which they fill without spilling
template <int NT, bool FULL>
__global__ void __launch_bounds__(kLaneWarps * 32, FULL ? 20 : 12)
potrs_lane_kernel(int n_, int alay, int64_t batch, const double* __restrict__ L,
                  double* __restrict__ B, const int32_t* __restrict__ zinfo) {
  constexpr int P = NT + 1;                     // pitch of a system's staged column
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n = FULL ? NT : n_;
  const int64_t s0 = (static_cast<int64_t>(blockIdx.x) * kLaneWarps + warp) * 32;
  if (s0 >= batch) return;                      // whole warp; no block barrier below
  const int nsys = batch - s0 < 32 ? static_cast<int>(batch - s0) : 32;
  const int64_t s = s0 + lane;
  const bool valid = lane < nsys;
  const int64_t nn = static_cast<int64_t>(n) * n;
  double* const buf = reinterpret_cast<double*>(smem_raw) + warp * 32 * P;
  double* const Bs = B + s * n;                 // this lane's b, x (and the reciprocals)

  // rows r0..n-1 of column c of the warp's systems into the buffer; lane = row
  auto stage = [&](int c, int r0) {
    const int i = r0 + lane;
    if (i < n) {
      const int64_t off =
          alay == kColMajor ? static_cast<int64_t>(c) * n + i : static_cast<int64_t>(i) * n + c;
      double* dst = buf + i;
      const double* src = L + s0 * nn + off;
      for (int j = 0; j < nsys; ++j) cp_async_elem<double>(dst + j * P, src + j * nn);
    }
    cp_async_commit();
  };

  double y[NT];
#pragma unroll
  for (int i = 0; i < NT; ++i) y[i] = (valid && (FULL || i < n)) ? Bs[i] : 0.0;

  const double* const col = buf + lane * P;
  // forward: L y = b by columns; 1/l_kk goes to slot k of B
#pragma unroll
  for (int k = 0; k < NT; ++k) {
    if (!FULL && k >= n) break;
    stage(k, k);
    cp_async_wait_group<0>();
    __syncwarp();
    const double rk = rcp_rn<double>(col[k]);
    if (valid) Bs[k] = rk;
    y[k] = y[k] * rk;
#pragma unroll
    for (int i = k + 1; i < NT; ++i)
      if (FULL || i < n) y[i] = fma_rn<double>(-col[i], y[k], y[i]);
    __syncwarp();                               // the buffer is restaged next step
  }

  // backward: L^T x = y, x_i from column i of L (rows below the diagonal)
#pragma unroll
  for (int i = NT - 1; i >= 0; --i) {
    if (!FULL && i >= n) continue;
    stage(i, i + 1);
    const double ri = valid ? Bs[i] : 1.0;
    cp_async_wait_group<0>();
    __syncwarp();
    double acc = y[i];
#pragma unroll
    for (int k = NT - 1; k > i; --k)
      if (FULL || k < n) acc = fma_rn<double>(-col[k], y[k], acc);
    y[i] = acc * ri;
    __syncwarp();
  }

  if (!valid) return;
  const bool zero_x = zinfo != nullptr && __ldg(zinfo + s) != 0;
#pragma unroll
  for (int i = 0; i < NT; ++i)
    if (FULL || i < n) Bs[i] = zero_x ? 0.0 : y[i];
}

template <int NT>
cudaError_t launch_nt(int alay, int n, int64_t batch, const double* L, double* B,
                      const int32_t* zinfo, cudaStream_t stream) {
  constexpr int per_block = kLaneWarps * 32;
  const int64_t blocks = (batch + per_block - 1) / per_block;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  const size_t bytes = static_cast<size_t>(kLaneWarps) * 32 * (NT + 1) * sizeof(double);
  cudaError_t e;
  if (n == NT) {
    e = cudaFuncSetAttribute(potrs_lane_kernel<NT, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (e != cudaSuccess) return e;
    potrs_lane_kernel<NT, true><<<static_cast<unsigned>(blocks), per_block, bytes, stream>>>(
        n, alay, batch, L, B, zinfo);
  } else {
    e = cudaFuncSetAttribute(potrs_lane_kernel<NT, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (e != cudaSuccess) return e;
    potrs_lane_kernel<NT, false><<<static_cast<unsigned>(blocks), per_block, bytes, stream>>>(
        n, alay, batch, L, B, zinfo);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_potrs_lane(int layout, int n, int nrhs, int64_t batch, const double* L,
                              double* B, const int32_t* zinfo, cudaStream_t stream) {
  if (n < 1 || n > 32 || nrhs != 1) return cudaErrorInvalidValue;
  const int alay = layout & 1;   // the factor's storage order (one right-hand side: B has none)
  if (n <= 8) return launch_nt<8>(alay, n, batch, L, B, zinfo, stream);
  if (n <= 16) return launch_nt<16>(alay, n, batch, L, B, zinfo, stream);
  return launch_nt<32>(alay, n, batch, L, B, zinfo, stream);
}

}  // namespace bsolve
