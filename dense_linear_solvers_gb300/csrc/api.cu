// C ABI of libbsolve.so: argument checks and dispatch to the kernel launchers.
// See include/bsolve.h for the contract of every entry point.
#include <atomic>
#include <cstdint>
#include <initializer_list>
#include <utility>

#include <cuda_runtime.h>

#include "bsolve.h"
#include "kernels.h"

namespace {

thread_local int g_last_cuda_error = 0;

constexpr int kMaxLuN = 128;
constexpr int kMaxCholN = 256;       // beyond kMaxLuN: the cluster factor and the big solve
constexpr int kMaxRegN = 32;
constexpr int kMaxNrhs = 8;          // right-hand sides a fused kernel holds
constexpr int kMaxNrhsAny = 65536;   // beyond kMaxNrhs: factor, then a chunked solve
constexpr int kMaxBdsvBs = 8;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Whether the byte ranges [a, a + na) and [b, b + nb) share a byte.
bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// Whether the byte ranges are pairwise disjoint: the operands of one call must not alias.
using Range = std::pair<const void*, size_t>;
bool disjoint(std::initializer_list<Range> rs) {
  for (auto a = rs.begin(); a != rs.end(); ++a)
    for (auto b = a + 1; b != rs.end(); ++b)
      if (overlap(a->first, a->second, b->first, b->second)) return false;
  return true;
}

// Systems a batched operand holds: the batch, rounded up to whole blocks of an
// interleaved layout (ilv > 1).
size_t held(int64_t batch, int64_t ilv) {
  return static_cast<size_t>(ilv > 1 ? (batch + ilv - 1) / ilv * ilv : batch);
}

// The four operands of an LU call (A, B, ipiv, info) do not alias.
bool lu_disjoint(bs_dtype dtype, int n, int nrhs, int64_t batch, int64_t ilv, const void* A,
                 const void* B, const void* ipiv, const void* info) {
  const size_t es = dtype == BS_FP32 ? 4 : 8, h = held(batch, ilv);
  return disjoint({{A, h * n * n * es}, {B, h * n * nrhs * es}, {ipiv, h * n * 4},
                   {info, static_cast<size_t>(batch) * 4}});
}

// The three operands of a Cholesky call (A, B, info) do not alias.
bool chol_disjoint(bs_dtype dtype, int n, int nrhs, int64_t batch, int64_t ilv, const void* A,
                   const void* B, const void* info) {
  const size_t es = dtype == BS_FP32 ? 4 : 8, h = held(batch, ilv);
  return disjoint({{A, h * n * n * es}, {B, h * n * nrhs * es},
                   {info, static_cast<size_t>(batch) * 4}});
}

bs_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return BS_OK;
  g_last_cuda_error = static_cast<int>(e);
  return BS_ERR_CUDA;
}

bool lu_supported(bs_dtype dtype, bs_layout layout, int n, int nrhs) {
  return (dtype == BS_FP32 || dtype == BS_FP64) &&
         (layout == BS_ROW_MAJOR || layout == BS_COL_MAJOR) && n >= 1 && n <= kMaxLuN &&
         nrhs >= 1 && nrhs <= kMaxNrhsAny;
}

bool chol_supported(bs_dtype dtype, bs_layout layout, bs_fill fill, int n, int nrhs) {
  return (dtype == BS_FP32 || dtype == BS_FP64) &&
         (layout == BS_ROW_MAJOR || layout == BS_COL_MAJOR) &&
         (fill == BS_LOWER || fill == BS_UPPER) && n >= 1 &&
         n <= kMaxCholN && nrhs >= 1 && nrhs <= kMaxNrhsAny;
}

// Packed storage-order code of the Cholesky kernels: bit 0 for A (or the factor), bit 1 for
// B. Upper fill in one order is the lower fill of the mirrored matrix, i.e. A read in the
// other order (cuSolverDx docs, "Cholesky Factorization": A = U^T U with U = L^T).
int chol_layouts(bs_layout layout, bs_fill fill) {
  const int a = fill == BS_LOWER ? static_cast<int>(layout) : 1 - static_cast<int>(layout);
  return a | (static_cast<int>(layout) << 1);
}

bool bdsv_supported(bs_dtype dtype, int nbr, int bs) {
  return (dtype == BS_FP32 || dtype == BS_FP64) && nbr >= 1 && bs >= 1 && bs <= kMaxBdsvBs;
}

// The row-major reading of TDLS (TDLS API, "solver_static.hpp File Reference"): the factor
// of S, the row-major array read column-major (P A^T = L U), by the plain factor kernels
// (or the one-CTA kernel under a threshold, an interleaved layout or RUDA's scaling), then
// the mirror solve U^T z = b, L^T w = z, x = P^T w, which writes X as zeros where
// info != 0. il: the element stride of an interleaved batched layout (1: plain).
bs_status getrf_getrs_mirror(bs_dtype dtype, int n, int nrhs, int64_t batch, void* A, void* B,
                             int32_t* ipiv, int32_t* info, double tau, int64_t il, int scaling,
                             void* stream) {
  if (n < 0 || nrhs < 0 || batch < 0) return BS_ERR_INVALID_ARG;
  if (!lu_supported(dtype, BS_ROW_MAJOR, n, nrhs)) return BS_ERR_UNSUPPORTED;
  if (batch == 0) return BS_OK;
  if (!A || !B || !ipiv || !info) return BS_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(ipiv) || !aligned16(info))
    return BS_ERR_INVALID_ARG;
  if (!lu_disjoint(dtype, n, nrhs, batch, il, A, B, ipiv, info)) return BS_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (tau == 1.0 && il == 1 && !scaling) {
    const bs_status st = bs_getrf_batched(dtype, BS_COL_MAJOR, n, batch, A, ipiv, info, stream);
    if (st != BS_OK) return st;
  } else {
    e = dtype == BS_FP32
            ? bsolve::launch_lu_smem_ex<float>(BS_COL_MAJOR, n, 0, batch, static_cast<float*>(A),
                                               nullptr, ipiv, info, tau, 0, s, il, scaling)
            : bsolve::launch_lu_smem_ex<double>(BS_COL_MAJOR, n, 0, batch,
                                                static_cast<double*>(A), nullptr, ipiv, info,
                                                tau, 0, s, il, scaling);
    if (e != cudaSuccess) return from_cuda(e);
  }
  const int code = BS_COL_MAJOR | (BS_ROW_MAJOR << 1);
  e = dtype == BS_FP32
          ? bsolve::launch_getrs_mirror<float>(code, n, nrhs, batch, static_cast<const float*>(A),
                                               ipiv, static_cast<float*>(B), info, s, il)
          : bsolve::launch_getrs_mirror<double>(code, n, nrhs, batch,
                                                static_cast<const double*>(A), ipiv,
                                                static_cast<double*>(B), info, s, il);
  return from_cuda(e);
}

// The interleaved batched layout (TDLS API, "solver_static.hpp File Reference": element e
// of system s at base_s[e * ilv], base_s = (s / ilv) * ilv * size + s % ilv; AoSoA, SoA
// when ilv >= batch) for A, B and ipiv; info one entry per system. The fused kernels with
// a stride: the register tier for n <= 32, one CTA per system above.
bs_status getrf_getrs_il(bs_dtype dtype, bs_layout layout, int n, int nrhs, int64_t batch,
                         int64_t ilv, void* A, void* B, int32_t* ipiv, int32_t* info,
                         void* stream) {
  if (n < 0 || nrhs < 0 || batch < 0) return BS_ERR_INVALID_ARG;
  if (!lu_supported(dtype, layout, n, nrhs) || nrhs > kMaxNrhs) return BS_ERR_UNSUPPORTED;
  if (batch == 0) return BS_OK;
  if (!A || !B || !ipiv || !info) return BS_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(ipiv) || !aligned16(info))
    return BS_ERR_INVALID_ARG;
  if (!lu_disjoint(dtype, n, nrhs, batch, ilv, A, B, ipiv, info)) return BS_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (n <= kMaxRegN) {
    e = dtype == BS_FP32
            ? bsolve::launch_lu_reg_il<float>(layout, n, nrhs, batch, ilv, static_cast<float*>(A),
                                              static_cast<float*>(B), ipiv, info, s)
            : bsolve::launch_lu_reg_il<double>(layout, n, nrhs, batch, ilv,
                                               static_cast<double*>(A), static_cast<double*>(B),
                                               ipiv, info, s);
  } else {
    e = dtype == BS_FP32
            ? bsolve::launch_lu_smem_ex<float>(layout, n, nrhs, batch, static_cast<float*>(A),
                                               static_cast<float*>(B), ipiv, info, 1.0, 0, s, ilv)
            : bsolve::launch_lu_smem_ex<double>(layout, n, nrhs, batch, static_cast<double*>(A),
                                                static_cast<double*>(B), ipiv, info, 1.0, 0, s,
                                                ilv);
  }
  return from_cuda(e);
}

bs_status potrf_potrs_il(bs_dtype dtype, bs_layout layout, bs_fill fill, int n, int nrhs,
                         int64_t batch, int64_t ilv, void* A, void* B, int32_t* info,
                         void* stream) {
  if (n < 0 || nrhs < 0 || batch < 0) return BS_ERR_INVALID_ARG;
  if (!chol_supported(dtype, layout, fill, n, nrhs) || nrhs > kMaxNrhs || n > kMaxLuN)
    return BS_ERR_UNSUPPORTED;
  if (batch == 0) return BS_OK;
  if (!A || !B || !info) return BS_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(info)) return BS_ERR_INVALID_ARG;
  if (!chol_disjoint(dtype, n, nrhs, batch, ilv, A, B, info)) return BS_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int code = chol_layouts(layout, fill);
  cudaError_t e;
  if (n <= kMaxRegN) {
    e = dtype == BS_FP32
            ? bsolve::launch_chol_sys<float>(code, n, nrhs, batch, static_cast<float*>(A),
                                             static_cast<float*>(B), info, s, ilv)
            : bsolve::launch_chol_sys<double>(code, n, nrhs, batch, static_cast<double*>(A),
                                              static_cast<double*>(B), info, s, ilv);
  } else {
    e = dtype == BS_FP32
            ? bsolve::launch_chol_smem_ex<float>(code, n, nrhs, batch, static_cast<float*>(A),
                                                 static_cast<float*>(B), info, 0, s, ilv)
            : bsolve::launch_chol_smem_ex<double>(code, n, nrhs, batch, static_cast<double*>(A),
                                                  static_cast<double*>(B), info, 0, s, ilv);
  }
  return from_cuda(e);
}

// ---------------------------------------------------------------- host-resident batches
// One operand of a host pipeline: the host array, its bytes per system, and whether it is
// copied in (H2D) and out (D2H).
struct HostOperand {
  char* host;
  size_t per_sys;
  bool in, out;
};

constexpr size_t kWorkAlign = 256;

size_t round_up(size_t x) { return (x + kWorkAlign - 1) / kWorkAlign * kWorkAlign; }

// Bytes of one slot of the workspace (a chunk of every operand, each 256-byte aligned);
// the workspace holds two slots. A size past kTooBig (no workspace is that large) is
// returned as kTooBig, so that no product or sum below can wrap around.
constexpr size_t kTooBig = SIZE_MAX / 4;
size_t slot_bytes(const HostOperand* ops, int nops, int64_t chunk) {
  const size_t c = static_cast<size_t>(chunk);
  size_t b = 0;
  for (int i = 0; i < nops; ++i) {
    const size_t per = ops[i].per_sys;
    if (per != 0 && c > (kTooBig - b) / per / 2) return kTooBig;
    b += round_up(per * c);
  }
  return b < kTooBig ? b : kTooBig;
}

// The batch in chunks of `chunk` systems; chunk c runs its copies in, its solve and its
// copies out on stream c % 2 with workspace slot c % 2, so that one chunk's copies
// overlap the other stream's solve and copies, and a slot is reused only after its
// stream has finished with it (stream order: no event needed). `call` gets the device
// pointers of the operands, the chunk's system count and the stream.
// Slot 1 starts `stride` bytes after slot 0 (0: right after it, i.e. at the slot size).
template <class Call>
bs_status host_pipeline(int64_t batch, int64_t chunk, HostOperand* ops, int nops, void* work,
                        size_t work_bytes, void* stream0, void* stream1, Call call,
                        size_t stride = 0) {
  if (batch < 0 || chunk < 1) return BS_ERR_INVALID_ARG;
  if (batch == 0) return BS_OK;
  if (!work || (reinterpret_cast<uintptr_t>(work) % kWorkAlign) != 0) return BS_ERR_INVALID_ARG;
  for (int i = 0; i < nops; ++i) {
    if (!ops[i].host) return BS_ERR_INVALID_ARG;
    // the extent of a host array must be representable before the alias test below
    if (ops[i].per_sys != 0 && static_cast<size_t>(batch) > kTooBig / ops[i].per_sys)
      return BS_ERR_INVALID_ARG;
    for (int j = 0; j < i; ++j)   // the host arrays do not alias
      if (overlap(ops[i].host, ops[i].per_sys * batch, ops[j].host, ops[j].per_sys * batch))
        return BS_ERR_INVALID_ARG;
  }
  const size_t slot = slot_bytes(ops, nops, chunk);
  if (slot >= kTooBig) return BS_ERR_INVALID_ARG;
  if (stride == 0) stride = slot;
  if (stride < slot || stride % kWorkAlign != 0 || work_bytes < stride ||
      work_bytes - stride < slot)
    return BS_ERR_INVALID_ARG;
  cudaStream_t st[2] = {static_cast<cudaStream_t>(stream0), static_cast<cudaStream_t>(stream1)};
  char* dev[8];
  for (int64_t c0 = 0, c = 0; c0 < batch; c0 += chunk, ++c) {
    const int64_t m = batch - c0 < chunk ? batch - c0 : chunk;
    cudaStream_t s = st[c & 1];
    char* base = static_cast<char*>(work) + (c & 1) * stride;
    for (int i = 0; i < nops; ++i) {
      dev[i] = base;
      base += round_up(ops[i].per_sys * static_cast<size_t>(chunk));
      if (ops[i].in) {
        const cudaError_t e = cudaMemcpyAsync(dev[i], ops[i].host + c0 * ops[i].per_sys,
                                              m * ops[i].per_sys, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return from_cuda(e);
      }
    }
    const bs_status r = call(dev, m, s);
    if (r != BS_OK) return r;
    for (int i = 0; i < nops; ++i) {
      if (!ops[i].out) continue;
      const cudaError_t e = cudaMemcpyAsync(ops[i].host + c0 * ops[i].per_sys, dev[i],
                                            m * ops[i].per_sys, cudaMemcpyDeviceToHost, s);
      if (e != cudaSuccess) return from_cuda(e);
    }
  }
  return BS_OK;
}

size_t elem_size(bs_dtype dtype) { return dtype == BS_FP32 ? 4 : 8; }

// Workspace bytes of the host-resident LU for a chunk (2 * kTooBig when too large).
size_t lu_host_bytes(bs_dtype dtype, int n, int nrhs, int64_t chunk) {
  HostOperand ops[4] = {{nullptr, elem_size(dtype) * n * n, true, true},
                        {nullptr, elem_size(dtype) * n * nrhs, true, true},
                        {nullptr, sizeof(int32_t) * n, false, true},
                        {nullptr, sizeof(int32_t), false, true}};
  return 2 * slot_bytes(ops, 4, chunk);
}

// Scratch of the entry point that takes no workspace: one static device array, placed by
// the driver when the library's module loads (no call allocates). Its two chunk slots sit
// at fixed offsets, 0 and half the array, whatever the shape of a call, so that calls
// queued one after another on the same two streams (in the same order) never let one
// call's chunk overwrite a slot that the other stream is still reading.
constexpr size_t kStaticScratchBytes = size_t(64) << 20;
constexpr size_t kStaticSlotBytes = kStaticScratchBytes / 2;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// The device address of g_static_scratch on the current device. In host code the array's
// name is only a host-side stand-in, so its address is looked up once per device (with
// that device current) and kept; later calls on that device reuse it.
constexpr int kMaxDevices = 64;
std::atomic<void*> g_static_scratch_ptr[kMaxDevices];

cudaError_t static_scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void* p = g_static_scratch_ptr[dev].load(std::memory_order_acquire);
  if (!p) {
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    g_static_scratch_ptr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return cudaSuccess;
}

// The options a split call takes, validated as the fused _ex calls validate them.
struct SplitOpts {
  double tau;
  int contract, mirror, scaling;
  int64_t il;   // element stride of the batched layout (1: plain)
};

bs_status split_opts(const bs_options* opts, SplitOpts* o) {
  o->tau = opts ? opts->pivot_threshold : 1.0;
  o->contract = opts ? opts->status_contract : BS_CONTRACT_DEFAULT;
  o->mirror = opts ? opts->transposed_factor : 0;
  o->scaling = opts ? opts->scaling : 0;
  const int64_t ilv = opts ? opts->interleave : 0;
  if (!(o->tau > 0.0 && o->tau <= 1.0)) return BS_ERR_INVALID_ARG;
  if (o->contract != BS_CONTRACT_DEFAULT && o->contract != BS_CONTRACT_RUDA)
    return BS_ERR_INVALID_ARG;
  if ((o->mirror != 0 && o->mirror != 1) || ilv < 0 || (o->scaling != 0 && o->scaling != 1))
    return BS_ERR_INVALID_ARG;
  o->il = ilv > 1 ? ilv : 1;
  // the RUDA contract and the scaling span the factor and the solve: fused calls only
  if (o->contract != BS_CONTRACT_DEFAULT || o->scaling) return BS_ERR_UNSUPPORTED;
  return BS_OK;
}

}  // namespace

extern "C" {

size_t bs_getrf_getrs_host_workspace(bs_dtype dtype, int n, int nrhs, int64_t chunk) {
  if (n < 1 || nrhs < 1 || chunk < 1) return 0;
  const size_t w = lu_host_bytes(dtype, n, nrhs, chunk);
  return w >= 2 * kTooBig ? 0 : w;
}

bs_status bs_getrf_getrs_batched_host(bs_dtype dtype, bs_layout layout, int n, int nrhs,
                                      int64_t batch, void* A, void* B, int32_t* ipiv,
                                      int32_t* info, void* work, size_t work_bytes,
                                      int64_t chunk, void* stream0, void* stream1) {
  if (n < 0 || nrhs < 0 || batch < 0) return BS_ERR_INVALID_ARG;
  if (!lu_supported(dtype, layout, n, nrhs)) return BS_ERR_UNSUPPORTED;
  const size_t es = elem_size(dtype);
  HostOperand ops[4] = {{static_cast<char*>(A), es * n * n, true, true},
                        {static_cast<char*>(B), es * n * nrhs, true, true},
                        {reinterpret_cast<char*>(ipiv), sizeof(int32_t) * n, false, true},
                        {reinterpret_cast<char*>(info), sizeof(int32_t), false, true}};
  return host_pipeline(batch, chunk, ops, 4, work, work_bytes, stream0, stream1,
                       [&](char** d, int64_t m, cudaStream_t s) {
                         return bs_getrf_getrs_batched(dtype, layout, n, nrhs, m, d[0], d[1],
                                                       reinterpret_cast<int32_t*>(d[2]),
                                                       reinterpret_cast<int32_t*>(d[3]), s);
                       });
}

bs_status bs_getrf_getrs_batched_host_static(bs_dtype dtype, bs_layout layout, int n, int nrhs,
                                             int64_t batch, void* A, void* B, int32_t* ipiv,
                                             int32_t* info, int64_t chunk, void* stream0,
                                             void* stream1) {
  if (n < 0 || nrhs < 0 || batch < 0 || chunk < 1) return BS_ERR_INVALID_ARG;
  if (!lu_supported(dtype, layout, n, nrhs)) return BS_ERR_UNSUPPORTED;
  if (batch == 0) return BS_OK;
  // the largest chunk, up to the requested one, whose slot fits half the static scratch
  int64_t c = chunk;
  while (c > 1 && lu_host_bytes(dtype, n, nrhs, c) / 2 > kStaticSlotBytes) c = c / 2;
  if (lu_host_bytes(dtype, n, nrhs, c) / 2 > kStaticSlotBytes) return BS_ERR_UNSUPPORTED;
  void* work = nullptr;
  const cudaError_t e = static_scratch_address(&work);
  if (e != cudaSuccess) return from_cuda(e);
  const size_t es = elem_size(dtype);
  HostOperand ops[4] = {{static_cast<char*>(A), es * n * n, true, true},
                        {static_cast<char*>(B), es * n * nrhs, true, true},
                        {reinterpret_cast<char*>(ipiv), sizeof(int32_t) * n, false, true},
                        {reinterpret_cast<char*>(info), sizeof(int32_t), false, true}};
  return host_pipeline(batch, c, ops, 4, work, kStaticScratchBytes, stream0, stream1,
                       [&](char** d, int64_t m, cudaStream_t s) {
                         return bs_getrf_getrs_batched(dtype, layout, n, nrhs, m, d[0], d[1],
                                                       reinterpret_cast<int32_t*>(d[2]),
                                                       reinterpret_cast<int32_t*>(d[3]), s);
                       },
                       kStaticSlotBytes);
}

size_t bs_potrf_potrs_host_workspace(bs_dtype dtype, int n, int nrhs, int64_t chunk) {
  if (n < 1 || nrhs < 1 || chunk < 1) return 0;
  HostOperand ops[3] = {{nullptr, elem_size(dtype) * n * n, true, true},
                        {nullptr, elem_size(dtype) * n * nrhs, true, true},
                        {nullptr, sizeof(int32_t), false, true}};
  const size_t slot = slot_bytes(ops, 3, chunk);
  return slot >= kTooBig ? 0 : 2 * slot;
}

bs_status bs_potrf_potrs_batched_host(bs_dtype dtype, bs_layout layout, bs_fill fill, int n,
                                      int nrhs, int64_t batch, void* A, void* B, int32_t* info,
                                      void* work, size_t work_bytes, int64_t chunk,
                                      void* stream0, void* stream1) {
  if (n < 0 || nrhs < 0 || batch < 0) return BS_ERR_INVALID_ARG;
  if (!chol_supported(dtype, layout, fill, n, nrhs)) return BS_ERR_UNSUPPORTED;
  const size_t es = elem_size(dtype);
  HostOperand ops[3] = {{static_cast<char*>(A), es * n * n, true, true},
                        {static_cast<char*>(B), es * n * nrhs, true, true},
                        {reinterpret_cast<char*>(info), sizeof(int32_t), false, true}};
  return host_pipeline(batch, chunk, ops, 3, work, work_bytes, stream0, stream1,
                       [&](char** d, int64_t m, cudaStream_t s) {
                         return bs_potrf_potrs_batched(dtype, layout, fill, n, nrhs, m, d[0],
                                                       d[1], reinterpret_cast<int32_t*>(d[2]),
                                                       s);
                       });
}

size_t bs_bdsv_host_workspace(bs_dtype dtype, int num_block_rows, int block_size,
                              int64_t chunk) {
  if (num_block_rows < 1 || block_size < 1 || chunk < 1) return 0;
  const size_t es = elem_size(dtype);
  HostOperand ops[3] = {
      {nullptr, es * num_block_rows * block_size * 3 * block_size, true, true},
      {nullptr, es * (num_block_rows + 2) * block_size, true, true},
      {nullptr, sizeof(int32_t), false, true}};
  const size_t slot = slot_bytes(ops, 3, chunk);
  return slot >= kTooBig ? 0 : 2 * slot;
}

bs_status bs_bdsv_batched_host(bs_dtype dtype, int num_block_rows, int block_size,
                               int64_t batch, void* strips, void* x_padded, int32_t* info,
                               void* work, size_t work_bytes, int64_t chunk, void* stream0,
                               void* stream1) {
  if (num_block_rows < 0 || block_size < 0 || batch < 0) return BS_ERR_INVALID_ARG;
  if (!bdsv_supported(dtype, num_block_rows, block_size)) return BS_ERR_UNSUPPORTED;
  const size_t es = elem_size(dtype);
  HostOperand ops[3] = {
      {static_cast<char*>(strips), es * num_block_rows * block_size * 3 * block_size, true,
       true},
      {static_cast<char*>(x_padded), es * (num_block_rows + 2) * block_size, true, true},
      {reinterpret_cast<char*>(info), sizeof(int32_t), false, true}};
  return host_pipeline(batch, chunk, ops, 3, work, work_bytes, stream0, stream1,
                       [&](char** d, int64_t m, cudaStream_t s) {
                         return bs_bdsv_batched(dtype, num_block_rows, block_size, m, d[0], d[1],
                                                reinterpret_cast<int32_t*>(d[2]), s);
                       });
}

bs_status bs_getrf_getrs_batched(bs_dtype dtype, bs_layout layout, int n, int nrhs,
                                 int64_t batch, void* A, void* B, int32_t* ipiv,
                                 int32_t* info, void* stream) {
  if (n < 0 || nrhs < 0 || batch < 0) return BS_ERR_INVALID_ARG;
  if (!lu_supported(dtype, layout, n, nrhs)) return BS_ERR_UNSUPPORTED;
  if (batch == 0) return BS_OK;
  if (!A || !B || !ipiv || !info) return BS_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(ipiv) || !aligned16(info))
    return BS_ERR_INVALID_ARG;
  if (!lu_disjoint(dtype, n, nrhs, batch, 1, A, B, ipiv, info)) return BS_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (nrhs > kMaxNrhs) {
    // more right-hand sides than a fused kernel holds: the factor, then the solve (which
    // zeroes X where info != 0); the same operations in the same order as the fused sweep
    const bs_status st = bs_getrf_batched(dtype, layout, n, batch, A, ipiv, info, stream);
    if (st != BS_OK) return st;
    e = dtype == BS_FP32
            ? bsolve::launch_getrs<float>(layout | (layout << 1), n, nrhs, batch,
                                          static_cast<const float*>(A), ipiv,
                                          static_cast<float*>(B), info, s)
            : bsolve::launch_getrs<double>(layout | (layout << 1), n, nrhs, batch,
                                           static_cast<const double*>(A), ipiv,
                                           static_cast<double*>(B), info, s);
  } else if (n <= kMaxRegN) {
    e = dtype == BS_FP32
            ? bsolve::launch_lu_reg<float>(layout, n, nrhs, batch, static_cast<float*>(A),
                                           static_cast<float*>(B), ipiv, info, s)
            : bsolve::launch_lu_reg<double>(layout, n, nrhs, batch, static_cast<double*>(A),
                                            static_cast<double*>(B), ipiv, info, s);
  } else {
    e = dtype == BS_FP32
            ? bsolve::launch_lu_smem<float>(layout, n, nrhs, batch, static_cast<float*>(A),
                                            static_cast<float*>(B), ipiv, info, s)
            : bsolve::launch_lu_smem<double>(layout, n, nrhs, batch, static_cast<double*>(A),
                                             static_cast<double*>(B), ipiv, info, s);
  }
  return from_cuda(e);
}

bs_status bs_potrf_potrs_batched(bs_dtype dtype, bs_layout layout, bs_fill fill, int n,
                                 int nrhs, int64_t batch, void* A, void* B, int32_t* info,
                                 void* stream) {
  if (n < 0 || nrhs < 0 || batch < 0) return BS_ERR_INVALID_ARG;
  if (!chol_supported(dtype, layout, fill, n, nrhs)) return BS_ERR_UNSUPPORTED;
  if (batch == 0) return BS_OK;
  if (!A || !B || !info) return BS_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(info)) return BS_ERR_INVALID_ARG;
  if (!chol_disjoint(dtype, n, nrhs, batch, 1, A, B, info)) return BS_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (nrhs > kMaxNrhs || n > kMaxLuN) {
    // the factor, then the solve that zeroes X where info != 0 (see the LU call); orders
    // beyond one CTA always run this way (the cluster factor, then the big solve)
    const bs_status st = bs_potrf_batched(dtype, layout, fill, n, batch, A, info, stream);
    if (st != BS_OK) return st;
    e = dtype == BS_FP32
            ? bsolve::launch_potrs<float>(chol_layouts(layout, fill), n, nrhs, batch,
                                          static_cast<const float*>(A), static_cast<float*>(B),
                                          info, s)
            : bsolve::launch_potrs<double>(chol_layouts(layout, fill), n, nrhs, batch,
                                           static_cast<const double*>(A),
                                           static_cast<double*>(B), info, s);
  } else if (n <= kMaxRegN) {
    e = dtype == BS_FP32
            ? bsolve::launch_chol_sys<float>(chol_layouts(layout, fill), n, nrhs, batch,
                                             static_cast<float*>(A), static_cast<float*>(B),
                                             info, s)
            : bsolve::launch_chol_sys<double>(chol_layouts(layout, fill), n, nrhs, batch,
                                              static_cast<double*>(A), static_cast<double*>(B),
                                              info, s);
  } else {
    e = dtype == BS_FP32
            ? bsolve::launch_chol_smem<float>(chol_layouts(layout, fill), n, nrhs, batch,
                                              static_cast<float*>(A), static_cast<float*>(B),
                                              info, s)
            : bsolve::launch_chol_smem<double>(chol_layouts(layout, fill), n, nrhs, batch,
                                               static_cast<double*>(A), static_cast<double*>(B),
                                               info, s);
  }
  return from_cuda(e);
}

bs_status bs_bdsv_batched(bs_dtype dtype, int num_block_rows, int block_size, int64_t batch,
                          void* strips, void* x_padded, int32_t* info, void* stream) {
  if (num_block_rows < 0 || block_size < 0 || batch < 0) return BS_ERR_INVALID_ARG;
  if (!bdsv_supported(dtype, num_block_rows, block_size)) return BS_ERR_UNSUPPORTED;
  if (batch == 0) return BS_OK;
  if (!strips || !x_padded || !info) return BS_ERR_INVALID_ARG;
  if (!aligned16(strips) || !aligned16(x_padded) || !aligned16(info)) return BS_ERR_INVALID_ARG;
  {
    const size_t es = dtype == BS_FP32 ? 4 : 8, b = static_cast<size_t>(batch);
    if (!disjoint({{strips, b * num_block_rows * block_size * 3 * block_size * es},
                   {x_padded, b * (num_block_rows + 2) * block_size * es}, {info, b * 4}}))
      return BS_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e =
      dtype == BS_FP32
          ? bsolve::launch_bdsv<float>(num_block_rows, block_size, batch,
                                       static_cast<float*>(strips),
                                       static_cast<float*>(x_padded), info, s)
          : bsolve::launch_bdsv<double>(num_block_rows, block_size, batch,
                                        static_cast<double*>(strips),
                                        static_cast<double*>(x_padded), info, s);
  return from_cuda(e);
}

bs_status bs_getrf_batched(bs_dtype dtype, bs_layout layout, int n, int64_t batch, void* A,
                           int32_t* ipiv, int32_t* info, void* stream) {
  if (n < 0 || batch < 0) return BS_ERR_INVALID_ARG;
  if (!lu_supported(dtype, layout, n, 1)) return BS_ERR_UNSUPPORTED;
  if (batch == 0) return BS_OK;
  if (!A || !ipiv || !info) return BS_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(ipiv) || !aligned16(info)) return BS_ERR_INVALID_ARG;
  {
    const size_t es = dtype == BS_FP32 ? 4 : 8, b = static_cast<size_t>(batch);
    if (!disjoint({{A, b * n * n * es}, {ipiv, b * n * 4}, {info, b * 4}}))
      return BS_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (n <= kMaxRegN) {
    e = dtype == BS_FP32
            ? bsolve::launch_lu_reg<float>(layout, n, 0, batch, static_cast<float*>(A), nullptr,
                                           ipiv, info, s)
            : bsolve::launch_lu_reg<double>(layout, n, 0, batch, static_cast<double*>(A),
                                            nullptr, ipiv, info, s);
  } else {
    e = dtype == BS_FP32
            ? bsolve::launch_lu_smem<float>(layout, n, 0, batch, static_cast<float*>(A), nullptr,
                                            ipiv, info, s)
            : bsolve::launch_lu_smem<double>(layout, n, 0, batch, static_cast<double*>(A),
                                             nullptr, ipiv, info, s);
  }
  return from_cuda(e);
}

bs_status bs_getrs_batched(bs_dtype dtype, bs_layout layout, int n, int nrhs, int64_t batch,
                           const void* LU, const int32_t* ipiv, void* B, void* stream) {
  if (n < 0 || nrhs < 0 || batch < 0) return BS_ERR_INVALID_ARG;
  if (!lu_supported(dtype, layout, n, nrhs)) return BS_ERR_UNSUPPORTED;
  if (batch == 0) return BS_OK;
  if (!LU || !ipiv || !B) return BS_ERR_INVALID_ARG;
  if (!aligned16(LU) || !aligned16(ipiv) || !aligned16(B)) return BS_ERR_INVALID_ARG;
  const size_t es = dtype == BS_FP32 ? 4 : 8;
  const size_t bbytes = static_cast<size_t>(batch) * n * nrhs * es;
  if (overlap(B, bbytes, LU, static_cast<size_t>(batch) * n * n * es) ||
      overlap(B, bbytes, ipiv, static_cast<size_t>(batch) * n * sizeof(int32_t)))
    return BS_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e =
      dtype == BS_FP32
          ? bsolve::launch_getrs<float>(layout | (layout << 1), n, nrhs, batch,
                                        static_cast<const float*>(LU), ipiv,
                                        static_cast<float*>(B), nullptr, s)
          : bsolve::launch_getrs<double>(layout | (layout << 1), n, nrhs, batch,
                                         static_cast<const double*>(LU), ipiv,
                                         static_cast<double*>(B), nullptr, s);
  return from_cuda(e);
}

bs_status bs_potrf_batched(bs_dtype dtype, bs_layout layout, bs_fill fill, int n, int64_t batch,
                           void* A, int32_t* info, void* stream) {
  if (n < 0 || batch < 0) return BS_ERR_INVALID_ARG;
  if (!chol_supported(dtype, layout, fill, n, 1)) return BS_ERR_UNSUPPORTED;
  if (batch == 0) return BS_OK;
  if (!A || !info) return BS_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(info)) return BS_ERR_INVALID_ARG;
  if (!disjoint({{A, static_cast<size_t>(batch) * n * n * (dtype == BS_FP32 ? 4 : 8)},
                 {info, static_cast<size_t>(batch) * 4}}))
    return BS_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (n > kMaxLuN) {
    e = dtype == BS_FP32
            ? bsolve::launch_chol_cluster<float>(chol_layouts(layout, fill), n, batch,
                                                 static_cast<float*>(A), info, s)
            : bsolve::launch_chol_cluster<double>(chol_layouts(layout, fill), n, batch,
                                                  static_cast<double*>(A), info, s);
  } else if (n <= kMaxRegN) {
    e = dtype == BS_FP32
            ? bsolve::launch_chol_sys<float>(chol_layouts(layout, fill), n, 0, batch,
                                             static_cast<float*>(A), nullptr, info, s)
            : bsolve::launch_chol_sys<double>(chol_layouts(layout, fill), n, 0, batch,
                                              static_cast<double*>(A), nullptr, info, s);
  } else {
    e = dtype == BS_FP32
            ? bsolve::launch_chol_smem<float>(chol_layouts(layout, fill), n, 0, batch,
                                              static_cast<float*>(A), nullptr, info, s)
            : bsolve::launch_chol_smem<double>(chol_layouts(layout, fill), n, 0, batch,
                                               static_cast<double*>(A), nullptr, info, s);
  }
  return from_cuda(e);
}

bs_status bs_potrs_batched(bs_dtype dtype, bs_layout layout, bs_fill fill, int n, int nrhs,
                           int64_t batch, const void* L, void* B, void* stream) {
  if (n < 0 || nrhs < 0 || batch < 0) return BS_ERR_INVALID_ARG;
  if (!chol_supported(dtype, layout, fill, n, nrhs)) return BS_ERR_UNSUPPORTED;
  if (batch == 0) return BS_OK;
  if (!L || !B) return BS_ERR_INVALID_ARG;
  if (!aligned16(L) || !aligned16(B)) return BS_ERR_INVALID_ARG;
  const size_t es = dtype == BS_FP32 ? 4 : 8;
  if (overlap(B, static_cast<size_t>(batch) * n * nrhs * es, L,
              static_cast<size_t>(batch) * n * n * es))
    return BS_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e =
      dtype == BS_FP32
          ? bsolve::launch_potrs<float>(chol_layouts(layout, fill), n, nrhs, batch,
                                        static_cast<const float*>(L), static_cast<float*>(B),
                                        nullptr, s)
          : bsolve::launch_potrs<double>(chol_layouts(layout, fill), n, nrhs, batch,
                                         static_cast<const double*>(L), static_cast<double*>(B),
                                         nullptr, s);
  return from_cuda(e);
}

bs_status bs_bdsv_factor_batched(bs_dtype dtype, int num_block_rows, int block_size,
                                 int64_t batch, void* strips, int32_t* info, void* stream) {
  if (num_block_rows < 0 || block_size < 0 || batch < 0) return BS_ERR_INVALID_ARG;
  if (!bdsv_supported(dtype, num_block_rows, block_size)) return BS_ERR_UNSUPPORTED;
  if (batch == 0) return BS_OK;
  if (!strips || !info) return BS_ERR_INVALID_ARG;
  if (!aligned16(strips) || !aligned16(info)) return BS_ERR_INVALID_ARG;
  if (!disjoint({{strips, static_cast<size_t>(batch) * num_block_rows * block_size * 3 *
                              block_size * (dtype == BS_FP32 ? 4 : 8)},
                 {info, static_cast<size_t>(batch) * 4}}))
    return BS_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e =
      dtype == BS_FP32
          ? bsolve::launch_bdsv_factor<float>(num_block_rows, block_size, batch,
                                              static_cast<float*>(strips), info, s)
          : bsolve::launch_bdsv_factor<double>(num_block_rows, block_size, batch,
                                               static_cast<double*>(strips), info, s);
  return from_cuda(e);
}

bs_status bs_bdsv_solve_batched(bs_dtype dtype, int num_block_rows, int block_size,
                                int64_t batch, const void* strips, void* x_padded,
                                void* stream) {
  if (num_block_rows < 0 || block_size < 0 || batch < 0) return BS_ERR_INVALID_ARG;
  if (!bdsv_supported(dtype, num_block_rows, block_size)) return BS_ERR_UNSUPPORTED;
  if (batch == 0) return BS_OK;
  if (!strips || !x_padded) return BS_ERR_INVALID_ARG;
  if (!aligned16(strips) || !aligned16(x_padded)) return BS_ERR_INVALID_ARG;
  const size_t es = dtype == BS_FP32 ? 4 : 8;
  const size_t sbytes = static_cast<size_t>(batch) * num_block_rows * block_size * 3 *
                        block_size * es;
  const size_t vbytes = static_cast<size_t>(batch) * (num_block_rows + 2) * block_size * es;
  if (overlap(x_padded, vbytes, strips, sbytes)) return BS_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e =
      dtype == BS_FP32
          ? bsolve::launch_bdsv_solve<float>(num_block_rows, block_size, batch,
                                             static_cast<const float*>(strips),
                                             static_cast<float*>(x_padded), s)
          : bsolve::launch_bdsv_solve<double>(num_block_rows, block_size, batch,
                                              static_cast<const double*>(strips),
                                              static_cast<double*>(x_padded), s);
  return from_cuda(e);
}

// bdmv with one output (two == false, y2_padded unused) or two
static bs_status bdmv_any(bs_dtype dtype, int num_block_rows, int block_size, int64_t batch,
                          const void* strips, const void* x_padded, void* y_padded,
                          void* y2_padded, bool two, void* stream) {
  if (num_block_rows < 0 || block_size < 0 || batch < 0) return BS_ERR_INVALID_ARG;
  if (!bdsv_supported(dtype, num_block_rows, block_size)) return BS_ERR_UNSUPPORTED;
  if (batch == 0) return BS_OK;
  if (!two) y2_padded = nullptr;
  if (!strips || !x_padded || !y_padded || (two && !y2_padded)) return BS_ERR_INVALID_ARG;
  if (!aligned16(strips) || !aligned16(x_padded) || !aligned16(y_padded) ||
      (y2_padded && !aligned16(y2_padded)))
    return BS_ERR_INVALID_ARG;
  const size_t es = dtype == BS_FP32 ? 4 : 8;
  const size_t sbytes = static_cast<size_t>(batch) * num_block_rows * block_size * 3 *
                        block_size * es;
  const size_t vbytes = static_cast<size_t>(batch) * (num_block_rows + 2) * block_size * es;
  if (overlap(y_padded, vbytes, strips, sbytes) || overlap(y_padded, vbytes, x_padded, vbytes))
    return BS_ERR_INVALID_ARG;
  if (y2_padded && !disjoint({{y2_padded, vbytes}, {strips, sbytes}, {x_padded, vbytes},
                              {y_padded, vbytes}}))
    return BS_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e =
      dtype == BS_FP32
          ? bsolve::launch_bdmv<float>(num_block_rows, block_size, batch,
                                       static_cast<const float*>(strips),
                                       static_cast<const float*>(x_padded),
                                       static_cast<float*>(y_padded),
                                       static_cast<float*>(y2_padded), s)
          : bsolve::launch_bdmv<double>(num_block_rows, block_size, batch,
                                        static_cast<const double*>(strips),
                                        static_cast<const double*>(x_padded),
                                        static_cast<double*>(y_padded),
                                        static_cast<double*>(y2_padded), s);
  return from_cuda(e);
}

bs_status bs_bdmv_batched(bs_dtype dtype, int num_block_rows, int block_size, int64_t batch,
                          const void* strips, const void* x_padded, void* y_padded,
                          void* stream) {
  return bdmv_any(dtype, num_block_rows, block_size, batch, strips, x_padded, y_padded, nullptr,
                  false, stream);
}

bs_status bs_bdmv2_batched(bs_dtype dtype, int num_block_rows, int block_size, int64_t batch,
                           const void* strips, const void* x_padded, void* y_padded,
                           void* y2_padded, void* stream) {
  return bdmv_any(dtype, num_block_rows, block_size, batch, strips, x_padded, y_padded,
                  y2_padded, true, stream);
}

bs_status bs_getrf_getrs_batched_ex(bs_dtype dtype, bs_layout layout, int n, int nrhs,
                                    int64_t batch, void* A, void* B, int32_t* ipiv,
                                    int32_t* info, const bs_options* opts, void* stream) {
  const double tau = opts ? opts->pivot_threshold : 1.0;
  const int contract = opts ? opts->status_contract : BS_CONTRACT_DEFAULT;
  const int mirror = opts ? opts->transposed_factor : 0;
  const int64_t ilv = opts ? opts->interleave : 0;
  const int scaling = opts ? opts->scaling : 0;
  if (!(tau > 0.0 && tau <= 1.0)) return BS_ERR_INVALID_ARG;
  if (contract != BS_CONTRACT_DEFAULT && contract != BS_CONTRACT_RUDA) return BS_ERR_INVALID_ARG;
  if (mirror != 0 && mirror != 1) return BS_ERR_INVALID_ARG;
  if (ilv < 0 || (scaling != 0 && scaling != 1)) return BS_ERR_INVALID_ARG;
  const int64_t il = ilv > 1 ? ilv : 1;   // element stride of the batched layout
  if (mirror && contract != BS_CONTRACT_DEFAULT) return BS_ERR_UNSUPPORTED;
  if (mirror && layout == BS_ROW_MAJOR)
    return getrf_getrs_mirror(dtype, n, nrhs, batch, A, B, ipiv, info, tau, il, scaling, stream);
  if (tau == 1.0 && contract == BS_CONTRACT_DEFAULT && !scaling)
    return il > 1 ? getrf_getrs_il(dtype, layout, n, nrhs, batch, il, A, B, ipiv, info, stream)
                  : bs_getrf_getrs_batched(dtype, layout, n, nrhs, batch, A, B, ipiv, info,
                                           stream);
  if (n < 0 || nrhs < 0 || batch < 0) return BS_ERR_INVALID_ARG;
  if (!lu_supported(dtype, layout, n, nrhs) || nrhs > kMaxNrhs) return BS_ERR_UNSUPPORTED;
  if (batch == 0) return BS_OK;
  if (!A || !B || !ipiv || !info) return BS_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(ipiv) || !aligned16(info))
    return BS_ERR_INVALID_ARG;
  if (!lu_disjoint(dtype, n, nrhs, batch, il, A, B, ipiv, info)) return BS_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int ruda = contract == BS_CONTRACT_RUDA;
  cudaError_t e =
      dtype == BS_FP32
          ? bsolve::launch_lu_smem_ex<float>(layout, n, nrhs, batch, static_cast<float*>(A),
                                             static_cast<float*>(B), ipiv, info, tau, ruda, s,
                                             il, scaling)
          : bsolve::launch_lu_smem_ex<double>(layout, n, nrhs, batch, static_cast<double*>(A),
                                              static_cast<double*>(B), ipiv, info, tau, ruda, s,
                                              il, scaling);
  return from_cuda(e);
}

bs_status bs_potrf_potrs_batched_ex(bs_dtype dtype, bs_layout layout, bs_fill fill, int n,
                                    int nrhs, int64_t batch, void* A, void* B, int32_t* info,
                                    const bs_options* opts, void* stream) {
  const double tau = opts ? opts->pivot_threshold : 1.0;
  const int contract = opts ? opts->status_contract : BS_CONTRACT_DEFAULT;
  const int mirror = opts ? opts->transposed_factor : 0;
  const int64_t ilv = opts ? opts->interleave : 0;
  if (!(tau > 0.0 && tau <= 1.0)) return BS_ERR_INVALID_ARG;
  if (contract != BS_CONTRACT_DEFAULT && contract != BS_CONTRACT_RUDA) return BS_ERR_INVALID_ARG;
  const int scaling = opts ? opts->scaling : 0;
  if ((mirror != 0 && mirror != 1) || ilv < 0 || (scaling != 0 && scaling != 1))
    return BS_ERR_INVALID_ARG;
  if (mirror || scaling) return BS_ERR_UNSUPPORTED;   // LU options
  const int64_t il = ilv > 1 ? ilv : 1;   // element stride of the batched layout
  if (contract == BS_CONTRACT_DEFAULT)   // the threshold has no meaning without pivoting
    return il > 1 ? potrf_potrs_il(dtype, layout, fill, n, nrhs, batch, il, A, B, info, stream)
                  : bs_potrf_potrs_batched(dtype, layout, fill, n, nrhs, batch, A, B, info,
                                           stream);
  if (n < 0 || nrhs < 0 || batch < 0) return BS_ERR_INVALID_ARG;
  if (!chol_supported(dtype, layout, fill, n, nrhs) || nrhs > kMaxNrhs || n > kMaxLuN)
    return BS_ERR_UNSUPPORTED;
  if (batch == 0) return BS_OK;
  if (!A || !B || !info) return BS_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(info)) return BS_ERR_INVALID_ARG;
  if (!chol_disjoint(dtype, n, nrhs, batch, il, A, B, info)) return BS_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e =
      dtype == BS_FP32
          ? bsolve::launch_chol_smem_ex<float>(chol_layouts(layout, fill), n, nrhs, batch,
                                               static_cast<float*>(A), static_cast<float*>(B),
                                               info, 1, s, il)
          : bsolve::launch_chol_smem_ex<double>(chol_layouts(layout, fill), n, nrhs, batch,
                                                static_cast<double*>(A),
                                                static_cast<double*>(B), info, 1, s, il);
  return from_cuda(e);
}

bs_status bs_getrf_batched_ex(bs_dtype dtype, bs_layout layout, int n, int64_t batch, void* A,
                              int32_t* ipiv, int32_t* info, const bs_options* opts,
                              void* stream) {
  SplitOpts o;
  const bs_status st = split_opts(opts, &o);
  if (st != BS_OK) return st;
  // the row-major reading factors S, the stored array read column-major
  const bs_layout fl = o.mirror ? BS_COL_MAJOR : layout;
  if (o.tau == 1.0 && o.il == 1)
    return bs_getrf_batched(dtype, fl, n, batch, A, ipiv, info, stream);
  if (n < 0 || batch < 0) return BS_ERR_INVALID_ARG;
  if (!lu_supported(dtype, fl, n, 1)) return BS_ERR_UNSUPPORTED;
  if (batch == 0) return BS_OK;
  if (!A || !ipiv || !info) return BS_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(ipiv) || !aligned16(info)) return BS_ERR_INVALID_ARG;
  if (!lu_disjoint(dtype, n, 0, batch, o.il, A, nullptr, ipiv, info)) return BS_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e =
      dtype == BS_FP32
          ? bsolve::launch_lu_smem_ex<float>(fl, n, 0, batch, static_cast<float*>(A), nullptr,
                                             ipiv, info, o.tau, 0, s, o.il, 0)
          : bsolve::launch_lu_smem_ex<double>(fl, n, 0, batch, static_cast<double*>(A), nullptr,
                                              ipiv, info, o.tau, 0, s, o.il, 0);
  return from_cuda(e);
}

bs_status bs_getrs_batched_ex(bs_dtype dtype, bs_layout layout, int n, int nrhs, int64_t batch,
                              const void* LU, const int32_t* ipiv, void* B,
                              const bs_options* opts, void* stream) {
  SplitOpts o;
  const bs_status st = split_opts(opts, &o);
  if (st != BS_OK) return st;
  const bool mirror = o.mirror && layout == BS_ROW_MAJOR;
  if (!mirror && o.il == 1)   // the threshold only shapes the factor the solve is given
    return bs_getrs_batched(dtype, layout, n, nrhs, batch, LU, ipiv, B, stream);
  if (n < 0 || nrhs < 0 || batch < 0) return BS_ERR_INVALID_ARG;
  if (!lu_supported(dtype, layout, n, nrhs)) return BS_ERR_UNSUPPORTED;
  if (batch == 0) return BS_OK;
  if (!LU || !ipiv || !B) return BS_ERR_INVALID_ARG;
  if (!aligned16(LU) || !aligned16(ipiv) || !aligned16(B)) return BS_ERR_INVALID_ARG;
  const size_t es = dtype == BS_FP32 ? 4 : 8, h = held(batch, o.il);
  const size_t bbytes = h * n * nrhs * es;
  if (overlap(B, bbytes, LU, h * n * n * es) || overlap(B, bbytes, ipiv, h * n * 4))
    return BS_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (mirror) {
    const int code = BS_COL_MAJOR | (BS_ROW_MAJOR << 1);
    e = dtype == BS_FP32
            ? bsolve::launch_getrs_mirror<float>(code, n, nrhs, batch,
                                                 static_cast<const float*>(LU), ipiv,
                                                 static_cast<float*>(B), nullptr, s, o.il)
            : bsolve::launch_getrs_mirror<double>(code, n, nrhs, batch,
                                                  static_cast<const double*>(LU), ipiv,
                                                  static_cast<double*>(B), nullptr, s, o.il);
  } else {
    e = dtype == BS_FP32
            ? bsolve::launch_getrs<float>(layout | (layout << 1), n, nrhs, batch,
                                          static_cast<const float*>(LU), ipiv,
                                          static_cast<float*>(B), nullptr, s, o.il)
            : bsolve::launch_getrs<double>(layout | (layout << 1), n, nrhs, batch,
                                           static_cast<const double*>(LU), ipiv,
                                           static_cast<double*>(B), nullptr, s, o.il);
  }
  return from_cuda(e);
}

bs_status bs_potrf_batched_ex(bs_dtype dtype, bs_layout layout, bs_fill fill, int n,
                              int64_t batch, void* A, int32_t* info, const bs_options* opts,
                              void* stream) {
  SplitOpts o;
  const bs_status st = split_opts(opts, &o);
  if (st != BS_OK) return st;
  if (o.mirror) return BS_ERR_UNSUPPORTED;   // an LU option
  if (o.il == 1) return bs_potrf_batched(dtype, layout, fill, n, batch, A, info, stream);
  if (n < 0 || batch < 0) return BS_ERR_INVALID_ARG;
  if (!chol_supported(dtype, layout, fill, n, 1) || n > kMaxLuN) return BS_ERR_UNSUPPORTED;
  if (batch == 0) return BS_OK;
  if (!A || !info) return BS_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(info)) return BS_ERR_INVALID_ARG;
  if (!chol_disjoint(dtype, n, 0, batch, o.il, A, nullptr, info)) return BS_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int code = chol_layouts(layout, fill);
  const cudaError_t e =
      dtype == BS_FP32
          ? bsolve::launch_chol_smem_ex<float>(code, n, 0, batch, static_cast<float*>(A),
                                               nullptr, info, 0, s, o.il)
          : bsolve::launch_chol_smem_ex<double>(code, n, 0, batch, static_cast<double*>(A),
                                                nullptr, info, 0, s, o.il);
  return from_cuda(e);
}

bs_status bs_potrs_batched_ex(bs_dtype dtype, bs_layout layout, bs_fill fill, int n, int nrhs,
                              int64_t batch, const void* L, void* B, const bs_options* opts,
                              void* stream) {
  SplitOpts o;
  const bs_status st = split_opts(opts, &o);
  if (st != BS_OK) return st;
  if (o.mirror) return BS_ERR_UNSUPPORTED;   // an LU option
  if (o.il == 1) return bs_potrs_batched(dtype, layout, fill, n, nrhs, batch, L, B, stream);
  if (n < 0 || nrhs < 0 || batch < 0) return BS_ERR_INVALID_ARG;
  if (!chol_supported(dtype, layout, fill, n, nrhs) || n > kMaxLuN) return BS_ERR_UNSUPPORTED;
  if (batch == 0) return BS_OK;
  if (!L || !B) return BS_ERR_INVALID_ARG;
  if (!aligned16(L) || !aligned16(B)) return BS_ERR_INVALID_ARG;
  const size_t es = dtype == BS_FP32 ? 4 : 8, h = held(batch, o.il);
  if (overlap(B, h * n * nrhs * es, L, h * n * n * es)) return BS_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int code = chol_layouts(layout, fill);
  const cudaError_t e =
      dtype == BS_FP32
          ? bsolve::launch_potrs<float>(code, n, nrhs, batch, static_cast<const float*>(L),
                                        static_cast<float*>(B), nullptr, s, o.il)
          : bsolve::launch_potrs<double>(code, n, nrhs, batch, static_cast<const double*>(L),
                                         static_cast<double*>(B), nullptr, s, o.il);
  return from_cuda(e);
}

const char* bs_status_string(bs_status status) {
  switch (status) {
    case BS_OK: return "BS_OK";
    case BS_ERR_INVALID_ARG: return "BS_ERR_INVALID_ARG";
    case BS_ERR_UNSUPPORTED: return "BS_ERR_UNSUPPORTED";
    case BS_ERR_CUDA: return "BS_ERR_CUDA";
    default: return "BS_UNKNOWN_STATUS";
  }
}

int bs_last_cuda_error(void) { return g_last_cuda_error; }

int bs_getrf_getrs_supported(bs_dtype dtype, bs_layout layout, int n, int nrhs) {
  return lu_supported(dtype, layout, n, nrhs) ? 1 : 0;
}

int bs_potrf_potrs_supported(bs_dtype dtype, bs_layout layout, bs_fill fill, int n, int nrhs) {
  return chol_supported(dtype, layout, fill, n, nrhs) ? 1 : 0;
}

int bs_bdsv_supported(bs_dtype dtype, int num_block_rows, int block_size) {
  return bdsv_supported(dtype, num_block_rows, block_size) ? 1 : 0;
}

int bs_version(void) { return 100; }

}  // extern "C"
