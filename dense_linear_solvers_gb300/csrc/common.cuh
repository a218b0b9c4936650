// Shared device helpers of the batched small dense solvers (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace bsolve {

enum Layout : int { kRowMajor = 0, kColMajor = 1 };

// Magnitude keys for the pivot search. A key orders |x| exactly (the bit pattern of a
// non-negative IEEE number is monotone in its value) with integer compares, keeping the
// comparisons off the floating-point pipes. Keys are offset by one so that 0 can mean
// "not a candidate":
//   candidate x finite or inf -> bits(|x|) + 1
//   candidate NaN             -> 1 (never beats a number; a scan "v > best" skips it)
//   NaN in the row in place   -> KEY_MAX (a scan seeded with it never moves on)
template <typename T> struct Traits;

template <> struct Traits<float> {
  using Key = uint32_t;
  static constexpr Key kKeyMax = 0xFFFFFFFFu;
  // bits of the smallest normal number: |pivot| below it is singular.
  static constexpr Key kFloorBits = 0x00800000u;
  static constexpr Key kInfBits = 0x7F800000u;
  __device__ __forceinline__ static Key mag_bits(float x) {
    return __float_as_uint(x) & 0x7FFFFFFFu;
  }
};

template <> struct Traits<double> {
  using Key = unsigned long long;
  static constexpr Key kKeyMax = 0xFFFFFFFFFFFFFFFFull;
  static constexpr Key kFloorBits = 0x0010000000000000ull;
  static constexpr Key kInfBits = 0x7FF0000000000000ull;
  __device__ __forceinline__ static Key mag_bits(double x) {
    return static_cast<Key>(__double_as_longlong(x)) & 0x7FFFFFFFFFFFFFFFull;
  }
};

// Candidate key of value x; in_place marks the row at the step's own position.
template <typename T>
__device__ __forceinline__ typename Traits<T>::Key pivot_key(T x, bool in_place) {
  using Tr = Traits<T>;
  const typename Tr::Key m = Tr::mag_bits(x);
  if (m > Tr::kInfBits) return in_place ? Tr::kKeyMax : typename Tr::Key(1);
  return m + 1;
}

// A pivot whose key is k is regular iff its magnitude is a normal number or inf
// (!(|p| >= smallest normal) is singular: zero, subnormal, NaN).
template <typename T>
__device__ __forceinline__ bool pivot_ok(typename Traits<T>::Key k) {
  using Tr = Traits<T>;
  return k != Tr::kKeyMax && k >= Tr::kFloorBits + 1;
}

// The pivot value of a regular pivot from its key (magnitude bits + 1) and sign bit.
template <typename T>
__device__ __forceinline__ T pivot_from_key(typename Traits<T>::Key k, unsigned sign);
template <>
__device__ __forceinline__ float pivot_from_key<float>(uint32_t k, unsigned sign) {
  return __uint_as_float((k - 1u) | (sign << 31));
}
template <>
__device__ __forceinline__ double pivot_from_key<double>(unsigned long long k, unsigned sign) {
  return __longlong_as_double(static_cast<long long>((k - 1ull) |
                                                     (static_cast<unsigned long long>(sign) << 63)));
}

template <typename T>
__device__ __forceinline__ T fma_rn(T a, T b, T c);
template <>
__device__ __forceinline__ float fma_rn<float>(float a, float b, float c) {
  return __fmaf_rn(a, b, c);
}
template <>
__device__ __forceinline__ double fma_rn<double>(double a, double b, double c) {
  return __fma_rn(a, b, c);
}

// Asynchronous global -> shared copies of one element (cp.async, 4 or 8 bytes; both
// addresses aligned to the element size). Every copy a thread issues is in flight at
// once; cp_async_wait_all() waits for the thread's own copies.
template <typename T>
__device__ __forceinline__ void cp_async_elem(T* smem_dst, const T* gmem_src) {
  const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(smem_dst));
  if constexpr (sizeof(T) == 8)
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(d), "l"(gmem_src) : "memory");
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
// Waits until at most N of the thread's committed groups are still in flight.
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;\n" ::: "memory");
}

// Correctly rounded reciprocal and square root (IEEE round to nearest, the same results
// as 1/x and sqrt(x) on the host, with shorter instruction sequences than a division).
template <typename T>
__device__ __forceinline__ T rcp_rn(T x);
template <>
__device__ __forceinline__ float rcp_rn<float>(float x) { return __frcp_rn(x); }
template <>
__device__ __forceinline__ double rcp_rn<double>(double x) { return __drcp_rn(x); }

template <typename T>
__device__ __forceinline__ T sqrt_rn(T x);
template <>
__device__ __forceinline__ float sqrt_rn<float>(float x) { return __fsqrt_rn(x); }
template <>
__device__ __forceinline__ double sqrt_rn<double>(double x) { return __dsqrt_rn(x); }

// Shuffle of a 64-bit integer key as two 32-bit halves.
__device__ __forceinline__ unsigned long long shfl_xor_u64(unsigned long long v, int m,
                                                           int width) {
  const unsigned lo = __shfl_xor_sync(0xFFFFFFFFu, static_cast<unsigned>(v), m, width);
  const unsigned hi = __shfl_xor_sync(0xFFFFFFFFu, static_cast<unsigned>(v >> 32), m, width);
  return (static_cast<unsigned long long>(hi) << 32) | lo;
}
__device__ __forceinline__ uint32_t shfl_xor_key(uint32_t v, int m, int width) {
  return __shfl_xor_sync(0xFFFFFFFFu, v, m, width);
}
__device__ __forceinline__ unsigned long long shfl_xor_key(unsigned long long v, int m,
                                                           int width) {
  return shfl_xor_u64(v, m, width);
}

}  // namespace bsolve
