// LU with partial pivoting + solve for FP32 systems of order 8 < n <= 16: two rows per
// lane, eight lanes per system, four systems per warp; the plain and the interleaved
// batched layouts.
//
// The register-row scheme of the TDLS CooperativeLUpp solver (TDLS API,
// "solver_static.hpp File Reference", Detailed Description: rows held in registers,
// "logical" row interchanges) with each lane holding physical rows t and t + 8 of its
// system. Against one row per lane (sixteen lanes per system), every warp instruction of
// the per-step pivot bookkeeping now serves four systems instead of two, and the
// pivot-row broadcast (one shared-memory store by the owning lane, one 16-byte load per
// chunk by all lanes) reaches four systems per access. The kernel was measured bound by
// the L1/shared data pipe (wavefronts) as much as by issue, so the rows are read and
// written with 32-byte global accesses where the layout allows it.
//
// Step k (fully unrolled, every register index static):
//   1. live keys: the magnitude bits with the top bit set while the row sits at a position
//      >= k (one LOP3 per row; NaN keys rank above inf); the group maximum over the eight
//      lanes by one full-warp redux.sync per group;
//   2. among the rows holding the maximum, the lowest current position (the lowest-row tie
//      rule) together with the holder's sign, packed as (position << 1 | sign), by a
//      second group reduction (minimum); a rare NaN candidate rewrites the keys first (a
//      NaN at the step's own position wins, one elsewhere ties with zero);
//   3. positions k and p exchange (bookkeeping only); the pivot row records its LAPACK
//      swap entry ipiv[k] = old position + 1 and the pivot reciprocal;
//   4. the lane owning the pivot row stores its columns > k (from the 16-byte chunk holding
//      k + 1) and its right-hand sides into a per-system shared buffer (double-buffered by
//      step parity, one __syncwarp per step); every row below the pivot scales its
//      column-k entry by the reciprocal and takes the rank-1 update chunk by chunk (packed
//      two-wide fused multiply-adds, each element still rounded once per update).
// Back substitution publishes x_i the same way, one __syncwarp per step. Each row is
// written once, at its final position.
//
// Arithmetic, operation by operation, as the CPU oracle: r = 1/pivot correctly rounded
// (r = 1 for a pivot below the smallest normal number, NaN included), l = a_ik * r, every
// update one fused multiply-add in increasing k, x_k = y_k * r_k.
#include "common.cuh"
#include "kernels.h"

namespace bsolve {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int NT = 16;               // order tier
constexpr int R = 2;                 // rows per lane
constexpr int G = NT / R;            // lanes per system
constexpr int GPW = 32 / G;          // systems per warp
constexpr uint32_t kAlive = 0x80000000u;
constexpr uint32_t kNanAbove = 0xFF800000u;   // live key of inf
constexpr uint32_t kRegular = 0x80800000u;    // live key of the smallest normal number
constexpr uint32_t kMax = 0xFFFFFFFFu;        // a NaN at the step's own position

// (x & 0x7FFFFFFF) | live on the raw bits, as one integer LOP3 (kept away from any
// floating-point rewrite that could canonicalise a NaN payload).
__device__ __forceinline__ uint32_t live_key(float x, uint32_t live) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(__float_as_uint(x)), "r"(0x7FFFFFFFu),
      "r"(live));
  return d;
}

// Maximum / minimum of v over the eight lanes of group g: one full-warp reduction per
// group, the other groups contributing the neutral value.
__device__ __forceinline__ uint32_t group_max(uint32_t v, int g) {
  uint32_t m = 0;
#pragma unroll
  for (int q = 0; q < GPW; ++q) {
    const uint32_t r = __reduce_max_sync(0xFFFFFFFFu, g == q ? v : 0u);
    m = g == q ? r : m;
  }
  return m;
}
__device__ __forceinline__ uint32_t group_min(uint32_t v, int g) {
  uint32_t m = 0;
#pragma unroll
  for (int q = 0; q < GPW; ++q) {
    const uint32_t r = __reduce_min_sync(0xFFFFFFFFu, g == q ? v : 0xFFFFFFFFu);
    m = g == q ? r : m;
  }
  return m;
}

__device__ __forceinline__ void st4(float* p, float a, float b, float c, float d) {
  *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
}
__device__ __forceinline__ float4 ld4(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
// d0 += a * b0, d1 += a * b1 in one packed two-wide FMA (each result rounded once).
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a, float b0, float b1) {
  const float2 r = __ffma2_rn(make_float2(a, a), make_float2(b0, b1), make_float2(d0, d1));
  d0 = r.x;
  d1 = r.y;
}
// 32-byte global accesses (sm_100 and later), for rows whose address is 32-byte aligned.
__device__ __forceinline__ void ld8(const float* p, float* r) {
  asm volatile("ld.global.nc.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3]), "=f"(r[4]), "=f"(r[5]),
                 "=f"(r[6]), "=f"(r[7])
               : "l"(p));
}
__device__ __forceinline__ void st8(float* p, const float* r) {
  asm volatile("st.global.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "f"(r[0]),
               "f"(r[1]), "f"(r[2]), "f"(r[3]), "f"(r[4]), "f"(r[5]), "f"(r[6]), "f"(r[7])
               : "memory");
}

// One right-hand-side row of RT floats from / to global memory (RT a tier: 1, 2, 4, 8).
template <int RT>
__device__ __forceinline__ void load_rhs(const float* p, float (&b)[RT]) {
  if constexpr (RT % 4 == 0) {
#pragma unroll
    for (int c = 0; c < RT; c += 4) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(p + c));
      b[c] = v.x; b[c + 1] = v.y; b[c + 2] = v.z; b[c + 3] = v.w;
    }
  } else if constexpr (RT == 2) {
    const float2 v = __ldg(reinterpret_cast<const float2*>(p));
    b[0] = v.x; b[1] = v.y;
  } else {
    b[0] = __ldg(p);
  }
}
// The same row through shared memory (16-byte aligned buffers).
template <int RT>
__device__ __forceinline__ void ld_rhs_shared(const float* p, float (&b)[RT]) {
  if constexpr (RT % 4 == 0) {
#pragma unroll
    for (int c = 0; c < RT; c += 4) {
      const float4 v = ld4(p + c);
      b[c] = v.x; b[c + 1] = v.y; b[c + 2] = v.z; b[c + 3] = v.w;
    }
  } else if constexpr (RT == 2) {
    const float2 v = *reinterpret_cast<const float2*>(p);
    b[0] = v.x; b[1] = v.y;
  } else {
    b[0] = p[0];
  }
}
template <int RT>
__device__ __forceinline__ void store_rhs(float* p, const float (&b)[RT]) {
  if constexpr (RT % 4 == 0) {
#pragma unroll
    for (int c = 0; c < RT; c += 4) st4(p + c, b[c], b[c + 1], b[c + 2], b[c + 3]);
  } else if constexpr (RT == 2) {
    *reinterpret_cast<float2*>(p) = make_float2(b[0], b[1]);
  } else {
    p[0] = b[0];
  }
}

// RT: right-hand-side tier (0: factor only). FULL: n == 16 and nrhs == RT (no guards).
// W32: 32-byte row accesses of A (FULL row-major with a 32-byte aligned A).
// IL: the interleaved batched layout (TDLS API, "solver_static.hpp File Reference": element
// e of system s at base_s[e * ilv], base_s = (s / ilv) * ilv * size + s % ilv, for A, B and
// ipiv; info one entry per system). kIlStaged: every block's sixteen systems fill whole
// 16-byte groups of one AoSoA block (ilv a multiple of 16, the batch's ragged tail left to
// a kIlElem launch) and are staged through shared memory with 16-byte accesses, each
// holding one element of four systems; kIlElem: every element is read and written on its
// own. first_block: the index of the launch's first block in the batch (a tail launch
// starts past the staged blocks).
constexpr int kIlNone = 0, kIlElem = 1, kIlStaged = 2;
template <int RT, int LAYOUT, bool FULL, bool W32, int IL>
__global__ void __launch_bounds__(kThreads, RT == 0 ? 8 : (RT <= 4 && IL != kIlElem ? 7 : 6))
lu_rows2_kernel(int n_, int nrhs_, int64_t batch, float* __restrict__ A, float* __restrict__ B,
                int32_t* __restrict__ ipiv, int32_t* __restrict__ info, int64_t ilv,
                int64_t first_block) {
  constexpr bool kSolve = RT > 0;
  constexpr bool staged = IL == kIlStaged;
  constexpr int RB = kSolve ? RT : 1;
  constexpr int WP = (NT + RB + 3) / 4 * 4;   // published row: A part, then B part
  __shared__ __align__(16) float prow[kWarps][GPW][2][WP];
  __shared__ __align__(16) float xbuf[kWarps][GPW][2][(RB + 3) / 4 * 4];
  // staging of an interleaved block: row r of the block's system j at j*SA + r*PA (A) and
  // j*SB + r*PB (B). Row pitches of 16-byte multiples let a lane move its row with 16-byte
  // accesses (PA = 20 words: eight consecutive rows hit distinct banks); the system strides
  // are 4 words off a multiple of 32 so that the element-wise transposition from and to the
  // 16-byte global vectors (one element of four systems each) spreads over the banks.
  constexpr int SPC = kWarps * GPW;          // systems of a thread block
  constexpr int PA = NT + 4, PB = (RB + 3) / 4 * 4;
  constexpr int SA = NT * PA + 4, SB = NT * PB + 4;
  __shared__ __align__(16) float st_a[staged ? SPC * SA : 4];
  __shared__ __align__(16) float st_b[staged ? SPC * SB : 4];
  __shared__ int32_t st_p[staged ? SPC * NT : 1];

  const int n = FULL ? NT : n_;
  const int nrhs = FULL ? RT : nrhs_;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane / G;
  const int t = lane % G;
  const int64_t bidx = first_block + blockIdx.x;
  const int64_t s = (bidx * kWarps + warp) * GPW + g;
  const bool valid = staged || s < batch;
  const int64_t sA = s * n * n;
  const int64_t sB = s * n * nrhs;
  // interleaved: the system's first element of A, B and ipiv (element stride ilv)
  const int64_t blk = IL ? s / ilv : 0;
  const int64_t sl = IL ? s - blk * ilv : 0;
  const int64_t eA = IL ? blk * ilv * n * n + sl : 0;
  const int64_t eB = IL ? blk * ilv * n * nrhs + sl : 0;
  const int64_t s_first = bidx * SPC;
  const int jl = warp * GPW + g;              // this group's system in the block
  const int64_t blk0 = staged ? s_first / ilv : 0;
  const int64_t sl0 = staged ? s_first - blk0 * ilv : 0;
  // staging passes: thread i moves the 16-byte vector q = i % PER (systems 4q..4q+3 of the
  // block) of elements i / PER + EPI * pass
  constexpr int PER = SPC / 4;                // 16-byte vectors per element
  constexpr int EPI = kThreads / PER;         // elements per pass
  const int q = threadIdx.x % PER, e0 = threadIdx.x / PER;
  if constexpr (staged) {
    const float* Ab = A + blk0 * ilv * n * n + sl0 + q * 4 + e0 * ilv;
    const int64_t step = EPI * ilv;
    if constexpr (FULL) {
      constexpr int kPassA = NT * NT / EPI;
      float4 v[kPassA];
#pragma unroll
      for (int it = 0; it < kPassA; ++it) v[it] = __ldg(reinterpret_cast<const float4*>(Ab + it * step));
#pragma unroll
      for (int it = 0; it < kPassA; ++it) {
        const int e = e0 + it * EPI;
        const int r = LAYOUT == kRowMajor ? e / NT : e % NT;
        const int c = LAYOUT == kRowMajor ? e % NT : e / NT;
        float* d = st_a + (q * 4) * SA + r * PA + c;
        d[0] = v[it].x;
        d[SA] = v[it].y;
        d[2 * SA] = v[it].z;
        d[3 * SA] = v[it].w;
      }
    } else {
      for (int e = e0, it = 0; e < n * n; e += EPI, ++it) {
        const int r = LAYOUT == kRowMajor ? e / n : e % n;
        const int c = LAYOUT == kRowMajor ? e % n : e / n;
        const float4 v = __ldg(reinterpret_cast<const float4*>(Ab + it * step));
        float* d = st_a + (q * 4) * SA + r * PA + c;
        d[0] = v.x;
        d[SA] = v.y;
        d[2 * SA] = v.z;
        d[3 * SA] = v.w;
      }
    }
    if constexpr (kSolve) {
      const float* Bb = B + blk0 * ilv * n * nrhs + sl0 + q * 4 + e0 * ilv;
#pragma unroll
      for (int e = e0, it = 0; e < n * nrhs; e += EPI, ++it) {
        const int r = LAYOUT == kRowMajor ? e / nrhs : e % n;
        const int c = LAYOUT == kRowMajor ? e % nrhs : e / n;
        const float4 v = __ldg(reinterpret_cast<const float4*>(Bb + it * step));
        float* d = st_b + (q * 4) * SB + r * PB + c;
        d[0] = v.x;
        d[SB] = v.y;
        d[2 * SB] = v.z;
        d[3 * SB] = v.w;
      }
    }
    __syncthreads();
  }

  float a[R][NT];
  float b[R][RB];
  int pos[R], ip[R];
  float rr[R];
  uint32_t okm[R];   // all ones for a real row of a real system
#pragma unroll
  for (int j = 0; j < R; ++j) {
    pos[j] = t + j * G;
    ip[j] = 0;
    rr[j] = 1.f;
    const bool row_ok = valid && (FULL || pos[j] < n);
    okm[j] = row_ok ? 0xFFFFFFFFu : 0u;
    const int row = pos[j];
    if (row_ok && staged) {
      const float* ra = st_a + jl * SA + row * PA;
      const float* rb = st_b + jl * SB + row * PB;
      if constexpr (FULL) {
#pragma unroll
        for (int c = 0; c < NT; c += 4) {
          const float4 v = ld4(ra + c);
          a[j][c] = v.x; a[j][c + 1] = v.y; a[j][c + 2] = v.z; a[j][c + 3] = v.w;
        }
        if constexpr (kSolve) ld_rhs_shared<RT>(rb, b[j]);
      } else {
#pragma unroll
        for (int c = 0; c < NT; ++c) a[j][c] = c < n ? ra[c] : 0.f;
#pragma unroll
        for (int c = 0; c < RT; ++c) b[j][c] = c < nrhs ? rb[c] : 0.f;
      }
    } else if (row_ok && IL == kIlElem) {
#pragma unroll
      for (int c = 0; c < NT; ++c)
        a[j][c] = (FULL || c < n)
                      ? A[eA + (LAYOUT == kRowMajor ? row * n + c : c * n + row) * ilv]
                      : 0.f;
#pragma unroll
      for (int c = 0; c < RT; ++c)
        b[j][c] = (FULL || c < nrhs)
                      ? B[eB + (LAYOUT == kRowMajor ? row * nrhs + c : c * n + row) * ilv]
                      : 0.f;
    } else if (row_ok) {
      if constexpr (LAYOUT == kRowMajor && FULL && IL == kIlNone) {
        const float* pa = A + sA + row * NT;
        if constexpr (W32) {
          ld8(pa, &a[j][0]);
          ld8(pa + 8, &a[j][8]);
        } else {
#pragma unroll
          for (int c = 0; c < NT; c += 4) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(pa + c));
            a[j][c] = v.x; a[j][c + 1] = v.y; a[j][c + 2] = v.z; a[j][c + 3] = v.w;
          }
        }
        if constexpr (kSolve) load_rhs<RT>(B + sB + row * RT, b[j]);
      } else {
#pragma unroll
        for (int c = 0; c < NT; ++c)
          a[j][c] = (FULL || c < n) ? A[sA + (LAYOUT == kRowMajor ? row * n + c : c * n + row)]
                                    : 0.f;
#pragma unroll
        for (int c = 0; c < RT; ++c)
          b[j][c] = (FULL || c < nrhs)
                        ? B[sB + (LAYOUT == kRowMajor ? row * nrhs + c : c * n + row)]
                        : 0.f;
      }
    } else {
#pragma unroll
      for (int c = 0; c < NT; ++c) a[j][c] = 0.f;
    }
    if (!row_ok || !kSolve) {
#pragma unroll
      for (int c = 0; c < RB; ++c) b[j][c] = 0.f;
    }
  }
  uint32_t fm = 0;   // bit k: the pivot of step k is singular

#pragma unroll
  for (int k = 0; k < NT; ++k) {
    if (!FULL && k >= n) break;
    uint32_t key[R];
#pragma unroll
    for (int j = 0; j < R; ++j)
      key[j] = live_key(a[j][k], static_cast<uint32_t>(k - 1 - pos[j]) & kAlive & okm[j]);
    uint32_t mk = group_max(key[0] > key[1] ? key[0] : key[1], g);
    if (__any_sync(0xFFFFFFFFu, mk > kNanAbove)) {
      // a NaN among some group's candidates (rare): the contract's keys
#pragma unroll
      for (int j = 0; j < R; ++j)
        if (key[j] > kNanAbove) key[j] = pos[j] == k ? kMax : kAlive;
      mk = group_max(key[0] > key[1] ? key[0] : key[1], g);
    }
    // the lowest current position among the holders of the maximum, with its sign
    uint32_t lc = 0xFFFFFFFFu;
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const uint32_t c = key[j] == mk ? ((static_cast<uint32_t>(pos[j]) << 1) |
                                         (__float_as_uint(a[j][k]) >> 31))
                                      : 0xFFFFFFFFu;
      lc = c < lc ? c : lc;
    }
    const uint32_t pc = group_min(lc, g);
    const int pos_p = static_cast<int>(pc >> 1);
    const bool ok = mk >= kRegular && mk != kMax;
    if (!ok) fm |= 1u << k;
    const float piv = __uint_as_float((mk & 0x7FFFFFFFu) | (pc << 31));
    const float r = ok ? 1.0f / piv : 1.0f;
    bool isp[R];
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const bool at_k = pos[j] == k, is_p = pos[j] == pos_p;
      isp[j] = is_p;
      pos[j] = at_k ? pos_p : pos[j];
      pos[j] = is_p ? k : pos[j];
      ip[j] = is_p ? pos_p + 1 : ip[j];
      rr[j] = is_p ? r : rr[j];
    }

    // publish the pivot row's columns > k (from the chunk holding k + 1) and its B part
    float* pr = prow[warp][g][k & 1];
    const int c1 = (k + 1) & ~3;
#pragma unroll
    for (int j = 0; j < R; ++j) {
      if (isp[j]) {
#pragma unroll
        for (int c = 0; c < NT; c += 4)
          if (c >= c1) st4(pr + c, a[j][c], a[j][c + 1], a[j][c + 2], a[j][c + 3]);
        if constexpr (kSolve) store_rhs<RT>(pr + NT, b[j]);
      }
    }
    __syncwarp();
    float nl[R];
    bool up[R];
#pragma unroll
    for (int j = 0; j < R; ++j) {
      up[j] = pos[j] > k;
      const float l = a[j][k] * r;
      if (up[j]) a[j][k] = l;
      nl[j] = -l;
    }
    // rank-1 update, one 16-byte chunk of the pivot row at a time
#pragma unroll
    for (int c = 0; c < NT; c += 4) {
      if (c >= c1) {
        const float4 v = ld4(pr + c);
        const float u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < R; ++j) {
          if (up[j]) {
            if (c >= k + 1) {
              ffma2(a[j][c], a[j][c + 1], nl[j], u[0], u[1]);
              ffma2(a[j][c + 2], a[j][c + 3], nl[j], u[2], u[3]);
            } else {
#pragma unroll
              for (int q = 0; q < 4; ++q)
                if (c + q >= k + 1) a[j][c + q] = __fmaf_rn(nl[j], u[q], a[j][c + q]);
            }
          }
        }
        asm volatile("" ::: "memory");   // keep the chunks' loads apart (live registers)
      }
    }
    if constexpr (kSolve) {
      float ub[RT];
      ld_rhs_shared<RT>(pr + NT, ub);
#pragma unroll
      for (int j = 0; j < R; ++j) {
        if (up[j]) {
#pragma unroll
          for (int c = 0; c + 1 < RT; c += 2) ffma2(b[j][c], b[j][c + 1], nl[j], ub[c], ub[c + 1]);
          if constexpr (RT & 1) b[j][RT - 1] = __fmaf_rn(nl[j], ub[RT - 1], b[j][RT - 1]);
        }
      }
    }
  }

  // U x = y, from the last position
  if constexpr (kSolve) {
#pragma unroll
    for (int i = NT - 1; i >= 0; --i) {
      if (!FULL && i >= n) continue;
      float* xb = xbuf[warp][g][i & 1];
#pragma unroll
      for (int j = 0; j < R; ++j) {
        if (pos[j] == i) {
#pragma unroll
          for (int c = 0; c < RT; ++c) b[j][c] = b[j][c] * rr[j];
          store_rhs<RT>(xb, b[j]);
        }
      }
      __syncwarp();
      float x[RT];
      ld_rhs_shared<RT>(xb, x);
#pragma unroll
      for (int j = 0; j < R; ++j) {
        if (pos[j] < i) {
          const float nu = -a[j][i];
#pragma unroll
          for (int c = 0; c + 1 < RT; c += 2) ffma2(b[j][c], b[j][c + 1], nu, x[c], x[c + 1]);
          if constexpr (RT & 1) b[j][RT - 1] = __fmaf_rn(nu, x[RT - 1], b[j][RT - 1]);
        }
      }
    }
  }

  if (fm != 0) {   // the contract: X is zero where info != 0
#pragma unroll
    for (int j = 0; j < R; ++j)
#pragma unroll
      for (int c = 0; c < RB; ++c) b[j][c] = 0.f;
  }
  if constexpr (staged) {
#pragma unroll
    for (int j = 0; j < R; ++j) {
      if (!okm[j]) continue;
      const int row = pos[j];
      float* ra = st_a + jl * SA + row * PA;
      float* rb = st_b + jl * SB + row * PB;
      if constexpr (FULL) {
#pragma unroll
        for (int c = 0; c < NT; c += 4) st4(ra + c, a[j][c], a[j][c + 1], a[j][c + 2], a[j][c + 3]);
        if constexpr (kSolve) store_rhs<RT>(rb, b[j]);
      } else {
#pragma unroll
        for (int c = 0; c < NT; ++c)
          if (c < n) ra[c] = a[j][c];
#pragma unroll
        for (int c = 0; c < RT; ++c)
          if (c < nrhs) rb[c] = b[j][c];
      }
      st_p[jl * NT + row] = ip[j];
    }
    if (t == 0) info[s] = fm ? __ffs(static_cast<int>(fm)) : 0;
    __syncthreads();
    float* Ab = A + blk0 * ilv * n * n + sl0 + q * 4 + e0 * ilv;
    const int64_t step = EPI * ilv;
    if constexpr (FULL) {
#pragma unroll
      for (int it = 0; it < NT * NT / EPI; ++it) {
        const int e = e0 + it * EPI;
        const int r = LAYOUT == kRowMajor ? e / NT : e % NT;
        const int c = LAYOUT == kRowMajor ? e % NT : e / NT;
        const float* d = st_a + (q * 4) * SA + r * PA + c;
        st4(Ab + it * step, d[0], d[SA], d[2 * SA], d[3 * SA]);
      }
    } else {
      for (int e = e0, it = 0; e < n * n; e += EPI, ++it) {
        const int r = LAYOUT == kRowMajor ? e / n : e % n;
        const int c = LAYOUT == kRowMajor ? e % n : e / n;
        const float* d = st_a + (q * 4) * SA + r * PA + c;
        st4(Ab + it * step, d[0], d[SA], d[2 * SA], d[3 * SA]);
      }
    }
    if constexpr (kSolve) {
      float* Bb = B + blk0 * ilv * n * nrhs + sl0 + q * 4 + e0 * ilv;
#pragma unroll
      for (int e = e0, it = 0; e < n * nrhs; e += EPI, ++it) {
        const int r = LAYOUT == kRowMajor ? e / nrhs : e % n;
        const int c = LAYOUT == kRowMajor ? e % nrhs : e / n;
        const float* d = st_b + (q * 4) * SB + r * PB + c;
        st4(Bb + it * step, d[0], d[SB], d[2 * SB], d[3 * SB]);
      }
    }
    int32_t* Pb = ipiv + blk0 * ilv * n + sl0 + q * 4;
    for (int k = e0; k < n; k += EPI)
      *reinterpret_cast<int4*>(Pb + static_cast<int64_t>(k) * ilv) =
          make_int4(st_p[(q * 4) * NT + k], st_p[(q * 4 + 1) * NT + k],
                    st_p[(q * 4 + 2) * NT + k], st_p[(q * 4 + 3) * NT + k]);
    return;
  }
  if (!valid) return;
#pragma unroll
  for (int j = 0; j < R; ++j) {
    if (!okm[j]) continue;
    const int row = pos[j];   // the final position
    if constexpr (IL == kIlElem) {
#pragma unroll
      for (int c = 0; c < NT; ++c)
        if (FULL || c < n) A[eA + (LAYOUT == kRowMajor ? row * n + c : c * n + row) * ilv] = a[j][c];
#pragma unroll
      for (int c = 0; c < RT; ++c)
        if (FULL || c < nrhs)
          B[eB + (LAYOUT == kRowMajor ? row * nrhs + c : c * n + row) * ilv] = b[j][c];
      ipiv[blk * ilv * n + sl + static_cast<int64_t>(row) * ilv] = ip[j];
      continue;
    } else if constexpr (LAYOUT == kRowMajor && FULL) {
      float* pa = A + sA + row * NT;
      if constexpr (W32) {
        st8(pa, &a[j][0]);
        st8(pa + 8, &a[j][8]);
      } else {
#pragma unroll
        for (int c = 0; c < NT; c += 4) st4(pa + c, a[j][c], a[j][c + 1], a[j][c + 2], a[j][c + 3]);
      }
      if constexpr (kSolve) store_rhs<RT>(B + sB + row * RT, b[j]);
    } else {
#pragma unroll
      for (int c = 0; c < NT; ++c)
        if (FULL || c < n) A[sA + (LAYOUT == kRowMajor ? row * n + c : c * n + row)] = a[j][c];
#pragma unroll
      for (int c = 0; c < RT; ++c)
        if (FULL || c < nrhs) B[sB + (LAYOUT == kRowMajor ? row * nrhs + c : c * n + row)] = b[j][c];
    }
    ipiv[s * n + row] = ip[j];
  }
  if (t == 0) info[s] = fm ? __ffs(static_cast<int>(fm)) : 0;
}

// The staged instance takes whole interleaved blocks with the shared memory it needs for
// seven blocks per SM; the element-wise one the ragged tail (or every block when ilv is
// not a multiple of sixteen).
template <int RT, int LAYOUT, bool FULL>
cudaError_t launch_il(unsigned nb, int n, int nrhs, int64_t batch, int64_t ilv, float* A,
                      float* B, int32_t* ipiv, int32_t* info, cudaStream_t stream) {
  constexpr int per_block = kWarps * GPW;
  const int64_t whole = ilv % per_block == 0 ? batch / per_block : 0;
  if (whole > 0) {
    auto kern = lu_rows2_kernel<RT, LAYOUT, FULL, false, kIlStaged>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>(whole), kThreads, 0, stream>>>(n, nrhs, batch, A, B, ipiv,
                                                                info, ilv, 0);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (nb > whole)
    lu_rows2_kernel<RT, LAYOUT, FULL, false, kIlElem>
        <<<static_cast<unsigned>(nb - whole), kThreads, 0, stream>>>(n, nrhs, batch, A, B,
                                                                    ipiv, info, ilv, whole);
  return cudaGetLastError();
}

template <int RT, int LAYOUT>
cudaError_t launch_tier(int n, int nrhs, int64_t batch, int64_t ilv, float* A, float* B,
                        int32_t* ipiv, int32_t* info, cudaStream_t stream) {
  constexpr int per_block = kWarps * GPW;
  const int64_t blocks = (batch + per_block - 1) / per_block;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  const unsigned nb = static_cast<unsigned>(blocks);
  const bool full = n == NT && nrhs == RT;
  if (ilv > 1) {
    if (full) return launch_il<RT, LAYOUT, true>(nb, n, nrhs, batch, ilv, A, B, ipiv, info, stream);
    return launch_il<RT, LAYOUT, false>(nb, n, nrhs, batch, ilv, A, B, ipiv, info, stream);
  } else if (full) {
    if (LAYOUT == kRowMajor && reinterpret_cast<uintptr_t>(A) % 32 == 0)
      lu_rows2_kernel<RT, LAYOUT, true, true, kIlNone><<<nb, kThreads, 0, stream>>>(
          n, nrhs, batch, A, B, ipiv, info, 1, 0);
    else
      lu_rows2_kernel<RT, LAYOUT, true, false, kIlNone><<<nb, kThreads, 0, stream>>>(
          n, nrhs, batch, A, B, ipiv, info, 1, 0);
  } else {
    lu_rows2_kernel<RT, LAYOUT, false, false, kIlNone><<<nb, kThreads, 0, stream>>>(
        n, nrhs, batch, A, B, ipiv, info, 1, 0);
  }
  return cudaGetLastError();
}

template <int LAYOUT>
cudaError_t launch_layout(int n, int nrhs, int64_t batch, int64_t ilv, float* A, float* B,
                          int32_t* ipiv, int32_t* info, cudaStream_t stream) {
  if (nrhs == 0) return launch_tier<0, LAYOUT>(n, nrhs, batch, ilv, A, B, ipiv, info, stream);
  if (nrhs <= 1) return launch_tier<1, LAYOUT>(n, nrhs, batch, ilv, A, B, ipiv, info, stream);
  if (nrhs <= 2) return launch_tier<2, LAYOUT>(n, nrhs, batch, ilv, A, B, ipiv, info, stream);
  if (nrhs <= 4) return launch_tier<4, LAYOUT>(n, nrhs, batch, ilv, A, B, ipiv, info, stream);
  return launch_tier<8, LAYOUT>(n, nrhs, batch, ilv, A, B, ipiv, info, stream);
}

}  // namespace

cudaError_t launch_lu_rows2(int layout, int n, int nrhs, int64_t batch, float* A, float* B,
                            int32_t* ipiv, int32_t* info, cudaStream_t stream, int64_t ilv) {
  if (n <= G || n > NT || nrhs < 0 || nrhs > 8 || ilv < 1) return cudaErrorInvalidValue;
  if (layout == kRowMajor)
    return launch_layout<kRowMajor>(n, nrhs, batch, ilv, A, B, ipiv, info, stream);
  return launch_layout<kColMajor>(n, nrhs, batch, ilv, A, B, ipiv, info, stream);
}

}  // namespace bsolve
