// Device helpers shared by the verify kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cooperative_groups.h>
#include <math_constants.h>
#include <stdint.h>

#include "spec_verify.h"

namespace sv {

namespace cg = cooperative_groups;

// Debug builds (-DSV_DEBUG): index checks on computed and data-dependent
// accesses.  A failed check sets a bit in this translation unit's debug word
// (read through sv_debug_flags) and the caller skips the access; nothing
// traps.  Release builds compile the checks away.
constexpr unsigned kDebugIndex = 1u;  // an index outside its buffer
#ifdef SV_DEBUG
static __device__ unsigned int g_sv_debug_word;
__device__ __forceinline__ bool sv_check(bool ok, unsigned bit) {
  if (!ok) atomicOr(&g_sv_debug_word, bit);
  return ok;
}
#else
__device__ __forceinline__ constexpr bool sv_check(bool, unsigned) { return true; }
#endif
// 0 <= i < n, checked in debug builds.
__device__ __forceinline__ bool sv_in(long long i, long long n) { return sv_check(i >= 0 && i < n, kDebugIndex); }

// Masses of the top-p search are summed exactly as integers: each
// exp((l - m)/T) in (0, 1] is rounded to a multiple of 2^-40.  With at most
// 2^24 elements the sums stay below 2^64 and the result does not depend on
// the order of accumulation.
constexpr float kFixScale = 1099511627776.0f;  // 2^40
constexpr double kFixInv = 1.0 / 1099511627776.0;

// Per-row result of the statistics pass, consumed by the decision/sampling
// pass.  e_j = exp2(l_j * c - mc) is the unnormalised weight of id j
// (c = log2(e) / T); the row's distribution is e_j / K over the kept ids.
struct __align__(32) RowStats {
  float m;         // largest logit of the row
  float mc;        // m * c, the offset used by every exp2 of this row
  float e_query;   // e at the row's query id if it is kept, else 0
  uint32_t tau;    // order key of the top-p threshold (0: every id kept)
  double K;        // kept mass sum(e_j over kept j)
  int32_t cut;     // ties at tau are kept iff their secondary id <= cut
  uint32_t status; // SV_ROW_* bits
};
static_assert(sizeof(RowStats) == 32, "RowStats layout");

// ---------------------------------------------------------------- loads ----

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Element traits: float rows and bf16 rows (stored as raw uint16 bits).
template <typename E> struct Elem;

template <> struct Elem<float> {
  static constexpr int kPerVec = 4;  // elements per 16-byte vector
  static constexpr uint32_t kNegInfBits = 0xff800000u;
  __device__ __forceinline__ static float at(const uint4& v, int i) {
    const uint32_t w = i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
    return __uint_as_float(w);
  }
  __device__ __forceinline__ static float load(const float* p) { return __ldg(p); }
  __device__ __forceinline__ static uint4 neg_inf_vec() {
    return make_uint4(kNegInfBits, kNegInfBits, kNegInfBits, kNegInfBits);
  }
};

template <> struct Elem<uint16_t> {
  static constexpr int kPerVec = 8;
  __device__ __forceinline__ static float at(const uint4& v, int i) {
    const uint32_t w = (i >> 1) == 0 ? v.x : (i >> 1) == 1 ? v.y : (i >> 1) == 2 ? v.z : v.w;
    return (i & 1) ? __uint_as_float(w & 0xffff0000u) : __uint_as_float(w << 16);
  }
  __device__ __forceinline__ static float load(const uint16_t* p) {
    return __uint_as_float(static_cast<uint32_t>(__ldg(p)) << 16);
  }
  __device__ __forceinline__ static uint4 neg_inf_vec() {
    const uint32_t w = 0xff80ff80u;
    return make_uint4(w, w, w, w);
  }
};

// A row split into a scalar head (until the first 16-byte boundary), a body
// of aligned 16-byte vectors and a scalar tail.
struct RowSplit {
  int head;  // elements before the first aligned vector
  int nvec;  // aligned vectors
  int tail0; // first tail element
};

template <typename E>
__device__ __forceinline__ RowSplit split_row(const E* p, int len) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  int head = static_cast<int>(((16u - (a & 15u)) & 15u) / sizeof(E));
  head = min(head, len);
  RowSplit s;
  s.head = head;
  s.nvec = (len - head) / Elem<E>::kPerVec;
  s.tail0 = head + s.nvec * Elem<E>::kPerVec;
  return s;
}

// Unpack a 16-byte vector into floats.
template <typename E>
__device__ __forceinline__ void unpack(const uint4& v, float* out) {
#pragma unroll
  for (int i = 0; i < Elem<E>::kPerVec; ++i) out[i] = Elem<E>::at(v, i);
}

// ------------------------------------------------------------ arithmetic ----

// Hardware base-2 exponential (MUFU), flushes subnormal results to zero.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Weight of a logit given the row offset: exp2(l * c - mc).  -inf -> 0.
__device__ __forceinline__ float weight(float l, float c, float mc) {
  return ex2(fmaf(l, c, -mc));
}

// Monotone map float -> uint32: a > b  <=>  key(a) > key(b); -0 and +0 share
// a key (they are equal logits).
__device__ __forceinline__ uint32_t order_key(float v) {
  uint32_t u = __float_as_uint(v);
  u = (u == 0x80000000u) ? 0u : u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ unsigned long long to_fixed(float e) {
  return __float2ull_rn(e * kFixScale);
}

// Is id j (with tie key `sec`) inside the kept set of a filtered row?
__device__ __forceinline__ bool kept(uint32_t key, int32_t sec, uint32_t tau, int32_t cut) {
  return key > tau || (key == tau && sec <= cut);
}

// ------------------------------------------------------------ reductions ----

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

__device__ __forceinline__ int warp_max_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide reductions; `scratch` holds >= 32 entries; result in every thread.
template <int THREADS>
__device__ __forceinline__ float block_max(float v, float* scratch) {
  v = warp_max(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) scratch[w] = v;
  __syncthreads();
  v = l < THREADS / 32 ? scratch[l] : -CUDART_INF_F;
  return warp_max(v);
}

template <int THREADS>
__device__ __forceinline__ float block_sum(float v, float* scratch) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) scratch[w] = v;
  __syncthreads();
  v = l < THREADS / 32 ? scratch[l] : 0.0f;
  return warp_sum(v);
}

template <int THREADS>
__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v,
                                                            unsigned long long* scratch) {
  v = warp_sum_u64(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) scratch[w] = v;
  __syncthreads();
  v = l < THREADS / 32 ? scratch[l] : 0ull;
  return warp_sum_u64(v);
}

template <int THREADS>
__device__ __forceinline__ unsigned long long block_max_u64(unsigned long long v,
                                                            unsigned long long* scratch) {
  v = warp_max_u64(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) scratch[w] = v;
  __syncthreads();
  v = l < THREADS / 32 ? scratch[l] : 0ull;
  return warp_max_u64(v);
}

template <int THREADS>
__device__ __forceinline__ int block_max_i(int v, int* scratch) {
  v = warp_max_i(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) scratch[w] = v;
  __syncthreads();
  v = l < THREADS / 32 ? scratch[l] : INT32_MIN;
  return warp_max_i(v);
}

// Exclusive prefix sum of one double per thread (block order); also returns
// the block total.
template <int THREADS>
__device__ __forceinline__ double block_exclusive_scan_d(double v, double* scratch, double* total) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  double x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, x, o);
    if (l >= o) x += y;
  }
  __syncthreads();
  if (l == 31) scratch[w] = x;
  __syncthreads();
  if (w == 0) {
    double s = l < THREADS / 32 ? scratch[l] : 0.0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, s, o);
      if (l >= o) s += y;
    }
    if (l < THREADS / 32) scratch[l] = s;  // inclusive warp totals
  }
  __syncthreads();
  const double before = w > 0 ? scratch[w - 1] : 0.0;
  *total = scratch[THREADS / 32 - 1];
  return before + x - v;
}

// Pack (value, index) so that the unsigned maximum is the largest value with
// the smallest index.
__device__ __forceinline__ unsigned long long argmax_pack(float v, int idx) {
  return (static_cast<unsigned long long>(order_key(v)) << 32) |
         static_cast<unsigned long long>(0xffffffffu - static_cast<uint32_t>(idx));
}
__device__ __forceinline__ int argmax_index(unsigned long long packed) {
  return static_cast<int>(0xffffffffu - static_cast<uint32_t>(packed & 0xffffffffull));
}

}  // namespace sv
