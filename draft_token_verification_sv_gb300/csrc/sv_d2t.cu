// EAGLE3 small-vocabulary mapping: scatter draft logits into the target
// vocabulary and build the inverse map.
//
// Source: "SSD: extending the engine with new models and an EAGLE3 draft"
// §六: the draft lm_head covers only draft_vocab_size ids; d2t/t2d map the
// small-vocabulary logits back into the full target vocabulary.
#include "sv_internal.h"

#include <cstring>

namespace sv {

// Gather form: every output element is written exactly once,
// out[r, t] = t2d[t] >= 0 ? in[r, t2d[t]] : fill.  Each thread owns U
// 16-byte output vectors of its row (strided by the block, so every load and
// store is coalesced); all their t2d entries are loaded before any value is
// gathered, and every gather before any store.
template <typename E, int THREADS, int U>
__global__ void __launch_bounds__(THREADS)
scatter_gather_kernel(const E* __restrict__ in, int64_t in_stride, const int32_t* __restrict__ t2d,
                      int vd, int V, E fill, E* __restrict__ out, int64_t out_stride, int tiles) {
  constexpr int EPV = Elem<E>::kPerVec;
  const int row = blockIdx.x / tiles;
  const int tile = blockIdx.x - row * tiles;
  const E* src = in + static_cast<int64_t>(row) * in_stride;
  E* dst = out + static_cast<int64_t>(row) * out_stride;
  const bool vec_ok = ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(t2d)) & 15u) == 0;
  const int v0 = tile * THREADS * U + static_cast<int>(threadIdx.x);
  if (vec_ok) {
    int32_t ids[U][EPV];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int t0 = (v0 + u * THREADS) * EPV;
#pragma unroll
      for (int q = 0; q < EPV / 4; ++q) {
        const int4 w = t0 + EPV <= V ? __ldg(reinterpret_cast<const int4*>(t2d + t0) + q) : make_int4(-1, -1, -1, -1);
        ids[u][4 * q + 0] = w.x;
        ids[u][4 * q + 1] = w.y;
        ids[u][4 * q + 2] = w.z;
        ids[u][4 * q + 3] = w.w;
      }
    }
    E vals[U][EPV];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        const int j = ids[u][e];
        vals[u][e] = (j >= 0 && j < vd) ? src[j] : fill;
      }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int t0 = (v0 + u * THREADS) * EPV;
      if (t0 + EPV <= V) {
        *reinterpret_cast<uint4*>(dst + t0) = *reinterpret_cast<const uint4*>(vals[u]);
      } else {
        for (int t = t0; t < V; ++t) {
          const int j = t2d[t];
          dst[t] = (j >= 0 && j < vd) ? src[j] : fill;
        }
      }
    }
  } else {
    for (int u = 0; u < U; ++u) {
      const int t0 = (v0 + u * THREADS) * EPV;
      for (int t = t0; t < min(V, t0 + EPV); ++t) {
        const int j = t2d[t];
        dst[t] = (j >= 0 && j < vd) ? src[j] : fill;
      }
    }
  }
}

// Sum of one int per thread, valid in every thread (shared counter: zeroed,
// added to, read; three barriers).
template <int THREADS>
__device__ __forceinline__ int block_sum_i(int v, int* counter) {
  if (threadIdx.x == 0) *counter = 0;
  __syncthreads();
  if (v) atomicAdd(counter, v);
  __syncthreads();
  const int r = *counter;
  __syncthreads();
  return r;
}

// Scatter form (no t2d): one block per row.  When d2t is strictly
// increasing within [0, V) (checked by the block over the whole map, which
// stays in L2), the row is built in shared-memory tiles of kTile ids: a
// tile is set to `fill`, the draft values whose ids fall in it (a contiguous
// run of draft ids, the run advancing tile by tile) are placed, and the tile
// is written out once with 16-byte stores.  Otherwise the block fills the
// row, then writes the draft values at their target ids (the barrier orders
// the two phases; every row is written twice).
template <typename E, int THREADS>
__global__ void __launch_bounds__(THREADS)
scatter_fill_kernel(const E* __restrict__ in, int64_t in_stride, const int32_t* __restrict__ d2t,
                    int vd, int V, E fill, E* __restrict__ out, int64_t out_stride) {
  constexpr int EPV = Elem<E>::kPerVec;
  constexpr int kTile = 8192;
  __shared__ __align__(16) E tile[kTile];
  __shared__ int s_a;
  const int row = blockIdx.x;
  const E* src = in + static_cast<int64_t>(row) * in_stride;
  E* dst = out + static_cast<int64_t>(row) * out_stride;
  int bad = 0;
  for (int j = threadIdx.x; j < vd; j += THREADS) {
    const int x = __ldg(d2t + j);
    if (x < 0 || x >= V || (j + 1 < vd && __ldg(d2t + j + 1) <= x)) bad = 1;
  }
  if (__syncthreads_or(bad)) {
    E fv[EPV];
#pragma unroll
    for (int e = 0; e < EPV; ++e) fv[e] = fill;
    const uint4 fvec = *reinterpret_cast<const uint4*>(fv);
    const RowSplit rs = split_row(dst, V);
    uint4* dv = reinterpret_cast<uint4*>(dst + rs.head);
    for (int v = threadIdx.x; v < rs.nvec; v += THREADS) dv[v] = fvec;
    for (int t = threadIdx.x; t < rs.head; t += THREADS) dst[t] = fill;
    for (int t = rs.tail0 + threadIdx.x; t < V; t += THREADS) dst[t] = fill;
    __syncthreads();
    for (int j = threadIdx.x; j < vd; j += THREADS) {
      const int x = __ldg(d2t + j);
      if (x >= 0 && sv_in(x, V)) dst[x] = src[j];
    }
    return;
  }
  const bool vec_ok = (reinterpret_cast<uintptr_t>(dst) & 15u) == 0;
  int a = 0;  // the first draft id whose target id is at or past this tile
  for (int t0 = 0; t0 < V; t0 += kTile) {
    const int n = min(kTile, V - t0);
    for (int i = threadIdx.x; i < n; i += THREADS) tile[i] = fill;
    __syncthreads();
    // The draft ids of this tile are a contiguous run from a (d2t is
    // increasing), at most n of them: place them and count them.
    const int m = min(n, vd - a);
    int cnt = 0;
    for (int i = threadIdx.x; i < m; i += THREADS) {
      const int x = __ldg(d2t + a + i) - t0;
      if (x < n) {
        if (sv_in(x, n)) tile[x] = src[a + i];
        ++cnt;
      }
    }
    const int run = block_sum_i<THREADS>(cnt, &s_a);  // its barriers also publish the tile
    if (vec_ok && (n % EPV) == 0 && (t0 % EPV) == 0) {
      const uint4* tv = reinterpret_cast<const uint4*>(tile);
      uint4* dv = reinterpret_cast<uint4*>(dst + t0);
      for (int v = threadIdx.x; v < n / EPV; v += THREADS) dv[v] = tv[v];
    } else {
      for (int i = threadIdx.x; i < n; i += THREADS) dst[t0 + i] = tile[i];
    }
    __syncthreads();
    a += run;
  }
}

__global__ void t2d_fill_kernel(int32_t* t2d, int V, int32_t* status) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t < V) t2d[t] = -1;
  if (t == 0 && status) *status = 0;
}

__global__ void t2d_set_kernel(const int32_t* d2t, int vd, int V, int32_t* t2d, int32_t* status) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= vd) return;
  const int x = d2t[j];
  if (x < 0 || x >= V) {
    if (status) atomicOr(status, 1);
    return;
  }
  const int old = atomicCAS(t2d + x, -1, j);
  if (old != -1 && status) atomicOr(status, 2);
}

template <typename E>
static E to_elem(float f);
template <>
float to_elem<float>(float f) {
  return f;
}
template <>
uint16_t to_elem<uint16_t>(float f) {
  // Round to nearest even; infinities and NaN keep their class.
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u) return static_cast<uint16_t>((u >> 16) | ((u & 0xffffu) ? 0x40u : 0u));
  u += 0x7fffu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

template <typename E>
static sv_status scatter_impl(const void* in, int64_t in_stride, const int32_t* d2t,
                              const int32_t* t2d, int rows, int vd, int V, float fill, void* out,
                              int64_t out_stride, cudaStream_t stream) {
  constexpr int kThreads = 256;
  if (rows == 0) return SV_OK;
  const E f = to_elem<E>(fill);
  if (t2d) {
    constexpr int kU = 8;
    const int nv = (V + Elem<E>::kPerVec - 1) / Elem<E>::kPerVec;
    const int tiles = (nv + kThreads * kU - 1) / (kThreads * kU);
    if (static_cast<long long>(rows) * tiles > INT32_MAX) return SV_ERR_UNSUPPORTED;
    scatter_gather_kernel<E, kThreads, kU><<<static_cast<unsigned>(rows) * tiles, kThreads, 0, stream>>>(
        static_cast<const E*>(in), in_stride, t2d, vd, V, f, static_cast<E*>(out), out_stride, tiles);
  } else {
    scatter_fill_kernel<E, 1024><<<rows, 1024, 0, stream>>>(static_cast<const E*>(in), in_stride, d2t,
                                                            vd, V, f, static_cast<E*>(out), out_stride);
  }
  if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  note_launch(stream);
  return SV_OK;
}

sv_status d2t_scatter(const void* in, int64_t in_stride, const int32_t* d2t, const int32_t* t2d,
                      int rows, int vd, int v, sv_dtype dtype, float fill, void* out,
                      int64_t out_stride, cudaStream_t stream) {
  return dtype == SV_BF16
             ? scatter_impl<uint16_t>(in, in_stride, d2t, t2d, rows, vd, v, fill, out, out_stride, stream)
             : scatter_impl<float>(in, in_stride, d2t, t2d, rows, vd, v, fill, out, out_stride, stream);
}

sv_status build_t2d(const int32_t* d2t, int vd, int v, int32_t* t2d, int32_t* status,
                    cudaStream_t stream) {
  t2d_fill_kernel<<<(v + 255) / 256, 256, 0, stream>>>(t2d, v, status);
  if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  note_launch(stream);
  if (vd > 0) {
    t2d_set_kernel<<<(vd + 255) / 256, 256, 0, stream>>>(d2t, vd, v, t2d, status);
    if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
    note_launch(stream);
  }
  return SV_OK;
}

}  // namespace sv
