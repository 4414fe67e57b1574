// Top-k node expansion of a draft token tree: the k ids with the highest
// logits of each row, in descending logit order, equal logits by lower id.
//
// Source: "A 2.16x speculative-decoding speedup from a 1-layer Llama draft"
// §5 (the draft tree grows every node into its top_k draft tokens: total
// tokens, depth, top_k).
//
// One 512-thread block per row streams the row once (16-byte loads, eight
// vectors per thread in flight).  After the first batch of vectors the block
// fixes a lower bound T on the row's k-th largest logit: the k-th largest of
// the 512 lane maxima (k distinct logits reach it).  Every logit >= T, the
// first batch's included, goes into a shared candidate list as a packed
// (order key, ~id) word; a vector whose maximum is below T costs one
// comparison.  The candidates are distinct words, and the k largest of them
// are the answer: each candidate's rank is counted directly when there are
// at most 512, otherwise k rounds of a block-wide maximum below the previous
// winner pick them.  A row whose candidates overflow the list (ties or -inf
// at T, rising rows) is selected by those k rounds over the whole row.
#include <cuda_bf16.h>

#include "sv_internal.h"

namespace sv {

constexpr int kKThreads = 512;
constexpr int kKUnroll = 8;
constexpr int kKCap = 2048;  // shared candidate list

__device__ __forceinline__ float value_of_key(uint32_t key) {
  return __uint_as_float(key & 0x80000000u ? (key & 0x7fffffffu) : ~key);
}

// The largest logit of one 16-byte vector (bf16: packed maxima, two logits
// per instruction; a NaN never hides a number).
template <typename E>
__device__ __forceinline__ float vec_max(const uint4& w) {
  if constexpr (sizeof(E) == 2) {
    auto h = [](uint32_t x) {
      __nv_bfloat162 r;
      memcpy(&r, &x, sizeof(r));
      return r;
    };
    const __nv_bfloat162 m = __hmax2(__hmax2(h(w.x), h(w.y)), __hmax2(h(w.z), h(w.w)));
    return fmaxf(__low2float(m), __high2float(m));
  } else {
    return fmaxf(fmaxf(__uint_as_float(w.x), __uint_as_float(w.y)),
                 fmaxf(__uint_as_float(w.z), __uint_as_float(w.w)));
  }
}

// The warp's 32 values sorted in descending order across the lanes (bitonic).
__device__ __forceinline__ float warp_sort_desc(float x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const float o = __shfl_xor_sync(0xffffffffu, x, stride);
      const bool desc = (lane & size) == 0;
      const bool low = (lane & stride) == 0;
      x = (low == desc) ? fmaxf(x, o) : fminf(x, o);
    }
  }
  return x;
}

// Appends every logit >= thr of one vector to the shared candidate list.  A
// rare path, kept out of line: inlined at every vector of the unrolled loop it
// slows the streaming loop about twofold.
template <typename E>
__device__ __noinline__ void offer_vec(uint4 w, int id0, float thr, unsigned long long* key, int* count) {
#pragma unroll 1
  for (int e = 0; e < Elem<E>::kPerVec; ++e) {
    const float x = Elem<E>::at(w, e);
    if (x >= thr) {
      const int p = atomicAdd(count, 1);
      if (p < kKCap) key[p] = argmax_pack(x, id0 + e);
    }
  }
}

__device__ __forceinline__ void offer_one(float x, int j, float thr, unsigned long long* key, int* count) {
  if (x >= thr) {
    const int p = atomicAdd(count, 1);
    if (p < kKCap) key[p] = argmax_pack(x, j);
  }
}

// The largest packed word of this thread's share of the row below `below`.
template <typename E>
__device__ __noinline__ unsigned long long row_max_below(const E* row, RowSplit rs, int V, unsigned long long below) {
  constexpr int EPV = Elem<E>::kPerVec;
  const uint4* vp = reinterpret_cast<const uint4*>(row + rs.head);
  unsigned long long best = 0;
  auto take = [&](float x, int j) {
    if (!(x == x)) return;
    const unsigned long long w = argmax_pack(x, j);
    if (w < below && w > best) best = w;
  };
  for (int j = threadIdx.x; j < rs.head; j += kKThreads) take(Elem<E>::load(row + j), j);
  for (int v = threadIdx.x; v < rs.nvec; v += kKThreads) {
    const uint4 w = ldg_stream(vp + v);
#pragma unroll
    for (int e = 0; e < EPV; ++e) take(Elem<E>::at(w, e), rs.head + v * EPV + e);
  }
  for (int j = rs.tail0 + static_cast<int>(threadIdx.x); j < V; j += kKThreads) take(Elem<E>::load(row + j), j);
  return best;
}

template <typename E>
__global__ void __launch_bounds__(kKThreads, 2) topk_kernel(const E* __restrict__ logits, int64_t stride, int V,
                                                         int k, int32_t* __restrict__ out_ids,
                                                         float* __restrict__ out_vals) {
  constexpr int EPV = Elem<E>::kPerVec;
  constexpr int kBatch = kKThreads * kKUnroll;
  __shared__ unsigned long long s_key[kKCap];
  __shared__ unsigned long long s_red[32];
  __shared__ __align__(16) float s_top[(kKThreads / 32) * SV_MAX_TOPK];
  __shared__ uint32_t s_thr;
  __shared__ int s_cnt;
  const int r = blockIdx.x;
  const E* row = logits + static_cast<int64_t>(r) * stride;
  const RowSplit rs = split_row(row, V);
  const uint4* vp = reinterpret_cast<const uint4*>(row + rs.head);
  if (threadIdx.x == 0) {
    s_cnt = 0;
    s_thr = 0;
  }

  uint4 w[kKUnroll];
#pragma unroll
  for (int u = 0; u < kKUnroll; ++u) {
    const int v = threadIdx.x + u * kKThreads;
    w[u] = v < rs.nvec ? ldg_stream(vp + v) : Elem<E>::neg_inf_vec();
  }
  float m = -CUDART_INF_F;
#pragma unroll
  for (int u = 0; u < kKUnroll; ++u) m = fmaxf(m, vec_max<E>(w[u]));
  // The k-th largest of the 512 lane maxima: each warp's top k, then each
  // of those values counted against all of them.
  const float srt = warp_sort_desc(m);
  const int lane = threadIdx.x & 31, nt = (kKThreads / 32) * k;
  if (lane < k) s_top[(threadIdx.x >> 5) * k + lane] = srt;
  __syncthreads();
  if (static_cast<int>(threadIdx.x) < nt) {
    const float c = s_top[threadIdx.x];
    const float4* t4 = reinterpret_cast<const float4*>(s_top);  // nt is a multiple of 16
    int ge = 0;
#pragma unroll 4
    for (int j = 0; j < nt / 4; ++j) {
      const float4 q = t4[j];
      ge += (q.x >= c) + (q.y >= c) + (q.z >= c) + (q.w >= c);
    }
    if (ge >= k) atomicMax(&s_thr, order_key(c));
  }
  __syncthreads();
  const float thr = value_of_key(s_thr);

#pragma unroll
  for (int u = 0; u < kKUnroll; ++u) {
    const int v = threadIdx.x + u * kKThreads;
    if (v < rs.nvec && vec_max<E>(w[u]) >= thr) offer_vec<E>(w[u], rs.head + v * EPV, thr, s_key, &s_cnt);
  }
  for (int j = threadIdx.x; j < rs.head; j += kKThreads) offer_one(Elem<E>::load(row + j), j, thr, s_key, &s_cnt);
  for (int j = rs.tail0 + static_cast<int>(threadIdx.x); j < V; j += kKThreads)
    offer_one(Elem<E>::load(row + j), j, thr, s_key, &s_cnt);
  // Whole batches without bounds checks, then the last one with them.
  const int full_end = rs.nvec - kBatch;  // v0 <= full_end: the batch is in range
  int v0 = threadIdx.x + kBatch;
  for (; v0 <= full_end; v0 += kBatch) {
#pragma unroll
    for (int u = 0; u < kKUnroll; ++u) w[u] = ldg_stream(vp + v0 + u * kKThreads);
#pragma unroll
    for (int u = 0; u < kKUnroll; ++u)
      if (vec_max<E>(w[u]) >= thr) offer_vec<E>(w[u], rs.head + (v0 + u * kKThreads) * EPV, thr, s_key, &s_cnt);
  }
  if (v0 < rs.nvec) {
#pragma unroll
    for (int u = 0; u < kKUnroll; ++u) {
      const int v = v0 + u * kKThreads;
      w[u] = v < rs.nvec ? ldg_stream(vp + v) : Elem<E>::neg_inf_vec();
    }
#pragma unroll
    for (int u = 0; u < kKUnroll; ++u) {
      const int v = v0 + u * kKThreads;
      if (v < rs.nvec && vec_max<E>(w[u]) >= thr) offer_vec<E>(w[u], rs.head + v * EPV, thr, s_key, &s_cnt);
    }
  }
  __syncthreads();
  const int n = s_cnt;
  int32_t* oi = out_ids + static_cast<int64_t>(r) * k;
  float* ov = out_vals ? out_vals + static_cast<int64_t>(r) * k : nullptr;
  if (n <= kKThreads) {
    if (static_cast<int>(threadIdx.x) < n) {
      const unsigned long long mine = s_key[threadIdx.x];
      int rank = 0;
      for (int j = 0; j < n; ++j) rank += s_key[j] > mine;
      if (rank < k) {
        const int id = argmax_index(mine);
        oi[rank] = sv_in(id, V) ? id : -1;
        if (ov) ov[rank] = value_of_key(static_cast<uint32_t>(mine >> 32));
      }
    } else if (static_cast<int>(threadIdx.x) < k) {  // fewer than k logits that are not NaN
      oi[threadIdx.x] = -1;
      if (ov) ov[threadIdx.x] = CUDART_NAN_F;
    }
    return;
  }
  unsigned long long prev = ~0ull;
  for (int q = 0; q < k; ++q) {
    unsigned long long best = 0;
    if (n <= kKCap) {
      for (int j = threadIdx.x; j < n; j += kKThreads) {
        const unsigned long long x = s_key[j];
        if (x < prev && x > best) best = x;
      }
    } else {
      best = row_max_below(row, rs, V, prev);
    }
    prev = block_max_u64<kKThreads>(best, s_red);
    if (threadIdx.x == 0) {
      oi[q] = prev ? argmax_index(prev) : -1;
      if (ov) ov[q] = prev ? value_of_key(static_cast<uint32_t>(prev >> 32)) : CUDART_NAN_F;
    }
  }
}

template <typename E>
static sv_status launch_topk_typed(const sv_topk_desc& d, const void* logits, int32_t* ids, float* vals,
                                   cudaStream_t stream) {
  const E* l = static_cast<const E*>(logits);
  topk_kernel<E><<<d.rows, kKThreads, 0, stream>>>(l, d.row_stride, d.vocab, d.k, ids, vals);
  if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  note_launch(stream);
  return SV_OK;
}

sv_status topk_rows(const sv_topk_desc& d, const void* logits, int32_t* out_ids, float* out_vals,
                    cudaStream_t stream) {
  if (d.rows == 0) return SV_OK;
  start_phases(stream);
  return d.dtype == SV_BF16 ? launch_topk_typed<uint16_t>(d, logits, out_ids, out_vals, stream)
                            : launch_topk_typed<float>(d, logits, out_ids, out_vals, stream);
}

}  // namespace sv
