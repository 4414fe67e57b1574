// Decision and draw of the sampling verify: accept/reject per draft, first
// rejection, and the resample / bonus draw by inverse CDF.
//
// Source: "LLM inference acceleration in practice: draft models and
// speculative sampling explained" (mlqm.cn) §3.1 (accept with min(1, p/q);
// on the first rejection sample from norm(max(0, p - q)); after γ
// acceptances sample the extra token from p) and §4.2 (the accept loop of
// generate()).  The uniforms are supplied by the caller.
//
// The accept/reject decisions of a batch row (decide_batch in sv_rows.cuh:
// the first rejection k, the status bits and the draw rows) are made by the
// statistics pass when it has a last block per row anyway (top-p), else by
// warp 0 of every block here.  The vocabulary
// of a batch row is cut into segments of NC chunks of 2048 ids, one thread
// block per (row, segment), with no cooperation between the blocks of a row
// while they stream.  Every block reads the record, then loads its segment of
// target row k (and of draft row k when drawing from the residual) with every
// 16-byte load of the segment issued before the first is used, and writes one
// draw-weight sum per chunk.  The last block of the row to finish (a counter
// per row) scans the chunk sums, finds the chunk that holds u * total and
// rescans that one chunk (from L2) with a block-wide prefix scan to pick the
// token.
#include "sv_rows.cuh"

namespace sv {

constexpr int kDThreads = 256;
constexpr int kDEPT = 8;                    // consecutive ids per thread per chunk
constexpr int kDChunk = kDThreads * kDEPT;  // 2048 ids per chunk
constexpr int kDWarps = kDThreads / 32;
constexpr int kDMaxNC = 8;                  // chunks per block (at most)

struct DecideShared {
  DecideRecord rec;
  float wsum[kDMaxNC][kDWarps];
  DrawSide pt, pd;
  double scan[32];
  int red_i[32];
  int k;
  unsigned status;
  int last;
  int chunk;
  int tok;
  int best;
  double carry;
  double target;
  double total;
};

// Raw 16-byte vectors of 8 consecutive logits: one for bf16, two for f32.
template <typename E>
struct Raw8 {
  static constexpr int kVec = sizeof(E) == 2 ? 1 : 2;
  uint4 v[kVec];
};

template <typename E>
__device__ __forceinline__ void raw_load(Raw8<E>& r, const E* p) {
#pragma unroll
  for (int i = 0; i < Raw8<E>::kVec; ++i) r.v[i] = __ldcg(reinterpret_cast<const uint4*>(p) + i);
}

template <typename E>
__device__ __forceinline__ float raw_at(const Raw8<E>& r, int e) {
  if constexpr (sizeof(E) == 2) {
    return Elem<uint16_t>::at(r.v[0], e);
  } else {
    return Elem<float>::at(r.v[e >> 2], e & 3);
  }
}

// Normalised filtered probability of id j with logit x (0 if filtered out).
__device__ __forceinline__ float prob_of(float x, int j, float c, const DrawSide& s) {
  if (s.tau != 0u && !kept(order_key(x), j, s.tau, s.cut)) return 0.0f;
  return weight(x, c, s.mc) * s.invK;
}

// Draw weight of id j: p(j) (bonus) or max(0, p(j) - q(j)) (residual; ld is
// -inf where the draft row has no entry for j).
__device__ __forceinline__ float draw_weight(float lt, float ld, int j, bool resid, float c, const DrawSide& pt,
                                             const DrawSide& pd) {
  const float p = prob_of(lt, j, c, pt);
  if (!resid) return p;
  const float q = ld > -CUDART_INF_F ? prob_of(ld, j, c, pd) : 0.0f;
  return fmaxf(0.0f, p - q);
}

struct RowView {
  const void* trow;
  const void* drow;
  bool fast;  // 16-byte aligned rows and V a multiple of 8: whole-vector loads
};

// Draw weights of the 8 ids of chunk `ch` owned by this thread (any layout).
template <typename ET, typename ED>
__device__ __forceinline__ void chunk_weights(const DecideParams& P, const RowView& R, int ch, bool resid,
                                              const DrawSide& pt, const DrawSide& pd, float* w) {
  const int j0 = ch * kDChunk + static_cast<int>(threadIdx.x) * kDEPT;
  const ET* trow = static_cast<const ET*>(R.trow);
  const ED* drow = static_cast<const ED*>(R.drow);
  float lt[8], ld[8];
  if (R.fast && j0 < P.V) {
    Raw8<ET> rt;
    raw_load(rt, trow + j0);
#pragma unroll
    for (int e = 0; e < 8; ++e) lt[e] = raw_at(rt, e);
    if (resid && !P.t2d) {
      Raw8<ED> rd;
      raw_load(rd, drow + j0);
#pragma unroll
      for (int e = 0; e < 8; ++e) ld[e] = raw_at(rd, e);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) lt[e] = j0 + e < P.V ? Elem<ET>::load(trow + j0 + e) : -CUDART_INF_F;
    if (resid && !P.t2d) {
#pragma unroll
      for (int e = 0; e < 8; ++e) ld[e] = j0 + e < P.V ? Elem<ED>::load(drow + j0 + e) : -CUDART_INF_F;
    }
  }
  if (resid && P.t2d) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int jd = j0 + e < P.V ? __ldg(P.t2d + j0 + e) : -1;
      ld[e] = (jd >= 0 && sv_in(jd, P.Vd)) ? Elem<ED>::load(drow + jd) : -CUDART_INF_F;
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e)
    w[e] = j0 + e < P.V ? draw_weight(lt[e], resid ? ld[e] : -CUDART_INF_F, j0 + e, resid, P.c, pt, pd) : 0.0f;
}

// Per-thread draw-weight sums of the NC chunks c0.. of this block with every
// load of the segment in flight together (R.fast only); groups of 8 ids past
// the row add nothing.  lp: the largest id with a positive weight.
template <typename ET, typename ED, int NC>
__device__ __forceinline__ void segment_sums_fast(const DecideParams& P, const RowView& R, int c0, bool resid,
                                                  const DrawSide& pt, const DrawSide& pd, float* part, int& lp) {
  const ET* trow = static_cast<const ET*>(R.trow);
  const ED* drow = static_cast<const ED*>(R.drow);
  const int tj = static_cast<int>(threadIdx.x) * kDEPT;
  Raw8<ET> rt[NC];
  bool ok[NC];
#pragma unroll
  for (int q = 0; q < NC; ++q) {
    const int j0 = (c0 + q) * kDChunk + tj;
    ok[q] = j0 < P.V;  // V is a multiple of 8: a group is wholly in or out
    raw_load(rt[q], trow + (ok[q] ? j0 : 0));
  }
  float ld[NC][8];
  if (resid) {
    if (P.t2d) {
      int4 m[NC][2];
#pragma unroll
      for (int q = 0; q < NC; ++q) {
        const int4* src = reinterpret_cast<const int4*>(P.t2d + (ok[q] ? (c0 + q) * kDChunk + tj : 0));
        m[q][0] = __ldg(src);
        m[q][1] = __ldg(src + 1);
      }
#pragma unroll
      for (int q = 0; q < NC; ++q) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int4& v = m[q][e >> 2];
          const int jd = (e & 3) == 0 ? v.x : (e & 3) == 1 ? v.y : (e & 3) == 2 ? v.z : v.w;
          ld[q][e] = (jd >= 0 && sv_in(jd, P.Vd)) ? Elem<ED>::load(drow + jd) : -CUDART_INF_F;
        }
      }
    } else {
      Raw8<ED> rd[NC];
#pragma unroll
      for (int q = 0; q < NC; ++q) raw_load(rd[q], drow + (ok[q] ? (c0 + q) * kDChunk + tj : 0));
#pragma unroll
      for (int q = 0; q < NC; ++q) {
#pragma unroll
        for (int e = 0; e < 8; ++e) ld[q][e] = raw_at(rd[q], e);
      }
    }
  }
#pragma unroll
  for (int q = 0; q < NC; ++q) {
    const int j0 = (c0 + q) * kDChunk + tj;
    float s = 0.0f;
    if (ok[q]) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float w = draw_weight(raw_at(rt[q], e), resid ? ld[q][e] : -CUDART_INF_F, j0 + e, resid, P.c, pt, pd);
        s += w;
        if (w > 0.0f) lp = j0 + e;
      }
    }
    part[q] = s;
  }
}

// Block sum of one float per thread; the result is valid in thread 0.
__device__ __forceinline__ float block_sum_to0(float v, DecideShared& sh) {
  v = warp_sum(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) sh.wsum[0][warp] = v;
  __syncthreads();
  float s = 0.0f;
  if (threadIdx.x == 0)
    for (int w = 0; w < kDWarps; ++w) s += sh.wsum[0][w];
  return s;
}

template <typename ET, typename ED, int NC>
__global__ void __launch_bounds__(kDThreads, NC >= 8 ? 2 : 4) decide_kernel(DecideParams P, int nseg) {
  __shared__ DecideShared sh;
  const int b = blockIdx.x / nseg;
  const int seg = blockIdx.x - b * nseg;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = P.G, V = P.V;
  const int nchunks = (V + kDChunk - 1) / kDChunk;

  // The batch row's decisions: made by the statistics pass (one thread
  // fetches the record), or here by warp 0.
  if (P.rec) {
    if (tid < 3) reinterpret_cast<uint4*>(&sh.rec)[tid] = __ldcg(reinterpret_cast<const uint4*>(P.rec + b) + tid);
  } else if (warp == 0) {
    const DecideRecord r0 = decide_batch(P.dec, b);
    if (lane == 0) sh.rec = r0;
  }
  __syncthreads();
  const DecideRecord rc = sh.rec;
  const unsigned status = rc.status;
  int32_t* out = P.out_tokens + static_cast<int64_t>(b) * (G + 1);
  if (status & (SV_ROW_BAD_DRAFT_ID | SV_ROW_EMPTY)) {
    if (seg == 0) {
      for (int i = tid; i <= G; i += kDThreads) out[i] = -1;
      if (tid == 0) {
        if (P.num_accepted) P.num_accepted[b] = 0;
        if (P.row_status) P.row_status[b] = static_cast<int32_t>(status);
        if (P.out_prob) P.out_prob[b] = 0.0f;
      }
    }
    return;
  }
  const int k = rc.k;
  bool resid = k < G;
  const DrawSide pt = rc.pt;
  const DrawSide pd = rc.pd;
  RowView R;
  R.trow = static_cast<const ET*>(P.target) + (static_cast<int64_t>(b) * (G + 1) + k) * P.t_stride;
  R.drow = resid ? static_cast<const void*>(static_cast<const ED*>(P.draft) +
                                            (static_cast<int64_t>(b) * G + k) * P.d_stride)
                 : nullptr;
  R.fast = (V % 8) == 0 && (reinterpret_cast<uintptr_t>(R.trow) & 15u) == 0 &&
           (!resid || P.t2d || (reinterpret_cast<uintptr_t>(R.drow) & 15u) == 0);

  // This block's chunks: per-chunk weight sums and the last positive id.
  const int c0 = seg * NC;
  float part[NC];
  int lp = -1;
  if (R.fast) {
    segment_sums_fast<ET, ED, NC>(P, R, c0, resid, pt, pd, part, lp);
  } else {
#pragma unroll 1
    for (int q = 0; q < NC; ++q) {
      part[q] = 0.0f;
      if (c0 + q >= nchunks) continue;
      float w[8];
      chunk_weights<ET, ED>(P, R, c0 + q, resid, pt, pd, w);
      const int j0 = (c0 + q) * kDChunk + tid * kDEPT;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        part[q] += w[e];
        if (w[e] > 0.0f) lp = j0 + e;
      }
    }
  }
#pragma unroll
  for (int q = 0; q < NC; ++q) {
    const float v = warp_sum(part[q]);
    if (lane == 0) sh.wsum[q][warp] = v;
  }
  lp = warp_max_i(lp);
  if (lane == 0) sh.red_i[warp] = lp;
  __syncthreads();
  float* csum = P.chunk_sums + static_cast<int64_t>(b) * nchunks;
  int32_t* slast = P.seg_last + static_cast<int64_t>(b) * nseg;
  if (tid < NC && c0 + tid < nchunks) {
    float v = 0.0f;
#pragma unroll
    for (int w = 0; w < kDWarps; ++w) v += sh.wsum[tid][w];
    csum[c0 + tid] = v;
  }
  if (tid == 32) {
    int l2 = -1;
    for (int w = 0; w < kDWarps; ++w) l2 = max(l2, sh.red_i[w]);
    slast[seg] = l2;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) sh.last = atomicAdd(P.counters + b, 1u) == static_cast<unsigned>(nseg - 1);
  __syncthreads();
  if (!sh.last) return;
  __threadfence();

  // The row's last block: the total, and the chunk that holds u * total.
  const float u = P.u_resample ? P.u_resample[b] : 0.0f;
  bool fallback = false;
  for (int attempt = 0; attempt < 2; ++attempt) {
    if (warp == 0) {
      const int per = (nchunks + 31) / 32;
      const int q0 = min(nchunks, lane * per), q1 = min(nchunks, q0 + per);
      double s = 0.0;
      for (int q = q0; q < q1; ++q) s += static_cast<double>(__ldcg(csum + q));
      double incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const double total = __shfl_sync(0xffffffffu, incl, 31);
      const double target = static_cast<double>(u) * total;
      const unsigned hb = __ballot_sync(0xffffffffu, s > 0.0 && incl > target && incl - s <= target);
      int lq = -1;
      for (int sg = lane; sg < nseg; sg += 32) lq = max(lq, __ldcg(slast + sg));
      lq = warp_max_i(lq);
      int chunk = -1;
      double carry = 0.0;
      if (hb) {
        const int wl = __ffs(hb) - 1;
        if (lane == wl) {
          double cc = incl - s;
          for (int q = q0; q < q1; ++q) {
            const double s2 = static_cast<double>(__ldcg(csum + q));
            if (s2 > 0.0 && cc + s2 > target) {
              chunk = q;
              break;
            }
            cc += s2;
          }
          carry = cc;
        }
        chunk = __shfl_sync(0xffffffffu, chunk, wl);
        carry = __shfl_sync(0xffffffffu, carry, wl);
      }
      if (lane == 0) {
        sh.total = total;
        sh.target = target;
        sh.chunk = chunk;
        sh.carry = carry;
        sh.tok = lq;
      }
    }
    __syncthreads();
    if (sh.total > 0.0 || !resid) break;
    // Residual mass 0 (possible only through rounding): draw from p_k.  This
    // block recomputes the chunk sums of p_k by itself.
    resid = false;
    fallback = true;
    int lpf = -1;
#pragma unroll 1
    for (int ch = 0; ch < nchunks; ++ch) {
      float w[8];
      chunk_weights<ET, ED>(P, R, ch, false, pt, pd, w);
      float s = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        s += w[e];
        if (w[e] > 0.0f) lpf = ch * kDChunk + tid * kDEPT + e;
      }
      s = block_sum_to0(s, sh);
      if (tid == 0) csum[ch] = s;
    }
    lpf = block_max_i<kDThreads>(lpf, sh.red_i);
    for (int sg = tid; sg < nseg; sg += kDThreads) slast[sg] = sg == 0 ? lpf : -1;
    __syncthreads();
  }
  if (sh.total > 0.0 && sh.chunk >= 0 && sv_in(sh.chunk, nchunks)) {
    // Rescan the chunk that holds the draw: the thread whose ids span
    // u * total (in block order) finds the id.
    const int j0 = sh.chunk * kDChunk + tid * kDEPT;
    float w[8];
    chunk_weights<ET, ED>(P, R, sh.chunk, resid, pt, pd, w);
    float mine = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) mine += w[e];
    double tot;
    const double excl = block_exclusive_scan_d<kDThreads>(static_cast<double>(mine), sh.scan, &tot);
    if (tid == 0) sh.best = INT32_MAX;
    __syncthreads();
    const double rem = sh.target - (sh.carry + excl);
    if (rem < static_cast<double>(mine)) {
      const float remf = static_cast<float>(rem);
      float run = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        run += w[e];
        if (w[e] > 0.0f && run > remf) {
          atomicMin(&sh.best, j0 + e);
          break;
        }
      }
    }
    __syncthreads();
    if (tid == 0 && sh.best != INT32_MAX) sh.tok = sh.best;
    __syncthreads();
  }
  const int tok = sv_in(sh.tok, V) ? sh.tok : -1;
  for (int i = tid; i <= G; i += kDThreads)
    out[i] = i < k ? P.ids[static_cast<int64_t>(b) * G + i] : (i == k ? tok : -1);
  if (tid == 0) {
    if (P.num_accepted) P.num_accepted[b] = k;
    if (P.row_status) P.row_status[b] = static_cast<int32_t>(status | (fallback ? SV_ROW_RESAMPLE_FALLBACK : 0u));
    if (P.out_prob) {
      float pr = 0.0f;
      if (!resid && tok >= 0) pr = prob_of(Elem<ET>::load(static_cast<const ET*>(R.trow) + tok), tok, P.c, pt);
      P.out_prob[b] = pr;
    }
  }
}

size_t decide_scratch_bytes(int B, int V) {
  const size_t chunks = static_cast<size_t>(B) * static_cast<size_t>((V + kDChunk - 1) / kDChunk);
  return align_up(chunks * sizeof(float), 256) + align_up(chunks * sizeof(int32_t), 256) +
         align_up(static_cast<size_t>(B) * sizeof(unsigned), 256);
}

template <typename ET, typename ED, int NC>
static sv_status launch_decide_typed(DecideParams P, void* scratch, cudaStream_t stream) {
  const int nchunks = (P.V + kDChunk - 1) / kDChunk;
  const int nseg = (nchunks + NC - 1) / NC;
  const size_t chunks = static_cast<size_t>(P.B) * nchunks;
  char* s = static_cast<char*>(scratch);
  P.chunk_sums = reinterpret_cast<float*>(s);
  P.seg_last = reinterpret_cast<int32_t*>(s + align_up(chunks * sizeof(float), 256));
  P.counters = reinterpret_cast<unsigned*>(s + align_up(chunks * sizeof(float), 256) +
                                           align_up(chunks * sizeof(int32_t), 256));
  const size_t blocks = static_cast<size_t>(P.B) * nseg;
  if (blocks > INT32_MAX) return SV_ERR_UNSUPPORTED;
  if (cudaMemsetAsync(P.counters, 0, static_cast<size_t>(P.B) * sizeof(unsigned), stream) != cudaSuccess)
    return SV_ERR_CUDA;
  decide_kernel<ET, ED, NC><<<static_cast<unsigned>(blocks), kDThreads, 0, stream>>>(P, nseg);
  if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  note_launch(stream);
  return SV_OK;
}

// Chunks per block: the most (8 for two bf16 rows, else 4) that still gives
// the launch about four blocks per SM; fewer chunks per block otherwise, so
// small batches still spread over the GPU.
static int chunks_per_block(int B, int V, int nc_max) {
  // SM count per device, cached; concurrent callers store the same value.
  static std::atomic<int> sms[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  int n = sms[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    sms[dev].store(n, std::memory_order_relaxed);
  }
  const long long want = 4LL * n;
  const int nchunks = (V + kDChunk - 1) / kDChunk;
  int nc = nc_max;
  while (nc > 2 && static_cast<long long>(B) * ((nchunks + nc - 1) / nc) < want) nc /= 2;
  return nc;
}

sv_status launch_decide(const DecideParams& P, sv_dtype td, sv_dtype dd, void* scratch, cudaStream_t stream) {
  if (P.B == 0) return SV_OK;
  const bool tb = td == SV_BF16, db = dd == SV_BF16;
  const int nc = chunks_per_block(P.B, P.V, 4);
  if (tb && db) {
    if (nc == 8) return launch_decide_typed<uint16_t, uint16_t, 8>(P, scratch, stream);
    if (nc == 4) return launch_decide_typed<uint16_t, uint16_t, 4>(P, scratch, stream);
    return launch_decide_typed<uint16_t, uint16_t, 2>(P, scratch, stream);
  }
  if (tb) {
    if (nc == 4) return launch_decide_typed<uint16_t, float, 4>(P, scratch, stream);
    return launch_decide_typed<uint16_t, float, 2>(P, scratch, stream);
  }
  if (db) {
    if (nc == 4) return launch_decide_typed<float, uint16_t, 4>(P, scratch, stream);
    return launch_decide_typed<float, uint16_t, 2>(P, scratch, stream);
  }
  if (nc == 4) return launch_decide_typed<float, float, 4>(P, scratch, stream);
  return launch_decide_typed<float, float, 2>(P, scratch, stream);
}

}  // namespace sv
