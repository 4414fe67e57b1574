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
//
// EAGLE3 draft rows (a d2t map; "SSD: extending the engine with new models
// and an EAGLE3 draft" §六): when d2t is strictly increasing, the draft ids
// whose target ids fall in a block's segment form one contiguous range
// (tabulated per call by d2t_range_kernel), so the block reads that range of
// the draft row and of d2t with plain coalesced loads and applies
// max(0, p - q) in shared memory, instead of a t2d lookup and a dependent
// gather per target id.  Per-id weights and the order of every sum are those
// of the t2d path, which stays in use for any other d2t.
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
  int a0, a1;     // this segment's draft-id range (draft-range table)
  unsigned bad;   // entries of d2t that break the table
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
// load of the segment in flight together (R.fast, draft rows without t2d
// only); groups of 8 ids past the row add nothing.  lp: the largest id with
// a positive weight.
template <typename ET, typename ED, int NC, bool MAY_RESID = true>
__device__ __forceinline__ void segment_sums_fast(const DecideParams& P, const RowView& R, int c0, bool resid,
                                                  const DrawSide& pt, const DrawSide& pd, float* part, int& lp) {
  const ET* trow = static_cast<const ET*>(R.trow);
  const ED* drow = static_cast<const ED*>(R.drow);
  const int tj = static_cast<int>(threadIdx.x) * kDEPT;
  // Chunks in flight together: all of them, or two at a time for fp32 target
  // rows, whose raw vectors with the draft's would not fit the registers.
  constexpr int kGrp = (sizeof(ET) == 4 && NC > 2) ? 2 : NC;
#pragma unroll
  for (int g0 = 0; g0 < NC; g0 += kGrp) {
    Raw8<ET> rt[kGrp];
    bool ok[kGrp];
#pragma unroll
    for (int q = 0; q < kGrp; ++q) {
      const int j0 = (c0 + g0 + q) * kDChunk + tj;
      ok[q] = j0 < P.V;  // V is a multiple of 8: a group is wholly in or out
      raw_load(rt[q], trow + (ok[q] ? j0 : 0));
    }
    float ld[kGrp][8];
    if (MAY_RESID && resid) {
      Raw8<ED> rd[kGrp];
#pragma unroll
      for (int q = 0; q < kGrp; ++q) raw_load(rd[q], drow + (ok[q] ? (c0 + g0 + q) * kDChunk + tj : 0));
#pragma unroll
      for (int q = 0; q < kGrp; ++q) {
#pragma unroll
        for (int e = 0; e < 8; ++e) ld[q][e] = raw_at(rd[q], e);
      }
    }
#pragma unroll
    for (int q = 0; q < kGrp; ++q) {
      const int j0 = (c0 + g0 + q) * kDChunk + tj;
      float s = 0.0f;
      if (ok[q]) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float w =
              draw_weight(raw_at(rt[q], e), resid ? ld[q][e] : -CUDART_INF_F, j0 + e, resid, P.c, pt, pd);
          s += w;
          if (w > 0.0f) lp = j0 + e;
        }
      }
      part[g0 + q] = s;
    }
  }
}

// Residual draw weights of this block's segment through the draft-range
// table: p(j) of the target segment into wbuf (shared memory), then for every
// draft id jd whose target id x = d2t[jd] lies in the segment (the ids
// [d2t_first[seg], d2t_first[seg + 1])) wbuf[x] = max(0, p(x) - q(jd)); ids
// without a draft entry keep p(x) = max(0, p(x) - 0).  Per-thread sums then
// run over the thread's own ids in id order, as in segment_sums_fast.
// 16-byte asynchronous copy global -> shared (L2 only), and the wait for all
// of this thread's copies.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

template <typename ET, typename ED, int NC>
__device__ __forceinline__ void segment_sums_compact(const DecideParams& P, const RowView& R, int a0, int a1,
                                                     int c0, const DrawSide& pt, const DrawSide& pd, float* wbuf,
                                                     float* part, int& lp) {
  const ET* trow = static_cast<const ET*>(R.trow);
  const ED* drow = static_cast<const ED*>(R.drow);
  const int tid = static_cast<int>(threadIdx.x);
  const int tj = tid * kDEPT;
  const int s0 = c0 * kDChunk;
  bool ok[NC];
#pragma unroll
  for (int q = 0; q < NC; ++q) ok[q] = (c0 + q) * kDChunk + tj < P.V;  // V is a multiple of 8
  // fp32 targets land in wbuf by asynchronous copies (no registers held while
  // in flight) and are turned into p(j) in place; bf16 targets come through
  // registers.
  Raw8<ET> rt[sizeof(ET) == 2 ? NC : 1];
  if constexpr (sizeof(ET) == 4) {
#pragma unroll
    for (int q = 0; q < NC; ++q) {
      float* dst = wbuf + q * kDChunk + tj;
      if (ok[q]) {
        const ET* src = trow + (c0 + q) * kDChunk + tj;
        cp_async16(dst, src);
        cp_async16(dst + 4, src + 4);
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  } else {
#pragma unroll
    for (int q = 0; q < NC; ++q) raw_load(rt[q], trow + (ok[q] ? (c0 + q) * kDChunk + tj : 0));
  }
  // The first draft ids of the range, loaded while the target is in flight.
  constexpr int kPre = 8;
  int xd[kPre];
  float ldv[kPre];
#pragma unroll
  for (int u = 0; u < kPre; ++u) {
    const int jd = a0 + u * kDThreads + tid;
    xd[u] = -1;
    ldv[u] = -CUDART_INF_F;
    if (jd < a1) {
      xd[u] = __ldg(P.d2t + jd);
      ldv[u] = Elem<ED>::load(drow + jd);
    }
  }
  if constexpr (sizeof(ET) == 4) cp_async_wait_all();
#pragma unroll
  for (int q = 0; q < NC; ++q) {
    const int j0 = (c0 + q) * kDChunk + tj;
    float4* slot = reinterpret_cast<float4*>(wbuf + q * kDChunk + tj);
    float x[8];
    if constexpr (sizeof(ET) == 4) {
      const float4 lo = ok[q] ? slot[0] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      const float4 hi = ok[q] ? slot[1] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      x[0] = lo.x; x[1] = lo.y; x[2] = lo.z; x[3] = lo.w;
      x[4] = hi.x; x[5] = hi.y; x[6] = hi.z; x[7] = hi.w;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = raw_at(rt[q], e);
    }
    float w[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) w[e] = ok[q] ? fmaxf(0.0f, prob_of(x[e], j0 + e, P.c, pt)) : 0.0f;
    slot[0] = make_float4(w[0], w[1], w[2], w[3]);
    slot[1] = make_float4(w[4], w[5], w[6], w[7]);
  }
  __syncthreads();
  constexpr int kSeg = NC * kDChunk;
  auto apply = [&](int x, float ld) {
    const int t = x - s0;
    if (ld > -CUDART_INF_F && sv_in(t, kSeg)) {
      const float qv = prob_of(ld, x, P.c, pd);
      wbuf[t] = fmaxf(0.0f, wbuf[t] - qv);
    }
  };
#pragma unroll
  for (int u = 0; u < kPre; ++u)
    if (xd[u] >= 0) apply(xd[u], ldv[u]);
#pragma unroll 4
  for (int jd = a0 + kPre * kDThreads + tid; jd < a1; jd += kDThreads) apply(__ldg(P.d2t + jd), Elem<ED>::load(drow + jd));
  __syncthreads();
#pragma unroll
  for (int q = 0; q < NC; ++q) {
    const int j0 = (c0 + q) * kDChunk + tj;
    float s = 0.0f;
    if (ok[q]) {
      const float4* src = reinterpret_cast<const float4*>(wbuf + q * kDChunk + tj);
      const float4 lo = src[0], hi = src[1];
      const float w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        s += w[e];
        if (w[e] > 0.0f) lp = j0 + e;
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

// COMPACT: the draft-range table is in use (d2t with t2d); the block then
// holds NC * kDChunk floats of dynamic shared memory.
template <typename ET, typename ED, int NC, bool COMPACT>
__global__ void __launch_bounds__(kDThreads, COMPACT ? (NC >= 8 ? 3 : 5) : (NC >= 8 ? 2 : 4)) decide_kernel(DecideParams P, int nseg) {
  __shared__ DecideShared sh;
  extern __shared__ __align__(16) float wbuf[];
  const int b = blockIdx.x / nseg;
  const int seg = blockIdx.x - b * nseg;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = P.G, V = P.V;
  const int nchunks = (V + kDChunk - 1) / kDChunk;

  // This segment's draft range and the table's validity, fetched together
  // with the record.
  if constexpr (COMPACT) {
    if (tid == 32) sh.a0 = __ldg(P.d2t_first + seg);
    if (tid == 33) sh.a1 = __ldg(P.d2t_first + seg + 1);
    if (tid == 34) sh.bad = __ldcg(P.counters + P.B);
  }

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
  // The draft-range table is usable when d2t is strictly increasing within
  // [0, V) (no entry counted by d2t_range_kernel).
  bool compact = false;
  if constexpr (COMPACT) compact = resid && R.fast && sh.bad == 0u;
  if (compact) {
    segment_sums_compact<ET, ED, NC>(P, R, sh.a0, sh.a1, c0, pt, pd, wbuf, part, lp);
  } else if (COMPACT && R.fast && !resid) {
    segment_sums_fast<ET, ED, NC, false>(P, R, c0, false, pt, pd, part, lp);
  } else if (!COMPACT && R.fast && !(resid && P.t2d)) {
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
  // One fence on each side, by the thread that counts the block (the
  // barriers order the other threads' writes and reads around it).
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const bool last = atomicAdd(P.counters + b, 1u) == static_cast<unsigned>(nseg - 1);
    if (last) __threadfence();
    sh.last = last;
  }
  __syncthreads();
  if (!sh.last) return;

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
  const size_t nchunks = static_cast<size_t>((V + kDChunk - 1) / kDChunk);
  const size_t chunks = static_cast<size_t>(B) * nchunks;
  return align_up(chunks * sizeof(float), 256) + align_up(chunks * sizeof(int32_t), 256) +
         align_up((static_cast<size_t>(B) + 1) * sizeof(unsigned), 256) + align_up((nchunks + 2) * sizeof(int32_t), 256);
}

// The draft-range table of the draw: first[s] = the first draft id whose
// target id is at least s * seg_ids, for s = 0..nseg (Vd when none).  It is
// meaningful when d2t is strictly increasing with every entry in [0, V); each
// entry that breaks this adds one to *bad (zero before the launch), and the
// draw then uses t2d instead.  One thread per draft id (at least nseg + 1).
__global__ void d2t_range_kernel(const int32_t* __restrict__ d2t, int Vd, int V, int seg_ids, int nseg,
                                 int32_t* __restrict__ first, unsigned* bad) {
  const int jd = static_cast<int>(blockIdx.x * blockDim.x + threadIdx.x);
  if (Vd == 0) {
    if (jd <= nseg) first[jd] = 0;
    return;
  }
  if (jd >= Vd) return;
  const int x = d2t[jd];
  const int xp = jd > 0 ? d2t[jd - 1] : -1;
  if (x < 0 || x >= V || x <= xp) {
    atomicAdd(bad, 1u);
    return;
  }
  const int cur = x / seg_ids;
  const int prev = xp >= 0 ? xp / seg_ids : -1;
  for (int s = prev + 1; s <= cur && s <= nseg; ++s) first[s] = jd;
  if (jd == Vd - 1)
    for (int s = cur + 1; s <= nseg; ++s) first[s] = Vd;
}

template <typename ET, typename ED, int NC>
static sv_status launch_decide_typed(DecideParams P, void* scratch, cudaStream_t stream) {
  static FuncAttrCache cache;
  const int nchunks = (P.V + kDChunk - 1) / kDChunk;
  const int nseg = (nchunks + NC - 1) / NC;
  const size_t chunks = static_cast<size_t>(P.B) * nchunks;
  char* s = static_cast<char*>(scratch);
  const size_t o_last = align_up(chunks * sizeof(float), 256);
  const size_t o_cnt = o_last + align_up(chunks * sizeof(int32_t), 256);
  const size_t o_first = o_cnt + align_up((static_cast<size_t>(P.B) + 1) * sizeof(unsigned), 256);
  P.chunk_sums = reinterpret_cast<float*>(s);
  P.seg_last = reinterpret_cast<int32_t*>(s + o_last);
  P.counters = reinterpret_cast<unsigned*>(s + o_cnt);
  P.d2t_first = reinterpret_cast<int32_t*>(s + o_first);
  const size_t blocks = static_cast<size_t>(P.B) * nseg;
  if (blocks > INT32_MAX) return SV_ERR_UNSUPPORTED;
  const bool table = P.t2d != nullptr && P.d2t != nullptr && P.G > 0;
  if (!table) P.d2t = nullptr;
  const size_t smem = table ? static_cast<size_t>(NC) * kDChunk * sizeof(float) : 0;
  auto kern = table ? decide_kernel<ET, ED, NC, true> : decide_kernel<ET, ED, NC, false>;
  if (table && !cache.ensure(reinterpret_cast<const void*>(kern), smem, false)) return SV_ERR_CUDA;
  if (cudaMemsetAsync(P.counters, 0, (static_cast<size_t>(P.B) + 1) * sizeof(unsigned), stream) != cudaSuccess)
    return SV_ERR_CUDA;
  if (table) {
    const int n = std::max(P.Vd, nseg + 1);
    d2t_range_kernel<<<(n + 255) / 256, 256, 0, stream>>>(P.d2t, P.Vd, P.V, NC * kDChunk, nseg, P.d2t_first,
                                                          P.counters + P.B);
    if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
    note_launch(stream);
  }
  kern<<<static_cast<unsigned>(blocks), kDThreads, smem, stream>>>(P, nseg);
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
