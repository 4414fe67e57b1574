// Decision and draw of the sampling verify: accept/reject per draft, first
// rejection, and the resample / bonus draw by inverse CDF.
//
// Source: "LLM inference acceleration in practice: draft models and
// speculative sampling explained" (mlqm.cn) §3.1 (accept with min(1, p/q);
// on the first rejection sample from norm(max(0, p - q)); after γ
// acceptances sample the extra token from p) and §4.2 (the accept loop of
// generate()).  The uniforms are supplied by the caller.
//
// One thread-block cluster per batch row.  Every block evaluates the
// decisions (a few scalars per row, from the statistics pass), then draws
// over its own contiguous segment of the vocabulary: per 4096-id chunk it
// sums the draw weights (8 contiguous ids per thread, 16-byte loads).  The
// segment totals are exchanged through distributed shared memory; the block
// whose segment holds u * total rescans the one chunk that holds it with a
// block-wide prefix scan and writes the row's outputs.
#include "sv_rows.cuh"

namespace sv {

constexpr int kDThreads = 512;
constexpr int kDEPT = 8;
constexpr int kDChunk = kDThreads * kDEPT;

struct DecideShared {
  float red[32];
  double scan[32];
  double seg_total;
  int seg_last;
  unsigned char acc[SV_MAX_GAMMA];
  int k;
  unsigned status;
  int writer;
  int tok;
  int chunk;
  double carry;
  double target;
};

// Eight consecutive logits starting at j0 (a multiple of 8); -inf past V.
template <typename E>
__device__ __forceinline__ void load8(const E* row, int j0, int V, bool aligned, float* out) {
  if (aligned && j0 + 8 <= V) {
    if constexpr (sizeof(E) == 2) {
      const uint4 w = ldg_stream(row + j0);
#pragma unroll
      for (int e = 0; e < 8; ++e) out[e] = Elem<uint16_t>::at(w, e);
    } else {
      const uint4 a = ldg_stream(row + j0), b = ldg_stream(row + j0 + 4);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        out[e] = Elem<float>::at(a, e);
        out[e + 4] = Elem<float>::at(b, e);
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) out[e] = j0 + e < V ? Elem<E>::load(row + j0 + e) : -CUDART_INF_F;
  }
}

struct DrawSide {
  float mc, invK;
  uint32_t tau;
  int32_t cut;
};

// Draw weights of ids j0..j0+7: p(j) (bonus) or max(0, p(j) - q(j)).
template <typename ET, typename ED>
__device__ __forceinline__ void weights8(const ET* trow, const ED* drow, const int32_t* t2d, int V, int Vd,
                                         bool t_al, bool d_al, bool resid, float c, const DrawSide& pt,
                                         const DrawSide& pd, int j0, float* w) {
  float lt[8];
  load8<ET>(trow, j0, V, t_al, lt);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int j = j0 + e;
    w[e] = (j < V && kept(order_key(lt[e]), j, pt.tau, pt.cut)) ? weight(lt[e], c, pt.mc) * pt.invK : 0.0f;
  }
  if (!resid) return;
  float ld[8];
  if (t2d) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int j = j0 + e;
      const int jd = j < V ? __ldg(t2d + j) : -1;
      ld[e] = (jd >= 0 && jd < Vd) ? Elem<ED>::load(drow + jd) : -CUDART_INF_F;
    }
  } else {
    load8<ED>(drow, j0, V, d_al, ld);
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int j = j0 + e;
    const float q = (ld[e] > -CUDART_INF_F && kept(order_key(ld[e]), j, pd.tau, pd.cut))
                        ? weight(ld[e], c, pd.mc) * pd.invK
                        : 0.0f;
    w[e] = fmaxf(0.0f, w[e] - q);
  }
}

template <typename ET, typename ED>
__global__ void __launch_bounds__(kDThreads) decide_kernel(DecideParams P, int cld) {
  extern __shared__ float chunk_sums[];
  __shared__ DecideShared sh;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int b = blockIdx.x / cld;
  const int tid = threadIdx.x;
  const int G = P.G;
  const RowStats* ts = P.t_stats + static_cast<int64_t>(b) * (G + 1);
  const RowStats* ds = P.d_stats + static_cast<int64_t>(b) * G;
  if (tid == 0) sh.status = 0;
  __syncthreads();
  // Decisions (identical in every block of the cluster).
  for (int i = tid; i <= G; i += kDThreads) {
    uint32_t st = ts[i].status;
    if (i < G) {
      st |= ds[i].status;
      const int x = P.ids[static_cast<int64_t>(b) * G + i];
      if (x < 0 || x >= P.V) st |= SV_ROW_BAD_DRAFT_ID;
      const double p = ts[i].K > 0.0 ? static_cast<double>(ts[i].e_query) / ts[i].K : 0.0;
      const double q = ds[i].K > 0.0 ? static_cast<double>(ds[i].e_query) / ds[i].K : 0.0;
      const double u = static_cast<double>(P.u_accept[static_cast<int64_t>(b) * G + i]);
      sh.acc[i] = (u * q < p) ? 1 : 0;
      if (rank == 0 && P.p_draft) P.p_draft[static_cast<int64_t>(b) * G + i] = static_cast<float>(p);
      if (rank == 0 && P.q_draft) P.q_draft[static_cast<int64_t>(b) * G + i] = static_cast<float>(q);
    }
    if (st) atomicOr(&sh.status, st);
  }
  __syncthreads();
  int32_t* out = P.out_tokens + static_cast<int64_t>(b) * (G + 1);
  if (sh.status & (SV_ROW_BAD_DRAFT_ID | SV_ROW_EMPTY)) {
    // Uniform over the cluster, before any distributed shared memory access.
    if (rank == 0) {
      for (int i = tid; i <= G; i += kDThreads) out[i] = -1;
      if (tid == 0) {
        if (P.num_accepted) P.num_accepted[b] = 0;
        if (P.row_status) P.row_status[b] = static_cast<int32_t>(sh.status);
        if (P.out_prob) P.out_prob[b] = 0.0f;
      }
    }
    return;
  }
  if (tid == 0) {
    int k = G;
    for (int i = 0; i < G; ++i)
      if (!sh.acc[i]) {
        k = i;
        break;
      }
    sh.k = k;
  }
  __syncthreads();
  const int k = sh.k;
  const float u = P.u_resample ? P.u_resample[b] : 0.0f;
  const RowStats& st = ts[k];
  const ET* trow = reinterpret_cast<const ET*>(P.target) + (static_cast<int64_t>(b) * (G + 1) + k) * P.t_stride;
  const ED* drow = k < G ? reinterpret_cast<const ED*>(P.draft) + (static_cast<int64_t>(b) * G + k) * P.d_stride
                         : nullptr;
  const DrawSide pt{st.mc, static_cast<float>(1.0 / st.K), st.tau, st.cut};
  DrawSide pd{0.0f, 0.0f, 0u, 0};
  if (k < G) pd = DrawSide{ds[k].mc, static_cast<float>(1.0 / ds[k].K), ds[k].tau, ds[k].cut};
  const bool t_al = (reinterpret_cast<uintptr_t>(trow) & 15u) == 0;
  const bool d_al = drow && (reinterpret_cast<uintptr_t>(drow) & 15u) == 0;
  const int V = P.V;
  const int nchunks = (V + kDChunk - 1) / kDChunk;
  const int cpc = (nchunks + cld - 1) / cld;
  const int c0 = min(nchunks, rank * cpc), c1 = min(nchunks, c0 + cpc);
  const int warp = tid >> 5, lane = tid & 31;

  bool resid = k < G;
  bool fallback = false;
  double R = 0.0;
  int last = -1;
  for (int attempt = 0; attempt < 2; ++attempt) {
    // Pass 1: chunk sums of this block's segment.
    double seg = 0.0;
    int lp = -1;
    for (int ci = c0; ci < c1; ++ci) {
      const int j0 = ci * kDChunk + tid * kDEPT;
      float w[kDEPT];
      weights8<ET, ED>(trow, drow, P.t2d, V, P.Vd, t_al, d_al, resid, P.c, pt, pd, j0, w);
      float part = 0.0f;
#pragma unroll
      for (int e = 0; e < kDEPT; ++e) {
        part += w[e];
        if (w[e] > 0.0f) lp = j0 + e;
      }
      part = warp_sum(part);
      if (lane == 0) sh.red[warp] = part;
      __syncthreads();
      if (warp == 0) {
        float s = lane < kDThreads / 32 ? sh.red[lane] : 0.0f;
        s = warp_sum(s);
        if (lane == 0) {
          chunk_sums[ci - c0] = s;
          seg += static_cast<double>(s);
        }
      }
      __syncthreads();
    }
    {
      __shared__ int s_red_i[32];
      lp = block_max_i<kDThreads>(lp, s_red_i);
    }
    if (tid == 0) {
      sh.seg_total = seg;
      sh.seg_last = lp;
    }
    __syncthreads();
    cluster.sync();
    R = 0.0;
    last = -1;
    for (int q = 0; q < cld; ++q) {
      const DecideShared* p = cluster.map_shared_rank(&sh, q);
      R += p->seg_total;
      last = max(last, p->seg_last);
    }
    if (R > 0.0 || !resid) break;
    // Residual mass 0 (possible only through rounding): draw from p_k.
    resid = false;
    fallback = true;
    cluster.sync();  // peers have read this block's totals
  }
  if (tid == 0) {
    sh.writer = 0;
    sh.tok = last;
    sh.chunk = -1;
    if (R > 0.0) {
      const double target = static_cast<double>(u) * R;
      double cum = 0.0;
      for (int q = 0; q < cld; ++q) {
        const double tq = cluster.map_shared_rank(&sh, q)->seg_total;
        if (cum + tq > target && tq > 0.0) {
          sh.writer = q;
          if (q == rank) {
            // Find the chunk inside this block's segment.
            double cc = cum;
            for (int ci = c0; ci < c1; ++ci) {
              const double s = chunk_sums[ci - c0];
              if (cc + s > target && s > 0.0f) {
                sh.chunk = ci;
                sh.carry = cc;
                break;
              }
              cc += s;
            }
          }
          break;
        }
        cum += tq;
      }
      sh.target = target;
    }
  }
  __syncthreads();
  if (sh.chunk >= 0) {
    // Rescan the chunk that holds the draw.
    const int j0 = sh.chunk * kDChunk + tid * kDEPT;
    float w[kDEPT];
    weights8<ET, ED>(trow, drow, P.t2d, V, P.Vd, t_al, d_al, resid, P.c, pt, pd, j0, w);
    float part = 0.0f;
    int lp = -1;
#pragma unroll
    for (int e = 0; e < kDEPT; ++e) {
      part += w[e];
      if (w[e] > 0.0f) lp = j0 + e;
    }
    double tot;
    const double excl = block_exclusive_scan_d<kDThreads>(static_cast<double>(part), sh.scan, &tot);
    __shared__ int s_best;
    if (tid == 0) s_best = INT32_MAX;
    __syncthreads();
    double run = sh.carry + excl;
#pragma unroll
    for (int e = 0; e < kDEPT; ++e) {
      run += w[e];
      if (w[e] > 0.0f && run > sh.target) {
        atomicMin(&s_best, j0 + e);
        break;
      }
    }
    __shared__ int s_red_i2[32];
    lp = block_max_i<kDThreads>(lp, s_red_i2);
    __syncthreads();
    if (tid == 0) sh.tok = s_best != INT32_MAX ? s_best : lp;
    __syncthreads();
  }
  if (rank == sh.writer) {
    const int tok = sh.tok;
    for (int i = tid; i <= G; i += kDThreads)
      out[i] = i < k ? P.ids[static_cast<int64_t>(b) * G + i] : (i == k ? tok : -1);
    if (tid == 0) {
      if (P.num_accepted) P.num_accepted[b] = k;
      if (P.row_status)
        P.row_status[b] = static_cast<int32_t>(sh.status | (fallback ? SV_ROW_RESAMPLE_FALLBACK : 0u));
      if (P.out_prob) {
        float pr = 0.0f;
        if (!resid && tok >= 0) {
          const float x = Elem<ET>::load(trow + tok);
          if (kept(order_key(x), tok, pt.tau, pt.cut)) pr = weight(x, P.c, pt.mc) * pt.invK;
        }
        P.out_prob[b] = pr;
      }
    }
  }
  // No block may leave while a peer can still read its shared memory.
  cluster.sync();
}

template <typename ET, typename ED>
static sv_status launch_decide_typed(const DecideParams& P, cudaStream_t stream) {
  const int nchunks = (P.V + kDChunk - 1) / kDChunk;
  const int cld = nchunks >= 8 ? 8 : (nchunks >= 4 ? 4 : (nchunks >= 2 ? 2 : 1));
  const int cpc = (nchunks + cld - 1) / cld;
  const size_t smem = align_up(static_cast<size_t>(cpc) * sizeof(float), 16);
  auto kern = decide_kernel<ET, ED>;
  static FuncAttrCache cache;
  if (smem > 48 * 1024 && !cache.ensure(reinterpret_cast<const void*>(kern), smem, false)) return SV_ERR_CUDA;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(P.B) * cld);
  cfg.blockDim = dim3(kDThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cld);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, P, cld) != cudaSuccess) return SV_ERR_CUDA;
  note_launch(stream);
  return SV_OK;
}

sv_status launch_decide(const DecideParams& P, sv_dtype td, sv_dtype dd, cudaStream_t stream) {
  if (P.B == 0) return SV_OK;
  const bool tb = td == SV_BF16, db = dd == SV_BF16;
  if (tb && db) return launch_decide_typed<uint16_t, uint16_t>(P, stream);
  if (tb) return launch_decide_typed<uint16_t, float>(P, stream);
  if (db) return launch_decide_typed<float, uint16_t>(P, stream);
  return launch_decide_typed<float, float>(P, stream);
}

}  // namespace sv
