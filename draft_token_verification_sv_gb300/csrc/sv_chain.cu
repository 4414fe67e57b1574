// Sampling verify of draft chains (temperature > 0) and draft-side sampling.
//
// Source: "LLM inference acceleration in practice: draft models and
// speculative sampling explained" (mlqm.cn), §3.1 (accept with min(1, p/q),
// resample from norm(max(0, p - q)) at the first rejection, bonus token from
// p after γ acceptances), §4.2 (generate(): temperature, _apply_top_p,
// softmax for every target and draft position; the accept loop), §6.2
// (batched verify, shared temperature and top_p).  The EAGLE3 small draft
// vocabulary follows "SSD: extending the engine with new models and an
// EAGLE3 draft" §六 (d2t/t2d).
//
// Two passes over device memory:
//   1. statistics: one pass over every logit row computes the row maximum,
//      the softmax normaliser and, when top_p < 1, the exact top-p threshold
//      (sv_topp.cu); it also evaluates the row's weight at its draft id.  In
//      the top-p pass, the block that writes the last statistic of a batch
//      row makes that row's accept/reject decisions (one warp) and records
//      the draw rows; without top-p the draw makes them.
//   2. draw (sv_decide.cu): blocks over segments of the vocabulary sum the
//      draw weights of the recorded rows per chunk; the last block of a batch
//      row draws by an inverse CDF within the one chunk that holds u * total.
#include "sv_rows.cuh"

#include <algorithm>
#include <cmath>

namespace sv {

// --------------------------------------------------- streaming statistics ----
// top_p == 1: one pass in registers; online max and a rescaled sum of
// exp2(l*c - m*c) in several independent fp32 accumulators per thread.

template <typename E, int THREADS, int UNROLL>
__global__ void __launch_bounds__(THREADS) stats_stream_kernel(StatsLaunch L) {
  constexpr int EPV = Elem<E>::kPerVec;
  __shared__ float s_red[32];
  int r = blockIdx.x;
  const RowSet& S = pick_set(L, r);
  const E* row = reinterpret_cast<const E*>(S.base) + static_cast<int64_t>(r) * S.stride;
  const float c = L.c;
  const RowSplit rs = split_row(row, S.len);
  const int nvec = rs.nvec;
  const uint4* vp = reinterpret_cast<const uint4*>(row + rs.head);

  float m = -CUDART_INF_F;
  float acc[EPV];
#pragma unroll
  for (int k = 0; k < EPV; ++k) acc[k] = 0.0f;

  for (int v0 = threadIdx.x; v0 < nvec; v0 += THREADS * UNROLL) {
    uint4 buf[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int v = v0 + u * THREADS;
      buf[u] = v < nvec ? ldg_stream(vp + v) : Elem<E>::neg_inf_vec();
    }
    float lm = -CUDART_INF_F;
#pragma unroll
    for (int u = 0; u < UNROLL; ++u)
#pragma unroll
      for (int k = 0; k < EPV; ++k) lm = fmaxf(lm, Elem<E>::at(buf[u], k));
    if (lm > m) {
      const float sc = ex2((m - lm) * c);  // m = -inf gives 0
#pragma unroll
      for (int k = 0; k < EPV; ++k) acc[k] *= sc;
      m = lm;
    }
    if (m > -CUDART_INF_F) {
      const float mc = m * c;
#pragma unroll
      for (int u = 0; u < UNROLL; ++u)
#pragma unroll
        for (int k = 0; k < EPV; ++k) acc[k] += ex2(fmaf(Elem<E>::at(buf[u], k), c, -mc));
    }
  }
  // Scalar head and tail (at most 2*EPV-2 elements in all).
  for (int t = static_cast<int>(threadIdx.x); t < rs.head + (S.len - rs.tail0); t += THREADS) {
    {
      const int j = t < rs.head ? t : rs.tail0 + (t - rs.head);
      const float x = Elem<E>::load(row + j);
      if (x > m) {
        const float sc = ex2((m - x) * c);
#pragma unroll
        for (int k = 0; k < EPV; ++k) acc[k] *= sc;
        m = x;
      }
      if (m > -CUDART_INF_F) acc[0] += ex2(fmaf(x, c, -m * c));
    }
  }
  float s = 0.0f;
#pragma unroll
  for (int k = 0; k < EPV; ++k) s += acc[k];
  const float M = block_max<THREADS>(m, s_red);
  const float scaled = (m > -CUDART_INF_F) ? s * ex2(fmaf(m, c, -M * c)) : 0.0f;
  const float tot = block_sum<THREADS>(scaled, s_red);
  if (threadIdx.x == 0) {
    RowStats st;
    st.m = M;
    st.mc = M * c;
    st.tau = 0u;
    st.cut = INT32_MAX;
    st.K = static_cast<double>(tot);
    st.status = 0u;
    st.e_query = 0.0f;
    if (!(M > -CUDART_INF_F)) st.status |= SV_ROW_EMPTY;
    const Query q = row_query(S, r);
    if (q.bad) st.status |= SV_ROW_BAD_DRAFT_ID;
    if (q.elem >= 0 && !(st.status & SV_ROW_EMPTY) && sv_in(q.elem, S.len))
      st.e_query = weight(Elem<E>::load(row + q.elem), c, st.mc);
    S.out[r] = st;
  }
  // Warp 0 alone (thread 0 wrote the statistics): count the row for its
  // batch row and, after the batch row's last one, make its decisions.
  if (L.dec.rec && threadIdx.x < 32) {
    bool last = false;
    if (threadIdx.x == 0) last = count_row(L.dec, S, r);
    if (__shfl_sync(0xffffffffu, last, 0)) {
      __threadfence();
      const DecideRecord rc = decide_batch(L.dec, r / S.per_group);
      if ((threadIdx.x & 31) == 0) L.dec.rec[r / S.per_group] = rc;
    }
  }
}

// ------------------------------------------------------------------ host ----

static constexpr int kStatsThreads = 512;
static constexpr int kStreamUnroll = 4;

template <typename E>
static sv_status launch_stream(const StatsLaunch& L, int rows, cudaStream_t stream) {
  if (rows == 0) return SV_OK;
  stats_stream_kernel<E, kStatsThreads, kStreamUnroll><<<rows, kStatsThreads, 0, stream>>>(L);
  if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  note_launch(stream);
  return SV_OK;
}

// One launch when both row sets share a dtype, else one per set.  top_p < 1
// selects the top-p kernel, whose scratch follows the row statistics.
sv_status launch_stats_sets(StatsLaunch L, sv_dtype d0, sv_dtype d1, bool topp, void* scratch,
                                   cudaStream_t stream) {
  auto one = [&](const StatsLaunch& X, sv_dtype dt, void* scr) -> sv_status {
    if (topp) return launch_topp_stats(X, dt, scr, stream);
    const int rows = X.set[0].rows + (X.nsets > 1 ? X.set[1].rows : 0);
    return dt == SV_BF16 ? launch_stream<uint16_t>(X, rows, stream) : launch_stream<float>(X, rows, stream);
  };
  if (L.nsets == 1 || d0 == d1) return one(L, d0, scratch);
  StatsLaunch a = L, b = L;
  a.nsets = 1;
  b.nsets = 1;
  b.set[0] = L.set[1];
  sv_status s = one(a, d0, scratch);
  if (s != SV_OK) return s;
  void* scr_b = topp ? static_cast<char*>(scratch) + topp_scratch_bytes(a.set[0].rows, a.set[0].len, 0, 0)
                     : scratch;
  return one(b, d1, scr_b);
}

static float log2e_over(double T) { return static_cast<float>(1.4426950408889634 / T); }

sv_status sampling_chain(const ChainArgs& a, cudaStream_t stream) {
  const sv_chain_desc& d = a.d;
  const int B = d.batch, G = d.gamma;
  if (B == 0) return SV_OK;
  WorkspaceLayout WL = chain_workspace_layout(d);
  RowStats* stats = reinterpret_cast<RowStats*>(static_cast<char*>(a.workspace) + WL.stats);
  const bool resident = d.top_p < 1.0f;
  StatsLaunch L{};
  L.c = log2e_over(d.temperature);
  L.top_p = d.top_p;
  RowSet& T = L.set[0];
  T.base = a.target;
  T.stride = d.target_row_stride;
  T.len = d.vocab;
  T.rows = B * (G + 1);
  T.per_group = G + 1;
  T.gamma = G;
  T.last_no_query = true;
  T.ids = G > 0 ? a.ids : nullptr;
  T.t2d = nullptr;
  T.sec = nullptr;
  T.vocab = d.vocab;
  T.out = stats;
  L.nsets = 1;
  int max_len = d.vocab;
  if (G > 0) {
    RowSet& D = L.set[1];
    D.base = a.draft;
    D.stride = d.draft_row_stride;
    D.len = d.draft_vocab;
    D.rows = B * G;
    D.per_group = G;
    D.gamma = G;
    D.last_no_query = false;
    D.ids = a.ids;
    D.t2d = a.d2t ? a.t2d : nullptr;
    D.sec = a.d2t;
    D.vocab = d.vocab;
    D.out = stats + static_cast<int64_t>(B) * (G + 1);
    L.nsets = 2;
    max_len = std::max(max_len, d.draft_vocab);
  }
  DecideRecord* rec = reinterpret_cast<DecideRecord*>(static_cast<char*>(a.workspace) + WL.records);
  unsigned* bcount = reinterpret_cast<unsigned*>(static_cast<char*>(a.workspace) + WL.counters);
  L.dec.t_stats = stats;
  L.dec.d_stats = stats + static_cast<int64_t>(B) * (G + 1);
  L.dec.ids = a.ids;
  L.dec.u_accept = a.u_accept;
  L.dec.p_draft = a.p_draft;
  L.dec.q_draft = a.q_draft;
  L.dec.rec = rec;
  L.dec.counters = bcount;
  L.dec.G = G;
  L.dec.V = d.vocab;
  L.dec.rows_per_batch = 2 * G + 1;
  // The top-p pass has a last block per row: it makes the decisions of a
  // batch row after the row's last statistic.  Otherwise the draw does.
  DecideIn in_draw = L.dec;
  if (!resident) L.dec.rec = nullptr;
  start_phases(stream);
  if (resident && cudaMemsetAsync(bcount, 0, static_cast<size_t>(B) * sizeof(unsigned), stream) != cudaSuccess)
    return SV_ERR_CUDA;
  void* scratch = static_cast<char*>(a.workspace) + WL.topp;
  sv_status s = launch_stats_sets(L, d.target_dtype, d.draft_dtype, resident, scratch, stream);
  if (s != SV_OK) return s;
  DecideParams P{};
  P.target = a.target;
  P.draft = a.draft;
  P.t_stride = d.target_row_stride;
  P.d_stride = d.draft_row_stride;
  P.B = B;
  P.G = G;
  P.V = d.vocab;
  P.Vd = d.draft_vocab;
  P.c = L.c;
  P.rec = resident ? rec : nullptr;
  P.dec = in_draw;
  P.ids = a.ids;
  P.u_resample = a.u_resample;
  P.t2d = a.d2t ? a.t2d : nullptr;
  P.d2t = a.d2t ? a.d2t : nullptr;
  P.out_tokens = a.out_tokens;
  P.num_accepted = a.num_accepted;
  P.row_status = a.row_status;
  return launch_decide(P, d.target_dtype, d.draft_dtype, static_cast<char*>(a.workspace) + WL.decide, stream);
}

// Sampling without top-p in one pass over each row (one block per row):
// every warp reduces whole chunks of 2048 ids to (chunk maximum m_c, sum of
// exp2((l - m_c) c)); the block combines the
// chunks into the row's maximum M and total S (double), takes the chunk
// holding u * S by a prefix over the chunks' masses in ascending id order,
// and rescans that chunk alone (just read: L2) with a block prefix scan in
// double.  Draw as the inverse CDF ("LLM inference acceleration in practice
// ..." §4.2 `multinomial`): the first id whose inclusive prefix exceeds u * S;
// zero-mass ids are never drawn; if rounding leaves u * S at or above the
// total, the last finite id.  Rows aligned to 16 bytes, V a multiple of the
// vector width and at most kSampleMaxChunks chunks.
constexpr int kSampleThreads = 512;
constexpr int kSampleChunk = 2048;
constexpr int kSampleMaxChunks = 512;

template <typename E>
__global__ void __launch_bounds__(kSampleThreads, 2) sample_stream_kernel(const E* __restrict__ logits, int64_t stride,
                                                                     int V, float c, const float* __restrict__ u,
                                                                     int32_t* out_tokens, float* out_prob) {
  constexpr int EPV = Elem<E>::kPerVec;
  constexpr int VPC = kSampleChunk / EPV;  // 16-byte vectors per chunk
  constexpr int VPL = VPC / 32;            // per lane
  constexpr int kWarps = kSampleThreads / 32;
  __shared__ float s_m[kSampleMaxChunks];
  __shared__ float s_s[kSampleMaxChunks];
  __shared__ float s_red[32];
  __shared__ double s_scan[32];
  __shared__ int s_chunk, s_tok, s_lastall, s_lastid;
  __shared__ int s_ri[32];
  __shared__ double s_target, s_carry, s_total;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = blockIdx.x;
  const E* row = logits + static_cast<int64_t>(r) * stride;
  const uint4* vp = reinterpret_cast<const uint4*>(row);
  const int nvec = V / EPV;
  const int nch = (V + kSampleChunk - 1) / kSampleChunk;

  // 1. Chunks, one warp each at a time (eight vectors per lane in flight).
  for (int ch = warp; ch < nch; ch += kWarps) {
    float m = -CUDART_INF_F, sacc = 0.0f;
#pragma unroll
    for (int h = 0; h < VPL; h += 8) {
      uint4 w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int v = ch * VPC + (h + i) * 32 + lane;
        w[i] = v < nvec ? ldg_stream(vp + v) : Elem<E>::neg_inf_vec();
      }
      float bm = -CUDART_INF_F;
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int e = 0; e < EPV; ++e) bm = fmaxf(bm, Elem<E>::at(w[i], e));
      if (bm > m) {
        sacc *= ex2((m - bm) * c);  // m = -inf gives 0
        m = bm;
      }
      if (m > -CUDART_INF_F) {
        const float mc = m * c;
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int e = 0; e < EPV; ++e) sacc += ex2(fmaf(Elem<E>::at(w[i], e), c, -mc));
      }
    }
    const float mw = warp_max(m);
    const float part = m > -CUDART_INF_F ? sacc * ex2((m - mw) * c) : 0.0f;
    const float sw = warp_sum(part);
    if (lane == 0) {
      s_m[ch] = mw;
      s_s[ch] = sw;
    }
  }
  __syncthreads();

  // 2. The row's maximum, then the chunk that holds u * S (one warp).
  float mloc = -CUDART_INF_F;
  for (int ch = tid; ch < nch; ch += kSampleThreads) mloc = fmaxf(mloc, s_m[ch]);
  const float M = block_max<kSampleThreads>(mloc, s_red);
  if (warp == 0) {
    const int per = (nch + 31) / 32;
    const int q0 = min(nch, lane * per), q1 = min(nch, q0 + per);
    double sl = 0.0;
    int lastc = -1;  // the last chunk with a finite logit
    for (int q = q0; q < q1; ++q) {
      if (s_m[q] > -CUDART_INF_F) {
        sl += static_cast<double>(s_s[q]) * static_cast<double>(ex2((s_m[q] - M) * c));
        lastc = q;
      }
    }
    double incl = sl;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const double total = __shfl_sync(0xffffffffu, incl, 31);
    const double target = static_cast<double>(u[r]) * total;
    const unsigned hb = __ballot_sync(0xffffffffu, sl > 0.0 && incl > target && incl - sl <= target);
    int chunk = -1;
    double carry = 0.0;
    if (hb) {
      const int wl = __ffs(hb) - 1;
      if (lane == wl) {
        double cc = incl - sl;
        for (int q = q0; q < q1; ++q) {
          const double s2 =
              s_m[q] > -CUDART_INF_F ? static_cast<double>(s_s[q]) * static_cast<double>(ex2((s_m[q] - M) * c)) : 0.0;
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
    lastc = warp_max_i(lastc);
    if (lane == 0) {
      s_chunk = chunk;
      s_carry = carry;
      s_target = target;
      s_total = total;
      s_lastall = lastc;  // the chunk; its last finite id is found below when needed
      s_lastid = -1;
      s_tok = INT32_MAX;
    }
  }
  __syncthreads();
  const int chunk = s_chunk;
  if (!(s_total > 0.0)) {
    if (tid == 0) {
      out_tokens[r] = -1;
      if (out_prob) out_prob[r] = 0.0f;
    }
    return;
  }

  // 3. The chunk that holds u * S, rescanned: the thread whose ids span it
  // finds the id.
  if (chunk >= 0) {
    const int v = chunk * VPC + tid;
    float wv[EPV];
    float mine = 0.0f;
    if (tid < VPC) {
      const uint4 w = v < nvec ? __ldcg(vp + v) : Elem<E>::neg_inf_vec();
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        const float x = Elem<E>::at(w, e);
        wv[e] = x > -CUDART_INF_F ? ex2((x - M) * c) : 0.0f;
        mine += wv[e];
      }
    } else {
#pragma unroll
      for (int e = 0; e < EPV; ++e) wv[e] = 0.0f;
    }
    double tot;
    const double excl = block_exclusive_scan_d<kSampleThreads>(static_cast<double>(mine), s_scan, &tot);
    const double rem = s_target - (s_carry + excl);
    if (tid < VPC && rem < static_cast<double>(mine)) {
      const float remf = static_cast<float>(rem);
      float run = 0.0f;
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        run += wv[e];
        if (wv[e] > 0.0f && run > remf) {
          atomicMin(&s_tok, v * EPV + e);
          break;
        }
      }
    }
    __syncthreads();
  }
  if (s_tok == INT32_MAX && s_lastall >= 0) {
    // Rounding left u * S at or past the total: the last id with a finite
    // logit, in the last chunk that has one.
    const int v = s_lastall * VPC + tid;
    int last = -1;
    if (tid < VPC && v < nvec) {
      const uint4 w = __ldcg(vp + v);
#pragma unroll
      for (int e = 0; e < EPV; ++e)
        if (Elem<E>::at(w, e) > -CUDART_INF_F) last = v * EPV + e;
    }
    last = block_max_i<kSampleThreads>(last, s_ri);
    if (tid == 0) s_lastid = last;
    __syncthreads();
  }
  if (tid == 0) {
    const int tok = s_tok != INT32_MAX ? s_tok : s_lastid;
    if (tok >= 0 && tok < V) {
      out_tokens[r] = tok;
      if (out_prob) {
        const float x = Elem<E>::load(row + tok);
        out_prob[r] = static_cast<float>(static_cast<double>(ex2((x - M) * c)) / s_total);
      }
    } else {
      out_tokens[r] = -1;
      if (out_prob) out_prob[r] = 0.0f;
    }
  }
}

sv_status sample_rows(const sv_sample_desc& d, const void* logits, const float* u,
                      int32_t* out_tokens, float* out_prob, void* workspace, cudaStream_t stream) {
  if (d.rows == 0) return SV_OK;
  {
    // Without top-p, aligned rows: one pass (sample_stream_kernel).
    const size_t es = d.dtype == SV_BF16 ? 2 : 4;
    const int epv = static_cast<int>(16 / es);
    const bool aligned = (reinterpret_cast<uintptr_t>(logits) & 15u) == 0 && (d.row_stride * es) % 16 == 0 &&
                         d.vocab % epv == 0;
    if (d.top_p >= 1.0f && aligned && d.vocab <= kSampleMaxChunks * kSampleChunk) {
      start_phases(stream);
      const float c = log2e_over(d.temperature);
      if (d.dtype == SV_BF16)
        sample_stream_kernel<uint16_t><<<d.rows, kSampleThreads, 0, stream>>>(
            static_cast<const uint16_t*>(logits), d.row_stride, d.vocab, c, u, out_tokens, out_prob);
      else
        sample_stream_kernel<float><<<d.rows, kSampleThreads, 0, stream>>>(
            static_cast<const float*>(logits), d.row_stride, d.vocab, c, u, out_tokens, out_prob);
      if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
      note_launch(stream);
      return SV_OK;
    }
  }
  RowStats* stats = static_cast<RowStats*>(workspace);
  StatsLaunch L{};
  L.c = log2e_over(d.temperature);
  L.top_p = d.top_p;
  L.nsets = 1;
  RowSet& T = L.set[0];
  T.base = logits;
  T.stride = d.row_stride;
  T.len = d.vocab;
  T.rows = d.rows;
  T.per_group = 1;
  T.gamma = 0;
  T.last_no_query = true;
  T.ids = nullptr;
  T.vocab = d.vocab;
  T.out = stats;
  DecideRecord* rec = reinterpret_cast<DecideRecord*>(static_cast<char*>(workspace) + sample_records_offset(d.rows));
  unsigned* bcount = reinterpret_cast<unsigned*>(static_cast<char*>(workspace) + sample_counters_offset(d.rows));
  L.dec.t_stats = stats;
  L.dec.d_stats = stats;
  L.dec.rec = rec;
  L.dec.counters = bcount;
  L.dec.G = 0;
  L.dec.V = d.vocab;
  L.dec.rows_per_batch = 1;
  const bool resident = d.top_p < 1.0f;
  DecideIn in_draw = L.dec;
  if (!resident) L.dec.rec = nullptr;
  start_phases(stream);
  if (resident && cudaMemsetAsync(bcount, 0, static_cast<size_t>(d.rows) * sizeof(unsigned), stream) != cudaSuccess)
    return SV_ERR_CUDA;
  void* scratch = static_cast<char*>(workspace) + sample_topp_offset(d.rows);
  sv_status s = launch_stats_sets(L, d.dtype, d.dtype, resident, scratch, stream);
  if (s != SV_OK) return s;
  DecideParams P{};
  P.target = logits;
  P.t_stride = d.row_stride;
  P.B = d.rows;
  P.G = 0;
  P.V = d.vocab;
  P.c = L.c;
  P.rec = resident ? rec : nullptr;
  P.dec = in_draw;
  P.u_resample = u;
  P.out_tokens = out_tokens;
  P.out_prob = out_prob;
  return launch_decide(P, d.dtype, d.dtype,
                       static_cast<char*>(workspace) + sample_topp_offset(d.rows) + sample_topp_bytes(d), stream);
}

}  // namespace sv

// ------------------------------------------------------ filtered probabilities ----
// p_j = softmax(top_p_filter(l / T))_j for every id of every row: the
// statistics pass, then one elementwise pass ("LLM inference acceleration in
// practice ..." §4.2: _apply_top_p followed by F.softmax).

namespace sv {

template <typename E>
__global__ void __launch_bounds__(256) probs_kernel(const E* __restrict__ logits, int64_t stride, int V,
                                                    const RowStats* __restrict__ stats, float c,
                                                    float* __restrict__ out, int64_t out_stride, int tiles) {
  const int row = blockIdx.x / tiles;
  const int tile = blockIdx.x - row * tiles;
  const RowStats st = stats[row];
  const E* src = logits + static_cast<int64_t>(row) * stride;
  float* dst = out + static_cast<int64_t>(row) * out_stride;
  const float invK = st.K > 0.0 ? static_cast<float>(1.0 / st.K) : 0.0f;
  const int base = tile * 256 * 8;
  for (int e = 0; e < 8; ++e) {
    const int j = base + e * 256 + threadIdx.x;
    if (j >= V) break;
    const float x = Elem<E>::load(src + j);
    const bool keep = !(st.status & SV_ROW_EMPTY) && kept(order_key(x), j, st.tau, st.cut);
    dst[j] = keep ? weight(x, c, st.mc) * invK : 0.0f;
  }
}

sv_status probs_rows(const sv_sample_desc& d, const void* logits, float* out, int64_t out_stride,
                     void* workspace, cudaStream_t stream) {
  if (d.rows == 0) return SV_OK;
  RowStats* stats = static_cast<RowStats*>(workspace);
  StatsLaunch L{};
  L.c = log2e_over(d.temperature);
  L.top_p = d.top_p;
  L.nsets = 1;
  RowSet& T = L.set[0];
  T.base = logits;
  T.stride = d.row_stride;
  T.len = d.vocab;
  T.rows = d.rows;
  T.per_group = 1;
  T.gamma = 0;
  T.last_no_query = true;
  T.ids = nullptr;
  T.vocab = d.vocab;
  T.out = stats;
  start_phases(stream);
  void* scratch = static_cast<char*>(workspace) + sample_topp_offset(d.rows);
  sv_status s = launch_stats_sets(L, d.dtype, d.dtype, d.top_p < 1.0f, scratch, stream);
  if (s != SV_OK) return s;
  const int tiles = (d.vocab + 2047) / 2048;
  const unsigned grid = static_cast<unsigned>(d.rows) * tiles;
  if (d.dtype == SV_BF16)
    probs_kernel<uint16_t><<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(logits), d.row_stride, d.vocab,
                                                     stats, L.c, out, out_stride, tiles);
  else
    probs_kernel<float><<<grid, 256, 0, stream>>>(static_cast<const float*>(logits), d.row_stride, d.vocab, stats,
                                                  L.c, out, out_stride, tiles);
  if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  note_launch(stream);
  return SV_OK;
}

}  // namespace sv
