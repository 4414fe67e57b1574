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

sv_status sample_rows(const sv_sample_desc& d, const void* logits, const float* u,
                      int32_t* out_tokens, float* out_prob, void* workspace, cudaStream_t stream) {
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
