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
//      (radix select over order keys with integer masses, rows held in the
//      shared memory of a thread-block cluster); it also evaluates the row's
//      weight at its draft id.
//   2. decision: one block per batch row turns those into p(x), q(x), finds
//      the first rejection and draws the resample/bonus token by an inverse
//      CDF over one (pair of) rows: chunk sums, then a block scan of the one
//      chunk that holds the draw.
#include "sv_internal.h"

#include <algorithm>
#include <cmath>

namespace sv {

// ------------------------------------------------------------- row sets ----

// A contiguous set of logit rows processed by the statistics pass.  Row r
// belongs to group b = r / per_group at position i = r % per_group.
struct RowSet {
  const void* base;
  int64_t stride;
  int len;             // elements per row
  int rows;
  int per_group;
  int gamma;           // ids are [groups, gamma]
  bool last_no_query;  // position per_group-1 has no query (target row γ)
  const int32_t* ids;  // query ids (target vocabulary) or nullptr
  const int32_t* t2d;  // query id -> row element (EAGLE3 draft rows) or nullptr
  const int32_t* sec;  // element -> tie key (d2t) or nullptr (the element index)
  int vocab;           // valid query ids are [0, vocab)
  RowStats* out;
};

struct StatsLaunch {
  RowSet set[2];
  int nsets;
  float c;             // log2(e) / T
  float top_p;
  int cl;              // cluster size (resident kernel)
  int slice;           // elements per cluster rank (resident kernel)
};

__device__ __forceinline__ const RowSet& pick_set(const StatsLaunch& L, int& r) {
  if (L.nsets > 1 && r >= L.set[0].rows) {
    r -= L.set[0].rows;
    return L.set[1];
  }
  return L.set[0];
}

// Resolve the query of row r: element index in the row (-1: none/unmapped),
// its tie key, and whether the id itself is invalid.
struct Query {
  int elem;
  int sec;
  bool bad;
};

__device__ __forceinline__ Query row_query(const RowSet& S, int r) {
  Query q{-1, -1, false};
  if (!S.ids) return q;
  const int b = r / S.per_group, i = r - b * S.per_group;
  if (S.last_no_query && i == S.per_group - 1) return q;
  const int x = S.ids[static_cast<int64_t>(b) * S.gamma + i];
  if (x < 0 || x >= S.vocab) {
    q.bad = true;
    return q;
  }
  q.sec = x;
  q.elem = S.t2d ? S.t2d[x] : x;
  if (q.elem >= S.len) q.elem = -1;  // a t2d entry outside the draft row maps nowhere
  return q;
}

__device__ __forceinline__ int tie_key(const RowSet& S, int j) { return S.sec ? __ldg(S.sec + j) : j; }

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
  const int nvec = S.len / EPV;
  const uint4* vp = reinterpret_cast<const uint4*>(row);

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
  {
    const int t = nvec * EPV + static_cast<int>(threadIdx.x);
    if (t < S.len) {
      const float x = Elem<E>::load(row + t);
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
    if (q.elem >= 0 && !(st.status & SV_ROW_EMPTY))
      st.e_query = weight(Elem<E>::load(row + q.elem), c, st.mc);
    S.out[r] = st;
  }
}

// ---------------------------------------------------- resident statistics ----
// top_p < 1: each row is split over a cluster of L.cl blocks, every block
// keeps its slice in shared memory.  After the maximum, radix passes over the
// order keys (8 bits per pass) build (mass, count) histograms; the cluster
// adds them through distributed shared memory and every block walks the bins
// from the top to find the bin holding the first rank whose cumulative mass
// exceeds top_p.  Masses are fixed-point integers so the totals are exact
// and identical in every block.  A partially kept group of equal logits is
// cut by a second radix select over the tie keys (lowest first).

constexpr float kFix39 = 549755813888.0f;  // 2^39: V <= 2^24 keeps sums < 2^63
constexpr double kFix39Inv = 1.0 / 549755813888.0;

__device__ __forceinline__ unsigned long long fixed39(float e) { return __float2ull_rn(e * kFix39); }

struct ResidentShared {
  unsigned long long h_mass[2][256];
  unsigned int h_cnt[2][256];
  unsigned long long t_mass[256];
  unsigned int t_cnt[256];
  unsigned long long red_u64[32];
  float red_f[32];
  float cta_max;
  int sel_bin;
  int found;
  unsigned long long sel_above;
};

template <int THREADS>
__device__ __forceinline__ void cluster_reduce_hist(cg::cluster_group& cluster, ResidentShared& sh,
                                                    int buf, int cl, bool with_mass) {
  __syncthreads();
  cluster.sync();
  for (int t = threadIdx.x; t < 256; t += THREADS) {
    unsigned long long ms = 0;
    unsigned int cs = 0;
    for (int q = 0; q < cl; ++q) {
      ResidentShared* peer = cluster.map_shared_rank(&sh, q);
      if (with_mass) ms += peer->h_mass[buf][t];
      cs += peer->h_cnt[buf][t];
    }
    sh.t_mass[t] = ms;
    sh.t_cnt[t] = cs;
  }
  __syncthreads();
}

// Walk bins from 255 down; find the first bin where above + mass > limit.
// Warp 0 only; result in sh.sel_bin / sh.sel_above / sh.found.
__device__ __forceinline__ void find_crossing_desc(ResidentShared& sh, unsigned long long above,
                                                   unsigned long long limit) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  unsigned long long local = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) local += sh.t_mass[255 - (lane * 8 + k)];
  unsigned long long incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  unsigned long long run = above + incl - local;
  int hit = -1;
  unsigned long long hit_above = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int bin = 255 - (lane * 8 + k);
    const unsigned long long ms = sh.t_mass[bin];
    if (hit < 0 && run + ms > limit) {
      hit = bin;
      hit_above = run;
    }
    run += ms;
  }
  const unsigned int ballot = __ballot_sync(0xffffffffu, hit >= 0);
  if (lane == 0) sh.found = ballot != 0;
  if (ballot) {
    const int src = __ffs(ballot) - 1;
    const int b = __shfl_sync(0xffffffffu, hit, src);
    const unsigned long long a = __shfl_sync(0xffffffffu, hit_above, src);
    if (lane == 0) {
      sh.sel_bin = b;
      sh.sel_above = a;
    }
  }
}

// Walk bins from 0 up; find the bin where the running count reaches `need`.
__device__ __forceinline__ void find_count_asc(ResidentShared& sh, unsigned int need) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  unsigned int local = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) local += sh.t_cnt[lane * 8 + k];
  unsigned int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  unsigned int run = incl - local;
  int hit = -1;
  unsigned int hit_before = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const unsigned int cnt = sh.t_cnt[lane * 8 + k];
    if (hit < 0 && run + cnt >= need) {
      hit = lane * 8 + k;
      hit_before = run;
    }
    run += cnt;
  }
  const unsigned int ballot = __ballot_sync(0xffffffffu, hit >= 0);
  if (lane == 0) sh.found = ballot != 0;
  if (ballot) {
    const int src = __ffs(ballot) - 1;
    const int b = __shfl_sync(0xffffffffu, hit, src);
    const unsigned int before = __shfl_sync(0xffffffffu, hit_before, src);
    if (lane == 0) {
      sh.sel_bin = b;
      sh.sel_above = before;
    }
  }
}

template <typename E, int THREADS>
__global__ void __launch_bounds__(THREADS) stats_resident_kernel(StatsLaunch L) {
  constexpr int EPV = Elem<E>::kPerVec;
  constexpr int kPasses = sizeof(E) == 2 ? 2 : 4;
  extern __shared__ __align__(16) unsigned char dyn_smem[];
  __shared__ ResidentShared sh;
  cg::cluster_group cluster = cg::this_cluster();
  const int cl = L.cl;
  const int rank = static_cast<int>(cluster.block_rank());
  int r = blockIdx.x / cl;
  const RowSet& S = pick_set(L, r);
  const E* row = reinterpret_cast<const E*>(S.base) + static_cast<int64_t>(r) * S.stride;
  const int lo = rank * L.slice;
  const int hi = min(S.len, lo + L.slice);
  const int n = max(0, hi - lo);
  E* sl = reinterpret_cast<E*>(dyn_smem);
  const float c = L.c;

  // 1. Stage the slice in shared memory; block maximum.
  const int nvec = n / EPV;
  const uint4* gv = reinterpret_cast<const uint4*>(row + lo);
  uint4* sv = reinterpret_cast<uint4*>(sl);
  float lm = -CUDART_INF_F;
  constexpr int U = 4;
  for (int v0 = threadIdx.x; v0 < nvec; v0 += THREADS * U) {
    uint4 buf[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + u * THREADS;
      buf[u] = v < nvec ? ldg_stream(gv + v) : Elem<E>::neg_inf_vec();
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + u * THREADS;
      if (v < nvec) sv[v] = buf[u];
#pragma unroll
      for (int k = 0; k < EPV; ++k) lm = fmaxf(lm, Elem<E>::at(buf[u], k));
    }
  }
  for (int t = nvec * EPV + static_cast<int>(threadIdx.x); t < n; t += THREADS) {
    sl[t] = row[lo + t];
    lm = fmaxf(lm, Elem<E>::load(row + lo + t));
  }
  lm = block_max<THREADS>(lm, sh.red_f);
  if (threadIdx.x == 0) sh.cta_max = lm;
  __syncthreads();
  cluster.sync();
  float M = -CUDART_INF_F;
  for (int q = 0; q < cl; ++q) M = fmaxf(M, cluster.map_shared_rank(&sh, q)->cta_max);
  const float mc = M * c;
  const bool empty = !(M > -CUDART_INF_F);

  auto value = [&](int t) -> float {
    if constexpr (sizeof(E) == 2) return __uint_as_float(static_cast<uint32_t>(sl[t]) << 16);
    else return sl[t];
  };

  uint32_t prefix = 0;
  unsigned long long above = 0, limit = 0, total = 0, grp_mass = 0;
  unsigned int grp_cnt = 0;
  bool keep_all = empty;
  int pass_no = 0;
  if (!empty) {
    for (int p = 0; p < kPasses; ++p, ++pass_no) {
      const int buf = pass_no & 1;
      const int sh_bits = 24 - 8 * p;
      for (int t = threadIdx.x; t < 256; t += THREADS) {
        sh.h_mass[buf][t] = 0;
        sh.h_cnt[buf][t] = 0;
      }
      __syncthreads();
      for (int t = threadIdx.x; t < n; t += THREADS) {
        const float x = value(t);
        const uint32_t key = order_key(x);
        if (p == 0 || (key >> (sh_bits + 8)) == prefix) {
          const int bin = (key >> sh_bits) & 255;
          const unsigned long long ef = fixed39(weight(x, c, mc));
          if (ef) atomicAdd(&sh.h_mass[buf][bin], ef);
          atomicAdd(&sh.h_cnt[buf][bin], 1u);
        }
      }
      cluster_reduce_hist<THREADS>(cluster, sh, buf, cl, true);
      if (p == 0) {
        unsigned long long part = 0;
        for (int t = threadIdx.x; t < 256; t += THREADS) part += sh.t_mass[t];
        total = block_sum_u64<THREADS>(part, sh.red_u64);
        limit = static_cast<unsigned long long>(floor(static_cast<double>(L.top_p) * static_cast<double>(total)));
      }
      find_crossing_desc(sh, above, limit);
      __syncthreads();
      if (!sh.found) {
        keep_all = true;
        break;
      }
      const int bin = sh.sel_bin;
      above = sh.sel_above;
      prefix = (prefix << 8) | static_cast<uint32_t>(bin);
      grp_mass = sh.t_mass[bin];
      grp_cnt = sh.t_cnt[bin];
      __syncthreads();
    }
  }
  const uint32_t tau = keep_all ? 0u : (sizeof(E) == 2 ? prefix << 16 : prefix);
  unsigned long long K = total;
  int32_t cut = INT32_MAX;
  if (!keep_all) {
    const unsigned long long e_tau = grp_mass / grp_cnt;
    unsigned long long nk = (limit - above) / e_tau + 1;
    if (nk >= grp_cnt) {
      nk = grp_cnt;
    } else {
      // nk-th smallest tie key among the elements equal to tau.
      uint32_t sp = 0;
      unsigned int need = static_cast<unsigned int>(nk);
      for (int q = 0; q < 3; ++q, ++pass_no) {
        const int buf = pass_no & 1;
        const int sb = 16 - 8 * q;
        for (int t = threadIdx.x; t < 256; t += THREADS) sh.h_cnt[buf][t] = 0;
        __syncthreads();
        for (int t = threadIdx.x; t < n; t += THREADS) {
          if (order_key(value(t)) != tau) continue;
          const uint32_t sec = static_cast<uint32_t>(tie_key(S, lo + t));
          if (q == 0 || (sec >> (sb + 8)) == sp) atomicAdd(&sh.h_cnt[buf][(sec >> sb) & 255], 1u);
        }
        cluster_reduce_hist<THREADS>(cluster, sh, buf, cl, false);
        find_count_asc(sh, need);
        __syncthreads();
        sp = (sp << 8) | static_cast<uint32_t>(sh.sel_bin);
        need -= static_cast<unsigned int>(sh.sel_above);
        __syncthreads();
      }
      cut = static_cast<int32_t>(sp);
    }
    K = above + nk * e_tau;
  }
  if (rank == 0 && threadIdx.x == 0) {
    RowStats st;
    st.m = M;
    st.mc = mc;
    st.tau = tau;
    st.cut = cut;
    st.K = static_cast<double>(K) * kFix39Inv;
    st.status = empty ? SV_ROW_EMPTY : 0u;
    st.e_query = 0.0f;
    const Query q = row_query(S, r);
    if (q.bad) st.status |= SV_ROW_BAD_DRAFT_ID;
    if (q.elem >= 0 && !empty) {
      const float x = Elem<E>::load(row + q.elem);
      if (kept(order_key(x), q.sec, tau, cut)) st.e_query = weight(x, c, mc);
    }
    S.out[r] = st;
  }
  // No block may leave while a peer can still read its shared memory.
  cluster.sync();
}

// ------------------------------------------------------ decision + draw ----

struct DecideParams {
  const void* target;
  const void* draft;
  int64_t t_stride, d_stride;
  int B, G, V, Vd;
  float c;
  const RowStats* t_stats;  // [B, G+1]
  const RowStats* d_stats;  // [B, G]
  const int32_t* ids;
  const float* u_accept;
  const float* u_resample;
  const int32_t* t2d;
  int32_t* out_tokens;
  int32_t* num_accepted;
  float* p_draft;
  float* q_draft;
  int32_t* row_status;
  float* out_prob;
};

// Weight of id j in the draw: p(j) (bonus), or max(0, p(j) - q(j)) (residual).
template <typename ET, typename ED, bool RESID>
struct DrawRow {
  const ET* t;
  const ED* d;
  const int32_t* t2d;
  int vd;  // draft row length (t2d entries at or beyond it map nowhere)
  float c, mct, invKt, mcd, invKd;
  uint32_t taut, taud;
  int32_t cutt, cutd;

  __device__ __forceinline__ float w(int j) const {
    const float lt = Elem<ET>::load(t + j);
    float p = 0.0f;
    if (kept(order_key(lt), j, taut, cutt)) p = weight(lt, c, mct) * invKt;
    if constexpr (!RESID) {
      return p;
    } else {
      const int jd = t2d ? __ldg(t2d + j) : j;
      float q = 0.0f;
      if (jd >= 0 && jd < vd) {
        const float ld = Elem<ED>::load(d + jd);
        if (kept(order_key(ld), j, taud, cutd)) q = weight(ld, c, mcd) * invKd;
      }
      return fmaxf(0.0f, p - q);
    }
  }
};

constexpr int kDrawThreads = 512;
constexpr int kDrawEPT = 8;                           // contiguous ids per thread per chunk
constexpr int kDrawChunk = kDrawThreads * kDrawEPT;   // 4096 ids per chunk
constexpr int kDrawUnroll = 2;                        // chunks in flight per iteration

struct DrawShared {
  float red[kDrawUnroll][32];
  double scan[32];
  int last_pos;
  int tok;
  int chunk;
  double carry;
  double target;
  double total;
  int k;
  unsigned int status;
  int fallback;
};

// Inverse-CDF draw over V weights: returns the smallest j whose inclusive
// prefix exceeds u * total, or -1 if the total is zero.
template <typename ET, typename ED, bool RESID>
__device__ int draw_inverse_cdf(const DrawRow<ET, ED, RESID>& R, int V, float u, float* chunk_sums,
                                DrawShared& sh) {
  const int nchunks = (V + kDrawChunk - 1) / kDrawChunk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int last_pos = -1;
  for (int c0 = 0; c0 < nchunks; c0 += kDrawUnroll) {
    float part[kDrawUnroll];
#pragma unroll
    for (int uu = 0; uu < kDrawUnroll; ++uu) {
      part[uu] = 0.0f;
      const int base = (c0 + uu) * kDrawChunk + threadIdx.x * kDrawEPT;
#pragma unroll
      for (int e = 0; e < kDrawEPT; ++e) {
        const int j = base + e;
        if (c0 + uu < nchunks && j < V) {
          const float x = R.w(j);
          part[uu] += x;
          if (x > 0.0f) last_pos = j;
        }
      }
    }
#pragma unroll
    for (int uu = 0; uu < kDrawUnroll; ++uu) {
      const float s = warp_sum(part[uu]);
      if (lane == 0) sh.red[uu][warp] = s;
    }
    __syncthreads();
    if (warp == 0) {
#pragma unroll
      for (int uu = 0; uu < kDrawUnroll; ++uu) {
        float s = lane < kDrawThreads / 32 ? sh.red[uu][lane] : 0.0f;
        s = warp_sum(s);
        if (lane == 0 && c0 + uu < nchunks) chunk_sums[c0 + uu] = s;
      }
    }
    __syncthreads();
  }
  // The last id with positive weight (fallback when rounding leaves the draw
  // at or past the end).
  {
    __shared__ int s_red_i[32];
    last_pos = block_max_i<kDrawThreads>(last_pos, s_red_i);
  }
  if (threadIdx.x == 0) {
    double total = 0.0;
    for (int ci = 0; ci < nchunks; ++ci) total += chunk_sums[ci];
    sh.total = total;
    sh.target = static_cast<double>(u) * total;
    sh.chunk = -1;
    double cum = 0.0;
    for (int ci = 0; ci < nchunks; ++ci) {
      const double next = cum + chunk_sums[ci];
      if (next > sh.target && chunk_sums[ci] > 0.0f) {
        sh.chunk = ci;
        sh.carry = cum;
        break;
      }
      cum = next;
    }
    sh.tok = INT32_MAX;
    sh.last_pos = last_pos;
  }
  __syncthreads();
  if (!(sh.total > 0.0)) return -1;
  if (sh.chunk < 0) return sh.last_pos;
  // Rescan the chunk that holds the draw.
  const int base = sh.chunk * kDrawChunk + threadIdx.x * kDrawEPT;
  float wv[kDrawEPT];
  float part = 0.0f;
  int lp = -1;
#pragma unroll
  for (int e = 0; e < kDrawEPT; ++e) {
    const int j = base + e;
    wv[e] = j < V ? R.w(j) : 0.0f;
    part += wv[e];
    if (wv[e] > 0.0f) lp = j;
  }
  double tot;
  const double excl = block_exclusive_scan_d<kDrawThreads>(static_cast<double>(part), sh.scan, &tot);
  double run = sh.carry + excl;
  const double target = sh.target;
#pragma unroll
  for (int e = 0; e < kDrawEPT; ++e) {
    run += wv[e];
    if (wv[e] > 0.0f && run > target) {
      atomicMin(&sh.tok, base + e);
      break;
    }
  }
  {
    __shared__ int s_red_i2[32];
    lp = block_max_i<kDrawThreads>(lp, s_red_i2);
  }
  __syncthreads();
  return sh.tok != INT32_MAX ? sh.tok : lp;
}

template <typename ET, typename ED>
__global__ void __launch_bounds__(kDrawThreads) decide_kernel(DecideParams P) {
  extern __shared__ float chunk_sums[];
  __shared__ DrawShared sh;
  __shared__ unsigned char s_acc[SV_MAX_GAMMA];
  const int b = blockIdx.x;
  const int G = P.G;
  const RowStats* ts = P.t_stats + static_cast<int64_t>(b) * (G + 1);
  const RowStats* ds = P.d_stats + static_cast<int64_t>(b) * G;
  if (threadIdx.x == 0) {
    sh.status = 0;
    sh.fallback = 0;
  }
  __syncthreads();
  for (int i = threadIdx.x; i <= G; i += kDrawThreads) {
    uint32_t st = ts[i].status;
    if (i < G) st |= ds[i].status;
    if (i < G) {
      const int x = P.ids[static_cast<int64_t>(b) * G + i];
      if (x < 0 || x >= P.V) st |= SV_ROW_BAD_DRAFT_ID;
      const double p = ts[i].K > 0.0 ? static_cast<double>(ts[i].e_query) / ts[i].K : 0.0;
      const double q = ds[i].K > 0.0 ? static_cast<double>(ds[i].e_query) / ds[i].K : 0.0;
      const double u = static_cast<double>(P.u_accept[static_cast<int64_t>(b) * G + i]);
      s_acc[i] = (u * q < p) ? 1 : 0;
      if (P.p_draft) P.p_draft[static_cast<int64_t>(b) * G + i] = static_cast<float>(p);
      if (P.q_draft) P.q_draft[static_cast<int64_t>(b) * G + i] = static_cast<float>(q);
    }
    if (st) atomicOr(&sh.status, st);
  }
  __syncthreads();
  int32_t* out = P.out_tokens + static_cast<int64_t>(b) * (G + 1);
  if (sh.status & (SV_ROW_BAD_DRAFT_ID | SV_ROW_EMPTY)) {
    for (int i = threadIdx.x; i <= G; i += kDrawThreads) out[i] = -1;
    if (threadIdx.x == 0) {
      if (P.num_accepted) P.num_accepted[b] = 0;
      if (P.row_status) P.row_status[b] = static_cast<int32_t>(sh.status);
      if (P.out_prob) P.out_prob[b] = 0.0f;
    }
    return;
  }
  if (threadIdx.x == 0) {
    int k = G;
    for (int i = 0; i < G; ++i)
      if (!s_acc[i]) {
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
  DrawRow<ET, ED, false> bonus{trow, nullptr, nullptr, 0, P.c, st.mc, static_cast<float>(1.0 / st.K),
                               0.0f, 0.0f, st.tau, 0u, st.cut, 0};
  int tok = -1;
  float prob = 0.0f;
  if (k < G) {
    const RowStats& sd = ds[k];
    const ED* drow = reinterpret_cast<const ED*>(P.draft) + (static_cast<int64_t>(b) * G + k) * P.d_stride;
    DrawRow<ET, ED, true> resid{trow, drow, P.t2d, P.Vd, P.c, st.mc, static_cast<float>(1.0 / st.K),
                                sd.mc, static_cast<float>(1.0 / sd.K), st.tau, sd.tau, st.cut, sd.cut};
    tok = draw_inverse_cdf(resid, P.V, u, chunk_sums, sh);
    if (tok < 0) {  // residual mass 0: draw from p_k
      if (threadIdx.x == 0) sh.fallback = 1;
      tok = draw_inverse_cdf(bonus, P.V, u, chunk_sums, sh);
    }
  } else {
    tok = draw_inverse_cdf(bonus, P.V, u, chunk_sums, sh);
    if (threadIdx.x == 0 && tok >= 0) prob = bonus.w(tok);
  }
  __syncthreads();
  for (int i = threadIdx.x; i <= G; i += kDrawThreads)
    out[i] = i < k ? P.ids[static_cast<int64_t>(b) * G + i] : (i == k ? tok : -1);
  if (threadIdx.x == 0) {
    if (P.num_accepted) P.num_accepted[b] = k;
    if (P.row_status)
      P.row_status[b] = static_cast<int32_t>(sh.status | (sh.fallback ? SV_ROW_RESAMPLE_FALLBACK : 0u));
    if (P.out_prob) P.out_prob[b] = prob;
  }
}

// ------------------------------------------------------------------ host ----

static constexpr int kStatsThreads = 512;
static constexpr int kStreamUnroll = 4;
static constexpr size_t kSliceBudget = 96 * 1024;  // two resident blocks per SM

static bool same_dtype_sets(sv_dtype a, sv_dtype b) { return a == b; }

template <typename E>
static sv_status launch_stats(const StatsLaunch& L, int rows, bool resident, cudaStream_t stream) {
  if (rows == 0) return SV_OK;
  if (!resident) {
    stats_stream_kernel<E, kStatsThreads, kStreamUnroll><<<rows, kStatsThreads, 0, stream>>>(L);
    if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
    note_launch(stream);
    return SV_OK;
  }
  const size_t smem = align_up(static_cast<size_t>(L.slice) * sizeof(E), 16);
  auto kern = stats_resident_kernel<E, kStatsThreads>;
  static FuncAttrCache cache;
  if (!cache.ensure(reinterpret_cast<const void*>(kern), smem, L.cl > 8)) return SV_ERR_CUDA;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(rows) * L.cl);
  cfg.blockDim = dim3(kStatsThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(L.cl);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, L) != cudaSuccess) return SV_ERR_CUDA;
  note_launch(stream);
  return SV_OK;
}

static sv_status launch_stats_sets(StatsLaunch L, sv_dtype d0, sv_dtype d1, bool resident,
                                   int max_len, cudaStream_t stream) {
  if (resident) {
    const size_t esz = 4;  // size the slice for the widest element type in use
    (void)esz;
    int cl = 1;
    auto slice_for = [&](int c) { return static_cast<int>(align_up((max_len + c - 1) / c, 8)); };
    auto bytes_for = [&](int c) {
      const size_t e = (d0 == SV_F32 || (L.nsets > 1 && d1 == SV_F32)) ? 4 : 2;
      return static_cast<size_t>(slice_for(c)) * e;
    };
    while (cl < 16 && bytes_for(cl) > kSliceBudget) cl *= 2;
    if (bytes_for(cl) > 200 * 1024) return SV_ERR_UNSUPPORTED;
    L.cl = cl;
    L.slice = slice_for(cl);
  }
  if (L.nsets == 1 || same_dtype_sets(d0, d1)) {
    const int rows = L.set[0].rows + (L.nsets > 1 ? L.set[1].rows : 0);
    return d0 == SV_BF16 ? launch_stats<uint16_t>(L, rows, resident, stream)
                         : launch_stats<float>(L, rows, resident, stream);
  }
  StatsLaunch a = L, b = L;
  a.nsets = 1;
  b.nsets = 1;
  b.set[0] = L.set[1];
  sv_status s = d0 == SV_BF16 ? launch_stats<uint16_t>(a, a.set[0].rows, resident, stream)
                              : launch_stats<float>(a, a.set[0].rows, resident, stream);
  if (s != SV_OK) return s;
  return d1 == SV_BF16 ? launch_stats<uint16_t>(b, b.set[0].rows, resident, stream)
                       : launch_stats<float>(b, b.set[0].rows, resident, stream);
}

template <typename ET, typename ED>
static sv_status launch_decide(const DecideParams& P, cudaStream_t stream) {
  const int nchunks = (P.V + kDrawChunk - 1) / kDrawChunk;
  const size_t smem = align_up(static_cast<size_t>(nchunks + kDrawUnroll) * sizeof(float), 16);
  auto kern = decide_kernel<ET, ED>;
  static FuncAttrCache cache;
  if (smem > 48 * 1024 && !cache.ensure(reinterpret_cast<const void*>(kern), smem, false)) return SV_ERR_CUDA;
  kern<<<P.B, kDrawThreads, smem, stream>>>(P);
  if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  note_launch(stream);
  return SV_OK;
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
  sv_status s = launch_stats_sets(L, d.target_dtype, d.draft_dtype, resident, max_len, stream);
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
  P.t_stats = stats;
  P.d_stats = stats + static_cast<int64_t>(B) * (G + 1);
  P.ids = a.ids;
  P.u_accept = a.u_accept;
  P.u_resample = a.u_resample;
  P.t2d = a.d2t ? a.t2d : nullptr;
  P.out_tokens = a.out_tokens;
  P.num_accepted = a.num_accepted;
  P.p_draft = a.p_draft;
  P.q_draft = a.q_draft;
  P.row_status = a.row_status;
  const bool tb = d.target_dtype == SV_BF16, db = d.draft_dtype == SV_BF16;
  if (tb && db) return launch_decide<uint16_t, uint16_t>(P, stream);
  if (tb) return launch_decide<uint16_t, float>(P, stream);
  if (db) return launch_decide<float, uint16_t>(P, stream);
  return launch_decide<float, float>(P, stream);
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
  sv_status s = launch_stats_sets(L, d.dtype, d.dtype, d.top_p < 1.0f, d.vocab, stream);
  if (s != SV_OK) return s;
  DecideParams P{};
  P.target = logits;
  P.t_stride = d.row_stride;
  P.B = d.rows;
  P.G = 0;
  P.V = d.vocab;
  P.c = L.c;
  P.t_stats = stats;
  P.d_stats = stats;
  P.u_resample = u;
  P.out_tokens = out_tokens;
  P.out_prob = out_prob;
  return d.dtype == SV_BF16 ? launch_decide<uint16_t, uint16_t>(P, stream)
                            : launch_decide<float, float>(P, stream);
}

}  // namespace sv
