// Speculative-sampling verify of draft token trees (T > 0).
//
// Sources: "LLM inference acceleration in practice: draft models and
// speculative sampling explained" §3.1 (one draft per position: accept with
// min(1, p/q), else draw from norm(max(0, p - q)); the bonus token from p)
// and §6.2 (draft and target share T and top_p); "A 2.16x speculative-
// decoding speedup from a 1-layer Llama draft" §5 (the draft token tree).
// The pages give no rule for several drafts at one position.  The rule used
// is sequential per-child rejection with a residual update: at an accepted
// node the residual r starts as p; children are tested in increasing node
// order, child x accepted iff u * q(x) < r(x); a rejection replaces r by
// norm(max(0, r - q)); the first accepted child becomes the node; when every
// child is rejected the last token is drawn from r, at a leaf from p.
//
// After j rejections at a node the residual has the closed form
//   r_j = max(0, p - c_j q) / W_j,  c_0 = 0, W_0 = 1,
//   c_{j+1} = c_j + W_j,  W_{j+1} = sum over ids of max(0, p - c_{j+1} q),
// because max(0, r_j - q) = max(0, p - (c_j + W_j) q) / W_j (where
// p - c_j q <= 0 both sides are 0).  So an accept test needs two logits and
// the scalars (c_j, W_j), and a rejection one pass over the node's target
// and draft rows for W_{j+1}.
//
// Launches: the statistics pass over every target and draft row (the
// streaming kernel, or the top-p kernel when top_p < 1) gives each row its
// exp2 offset, kept mass and top-p cut; then tree_sample_kernel walks each
// tree from the root, one cluster of CS thread blocks per tree (CS = 2 when
// the trees leave SMs idle, else 1).  A pass keeps per-chunk sums of
// max(0, p - c q) in shared memory; the final inverse-CDF draw reuses them
// and rescans only the chunk that holds u * total.  In a cluster every block
// runs the whole walk on the same data and takes the same decisions (the
// same double-precision arithmetic in the same order); only a pass is split:
// block r computes the chunks k = r (mod CS) and stores each chunk sum into
// every block's shared memory, and a cluster barrier ends the pass.
#include "sv_internal.h"
#include "sv_rows.cuh"

namespace sv {

constexpr int kTSThreads = 1024;
constexpr int kTSWarps = kTSThreads / 32;
constexpr int kTSMaxChunks = 256;
constexpr int kTSChunkUnit = 2048;  // ids; chunks are multiples of this

struct TreeSampleParams {
  const void* target;
  int64_t t_stride;
  const void* draft;
  int64_t d_stride;
  const RowStats* ts;  // [B * N] target rows
  const RowStats* ds;  // [B * N] draft rows
  const int32_t* parents;
  const int32_t* tokens;
  const float* u_accept;
  const float* u_final;
  int N, V, D;
  float c;     // log2(e) / T
  int chunk;   // ids per chunk
  int nchunks;
  int32_t* accept_len;
  int32_t* path;
  int32_t* out_tokens;
  int32_t* row_status;
};

// p or q of one row: exp2(l * c - mc) / K over the ids kept by (tau, cut)
// (tau = 0: every id).
struct RowDist {
  float mc, invK;
  uint32_t tau;
  int32_t cut;
  template <bool FILTERED = true>
  __device__ __forceinline__ float at(float l, int j, float c) const {
    if (FILTERED && !kept(order_key(l), j, tau, cut)) return 0.0f;
    return weight(l, c, mc) * invK;
  }
};

// p(x) of one id in double: exp2(l * c - mc) / K over the kept ids.
__device__ __forceinline__ double exact_prob(const RowDist& d, float l, int j, float c, double K) {
  if (d.tau != 0u && !kept(order_key(l), j, d.tau, d.cut)) return 0.0;
  if (!(K > 0.0) || !(l > -CUDART_INF_F)) return 0.0;
  return exp2(static_cast<double>(l) * static_cast<double>(c) - static_cast<double>(d.mc)) / K;
}

template <typename E>
struct NodeRows {
  const E* lt;
  const E* ld;
  RowDist p, q;
  bool vec;  // both rows start on a 16-byte boundary
};

struct TSShared {
  int first_child[SV_MAX_TREE_NODES];
  int next_sib[SV_MAX_TREE_NODES];
  int depth[SV_MAX_TREE_NODES];
  // Node n's accept test as a child of its parent, for every n > 0 (the
  // test does not depend on the path the walk takes): p(x_n) and q(x_n)
  // under the parent's rows, and the node's uniform.
  double test[SV_MAX_TREE_NODES][3];
  double chunk_sum[kTSMaxChunks];
  double red[32];
  double warp_before[32];  // the draw: prefix of the warps before each
  double tile_total;
  RowDist pd[2];
  double bcast_d;
  int bcast_i;
  int hit;
  int last_pos;
  uint32_t status;
};

// The coefficient c_j of the residual as an unevaluated sum of two floats,
// hi + lo == c_j to about 2^-48 relative, so that p - c_j q keeps the
// precision of p and q where they nearly cancel.
struct Coef {
  float hi, lo;
};
__device__ __forceinline__ Coef split_coef(double c) {
  Coef k;
  k.hi = static_cast<float>(c);
  k.lo = static_cast<float>(c - static_cast<double>(k.hi));
  return k;
}

// max(0, p - cj q) of id j: two fused multiply-adds with cj = hi + lo.
template <typename E, bool FILTERED = true>
__device__ __forceinline__ float resid(const NodeRows<E>& R, float lt, float ld, int j, float c, Coef cj) {
  const float q = R.q.template at<FILTERED>(ld, j, c);
  return fmaxf(0.0f, fmaf(-cj.lo, q, fmaf(-cj.hi, q, R.p.template at<FILTERED>(lt, j, c))));
}

// Sum of max(0, p - cj q) over [j0, j1) by one warp: 16-byte loads with four
// vectors of each row in flight per lane when both rows are aligned; the
// draft row is not read when cj == 0 (the weights are p).  Each lane sums in
// fp32 (at most a chunk's share of the ids); the caller adds the lanes in
// double.
template <typename E, bool FILTERED, bool PONLY>
__device__ __forceinline__ float chunk_residual(const NodeRows<E>& R, int j0, int j1, float c, Coef cj) {
  constexpr int EPV = Elem<E>::kPerVec;
  constexpr int U = 4;
  const int lane = threadIdx.x & 31;
  float s = 0.0f;
  auto one = [&](float lt, float ld, int j) {
    s += PONLY ? R.p.template at<FILTERED>(lt, j, c) : resid<E, FILTERED>(R, lt, ld, j, c, cj);
  };
  int tail = j0;
  if (R.vec) {
    // j0 is a multiple of 2048 ids, so a 16-byte boundary of both rows.
    const int nv = (j1 - j0) / EPV;
    const uint4* vt = reinterpret_cast<const uint4*>(R.lt + j0);
    const uint4* vd = reinterpret_cast<const uint4*>(R.ld + j0);
    int v = lane;
    for (; v + (U - 1) * 32 < nv; v += U * 32) {
      uint4 a[U], b[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        a[u] = __ldg(vt + v + u * 32);
        if (!PONLY) b[u] = __ldg(vd + v + u * 32);
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int e = 0; e < EPV; ++e)
          one(Elem<E>::at(a[u], e), PONLY ? 0.0f : Elem<E>::at(b[u], e), j0 + (v + u * 32) * EPV + e);
    }
    for (; v < nv; v += 32) {
      const uint4 a = __ldg(vt + v);
      const uint4 b = PONLY ? a : __ldg(vd + v);
#pragma unroll
      for (int e = 0; e < EPV; ++e) one(Elem<E>::at(a, e), Elem<E>::at(b, e), j0 + v * EPV + e);
    }
    tail = j0 + nv * EPV;
  }
  for (int j = tail + lane; j < j1; j += 32)
    one(Elem<E>::load(R.lt + j), PONLY ? 0.0f : Elem<E>::load(R.ld + j), j);
  return s;
}

// One pass over the node's rows: chunk_sum[k] = sum of max(0, p - cj q) over
// chunk k (one warp per chunk, fp32 per lane, double across lanes); returns
// the row total (double, the same in every thread).
template <typename E, int CS>
__device__ double residual_pass(const NodeRows<E>& R, const TreeSampleParams& P, Coef cj, TSShared& sh) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool filtered = (R.p.tau | R.q.tau) != 0u;
  int rank = 0;
  if constexpr (CS > 1) {
    // No block writes into another's chunk sums before every block of the
    // cluster is done reading the previous pass's (every block makes the
    // same sequence of passes, so the barriers pair up).
    rank = static_cast<int>(cg::this_cluster().block_rank());
    cg::this_cluster().sync();
  }
  for (int k = rank + CS * warp; k < P.nchunks; k += CS * kTSWarps) {
    const int j0 = k * P.chunk, j1 = min(P.V, j0 + P.chunk);
    float s;
    if (cj.hi == 0.0f)
      s = filtered ? chunk_residual<E, true, true>(R, j0, j1, P.c, cj) : chunk_residual<E, false, true>(R, j0, j1, P.c, cj);
    else
      s = filtered ? chunk_residual<E, true, false>(R, j0, j1, P.c, cj)
                   : chunk_residual<E, false, false>(R, j0, j1, P.c, cj);
    const double t = warp_sum_d(static_cast<double>(s));
    if (lane == 0) {
      if constexpr (CS > 1) {
        cg::cluster_group cl = cg::this_cluster();
#pragma unroll
        for (int r = 0; r < CS; ++r) *cl.map_shared_rank(&sh.chunk_sum[k], r) = t;
      } else {
        sh.chunk_sum[k] = t;
      }
    }
  }
  if constexpr (CS > 1) cg::this_cluster().sync();  // every block holds every chunk sum
  else __syncthreads();
  if (warp == 0) {
    double t = 0.0;
    for (int k = lane; k < P.nchunks; k += 32) t += sh.chunk_sum[k];
    t = warp_sum_d(t);
    if (lane == 0) sh.bcast_d = t;
  }
  __syncthreads();
  return sh.bcast_d;
}

// Inverse CDF over max(0, p - cj q) with the chunk sums of the last pass:
// the first id whose inclusive prefix exceeds u * total, in ascending id;
// if rounding leaves u * total at or above the last prefix, the last id of
// positive weight.
template <typename E>
__device__ int draw(const NodeRows<E>& R, const TreeSampleParams& P, Coef cj, double total, float u,
                    TSShared& sh) {
  const double target = static_cast<double>(u) * total;
  if (threadIdx.x < 32) {
    // Lane l owns a contiguous run of chunks; a warp scan of the run totals
    // finds the run, then its owner walks it.
    const int lane = threadIdx.x;
    const int per = (P.nchunks + 31) / 32;
    const int k0 = min(P.nchunks, lane * per), k1 = min(P.nchunks, k0 + per);
    double run = 0.0;
    int lastpos = -1;
    for (int k = k0; k < k1; ++k) {
      run += sh.chunk_sum[k];
      if (sh.chunk_sum[k] > 0.0) lastpos = k;
    }
    double incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const double excl = incl - run;
    const unsigned cross = __ballot_sync(0xffffffffu, incl > target && run > 0.0);
    const int last_lane = 31 - __clz(__ballot_sync(0xffffffffu, lastpos >= 0) | 1u);
    const int last_chunk = __shfl_sync(0xffffffffu, lastpos, last_lane);
    if (cross) {
      const int owner = __ffs(cross) - 1;
      if (lane == owner) {
        double before = excl;
        int k = k0;
        for (; k < k1 - 1; ++k) {
          if (before + sh.chunk_sum[k] > target && sh.chunk_sum[k] > 0.0) break;
          before += sh.chunk_sum[k];
        }
        sh.bcast_i = k;
        sh.bcast_d = before;
      }
    } else if (lane == 0) {
      sh.bcast_i = last_chunk;  // rounding: the last chunk of positive weight
      sh.bcast_d = -1.0;
    }
    if (lane == 0) {
      sh.hit = INT32_MAX;
      sh.last_pos = -1;
    }
  }
  __syncthreads();
  if (sh.bcast_i < 0) return -1;  // no positive weight (excluded by the callers)
  const int k = sh.bcast_i;
  double before = sh.bcast_d;
  const bool rounding = before < 0.0;
  const int j0 = k * P.chunk, j1 = min(P.V, j0 + P.chunk);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Tiles of 2 * kTSThreads ids, thread t holding ids 2t and 2t + 1 (ids
  // ascend with the thread index): a warp scan of the pairs, one warp's
  // scan of the warp totals, then the first id whose inclusive prefix
  // exceeds u * total.
  for (int t0 = j0; t0 < j1; t0 += 2 * kTSThreads) {
    const int ja = t0 + 2 * static_cast<int>(threadIdx.x), jb = ja + 1;
    const float wa = ja < j1 ? resid(R, Elem<E>::load(R.lt + ja), Elem<E>::load(R.ld + ja), ja, P.c, cj) : 0.0f;
    const float wb = jb < j1 ? resid(R, Elem<E>::load(R.lt + jb), Elem<E>::load(R.ld + jb), jb, P.c, cj) : 0.0f;
    const double mine = static_cast<double>(wa) + static_cast<double>(wb);
    double incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) sh.red[warp] = incl;
    if (wb > 0.0f) atomicMax(&sh.last_pos, jb);
    else if (wa > 0.0f) atomicMax(&sh.last_pos, ja);
    __syncthreads();
    if (warp == 0) {
      const double t = lane < kTSWarps ? sh.red[lane] : 0.0;
      double c = t;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, c, o);
        if (lane >= o) c += y;
      }
      sh.warp_before[lane] = c - t;
      if (lane == 31) sh.tile_total = c;
    }
    __syncthreads();
    if (!rounding) {
      const double ex = before + sh.warp_before[warp] + (incl - mine);  // before id ja
      if (wa > 0.0f && ex + wa > target) atomicMin(&sh.hit, ja);
      else if (wb > 0.0f && ex + static_cast<double>(wa) + wb > target) atomicMin(&sh.hit, jb);
    }
    __syncthreads();
    if (sh.hit != INT32_MAX) break;
    before += sh.tile_total;
  }
  return sh.hit != INT32_MAX ? sh.hit : sh.last_pos;
}

template <typename E, int CS>
__global__ void __launch_bounds__(kTSThreads) tree_sample_kernel(TreeSampleParams P) {
  __shared__ TSShared sh;
  const int b = blockIdx.x / CS;
  // Only the first block of a tree's cluster writes the tree's outputs (the
  // others hold the same values).
  bool writer = true;
  if constexpr (CS > 1) writer = cg::this_cluster().block_rank() == 0;
  const int N = P.N;
  const int64_t base = static_cast<int64_t>(b) * N;
  const int32_t* par = P.parents + base;
  const int32_t* tok = P.tokens + base;
  const int L = P.D + 1;
  if (threadIdx.x == 0) sh.status = 0;
  __syncthreads();
  uint32_t st = 0;
  for (int n = threadIdx.x; n < N; n += kTSThreads) {
    const int p = par[n];
    if (n == 0 ? p != -1 : (p < 0 || p >= n)) st |= SV_ROW_BAD_PARENT;
    if (n > 0 && (tok[n] < 0 || tok[n] >= P.V)) st |= SV_ROW_BAD_TOKEN;
    if ((P.ts[base + n].status | P.ds[base + n].status) & SV_ROW_EMPTY) st |= SV_ROW_EMPTY;
    sh.first_child[n] = -1;
    sh.next_sib[n] = -1;
  }
  if (st) atomicOr(&sh.status, st);
  __syncthreads();
  if (threadIdx.x == 0 && !(sh.status & SV_ROW_BAD_PARENT)) {
    // Children lists in increasing node order, and depths (parents[n] < n).
    uint32_t s = 0;
    sh.depth[0] = 0;
    for (int n = 1; n < N; ++n) {
      sh.depth[n] = sh.depth[par[n]] + 1;
      if (sh.depth[n] > P.D) s |= SV_ROW_DEPTH_EXCEEDED;
    }
    for (int n = N - 1; n >= 1; --n) {
      sh.next_sib[n] = sh.first_child[par[n]];
      sh.first_child[par[n]] = n;
    }
    sh.status |= s;
  }
  __syncthreads();
  uint32_t status = sh.status;
  int32_t* path = P.path + static_cast<int64_t>(b) * L;
  int32_t* out = P.out_tokens + static_cast<int64_t>(b) * L;
  if (status) {
    for (int i = threadIdx.x; writer && i < L; i += kTSThreads) {
      path[i] = -1;
      out[i] = -1;
    }
    if (writer && threadIdx.x == 0) {
      P.accept_len[b] = 0;
      if (P.row_status) P.row_status[b] = static_cast<int32_t>(status);
    }
    return;
  }

  const E* tgt = static_cast<const E*>(P.target);
  const E* dft = static_cast<const E*>(P.draft);
  // Every node's accept test inputs, all loads in flight together: p(x) and
  // q(x) from the parent rows' offsets and kept masses with the
  // double-precision exp2, and the node's uniform.
  for (int i = threadIdx.x; i < 3 * (N - 1); i += kTSThreads) {
    const int n = 1 + i / 3, which = i - 3 * (n - 1);
    double v = 0.0;
    if (which == 2) {
      v = static_cast<double>(P.u_accept[base + n]);
    } else {
      const int64_t prow = base + par[n];
      const int x = tok[n];
      const RowStats st = which == 0 ? P.ts[prow] : P.ds[prow];
      RowDist r;
      r.mc = st.mc;
      r.invK = 0.0f;
      r.tau = st.tau;
      r.cut = st.cut;
      if (sv_in(x, P.V))
        v = exact_prob(r, which == 0 ? Elem<E>::load(tgt + prow * P.t_stride + x) : Elem<E>::load(dft + prow * P.d_stride + x),
                       x, P.c, st.K);
    }
    sh.test[n][which] = v;
  }
  __syncthreads();
  int node = 0, d = 0;
  if (writer && threadIdx.x == 0) path[0] = 0;
  // Every iteration either moves one level down (parents[n] < n and depths
  // <= D were checked above) or returns: at most D + 1 iterations.
  for (;;) {
    const int64_t row = base + node;
    if (threadIdx.x < 2) {
      const RowStats s = threadIdx.x == 0 ? P.ts[row] : P.ds[row];
      RowDist r;
      r.mc = s.mc;
      r.invK = s.K > 0.0 ? static_cast<float>(1.0 / s.K) : 0.0f;
      r.tau = s.tau;
      r.cut = s.cut;
      sh.pd[threadIdx.x] = r;
    }
    __syncthreads();
    NodeRows<E> R;
    R.lt = tgt + row * P.t_stride;
    R.ld = dft + row * P.d_stride;
    R.p = sh.pd[0];
    R.q = sh.pd[1];
    R.vec = ((reinterpret_cast<uintptr_t>(R.lt) | reinterpret_cast<uintptr_t>(R.ld)) & 15u) == 0;
    double cj = 0.0, W = 1.0;
    bool sums_for_cj = false;  // chunk sums of the current residual are in shared memory
    int next = -1;
    for (int ch = sh.first_child[node]; ch >= 0; ch = sh.next_sib[ch]) {
      const double p = sh.test[ch][0], q = sh.test[ch][1], u = sh.test[ch][2];
      // Every thread evaluates the same test on the same values.
      if (u * q * W < fmax(0.0, p - cj * q)) {
        next = ch;
        break;
      }
      const double c_new = cj + W;
      const double W_new = residual_pass<E, CS>(R, P, split_coef(c_new), sh);
      if (W_new > 0.0) {
        cj = c_new;
        W = W_new;
        sums_for_cj = true;
      } else {
        status |= SV_ROW_RESAMPLE_FALLBACK;  // r kept; its sums are not in shared memory
        sums_for_cj = false;
      }
    }
    if (next >= 0) {
      node = next;
      ++d;
      if (writer && threadIdx.x == 0 && sv_in(d, L)) {
        path[d] = node;
        out[d - 1] = tok[node];
      }
      continue;
    }
    double total = sums_for_cj ? W : residual_pass<E, CS>(R, P, split_coef(cj), sh);
    const int y = draw(R, P, split_coef(cj), total, P.u_final[b], sh);
    if (writer && threadIdx.x == 0) {
      out[d] = y;
      P.accept_len[b] = d;
      if (P.row_status) P.row_status[b] = static_cast<int32_t>(status);
    }
    for (int i = d + 1 + threadIdx.x; writer && i < L; i += kTSThreads) {
      path[i] = -1;
      out[i] = -1;
    }
    return;
  }
}

size_t tree_sample_workspace_bytes(const sv_tree_sample_desc& d) {
  const size_t rows = static_cast<size_t>(d.batch) * d.nodes;
  size_t n = 2 * align_up(rows * sizeof(RowStats), 256);
  if (d.top_p < 1.0f) n += align_up(topp_scratch_bytes(static_cast<int>(rows), d.vocab, static_cast<int>(rows), d.vocab), 256);
  return n + 256;
}

sv_status tree_sample(const sv_tree_sample_desc& d, const void* target, const void* draft,
                      const int32_t* parents, const int32_t* tokens, const float* u_accept,
                      const float* u_final, int32_t* accept_len, int32_t* path, int32_t* out_tokens,
                      int32_t* row_status, void* workspace, cudaStream_t stream) {
  if (d.batch == 0) return SV_OK;
  const int rows = d.batch * d.nodes;
  RowStats* ts = static_cast<RowStats*>(workspace);
  RowStats* ds = reinterpret_cast<RowStats*>(static_cast<char*>(workspace) +
                                             align_up(static_cast<size_t>(rows) * sizeof(RowStats), 256));
  void* scratch = static_cast<char*>(workspace) + 2 * align_up(static_cast<size_t>(rows) * sizeof(RowStats), 256);
  StatsLaunch L{};
  L.c = static_cast<float>(1.4426950408889634 / static_cast<double>(d.temperature));
  L.top_p = d.top_p;
  L.nsets = 2;
  const void* bases[2] = {target, draft};
  const int64_t strides[2] = {d.target_row_stride, d.draft_row_stride};
  RowStats* outs[2] = {ts, ds};
  for (int i = 0; i < 2; ++i) {
    RowSet& S = L.set[i];
    S.base = bases[i];
    S.stride = strides[i];
    S.len = d.vocab;
    S.rows = rows;
    S.per_group = 1;
    S.gamma = 0;
    S.last_no_query = true;
    S.ids = nullptr;
    S.vocab = d.vocab;
    S.out = outs[i];
  }
  start_phases(stream);
  sv_status s = launch_stats_sets(L, d.dtype, d.dtype, d.top_p < 1.0f, scratch, stream);
  if (s != SV_OK) return s;
  TreeSampleParams P{};
  P.target = target;
  P.t_stride = d.target_row_stride;
  P.draft = draft;
  P.d_stride = d.draft_row_stride;
  P.ts = ts;
  P.ds = ds;
  P.parents = parents;
  P.tokens = tokens;
  P.u_accept = u_accept;
  P.u_final = u_final;
  P.N = d.nodes;
  P.V = d.vocab;
  P.D = d.max_depth;
  P.c = L.c;
  const int units = (d.vocab + kTSChunkUnit - 1) / kTSChunkUnit;
  const int per = (units + kTSMaxChunks - 1) / kTSMaxChunks;
  P.chunk = per * kTSChunkUnit;
  P.nchunks = (d.vocab + P.chunk - 1) / P.chunk;
  P.accept_len = accept_len;
  P.path = path;
  P.out_tokens = out_tokens;
  P.row_status = row_status;
  // A cluster of two blocks per tree while the trees leave SMs idle.
  static std::atomic<int> sms[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  int nsm = sms[dev].load(std::memory_order_relaxed);
  if (nsm == 0) {
    if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || nsm <= 0) nsm = 148;
    sms[dev].store(nsm, std::memory_order_relaxed);
  }
  const bool pair = 2LL * d.batch <= nsm;
  const bool bf = d.dtype == SV_BF16;
  if (pair) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * d.batch));
    cfg.blockDim = dim3(kTSThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = bf ? cudaLaunchKernelEx(&cfg, tree_sample_kernel<uint16_t, 2>, P)
                             : cudaLaunchKernelEx(&cfg, tree_sample_kernel<float, 2>, P);
    if (e != cudaSuccess) return SV_ERR_CUDA;
  } else if (bf) {
    tree_sample_kernel<uint16_t, 1><<<d.batch, kTSThreads, 0, stream>>>(P);
  } else {
    tree_sample_kernel<float, 1><<<d.batch, kTSThreads, 0, stream>>>(P);
  }
  if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  note_launch(stream);
  return SV_OK;
}

}  // namespace sv
