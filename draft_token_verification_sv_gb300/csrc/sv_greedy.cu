// Greedy (temperature 0) verify: argmax of every target row, then the
// per-group decision (chain prefix match or tree walk) by the last block of
// the group to finish, all in one launch.  One block streams a whole row
// when there are enough rows to fill the GPU; for small batches a row is cut
// into segments (one block each) so that every SM gets work: each segment
// block folds its packed (value, lowest index) maximum into the row's word
// with a 64-bit atomicMax, and the row's last segment block goes on with the
// row's result.
//
// Sources: "SSD: extending the engine with new models and an EAGLE3 draft"
// §七 (--temp 0 benchmarking); "A 2.16x speculative-decoding speedup from a
// 1-layer Llama draft", headline table ("Match = True": greedy speculative
// output equals greedy decoding) and §5 (draft token tree).
#include <cuda_bf16.h>

#include "sv_internal.h"

namespace sv {

enum class GreedyMode : int { kChain = 0, kTree = 1, kSample = 2 };

struct GreedyParams {
  const void* logits;
  int64_t stride;
  int V;
  int rows_per_group;  // γ+1 (chain), N (tree), 1 (sample)
  int groups;
  int32_t* g;          // [rows] argmax per row, -1 for a row with no finite logit
  unsigned int* counters;  // [groups], zero before the launch
  int nseg;                // segment blocks per row
  unsigned long long* rowmax;  // [rows] packed row maxima (nseg > 1), zero before the launch
  unsigned int* segcnt;        // [rows] finished segment blocks (nseg > 1), zero before the launch
  // chain
  const int32_t* draft_ids;
  int32_t* out_tokens;
  int32_t* num_accepted;
  float* p_draft;
  float* q_draft;
  int32_t* row_status;
  // tree
  const int32_t* parents;
  const int32_t* tokens;
  int32_t* accept_len;
  int32_t* path;
  int max_depth;
  // sample
  float* out_prob;
};

// The largest logit of one 16-byte vector (bf16: packed maxima, two logits
// per instruction; fp32: three-input maxima).  A NaN never hides a number,
// as with fmaxf.
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
    float m;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(m) : "f"(__uint_as_float(w.x)), "f"(__uint_as_float(w.y)),
        "f"(__uint_as_float(w.z)));
    return fmaxf(m, __uint_as_float(w.w));
  }
}

// Largest value with the lowest index over one row, packed (see argmax_pack);
// the result is valid in every thread.
// Segment `seg` of `nseg` covers an equal share of whole loop steps
// (THREADS * UNROLL 16-byte vectors) of the body, the last one to the end of
// the row; segment 0 adds the scalar head and the last segment the tail.
template <typename E, int THREADS, int UNROLL>
__device__ __forceinline__ unsigned long long row_argmax(const E* row, int V, int seg, int nseg,
                                                         unsigned long long* scratch) {
  constexpr int EPV = Elem<E>::kPerVec;
  constexpr int kStep = THREADS * UNROLL;
  const RowSplit rs = split_row(row, V);
  const int per_seg = ((rs.nvec + kStep - 1) / kStep + nseg - 1) / nseg;  // steps per segment
  const int v_lo = min(rs.nvec, seg * per_seg * kStep);
  const int nvec = seg == nseg - 1 ? rs.nvec : min(rs.nvec, v_lo + per_seg * kStep);
  const uint4* vp = reinterpret_cast<const uint4*>(row + rs.head);
  float bv = -CUDART_INF_F;
  int bi = 0x7fffffff;
  // Each thread visits its ids in increasing order (head, body, tail), so a
  // strict '>' keeps the lowest id among equal values.
  if (seg == 0 && static_cast<int>(threadIdx.x) < rs.head) {
    const float x = Elem<E>::load(row + threadIdx.x);
    if (x > bv) {
      bv = x;
      bi = threadIdx.x;
    }
  }
  for (int v0 = v_lo + static_cast<int>(threadIdx.x); v0 < nvec; v0 += kStep) {
    uint4 buf[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int v = v0 + u * THREADS;
      buf[u] = v < nvec ? ldg_stream(vp + v) : Elem<E>::neg_inf_vec();
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      // The vector's maximum by packed maxima (bf16: two logits per
      // instruction); its lowest index only when it beats the running one.
      const float vm = vec_max<E>(buf[u]);
      if (vm > bv) {
        float x[EPV];
        unpack<E>(buf[u], x);
        int first = EPV - 1;
#pragma unroll
        for (int i = EPV - 1; i >= 0; --i)
          if (x[i] == vm) first = i;
        bv = vm;
        bi = rs.head + (v0 + u * THREADS) * EPV + first;
      }
    }
  }
  const int tail = rs.tail0 + static_cast<int>(threadIdx.x);
  if (seg == nseg - 1 && tail < V) {
    const float x = Elem<E>::load(row + tail);
    if (x > bv) {
      bv = x;
      bi = tail;
    }
  }
  // A thread that saw only -inf proposes index 0 (np.argmax convention).
  const unsigned long long packed = bi == 0x7fffffff ? argmax_pack(-CUDART_INF_F, 0)
                                                     : argmax_pack(bv, bi);
  return block_max_u64<THREADS>(packed, scratch);
}

template <int THREADS>
__device__ void chain_decide(const GreedyParams& P, int b) {
  // Single thread: γ <= 64 comparisons.
  if (threadIdx.x != 0) return;
  const int G = P.rows_per_group - 1;
  const int32_t* g = P.g + static_cast<int64_t>(b) * (G + 1);
  const int32_t* ids = P.draft_ids + static_cast<int64_t>(b) * G;
  int32_t* out = P.out_tokens + static_cast<int64_t>(b) * (G + 1);
  uint32_t status = 0;
  for (int i = 0; i < G; ++i) {
    const int x = ids[i];
    if (x < 0 || x >= P.V) status |= SV_ROW_BAD_DRAFT_ID;
  }
  for (int i = 0; i <= G; ++i)
    if (__ldcg(g + i) < 0) status |= SV_ROW_EMPTY;
  int k = 0;
  if (!status) {
    k = G;
    for (int i = 0; i < G; ++i) {
      if (ids[i] != __ldcg(g + i)) {
        k = i;
        break;
      }
    }
    for (int i = 0; i < k; ++i) out[i] = ids[i];
    out[k] = __ldcg(g + k);
    for (int i = k + 1; i <= G; ++i) out[i] = -1;
  } else {
    for (int i = 0; i <= G; ++i) out[i] = -1;
  }
  P.num_accepted[b] = k;
  if (P.row_status) P.row_status[b] = static_cast<int32_t>(status);
  if (P.p_draft)
    for (int i = 0; i < G; ++i) P.p_draft[static_cast<int64_t>(b) * G + i] = 0.0f;
  if (P.q_draft)
    for (int i = 0; i < G; ++i) P.q_draft[static_cast<int64_t>(b) * G + i] = 0.0f;
}

template <int THREADS>
__device__ void tree_walk(const GreedyParams& P, int b) {
  // Nodes are handled in a block-strided loop (N <= SV_MAX_TREE_NODES).
  __shared__ int s_par[SV_MAX_TREE_NODES];
  __shared__ int s_tok[SV_MAX_TREE_NODES];
  __shared__ int s_g[SV_MAX_TREE_NODES];
  __shared__ int s_depth[SV_MAX_TREE_NODES];
  __shared__ unsigned char s_acc[SV_MAX_TREE_NODES];
  __shared__ unsigned int s_status;
  __shared__ unsigned long long s_red[32];
  const int N = P.rows_per_group;
  const int D = P.max_depth;
  const int64_t base = static_cast<int64_t>(b) * N;
  if (threadIdx.x == 0) s_status = 0;
  __syncthreads();
  for (int n = threadIdx.x; n < N; n += THREADS) {
    const int par = P.parents[base + n];
    const int tok = P.tokens[base + n];
    const int gv = __ldcg(P.g + base + n);
    s_par[n] = par;
    s_tok[n] = tok;
    s_g[n] = gv;
    s_acc[n] = n == 0 ? 1 : 0;
    s_depth[n] = 0;
    uint32_t st = 0;
    if (n == 0 ? par != -1 : (par < 0 || par >= n)) st |= SV_ROW_BAD_PARENT;
    if (n > 0 && (tok < 0 || tok >= P.V)) st |= SV_ROW_BAD_TOKEN;
    if (gv < 0) st |= SV_ROW_EMPTY;
    if (st) atomicOr(&s_status, st);
  }
  __syncthreads();
  if (!(s_status & SV_ROW_BAD_PARENT)) {
    for (int n = threadIdx.x; n < N; n += THREADS) {
      // parents[m] < m: the walk reaches the root; D+1 steps are enough to
      // tell that a node is deeper than D.
      int d = 0, cur = n;
      for (int step = 0; step <= D && cur > 0; ++step) {
        cur = s_par[cur];
        ++d;
      }
      if (cur > 0) atomicOr(&s_status, SV_ROW_DEPTH_EXCEEDED);
      s_depth[n] = d;
    }
  }
  __syncthreads();
  const uint32_t status = s_status;
  int32_t* out = P.out_tokens + static_cast<int64_t>(b) * (D + 1);
  int32_t* path = P.path + static_cast<int64_t>(b) * (D + 1);
  if (status) {
    for (int d = threadIdx.x; d <= D; d += THREADS) {
      out[d] = -1;
      path[d] = -1;
    }
    if (threadIdx.x == 0) {
      P.accept_len[b] = 0;
      if (P.row_status) P.row_status[b] = static_cast<int32_t>(status);
    }
    return;
  }
  // Level by level: a node is accepted iff its parent is and its token is
  // the argmax of the parent's row.
  for (int lvl = 1; lvl <= D; ++lvl) {
    __syncthreads();
    for (int n = threadIdx.x; n < N; n += THREADS)
      if (s_depth[n] == lvl) {
        const int par = s_par[n];
        s_acc[n] = (sv_in(par, N) && s_acc[par] && s_tok[n] == s_g[par]) ? 1 : 0;
      }
  }
  __syncthreads();
  unsigned long long key = 0;
  for (int n = threadIdx.x; n < N; n += THREADS)
    if (s_acc[n]) {
      const unsigned long long k =
          (static_cast<unsigned long long>(s_depth[n]) << 32) | (0xffffffffu - static_cast<uint32_t>(n));
      key = k > key ? k : key;
    }
  key = block_max_u64<THREADS>(key, s_red);
  const int best = static_cast<int>(0xffffffffu - static_cast<uint32_t>(key & 0xffffffffull));
  const int L = static_cast<int>(key >> 32);
  if (threadIdx.x == 0 && sv_in(best, N) && sv_in(L, D + 1)) {
    int cur = best;
    for (int d = L; d >= 0; --d) {  // L <= D steps
      if (!sv_in(cur, N)) break;
      path[d] = cur;
      if (d > 0) out[d - 1] = s_tok[cur];
      if (d > 0) cur = s_par[cur];
    }
    out[L] = s_g[best];
    for (int d = L + 1; d <= D; ++d) {
      path[d] = -1;
      out[d] = -1;
    }
    P.accept_len[b] = L;
    if (P.row_status) P.row_status[b] = 0;
  }
}

template <typename E, int THREADS, int UNROLL, GreedyMode MODE>
__global__ void __launch_bounds__(THREADS) greedy_kernel(GreedyParams P) {
  __shared__ unsigned long long s_red[32];
  __shared__ bool s_seg_last, s_last;
  const int row = blockIdx.x / P.nseg;
  const int seg = blockIdx.x - row * P.nseg;
  const E* rp = reinterpret_cast<const E*>(P.logits) + static_cast<int64_t>(row) * P.stride;
  unsigned long long best = row_argmax<E, THREADS, UNROLL>(rp, P.V, seg, P.nseg, s_red);
  if (P.nseg > 1) {
    // Fold into the row's maximum; the row's last segment block goes on.
    if (threadIdx.x == 0) {
      atomicMax(P.rowmax + row, best);
      __threadfence();
      s_seg_last = atomicAdd(P.segcnt + row, 1u) == static_cast<unsigned>(P.nseg - 1);
    }
    __syncthreads();
    if (!s_seg_last) return;
    __threadfence();
    best = __ldcg(P.rowmax + row);
  }
  const bool empty = (best >> 32) == static_cast<unsigned long long>(order_key(-CUDART_INF_F));
  const int idx = empty ? -1 : argmax_index(best);
  if constexpr (MODE == GreedyMode::kSample) {
    if (threadIdx.x == 0) {
      P.out_tokens[row] = empty ? -1 : idx;
      if (P.out_prob) P.out_prob[row] = empty ? 0.0f : 1.0f;
    }
    return;
  } else {
    const int group = row / P.rows_per_group;
    if (threadIdx.x == 0) {
      P.g[row] = idx;
      __threadfence();
      const unsigned int prev = atomicAdd(P.counters + group, 1u);
      s_last = prev == static_cast<unsigned int>(P.rows_per_group - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if constexpr (MODE == GreedyMode::kChain) chain_decide<THREADS>(P, group);
    else tree_walk<THREADS>(P, group);
  }
}

constexpr int kGThreads = 512;
constexpr int kGUnroll = 8;

// Segment blocks per row: 1 when the rows alone give every SM two blocks
// (measured: splitting rows then only adds the per-block reduction and
// atomics), else up to one segment per loop step so that small batches
// still spread over the GPU.
template <typename E>
static int greedy_segments(int rows, int V) {
  static std::atomic<int> sms[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  int n = sms[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    sms[dev].store(n, std::memory_order_relaxed);
  }
  const long long want = 2LL * n;
  if (rows <= 0 || rows >= want) return 1;
  constexpr int step = kGThreads * kGUnroll;
  const int max_seg = std::max(1, V / Elem<E>::kPerVec / step);
  return static_cast<int>(std::min<long long>(max_seg, (want + rows - 1) / rows));
}

// rows x nseg blocks; P.counters, P.rowmax and P.segcnt zeroed by the caller.
template <typename E, GreedyMode MODE>
static sv_status launch_greedy(const GreedyParams& P, int rows, cudaStream_t stream) {
  if (rows == 0) return SV_OK;
  const long long blocks = static_cast<long long>(rows) * P.nseg;
  if (blocks > INT32_MAX) return SV_ERR_UNSUPPORTED;
  greedy_kernel<E, kGThreads, kGUnroll, MODE><<<static_cast<unsigned>(blocks), kGThreads, 0, stream>>>(P);
  if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  note_launch(stream);
  return SV_OK;
}

sv_status greedy_chain(const sv_chain_desc& d, const void* target, const int32_t* ids,
                       int32_t* out_tokens, int32_t* num_accepted, float* p_draft, float* q_draft,
                       int32_t* row_status, void* workspace, cudaStream_t stream) {
  const int rows = d.batch * (d.gamma + 1);
  GreedyParams P{};
  P.logits = target;
  P.stride = d.target_row_stride;
  P.V = d.vocab;
  P.rows_per_group = d.gamma + 1;
  P.groups = d.batch;
  WorkspaceLayout L = chain_workspace_layout(d);
  char* ws = static_cast<char*>(workspace);
  P.counters = reinterpret_cast<unsigned int*>(ws + L.counters);
  // The row maxima and segment counters live in the statistics region,
  // which the greedy path does not otherwise use (12 bytes per row against
  // 32 per statistics row).
  P.nseg = d.target_dtype == SV_BF16 ? greedy_segments<uint16_t>(rows, d.vocab) : greedy_segments<float>(rows, d.vocab);
  P.rowmax = reinterpret_cast<unsigned long long*>(ws + L.stats);
  P.segcnt = reinterpret_cast<unsigned int*>(ws + L.stats + static_cast<size_t>(rows) * sizeof(unsigned long long));
  // The workspace is scratch shared with other calls: clear the counters
  // (and the row maxima) in one go.
  start_phases(stream);
  const size_t clear = P.nseg > 1 ? L.stats + static_cast<size_t>(rows) * 12 : static_cast<size_t>(d.batch) * 4;
  if (cudaMemsetAsync(ws, 0, clear, stream) != cudaSuccess) return SV_ERR_CUDA;
  P.g = reinterpret_cast<int32_t*>(ws + L.argmax);
  P.draft_ids = ids;
  P.out_tokens = out_tokens;
  P.num_accepted = num_accepted;
  P.p_draft = p_draft;
  P.q_draft = q_draft;
  P.row_status = row_status;
  return d.target_dtype == SV_BF16 ? launch_greedy<uint16_t, GreedyMode::kChain>(P, rows, stream)
                                   : launch_greedy<float, GreedyMode::kChain>(P, rows, stream);
}

sv_status greedy_tree(const sv_tree_desc& d, const void* logits, const int32_t* parents,
                      const int32_t* tokens, int32_t* accept_len, int32_t* path,
                      int32_t* out_tokens, int32_t* row_status, void* workspace,
                      cudaStream_t stream) {
  GreedyParams P{};
  P.logits = logits;
  P.stride = d.row_stride;
  P.V = d.vocab;
  P.rows_per_group = d.nodes;
  P.groups = d.batch;
  const int rows = d.batch * d.nodes;
  const TreeGreedyLayout TL = tree_greedy_layout(d.batch, d.nodes);
  char* ws = static_cast<char*>(workspace);
  P.counters = reinterpret_cast<unsigned int*>(ws);
  P.nseg = d.dtype == SV_BF16 ? greedy_segments<uint16_t>(rows, d.vocab) : greedy_segments<float>(rows, d.vocab);
  P.segcnt = reinterpret_cast<unsigned int*>(ws + TL.segcnt);
  P.rowmax = reinterpret_cast<unsigned long long*>(ws + TL.rowmax);
  start_phases(stream);
  // Counters, segment counters and row maxima are contiguous: one clear.
  const size_t clear = P.nseg > 1 ? TL.g : static_cast<size_t>(d.batch) * sizeof(uint32_t);
  if (cudaMemsetAsync(ws, 0, clear, stream) != cudaSuccess) return SV_ERR_CUDA;
  P.g = reinterpret_cast<int32_t*>(ws + TL.g);
  P.parents = parents;
  P.tokens = tokens;
  P.accept_len = accept_len;
  P.path = path;
  P.out_tokens = out_tokens;
  P.row_status = row_status;
  P.max_depth = d.max_depth;
  return d.dtype == SV_BF16 ? launch_greedy<uint16_t, GreedyMode::kTree>(P, rows, stream)
                            : launch_greedy<float, GreedyMode::kTree>(P, rows, stream);
}

sv_status greedy_sample(const sv_sample_desc& d, const void* logits, int32_t* out_tokens,
                        float* out_prob, cudaStream_t stream) {
  GreedyParams P{};
  P.logits = logits;
  P.stride = d.row_stride;
  P.V = d.vocab;
  P.rows_per_group = 1;
  P.groups = d.rows;
  P.nseg = 1;  // no workspace: whole rows
  P.out_tokens = out_tokens;
  P.out_prob = out_prob;
  return d.dtype == SV_BF16 ? launch_greedy<uint16_t, GreedyMode::kSample>(P, d.rows, stream)
                            : launch_greedy<float, GreedyMode::kSample>(P, d.rows, stream);
}

}  // namespace sv
