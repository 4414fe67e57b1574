// Greedy verify of draft token trees that reads only the rows on the
// accepted frontier, level by level, instead of every node row.
//
// Source: "A 2.16x speculative-decoding speedup from a 1-layer Llama draft",
// §5 (draft token tree: total_token nodes, depth, top_k children) and the
// headline table ("Match = True": greedy speculative output equals greedy
// decoding).  Same contract as the all-node verify: a node is accepted when
// its parent is accepted and its token is the argmax of the parent's row
// (lowest id on ties); the result is the deepest accepted node (lowest node
// id among equally deep ones), its root path and the bonus token.
//
// The accepted nodes of depth d (the frontier) are exactly the nodes whose
// rows the next level needs, so level d computes the argmax of the frontier
// rows only: one block per (tree, segment of the row), partial maxima merged
// with a global atomicMax, and the tree's last block of the level builds the
// next frontier (children whose token matches their parent's argmax) or, when
// it is empty, writes the result.  One launch per level (depth 0..D), so no
// block ever waits for another.  Rows off the walked path are never read:
// a row with no finite logit is reported only when the walk reads it.
#include "sv_internal.h"

namespace sv {

constexpr int kWThreads = 256;
constexpr int kWVecs = 8;                     // 16-byte vectors per thread per segment
constexpr int kWSegVec = kWThreads * kWVecs;  // vectors per segment

struct WalkTree {
  int32_t depth;     // depth of the current frontier
  int32_t nf;        // frontier size; 0 once the tree is done
  uint32_t status;   // SV_ROW_* bits
  uint32_t counter;  // segment blocks finished at this level
};

struct WalkParams {
  const void* logits;
  int64_t stride;
  int V, N, D, B, nseg;
  const int32_t* parents;
  const int32_t* tokens;
  int32_t* accept_len;
  int32_t* path;
  int32_t* out_tokens;
  int32_t* row_status;
  WalkTree* trees;               // [B]
  int32_t* frontier;             // [B, N]
  unsigned long long* best;      // [B, N] packed argmax of each node's row
};

__device__ __forceinline__ void write_invalid(const WalkParams& P, int b, uint32_t status) {
  const int L = P.D + 1;
  for (int d = threadIdx.x; d < L; d += blockDim.x) {
    P.path[static_cast<int64_t>(b) * L + d] = -1;
    P.out_tokens[static_cast<int64_t>(b) * L + d] = -1;
  }
  if (threadIdx.x == 0) {
    P.accept_len[b] = 0;
    if (P.row_status) P.row_status[b] = static_cast<int32_t>(status);
  }
}

// One block (32 threads) per tree: validate it and start the walk at the root.
__global__ void __launch_bounds__(32) walk_init_kernel(WalkParams P) {
  const int b = blockIdx.x;
  const int N = P.N, D = P.D;
  const int32_t* par = P.parents + static_cast<int64_t>(b) * N;
  const int32_t* tok = P.tokens + static_cast<int64_t>(b) * N;
  uint32_t st = 0;
  for (int n = threadIdx.x; n < N; n += 32) {
    const int p = par[n];
    if (n == 0 ? p != -1 : (p < 0 || p >= n)) st |= SV_ROW_BAD_PARENT;
    if (n > 0 && (tok[n] < 0 || tok[n] >= P.V)) st |= SV_ROW_BAD_TOKEN;
    P.best[static_cast<int64_t>(b) * N + n] = 0ull;
  }
  st = __reduce_or_sync(0xffffffffu, st);
  if (!(st & SV_ROW_BAD_PARENT)) {
    // parents[m] < m: walking up reaches the root; D+1 steps tell a node
    // deeper than D.
    uint32_t deep = 0;
    for (int n = threadIdx.x; n < N; n += 32) {
      int cur = n;
      for (int step = 0; step <= D && cur > 0; ++step) cur = par[cur];
      if (cur > 0) deep = SV_ROW_DEPTH_EXCEEDED;
    }
    st |= __reduce_or_sync(0xffffffffu, deep);
  }
  if (threadIdx.x == 0) {
    WalkTree t;
    t.depth = 0;
    t.nf = st ? 0 : 1;
    t.status = st;
    t.counter = 0;
    P.trees[b] = t;
    P.frontier[static_cast<int64_t>(b) * N] = 0;
  }
  if (st) write_invalid(P, b, st);
}

// Packed maximum (order key, lowest id) over this block's segment of a row.
template <typename E>
__device__ __forceinline__ unsigned long long segment_argmax(const E* row, int V, int seg, int nseg,
                                                             unsigned long long* scratch) {
  constexpr int EPV = Elem<E>::kPerVec;
  const RowSplit rs = split_row(row, V);
  const uint4* vp = reinterpret_cast<const uint4*>(row + rs.head);
  const int v0 = seg * kWSegVec, v1 = min(rs.nvec, v0 + kWSegVec);
  float bv = -CUDART_INF_F;
  int bi = 0x7fffffff;
  // Ids are visited in increasing order per thread: a strict '>' keeps the
  // lowest id among equal values.
  if (seg == 0 && static_cast<int>(threadIdx.x) < rs.head) {
    const float x = Elem<E>::load(row + threadIdx.x);
    if (x > bv) {
      bv = x;
      bi = threadIdx.x;
    }
  }
  uint4 w[kWVecs];
#pragma unroll
  for (int u = 0; u < kWVecs; ++u) {
    const int v = v0 + static_cast<int>(threadIdx.x) + u * kWThreads;
    w[u] = v < v1 ? ldg_stream(vp + v) : Elem<E>::neg_inf_vec();
  }
#pragma unroll
  for (int u = 0; u < kWVecs; ++u) {
    float x[EPV];
    unpack<E>(w[u], x);
    float vm = x[0];
#pragma unroll
    for (int i = 1; i < EPV; ++i) vm = fmaxf(vm, x[i]);
    if (vm > bv) {
      int first = EPV - 1;
#pragma unroll
      for (int i = EPV - 1; i >= 0; --i)
        if (x[i] == vm) first = i;
      bv = vm;
      bi = rs.head + (v0 + static_cast<int>(threadIdx.x) + u * kWThreads) * EPV + first;
    }
  }
  if (seg == nseg - 1) {
    const int t = rs.tail0 + static_cast<int>(threadIdx.x);
    if (t < V) {
      const float x = Elem<E>::load(row + t);
      if (x > bv) {
        bv = x;
        bi = t;
      }
    }
  }
  const unsigned long long packed = bi == 0x7fffffff ? argmax_pack(-CUDART_INF_F, 0) : argmax_pack(bv, bi);
  return block_max_u64<kWThreads>(packed, scratch);
}

template <typename E>
__global__ void __launch_bounds__(kWThreads) walk_level_kernel(WalkParams P, int level) {
  __shared__ unsigned long long s_red[32];
  __shared__ int s_last;
  __shared__ int s_nf;
  __shared__ uint32_t s_status;
  __shared__ int s_next_n;
  __shared__ int s_front[SV_MAX_TREE_NODES];
  __shared__ int s_g[SV_MAX_TREE_NODES];       // argmax of frontier nodes, -2 elsewhere
  const int b = blockIdx.x / P.nseg;
  const int seg = blockIdx.x - b * P.nseg;
  const int N = P.N;
  const int64_t tb = static_cast<int64_t>(b) * N;
  if (threadIdx.x == 0) {
    const WalkTree t = P.trees[b];
    s_nf = (t.nf > 0 && t.depth == level) ? t.nf : 0;
  }
  __syncthreads();
  const int nf = s_nf;
  if (nf == 0) return;
  for (int i = 0; i < nf; ++i) {
    const int node = __ldcg(P.frontier + tb + i);
    const E* row = reinterpret_cast<const E*>(P.logits) + (tb + node) * P.stride;
    const unsigned long long m = segment_argmax<E>(row, P.V, seg, P.nseg, s_red);
    if (threadIdx.x == 0) atomicMax(P.best + tb + node, m);
  }
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(&P.trees[b].counter, 1u) == static_cast<unsigned>(P.nseg - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // The tree's last block of this level: argmax of each frontier node, then
  // the next frontier or the result.
  for (int n = threadIdx.x; n < N; n += kWThreads) s_g[n] = -2;
  if (threadIdx.x == 0) {
    s_status = 0;
    s_next_n = 0;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < nf; i += kWThreads) {
    const int node = __ldcg(P.frontier + tb + i);
    s_front[i] = node;
    const unsigned long long m = atomicAdd(P.best + tb + node, 0ull);
    const bool empty = (m >> 32) == static_cast<unsigned long long>(order_key(-CUDART_INF_F));
    s_g[node] = empty ? -1 : argmax_index(m);
    if (empty) atomicOr(&s_status, SV_ROW_EMPTY);
  }
  __syncthreads();
  if (s_status) {
    if (threadIdx.x == 0) {
      WalkTree t = P.trees[b];
      t.nf = 0;
      t.status |= s_status;
      P.trees[b] = t;
    }
    write_invalid(P, b, s_status);
    return;
  }
  const int32_t* par = P.parents + tb;
  const int32_t* tok = P.tokens + tb;
  if (level < P.D) {
    for (int c = 1 + threadIdx.x; c < N; c += kWThreads) {
      const int p = par[c];
      if (sv_in(p, N) && s_g[p] >= 0 && tok[c] == s_g[p]) {
        const int slot = atomicAdd(&s_next_n, 1);
        P.frontier[tb + slot] = c;  // the frontier was copied to shared memory
      }
    }
  }
  __syncthreads();
  const int nn = s_next_n;
  if (threadIdx.x == 0) {
    WalkTree t = P.trees[b];
    t.counter = 0;
    if (nn > 0) {
      t.depth = level + 1;
      t.nf = nn;
    } else {
      t.nf = 0;
      // The deepest accepted nodes are the frontier: the lowest id wins.
      int best = s_front[0];
      for (int i = 1; i < nf; ++i) best = min(best, s_front[i]);
      const int L = P.D + 1;
      int32_t* path = P.path + static_cast<int64_t>(b) * L;
      int32_t* out = P.out_tokens + static_cast<int64_t>(b) * L;
      int cur = best;
      for (int d = level; d >= 0; --d) {
        if (!sv_in(cur, N) || !sv_in(d, L)) break;
        path[d] = cur;
        if (d > 0) out[d - 1] = tok[cur];
        if (d > 0) cur = par[cur];
      }
      out[level] = s_g[best];
      for (int d = level + 1; d < L; ++d) {
        path[d] = -1;
        out[d] = -1;
      }
      P.accept_len[b] = level;
      if (P.row_status) P.row_status[b] = 0;
    }
    P.trees[b] = t;
  }
}

inline size_t walk_trees_bytes(int B) { return align_up(static_cast<size_t>(B) * sizeof(WalkTree), 256); }
inline size_t walk_frontier_bytes(int B, int N) {
  return align_up(static_cast<size_t>(B) * N * sizeof(int32_t), 256);
}

size_t tree_walk_workspace_bytes(const sv_tree_desc& d) {
  return walk_trees_bytes(d.batch) + walk_frontier_bytes(d.batch, d.nodes) +
         align_up(static_cast<size_t>(d.batch) * d.nodes * sizeof(unsigned long long), 256);
}

sv_status greedy_tree_walk(const sv_tree_desc& d, const void* logits, const int32_t* parents,
                           const int32_t* tokens, int32_t* accept_len, int32_t* path,
                           int32_t* out_tokens, int32_t* row_status, void* workspace,
                           cudaStream_t stream) {
  WalkParams P{};
  P.logits = logits;
  P.stride = d.row_stride;
  P.V = d.vocab;
  P.N = d.nodes;
  P.D = d.max_depth;
  P.B = d.batch;
  const int epv = d.dtype == SV_BF16 ? 8 : 4;
  const long long nvec_max = d.vocab / epv + 1;  // any alignment of a row
  P.nseg = static_cast<int>((nvec_max + kWSegVec - 1) / kWSegVec);
  P.parents = parents;
  P.tokens = tokens;
  P.accept_len = accept_len;
  P.path = path;
  P.out_tokens = out_tokens;
  P.row_status = row_status;
  char* w = static_cast<char*>(workspace);
  P.trees = reinterpret_cast<WalkTree*>(w);
  P.frontier = reinterpret_cast<int32_t*>(w + walk_trees_bytes(d.batch));
  P.best = reinterpret_cast<unsigned long long*>(w + walk_trees_bytes(d.batch) +
                                                  walk_frontier_bytes(d.batch, d.nodes));
  const long long blocks = static_cast<long long>(d.batch) * P.nseg;
  if (blocks > INT32_MAX) return SV_ERR_UNSUPPORTED;
  start_phases(stream);
  walk_init_kernel<<<d.batch, 32, 0, stream>>>(P);
  if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  note_launch(stream);
  for (int level = 0; level <= d.max_depth; ++level) {
    if (d.dtype == SV_BF16)
      walk_level_kernel<uint16_t><<<static_cast<unsigned>(blocks), kWThreads, 0, stream>>>(P, level);
    else
      walk_level_kernel<float><<<static_cast<unsigned>(blocks), kWThreads, 0, stream>>>(P, level);
    if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
    note_launch(stream);
  }
  return SV_OK;
}

}  // namespace sv
