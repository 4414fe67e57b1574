// Row sets of the statistics pass and the per-row query lookup, shared by
// the streaming and the top-p statistics kernels.
#pragma once

#include "sv_internal.h"

#include <string.h>

namespace sv {

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

// What the draw needs of one of its rows: e_j / K = exp2(l_j * c - mc) * invK
// over the ids kept by (tau, cut).
struct DrawSide {
  float mc, invK;
  uint32_t tau;
  int32_t cut;
};

// The decisions of a batch row: k = first rejected draft (γ if none), the
// row's status bits, and the draw rows (target k; draft k when k < γ).
struct __align__(16) DecideRecord {
  int32_t k;
  uint32_t status;
  int32_t pad[2];
  DrawSide pt, pd;
};
static_assert(sizeof(DecideRecord) == 48, "DecideRecord layout");

// Decisions made by the statistics pass as soon as every statistic of a
// batch row is written (rec == nullptr: none).
struct DecideIn {
  const RowStats* t_stats;  // [B, G+1]
  const RowStats* d_stats;  // [B, G]
  const int32_t* ids;       // [B, G] or nullptr (G == 0)
  const float* u_accept;    // [B, G] or nullptr (G == 0)
  float* p_draft;           // [B, G] optional
  float* q_draft;           // [B, G] optional
  DecideRecord* rec;        // [B] (statistics pass: nullptr = no decisions there)
  unsigned* counters;       // [B] statistic rows finished per batch row, zero before the pass
  int G, V, rows_per_batch;
};

struct StatsLaunch {
  RowSet set[2];
  int nsets;
  float c;             // log2(e) / T
  float top_p;
  int nslices[2];      // top-p kernel: slices per row of each set
  float* summ;         // top-p kernel: per-slice summaries
  uint8_t* codes;      // top-p kernel: every logit's bin under its slice maximum, one byte each
  unsigned* counters;  // top-p kernel: finished slices per row
  DecideIn dec;
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
  q.elem = S.t2d ? (sv_in(x, S.vocab) ? S.t2d[x] : -1) : x;
  if (q.elem >= S.len) q.elem = -1;  // a t2d entry outside the draft row maps nowhere
  return q;
}

__device__ __forceinline__ int tie_key(const RowSet& S, int j) { return S.sec ? __ldg(S.sec + j) : j; }

// A row's statistics as written by another block of this launch (read
// through L2, never a stale L1 line).
__device__ __forceinline__ RowStats load_stats(const RowStats* p) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
  const uint4 a = __ldcg(q), b = __ldcg(q + 1);
  RowStats st;
  static_assert(sizeof(RowStats) == 2 * sizeof(uint4), "RowStats is two 16-byte words");
  memcpy(reinterpret_cast<char*>(&st), &a, sizeof(uint4));
  memcpy(reinterpret_cast<char*>(&st) + sizeof(uint4), &b, sizeof(uint4));
  return st;
}

// One warp: the decisions of batch row b ("LLM inference acceleration in
// practice ..." §3.1, §4.2): accept draft i iff u_i * q_i(x_i) < p_i(x_i)
// with p = e_query / K on each side, compared as u * e_q * K_t < e_t * K_d
// (both K > 0) to avoid divisions; k = the first rejection.  Writes p and q
// of every draft when asked; returns the batch row's record (every lane).
__device__ __forceinline__ DecideRecord decide_batch(const DecideIn& D, int b) {
  const int G = D.G, lane = threadIdx.x & 31;
  const RowStats* ts = D.t_stats + static_cast<int64_t>(b) * (G + 1);
  const RowStats* ds = D.d_stats + static_cast<int64_t>(b) * G;
  uint32_t status = 0;
  int k = G;
  bool found = false;
  DrawSide pt{0.0f, 0.0f, 0u, 0}, pd{0.0f, 0.0f, 0u, 0};
  for (int base = 0; base <= G; base += 32) {
    const int i = base + lane;
    bool rej = false;
    RowStats t{}, d{};
    if (i <= G) {
      t = load_stats(ts + i);
      status |= t.status;
      if (i < G) {
        d = load_stats(ds + i);
        status |= d.status;
        const int x = D.ids[static_cast<int64_t>(b) * G + i];
        if (x < 0 || x >= D.V) status |= SV_ROW_BAD_DRAFT_ID;
        const double u = static_cast<double>(D.u_accept[static_cast<int64_t>(b) * G + i]);
        const double et = t.K > 0.0 ? static_cast<double>(t.e_query) : 0.0;
        const double eq = d.K > 0.0 ? static_cast<double>(d.e_query) : 0.0;
        const double kt = t.K > 0.0 ? t.K : 1.0, kd = d.K > 0.0 ? d.K : 1.0;
        rej = !(u * eq * kt < et * kd);
        if (D.p_draft) D.p_draft[static_cast<int64_t>(b) * G + i] = static_cast<float>(et / kt);
        if (D.q_draft) D.q_draft[static_cast<int64_t>(b) * G + i] = static_cast<float>(eq / kd);
      }
    }
    const unsigned m = __ballot_sync(0xffffffffu, rej);
    int src = -1;
    if (!found && m) {
      k = base + __ffs(m) - 1;
      found = true;
      src = k - base;
    } else if (!found && G < base + 32) {
      src = G - base;  // every draft accepted: the bonus row
    }
    if (src >= 0) {
      const double Kt = __shfl_sync(0xffffffffu, t.K, src);
      const double Kd = __shfl_sync(0xffffffffu, d.K, src);
      float it = 0.0f, id = 0.0f;
      if (lane == 0) {
        it = Kt > 0.0 ? static_cast<float>(1.0 / Kt) : 0.0f;
        id = Kd > 0.0 ? static_cast<float>(1.0 / Kd) : 0.0f;
      }
      pt = DrawSide{__shfl_sync(0xffffffffu, t.mc, src), __shfl_sync(0xffffffffu, it, 0),
                    __shfl_sync(0xffffffffu, t.tau, src), __shfl_sync(0xffffffffu, t.cut, src)};
      pd = DrawSide{__shfl_sync(0xffffffffu, d.mc, src), __shfl_sync(0xffffffffu, id, 0),
                    __shfl_sync(0xffffffffu, d.tau, src), __shfl_sync(0xffffffffu, d.cut, src)};
    }
  }
  status = __reduce_or_sync(0xffffffffu, status);
  DecideRecord r;
  r.k = k;
  r.status = status;
  r.pad[0] = r.pad[1] = 0;
  r.pt = pt;
  r.pd = k < G ? pd : DrawSide{0.0f, 0.0f, 0u, 0};
  return r;
}

// Thread 0 of a block that has just written the statistics of row r of set
// S: counts the row for its batch row; true for the batch row's last one.
__device__ __forceinline__ bool count_row(const DecideIn& D, const RowSet& S, int r) {
  __threadfence();
  const unsigned prev = atomicAdd(D.counters + r / S.per_group, 1u);
  return prev == static_cast<unsigned>(D.rows_per_batch - 1);
}


// Inputs and outputs of the decision/draw pass (sv_decide.cu).
struct DecideParams {
  const void* target;
  const void* draft;
  int64_t t_stride, d_stride;
  int B, G, V, Vd;
  float c;
  const DecideRecord* rec;  // [B] written by the statistics pass, or nullptr:
  DecideIn dec;             // then the draw makes the decisions itself from these
  const int32_t* ids;
  const float* u_resample;
  const int32_t* t2d;
  const int32_t* d2t;       // with t2d: draft id -> target id
  int32_t* out_tokens;
  int32_t* num_accepted;
  int32_t* row_status;
  float* out_prob;
  // Scratch, set by launch_decide: per-chunk draw-weight sums, the last id
  // with a positive weight per block, finished blocks per row ([B], then one
  // word counting the d2t entries that break the draft-range table), and
  // per segment the first draft id whose target id lies in it or beyond.
  float* chunk_sums;
  int32_t* seg_last;
  unsigned* counters;
  int32_t* d2t_first;
};

// The decision/draw pass with `scratch` of decide_scratch_bytes(B, V) bytes.
sv_status launch_decide(const DecideParams& P, sv_dtype target_dtype, sv_dtype draft_dtype, void* scratch,
                        cudaStream_t stream);

// Top-p statistics of every row of L (sv_topp.cu), with `scratch` of
// topp_scratch_bytes(...) bytes (slice summaries and row counters).
sv_status launch_topp_stats(StatsLaunch L, sv_dtype dtype, void* scratch, cudaStream_t stream);
// Statistics of one or two row sets (sv_chain.cu): the streaming kernel, or
// the top-p kernel when `topp`, with its scratch at `scratch`.
sv_status launch_stats_sets(StatsLaunch L, sv_dtype d0, sv_dtype d1, bool topp, void* scratch,
                            cudaStream_t stream);

}  // namespace sv
