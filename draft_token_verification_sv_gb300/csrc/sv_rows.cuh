// Row sets of the statistics pass and the per-row query lookup, shared by
// the streaming and the top-p statistics kernels.
#pragma once

#include "sv_internal.h"

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

struct StatsLaunch {
  RowSet set[2];
  int nsets;
  float c;             // log2(e) / T
  float top_p;
  int nslices[2];      // top-p kernel: slices per row of each set
  float* summ;         // top-p kernel: per-slice summaries
  unsigned* counters;  // top-p kernel: finished slices per row
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


// Inputs and outputs of the decision/draw pass (sv_decide.cu).
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
  // Scratch, set by launch_decide: per-chunk draw-weight sums, the last id
  // with a positive weight per block, finished blocks per row.
  float* chunk_sums;
  int32_t* seg_last;
  unsigned* counters;
};

// The decision/draw pass with `scratch` of decide_scratch_bytes(B, V) bytes.
sv_status launch_decide(const DecideParams& P, sv_dtype target_dtype, sv_dtype draft_dtype, void* scratch,
                        cudaStream_t stream);

// Top-p statistics of every row of L (sv_topp.cu), with `scratch` of
// topp_scratch_bytes(...) bytes (slice summaries and row counters).
sv_status launch_topp_stats(StatsLaunch L, sv_dtype dtype, void* scratch, cudaStream_t stream);

}  // namespace sv
