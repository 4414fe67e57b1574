// Internal declarations shared by the library's translation units.
#pragma once

#include "sv_common.cuh"

#include <atomic>

namespace sv {

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Debug builds: every translation unit registers a reader of its debug
// word (returns it; clears it when asked).  sv_debug_flags ORs them.
using DebugReader = unsigned (*)(bool reset);
int register_debug_reader(DebugReader r);
unsigned read_debug_words(bool reset);

// Call once before the first device operation of a public call: records
// the caller's first phase event, if one is pending (sv_set_phase_events).
void start_phases(cudaStream_t stream);
// Call after every kernel launch: counts launches and records the caller's
// next phase event, if one is pending.
void note_launch(cudaStream_t stream);
// Drop any phase events left over when a call returns.
void end_call();

// Per-kernel cache of the attributes set with cudaFuncSetAttribute, per
// device, so a call only touches them when it needs more than any earlier
// call did (repeated calls, and calls under stream capture, make none).
struct FuncAttrCache {
  static constexpr int kMaxDevices = 64;
  std::atomic<size_t> smem[kMaxDevices] = {};
  std::atomic<int> nonportable[kMaxDevices] = {};
  bool ensure(const void* func, size_t dyn_smem, bool non_portable_cluster);
};

// Scratch of the top-p statistics kernel for two row sets (sv_topp.cu).
size_t topp_scratch_bytes(int rows0, int len0, int rows1, int len1);

// Scratch of the decision/draw kernel for B rows of V ids (sv_decide.cu).
size_t decide_scratch_bytes(int B, int V);

// Chain workspace: [counters: B u32][stats: B(2γ+1) RowStats][argmax: B(γ+1) i32]
//                  [decision records: B x 48 B][top-p scratch when T > 0 and
//                  top_p < 1][draw scratch when T > 0]
struct WorkspaceLayout {
  size_t counters, stats, argmax, records, topp, decide, total;
};

inline WorkspaceLayout chain_workspace_layout(const sv_chain_desc& d) {
  WorkspaceLayout L{};
  const size_t B = static_cast<size_t>(d.batch);
  const size_t G = static_cast<size_t>(d.gamma);
  L.counters = 0;
  L.stats = align_up(B * sizeof(uint32_t), 256);
  L.argmax = L.stats + align_up(B * (2 * G + 1) * sizeof(RowStats), 256);
  L.records = L.argmax + align_up(B * (G + 1) * sizeof(int32_t), 256);
  L.topp = L.records + align_up(B * 48, 256);
  L.decide = L.topp;
  if (d.temperature > 0.0f && d.top_p < 1.0f)
    L.decide += align_up(topp_scratch_bytes(d.batch * (d.gamma + 1), d.vocab, d.batch * d.gamma, d.draft_vocab), 256);
  L.total = L.decide;
  if (d.temperature > 0.0f) L.total += decide_scratch_bytes(d.batch, d.vocab);
  return L;
}

// Draft-side sampling / filtered probabilities:
//   [stats: R RowStats][counters: R u32][decision records: R x 48 B]
//   [top-p scratch when top_p < 1][draw scratch]
inline size_t sample_stats_bytes(int rows) { return align_up(static_cast<size_t>(rows) * sizeof(RowStats), 256); }
inline size_t sample_counters_offset(int rows) { return sample_stats_bytes(rows); }
inline size_t sample_records_offset(int rows) {
  return sample_counters_offset(rows) + align_up(static_cast<size_t>(rows) * sizeof(uint32_t), 256);
}
inline size_t sample_topp_offset(int rows) {
  return sample_records_offset(rows) + align_up(static_cast<size_t>(rows) * 48, 256);
}
inline size_t sample_topp_bytes(const sv_sample_desc& d) {
  return d.temperature > 0.0f && d.top_p < 1.0f ? align_up(topp_scratch_bytes(d.rows, d.vocab, 0, 0), 256) : 0;
}
inline size_t sample_workspace_bytes(const sv_sample_desc& d) {
  size_t n = sample_topp_offset(d.rows) + sample_topp_bytes(d);
  if (d.temperature > 0.0f) n += decide_scratch_bytes(d.rows, d.vocab);
  return n + 256;
}

inline size_t tree_counter_bytes(int batch) {
  return align_up(static_cast<size_t>(batch) * sizeof(uint32_t), 256);
}

// Greedy tree workspace: [group counters: B u32][segment counters: B*N u32]
// [row maxima: B*N u64][argmax: B*N i32]; the first three are cleared per call.
struct TreeGreedyLayout {
  size_t segcnt, rowmax, g, total;
};
inline TreeGreedyLayout tree_greedy_layout(int batch, int nodes) {
  const size_t rows = static_cast<size_t>(batch) * static_cast<size_t>(nodes);
  TreeGreedyLayout L{};
  L.segcnt = tree_counter_bytes(batch);
  L.rowmax = L.segcnt + align_up(rows * sizeof(uint32_t), 256);
  L.g = L.rowmax + align_up(rows * sizeof(unsigned long long), 256);
  L.total = L.g + align_up(rows * sizeof(int32_t), 256);
  return L;
}

// Entry points of the individual paths (arguments already validated).
sv_status greedy_chain(const sv_chain_desc& d, const void* target, const int32_t* ids,
                       int32_t* out_tokens, int32_t* num_accepted, float* p_draft, float* q_draft,
                       int32_t* row_status, void* workspace, cudaStream_t stream);
sv_status greedy_tree(const sv_tree_desc& d, const void* logits, const int32_t* parents,
                      const int32_t* tokens, int32_t* accept_len, int32_t* path,
                      int32_t* out_tokens, int32_t* row_status, void* workspace,
                      cudaStream_t stream);
sv_status greedy_sample(const sv_sample_desc& d, const void* logits, int32_t* out_tokens,
                        float* out_prob, cudaStream_t stream);
// Speculative-sampling tree verify (sv_tree_sample.cu).
size_t tree_sample_workspace_bytes(const sv_tree_sample_desc& d);
sv_status tree_sample(const sv_tree_sample_desc& d, const void* target, const void* draft,
                      const int32_t* parents, const int32_t* tokens, const float* u_accept,
                      const float* u_final, int32_t* accept_len, int32_t* path, int32_t* out_tokens,
                      int32_t* row_status, void* workspace, cudaStream_t stream);
// Top-k ids per row (sv_topk.cu).
sv_status topk_rows(const sv_topk_desc& d, const void* logits, int32_t* out_ids, float* out_vals,
                    cudaStream_t stream);
// Tree verify along the accepted frontier only (sv_tree_walk.cu).
size_t tree_walk_workspace_bytes(const sv_tree_desc& d);
sv_status greedy_tree_walk(const sv_tree_desc& d, const void* logits, const int32_t* parents,
                           const int32_t* tokens, int32_t* accept_len, int32_t* path,
                           int32_t* out_tokens, int32_t* row_status, void* workspace,
                           cudaStream_t stream);

struct ChainArgs {
  sv_chain_desc d;
  const void* target;
  const void* draft;
  const int32_t* d2t;
  const int32_t* t2d;
  const int32_t* ids;
  const float* u_accept;
  const float* u_resample;
  int32_t* out_tokens;
  int32_t* num_accepted;
  float* p_draft;
  float* q_draft;
  int32_t* row_status;
  void* workspace;
};
sv_status sampling_chain(const ChainArgs& a, cudaStream_t stream);

sv_status sample_rows(const sv_sample_desc& d, const void* logits, const float* u,
                      int32_t* out_tokens, float* out_prob, void* workspace, cudaStream_t stream);
sv_status probs_rows(const sv_sample_desc& d, const void* logits, float* out, int64_t out_stride,
                     void* workspace, cudaStream_t stream);

sv_status d2t_scatter(const void* in, int64_t in_stride, const int32_t* d2t, const int32_t* t2d,
                      int rows, int vd, int v, sv_dtype dtype, float fill, void* out,
                      int64_t out_stride, cudaStream_t stream);
sv_status build_t2d(const int32_t* d2t, int vd, int v, int32_t* t2d, int32_t* status,
                    cudaStream_t stream);

#ifdef SV_DEBUG
// This translation unit's debug word reader, registered at load time.
static unsigned read_this_debug_word(bool reset) {
  unsigned v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return ~0u;
  if (cudaMemcpyFromSymbol(&v, g_sv_debug_word, sizeof(v)) != cudaSuccess) return ~0u;
  if (reset) {
    const unsigned z = 0;
    if (cudaMemcpyToSymbol(g_sv_debug_word, &z, sizeof(z)) != cudaSuccess) return ~0u;
  }
  return v;
}
[[maybe_unused]] static const int g_debug_reader_registered = register_debug_reader(&read_this_debug_word);
#endif

}  // namespace sv
