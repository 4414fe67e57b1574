// C-ABI entry points: host-side argument checks, then dispatch to the paths.
// Nothing is launched and no memory is touched when a check fails.
#include "sv_internal.h"

#include <cmath>

using namespace sv;

namespace {

// Clears any pending phase events when a public call returns.
struct CallScope {
  ~CallScope() { sv::end_call(); }
};

// Logit pointers need element alignment only (bf16: 2 bytes, fp32: 4).
bool aligned_elem(const void* p, sv_dtype t) {
  return (reinterpret_cast<uintptr_t>(p) & (t == SV_BF16 ? 1u : 3u)) == 0;
}
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

bool valid_dtype(sv_dtype t) { return t == SV_F32 || t == SV_BF16; }

size_t esize(sv_dtype t) { return t == SV_BF16 ? 2 : 4; }

bool valid_stride(int64_t stride, int len, sv_dtype t) {
  (void)t;
  return stride >= len && stride <= (int64_t{1} << 40);
}

bool valid_vocab(int v) { return v >= 1 && v <= SV_MAX_VOCAB; }

bool chain_desc_ok(const sv_chain_desc* d, bool has_d2t) {
  if (!d) return false;
  if (d->batch < 0 || d->gamma < 0 || d->gamma > SV_MAX_GAMMA) return false;
  if (!valid_vocab(d->vocab)) return false;
  if (!valid_dtype(d->target_dtype) || !valid_dtype(d->draft_dtype)) return false;
  if (!std::isfinite(d->temperature) || d->temperature < 0.0f) return false;
  if (!(d->top_p > 0.0f && d->top_p <= 1.0f)) return false;
  if (!valid_stride(d->target_row_stride, d->vocab, d->target_dtype)) return false;
  const bool sampling = d->temperature > 0.0f;
  if (sampling && d->gamma > 0) {
    if (has_d2t ? !(d->draft_vocab >= 1 && d->draft_vocab <= d->vocab) : d->draft_vocab != d->vocab)
      return false;
    if (!valid_stride(d->draft_row_stride, d->draft_vocab, d->draft_dtype)) return false;
  }
  // Grid size: B*(2γ+1) rows, up to 16 blocks each.
  if (static_cast<int64_t>(d->batch) * (2 * d->gamma + 1) * 16 > INT32_MAX) return false;
  return true;
}

bool tree_desc_ok(const sv_tree_desc* d) {
  if (!d) return false;
  if (d->batch < 0 || d->nodes < 1 || d->nodes > SV_MAX_TREE_NODES) return false;
  if (d->max_depth < 0 || d->max_depth > SV_MAX_TREE_DEPTH) return false;
  if (!valid_vocab(d->vocab) || !valid_dtype(d->dtype)) return false;
  if (!valid_stride(d->row_stride, d->vocab, d->dtype)) return false;
  if (static_cast<int64_t>(d->batch) * d->nodes > INT32_MAX) return false;
  return true;
}

bool tree_sample_desc_ok(const sv_tree_sample_desc* d) {
  if (!d) return false;
  if (d->batch < 0 || d->nodes < 1 || d->nodes > SV_MAX_TREE_NODES) return false;
  if (d->max_depth < 0 || d->max_depth > SV_MAX_TREE_DEPTH) return false;
  if (!valid_vocab(d->vocab) || !valid_dtype(d->dtype)) return false;
  if (!std::isfinite(d->temperature) || !(d->temperature > 0.0f)) return false;
  if (!(d->top_p > 0.0f && d->top_p <= 1.0f)) return false;
  if (!valid_stride(d->target_row_stride, d->vocab, d->dtype)) return false;
  if (!valid_stride(d->draft_row_stride, d->vocab, d->dtype)) return false;
  // Statistics grid: 2*B*N rows, up to 16 blocks each.
  if (static_cast<int64_t>(d->batch) * d->nodes * 2 * 16 > INT32_MAX) return false;
  return true;
}

bool sample_desc_ok(const sv_sample_desc* d) {
  if (!d) return false;
  if (d->rows < 0 || !valid_vocab(d->vocab) || !valid_dtype(d->dtype)) return false;
  if (!std::isfinite(d->temperature) || d->temperature < 0.0f) return false;
  if (!(d->top_p > 0.0f && d->top_p <= 1.0f)) return false;
  if (!valid_stride(d->row_stride, d->vocab, d->dtype)) return false;
  if (static_cast<int64_t>(d->rows) * 16 > INT32_MAX) return false;
  return true;
}

}  // namespace

extern "C" {

int32_t sv_version(void) { return 100; }

const char* sv_status_string(sv_status s) {
  switch (s) {
    case SV_OK: return "ok";
    case SV_ERR_INVALID_ARGUMENT: return "invalid argument";
    case SV_ERR_UNSUPPORTED: return "unsupported configuration";
    case SV_ERR_CUDA: return "CUDA launch failed";
    case SV_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
  }
  return "unknown status";
}

size_t sv_chain_workspace_size(const sv_chain_desc* desc) {
  if (!chain_desc_ok(desc, desc && desc->draft_vocab != desc->vocab)) return 0;
  return chain_workspace_layout(*desc).total;
}

sv_status sv_verify_chain(const sv_chain_desc* desc, const void* target_logits,
                          const void* draft_logits, const int32_t* d2t, const int32_t* t2d,
                          const int32_t* draft_ids, const float* u_accept, const float* u_resample,
                          int32_t* out_tokens, int32_t* num_accepted, float* p_draft,
                          float* q_draft, int32_t* row_status, void* workspace,
                          size_t workspace_bytes, sv_stream_t stream) {
  CallScope scope;
  if (!chain_desc_ok(desc, d2t != nullptr)) return SV_ERR_INVALID_ARGUMENT;
  const sv_chain_desc& d = *desc;
  if (d.batch == 0) return SV_OK;
  const bool sampling = d.temperature > 0.0f;
  if (!target_logits || !aligned_elem(target_logits, d.target_dtype) || !out_tokens || !num_accepted ||
      !workspace)
    return SV_ERR_INVALID_ARGUMENT;
  if (d.gamma > 0 && !draft_ids) return SV_ERR_INVALID_ARGUMENT;
  if (sampling) {
    if (!u_resample) return SV_ERR_INVALID_ARGUMENT;
    if (d.gamma > 0) {
      if (!draft_logits || !aligned_elem(draft_logits, d.draft_dtype) || !u_accept)
        return SV_ERR_INVALID_ARGUMENT;
      if ((d2t == nullptr) != (t2d == nullptr)) return SV_ERR_INVALID_ARGUMENT;
    }
  }
  if (workspace_bytes < chain_workspace_layout(d).total) return SV_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!sampling)
    return greedy_chain(d, target_logits, draft_ids, out_tokens, num_accepted, p_draft, q_draft,
                        row_status, workspace, s);
  ChainArgs a{};
  a.d = d;
  a.target = target_logits;
  a.draft = draft_logits;
  a.d2t = d.gamma > 0 ? d2t : nullptr;
  a.t2d = d.gamma > 0 ? t2d : nullptr;
  a.ids = draft_ids;
  a.u_accept = u_accept;
  a.u_resample = u_resample;
  a.out_tokens = out_tokens;
  a.num_accepted = num_accepted;
  a.p_draft = p_draft;
  a.q_draft = q_draft;
  a.row_status = row_status;
  a.workspace = workspace;
  return sampling_chain(a, s);
}

size_t sv_tree_workspace_size(const sv_tree_desc* desc) {
  if (!tree_desc_ok(desc)) return 0;
  return tree_greedy_layout(desc->batch, desc->nodes).total;
}

sv_status sv_verify_tree(const sv_tree_desc* desc, const void* logits, const int32_t* parents,
                         const int32_t* tokens, int32_t* accept_len, int32_t* path,
                         int32_t* out_tokens, int32_t* row_status, void* workspace,
                         size_t workspace_bytes, sv_stream_t stream) {
  CallScope scope;
  if (!tree_desc_ok(desc)) return SV_ERR_INVALID_ARGUMENT;
  if (desc->batch == 0) return SV_OK;
  if (!logits || !aligned_elem(logits, desc->dtype) || !parents || !tokens || !accept_len || !path ||
      !out_tokens ||
      !workspace)
    return SV_ERR_INVALID_ARGUMENT;
  if (workspace_bytes < sv_tree_workspace_size(desc)) return SV_ERR_WORKSPACE_TOO_SMALL;
  return greedy_tree(*desc, logits, parents, tokens, accept_len, path, out_tokens, row_status,
                     workspace, reinterpret_cast<cudaStream_t>(stream));
}

size_t sv_tree_path_workspace_size(const sv_tree_desc* desc) {
  if (!tree_desc_ok(desc)) return 0;
  return tree_walk_workspace_bytes(*desc);
}

sv_status sv_verify_tree_path(const sv_tree_desc* desc, const void* logits, const int32_t* parents,
                              const int32_t* tokens, int32_t* accept_len, int32_t* path,
                              int32_t* out_tokens, int32_t* row_status, void* workspace,
                              size_t workspace_bytes, sv_stream_t stream) {
  CallScope scope;
  if (!tree_desc_ok(desc)) return SV_ERR_INVALID_ARGUMENT;
  if (desc->batch == 0) return SV_OK;
  if (!logits || !aligned_elem(logits, desc->dtype) || !parents || !tokens || !accept_len || !path ||
      !out_tokens || !workspace)
    return SV_ERR_INVALID_ARGUMENT;
  if (workspace_bytes < sv_tree_path_workspace_size(desc)) return SV_ERR_WORKSPACE_TOO_SMALL;
  return greedy_tree_walk(*desc, logits, parents, tokens, accept_len, path, out_tokens, row_status,
                          workspace, reinterpret_cast<cudaStream_t>(stream));
}

size_t sv_tree_sample_workspace_size(const sv_tree_sample_desc* desc) {
  if (!tree_sample_desc_ok(desc)) return 0;
  return tree_sample_workspace_bytes(*desc);
}

sv_status sv_verify_tree_sample(const sv_tree_sample_desc* desc, const void* target_logits,
                                const void* draft_logits, const int32_t* parents, const int32_t* tokens,
                                const float* u_accept, const float* u_final, int32_t* accept_len,
                                int32_t* path, int32_t* out_tokens, int32_t* row_status,
                                void* workspace, size_t workspace_bytes, sv_stream_t stream) {
  CallScope scope;
  if (!tree_sample_desc_ok(desc)) return SV_ERR_INVALID_ARGUMENT;
  if (desc->batch == 0) return SV_OK;
  if (!target_logits || !aligned_elem(target_logits, desc->dtype) || !draft_logits ||
      !aligned_elem(draft_logits, desc->dtype) || !parents || !tokens || !u_accept || !u_final ||
      !accept_len || !path || !out_tokens || !workspace)
    return SV_ERR_INVALID_ARGUMENT;
  if (workspace_bytes < sv_tree_sample_workspace_size(desc)) return SV_ERR_WORKSPACE_TOO_SMALL;
  return tree_sample(*desc, target_logits, draft_logits, parents, tokens, u_accept, u_final, accept_len, path,
                     out_tokens, row_status, workspace, reinterpret_cast<cudaStream_t>(stream));
}

sv_status sv_topk(const sv_topk_desc* desc, const void* logits, int32_t* out_ids, float* out_vals,
                  sv_stream_t stream) {
  CallScope scope;
  if (!desc || desc->rows < 0 || !valid_vocab(desc->vocab) || !valid_dtype(desc->dtype)) return SV_ERR_INVALID_ARGUMENT;
  if (desc->k < 1 || desc->k > SV_MAX_TOPK || desc->k > desc->vocab) return SV_ERR_INVALID_ARGUMENT;
  if (!valid_stride(desc->row_stride, desc->vocab, desc->dtype)) return SV_ERR_INVALID_ARGUMENT;
  if (desc->rows == 0) return SV_OK;
  if (!logits || !aligned_elem(logits, desc->dtype) || !out_ids) return SV_ERR_INVALID_ARGUMENT;
  return topk_rows(*desc, logits, out_ids, out_vals, reinterpret_cast<cudaStream_t>(stream));
}

sv_status sv_d2t_scatter(const void* draft_logits, int64_t in_row_stride, const int32_t* d2t,
                         const int32_t* t2d, int32_t rows, int32_t draft_vocab, int32_t vocab,
                         sv_dtype dtype, float fill, void* out, int64_t out_row_stride,
                         sv_stream_t stream) {
  CallScope scope;
  if (rows < 0 || !valid_vocab(vocab) || draft_vocab < 1 || draft_vocab > vocab || !valid_dtype(dtype))
    return SV_ERR_INVALID_ARGUMENT;
  if (!valid_stride(in_row_stride, draft_vocab, dtype) || !valid_stride(out_row_stride, vocab, dtype))
    return SV_ERR_INVALID_ARGUMENT;
  if (rows == 0) return SV_OK;
  if (!draft_logits || !d2t || !out || !aligned_elem(draft_logits, dtype) || !aligned_elem(out, dtype))
    return SV_ERR_INVALID_ARGUMENT;
  if (t2d && !aligned4(t2d)) return SV_ERR_INVALID_ARGUMENT;
  if (static_cast<int64_t>(rows) * ((vocab + 255) / 256) > INT32_MAX) return SV_ERR_INVALID_ARGUMENT;
  return d2t_scatter(draft_logits, in_row_stride, d2t, t2d, rows, draft_vocab, vocab, dtype, fill, out,
                     out_row_stride, reinterpret_cast<cudaStream_t>(stream));
}

sv_status sv_build_t2d(const int32_t* d2t, int32_t draft_vocab, int32_t vocab, int32_t* t2d,
                       int32_t* status, sv_stream_t stream) {
  CallScope scope;
  if (!valid_vocab(vocab) || draft_vocab < 0 || draft_vocab > vocab || !t2d) return SV_ERR_INVALID_ARGUMENT;
  if (draft_vocab > 0 && !d2t) return SV_ERR_INVALID_ARGUMENT;
  return build_t2d(d2t, draft_vocab, vocab, t2d, status, reinterpret_cast<cudaStream_t>(stream));
}

size_t sv_sample_workspace_size(const sv_sample_desc* desc) {
  if (!sample_desc_ok(desc)) return 0;
  return sample_workspace_bytes(*desc);
}

sv_status sv_sample(const sv_sample_desc* desc, const void* logits, const float* u,
                    int32_t* out_tokens, float* out_prob, void* workspace, size_t workspace_bytes,
                    sv_stream_t stream) {
  CallScope scope;
  if (!sample_desc_ok(desc)) return SV_ERR_INVALID_ARGUMENT;
  if (desc->rows == 0) return SV_OK;
  if (!logits || !aligned_elem(logits, desc->dtype) || !out_tokens) return SV_ERR_INVALID_ARGUMENT;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (desc->temperature == 0.0f) return greedy_sample(*desc, logits, out_tokens, out_prob, s);
  if (!u || !workspace) return SV_ERR_INVALID_ARGUMENT;
  if (workspace_bytes < sv_sample_workspace_size(desc)) return SV_ERR_WORKSPACE_TOO_SMALL;
  return sample_rows(*desc, logits, u, out_tokens, out_prob, workspace, s);
}

sv_status sv_softmax_topp(const sv_sample_desc* desc, const void* logits, float* out_probs,
                          int64_t out_row_stride, void* workspace, size_t workspace_bytes, sv_stream_t stream) {
  CallScope scope;
  if (!sample_desc_ok(desc) || desc->temperature == 0.0f) return SV_ERR_INVALID_ARGUMENT;
  if (out_row_stride < desc->vocab) return SV_ERR_INVALID_ARGUMENT;
  if (desc->rows == 0) return SV_OK;
  if (!logits || !aligned_elem(logits, desc->dtype) || !out_probs || !aligned4(out_probs) || !workspace)
    return SV_ERR_INVALID_ARGUMENT;
  if (workspace_bytes < sv_sample_workspace_size(desc)) return SV_ERR_WORKSPACE_TOO_SMALL;
  return probs_rows(*desc, logits, out_probs, out_row_stride, workspace, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

// ------------------------------------------------------- profiling hooks ----

#include <atomic>

namespace {
std::atomic<unsigned long long> g_launches{0};
thread_local void* const* t_events = nullptr;
thread_local int t_nevents = 0;
thread_local int t_next = 0;
}  // namespace

namespace sv {
static void record_phase(cudaStream_t stream) {
  if (!t_events || t_next >= t_nevents) return;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(stream, &cap);
  // Under capture the record must become a graph node that records the
  // event on every replay.
  cudaEventRecordWithFlags(static_cast<cudaEvent_t>(t_events[t_next]), stream,
                           cap == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : 0u);
  ++t_next;
}

void start_phases(cudaStream_t stream) {
  if (t_next == 0) record_phase(stream);
}

void note_launch(cudaStream_t stream) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (t_next == 0) record_phase(stream);  // a path that did not call start_phases
  record_phase(stream);
}

bool FuncAttrCache::ensure(const void* func, size_t dyn_smem, bool non_portable_cluster) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  if (non_portable_cluster && !nonportable[dev].load()) {
    if (cudaFuncSetAttribute(func, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
      return false;
    nonportable[dev].store(1);
  }
  size_t have = smem[dev].load();
  if (dyn_smem > have) {
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(dyn_smem)) !=
        cudaSuccess)
      return false;
    while (have < dyn_smem && !smem[dev].compare_exchange_weak(have, dyn_smem)) {
    }
  }
  return true;
}
void end_call() {
  t_events = nullptr;
  t_nevents = 0;
  t_next = 0;
}
}  // namespace sv

namespace {
constexpr int kMaxDebugReaders = 32;
sv::DebugReader g_debug_readers[kMaxDebugReaders];
std::atomic<int> g_debug_nreaders{0};
}  // namespace

namespace sv {
int register_debug_reader(DebugReader r) {
  const int i = g_debug_nreaders.fetch_add(1);
  if (i < kMaxDebugReaders) g_debug_readers[i] = r;
  return i;
}
unsigned read_debug_words(bool reset) {
  unsigned v = 0;
  const int n = g_debug_nreaders.load();
  for (int i = 0; i < n && i < kMaxDebugReaders; ++i) v |= g_debug_readers[i](reset);
  return v;
}
}  // namespace sv

extern "C" {
uint32_t sv_debug_flags(int32_t reset) { return sv::read_debug_words(reset != 0); }

void sv_set_phase_events(void* const* events, int32_t n) {
  if (!events || n <= 0) {
    sv::end_call();
    return;
  }
  t_events = events;
  t_nevents = n;
  t_next = 0;
}

uint64_t sv_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }
}
