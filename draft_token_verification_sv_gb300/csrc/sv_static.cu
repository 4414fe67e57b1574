// sv_verify_chain_static: sv_verify_chain for callers that cannot allocate
// device memory.
//
// Some callers may not call cudaMalloc at all: code running inside another
// runtime's memory pool or allocator, plugins loaded into a process whose
// device memory is owned by someone else, or serving loops that forbid new
// allocations once they are warmed up.  For them this entry point takes its
// scratch from an array compiled into this library instead of from a
// caller-provided workspace.  It allocates nothing and calls no allocating
// routine; it forwards to sv_verify_chain with that array as the workspace.
#include <mutex>

#include "sv_internal.h"

namespace {

// Scratch shared by every call on a device.  Every GPU that loads this
// library holds this array until the process exits.
constexpr size_t kStaticScratchBytes = size_t{16} << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
sv_status static_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return SV_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SV_OK;
}

}  // namespace

extern "C" {

size_t sv_static_scratch_bytes(void) { return kStaticScratchBytes; }

sv_status sv_verify_chain_static(const sv_chain_desc* desc, const void* target_logits,
                                 const void* draft_logits, const int32_t* d2t, const int32_t* t2d,
                                 const int32_t* draft_ids, const float* u_accept, const float* u_resample,
                                 int32_t* out_tokens, int32_t* num_accepted, float* p_draft, float* q_draft,
                                 int32_t* row_status, sv_stream_t stream) {
  // An empty batch needs no scratch: sv_verify_chain checks the descriptor
  // and returns without touching the device.
  if (desc && desc->batch == 0)
    return sv_verify_chain(desc, target_logits, draft_logits, d2t, t2d, draft_ids, u_accept, u_resample,
                           out_tokens, num_accepted, p_draft, q_draft, row_status, nullptr, 0, stream);
  const size_t need = sv_chain_workspace_size(desc);
  if (need == 0) return SV_ERR_INVALID_ARGUMENT;
  if (need > kStaticScratchBytes) return SV_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const sv_status s = static_scratch(&scratch);
  if (s != SV_OK) return s;
  return sv_verify_chain(desc, target_logits, draft_logits, d2t, t2d, draft_ids, u_accept, u_resample,
                         out_tokens, num_accepted, p_draft, q_draft, row_status, scratch, kStaticScratchBytes,
                         stream);
}

}  // extern "C"
