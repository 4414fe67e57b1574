/*
 * spec_verify.h -- the verify step of speculative decoding on one GPU.
 *
 * A plain C interface.  Every pointer argument is a DEVICE pointer owned by
 * the caller unless it is documented otherwise; the library allocates no
 * memory and keeps no state between calls beyond what the caller passes in,
 * so calls on different streams with different buffers may run concurrently.
 * Every call is asynchronous on `stream` (NULL = the legacy default stream).
 *
 * Error behaviour, for every entry point:
 *   - Arguments are checked on the host before anything is launched; a bad
 *     argument returns SV_ERR_INVALID_ARGUMENT and touches no memory.
 *   - A launch that the CUDA runtime rejects returns SV_ERR_CUDA.
 *   - Faults that depend on device data (a draft id outside the vocabulary,
 *     a malformed tree, a row with no finite logit) never trap: they are
 *     reported per batch row in `row_status` (bits SV_ROW_*); such rows emit
 *     num_accepted = 0 / accept_len = 0 and token -1.
 *   - No kernel spins on a flag or waits on another launch.
 *
 * Layouts: logits are row-major; a "row" is one position's logits over the
 * vocabulary.  Row strides are in ELEMENTS and at least the row length; any
 * such stride is accepted and logit pointers need only be aligned to their
 * element size (rows that start on a 16-byte boundary take the vectorised
 * path, others are read with a scalar head and tail).  Logits may be -inf
 * (probability 0); NaN logits are not supported.
 *
 * Sources (web pages):
 *  [P3] "LLM inference acceleration in practice: draft models and
 *       speculative sampling explained" (mlqm.cn/news/1205650), §3.1 the
 *       algorithm, §4.2 SpeculativeDecoder.generate() and _apply_top_p,
 *       §6.2 batching and shared temperature/top_p.
 *  [P2] "A 2.16x speculative-decoding speedup from a 1-layer Llama draft"
 *       (blog.bruce.linkpc.net), headline table ("Match = True") and §5,
 *       the draft token tree (total_token 32, depth 5, top_k 8).
 *  [P1] "SSD: extending the engine with new models and an EAGLE3 draft"
 *       (lpnh.cn/news/2716086), §六 EAGLE3 d2t/t2d small-vocabulary
 *       scatter, §七 greedy (--temp 0) benchmarking.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t. */
typedef struct CUstream_st* sv_stream_t;

typedef enum sv_status {
  SV_OK = 0,
  SV_ERR_INVALID_ARGUMENT = 1,
  SV_ERR_UNSUPPORTED = 2,        /* valid request outside what is implemented */
  SV_ERR_CUDA = 3,               /* the CUDA runtime rejected a launch */
  SV_ERR_WORKSPACE_TOO_SMALL = 4
} sv_status;

typedef enum sv_dtype { SV_F32 = 0, SV_BF16 = 1 } sv_dtype;

/* Per-batch-row status bits (row_status outputs). */
#define SV_ROW_BAD_DRAFT_ID 1        /* a draft id outside [0, vocab) */
#define SV_ROW_BAD_PARENT 2          /* tree: parents[0] != -1 or parents[n] not in [0, n) */
#define SV_ROW_DEPTH_EXCEEDED 4      /* tree: a node deeper than max_depth */
#define SV_ROW_BAD_TOKEN 8           /* tree: a node token (n >= 1) outside [0, vocab) */
#define SV_ROW_EMPTY 16              /* a logit row with no finite value */
#define SV_ROW_RESAMPLE_FALLBACK 32  /* informational: residual mass was 0, drew from p_k */

/* Limits checked on the host. */
#define SV_MAX_GAMMA 64
#define SV_MAX_VOCAB 16777216
#define SV_MAX_TOPK 16
#define SV_MAX_TREE_NODES 1024
#define SV_MAX_TREE_DEPTH 64

typedef struct sv_chain_desc {
  int32_t batch;              /* B >= 0 (0: nothing to do) */
  int32_t gamma;              /* γ in [0, SV_MAX_GAMMA]: draft tokens per row */
  int32_t vocab;              /* V in [1, SV_MAX_VOCAB]: target vocabulary */
  int32_t draft_vocab;        /* V_d: == vocab, or the EAGLE3 draft vocabulary when d2t != NULL */
  sv_dtype target_dtype, draft_dtype;
  float temperature;          /* T >= 0, finite; 0 selects greedy verify */
  float top_p;                /* (0, 1]; 1 filters nothing */
  int64_t target_row_stride;  /* elements between consecutive target rows */
  int64_t draft_row_stride;   /* elements between consecutive draft rows */
} sv_chain_desc;

/* Bytes of device workspace sv_verify_chain needs for `desc`.  Returns 0 for
 * an invalid descriptor.  The workspace is scratch: it needs no
 * initialisation and its contents are undefined after a call.  Calls that
 * may overlap on the device must use different workspaces. */
size_t sv_chain_workspace_size(const sv_chain_desc* desc);

/*
 * Verify a batch of γ-token draft chains.  [P3] §3.1 and §4.2 (steps 2-5 of
 * generate()), batched per [P3] §6.2; greedy per [P1] §七 / [P2] "Match".
 *
 * T > 0, for each batch row b:
 *   p_i = softmax(top_p_filter(target row i / T)) for i = 0..γ,
 *   q_i = softmax(top_p_filter(draft row i / T))  for i = 0..γ-1 (same T, top_p),
 *   top-p keeps rank r (logit descending, lower index first on ties) iff
 *   r == 0 or the softmax mass of ranks < r is <= top_p.
 *   Draft x_i = draft_ids[b, i] is accepted iff u_accept[b,i] * q_i(x_i) < p_i(x_i);
 *   k = the first rejected i (γ if none).  If k < γ the token at position k
 *   is drawn from max(0, p_k - q_k) (from p_k if that mass is 0), else the
 *   bonus token is drawn from p_γ; a draw from weights w with uniform u is
 *   the smallest id j with w_0 + ... + w_j > u * sum(w).
 * T == 0 (greedy): g_i = argmax of target row i (lowest id on ties); accept
 *   iff x_i == g_i; the token after the accepted prefix is g_k.  Draft
 *   logits, d2t/t2d and the uniforms are not read and may be NULL; top_p is
 *   ignored.
 *
 * EAGLE3 small draft vocabulary ([P1] §六): when d2t != NULL the draft rows
 * hold V_d = draft_vocab logits and d2t[j] is the target id of draft id j
 * (injective).  q is then the distribution of the scattered row (unmapped
 * ids have probability 0; top-p ties are ordered by target id); t2d, the
 * inverse map with -1 for unmapped ids (see sv_build_t2d), is required.
 *
 * Arguments (device pointers unless noted):
 *   desc           host pointer.
 *   target_logits  [B, γ+1] rows of V elements (target_dtype), row stride
 *                  target_row_stride; row b*(γ+1)+i is position i of row b.
 *   draft_logits   [B, γ] rows of V_d elements (draft_dtype).
 *   d2t            [V_d] int32 or NULL;  t2d [V] int32, required iff d2t.
 *   draft_ids      [B, γ] int32 target-vocabulary ids.
 *   u_accept       [B, γ] float in [0, 1);  u_resample [B] float in [0, 1).
 *   out_tokens     [B, γ+1] int32: accepted drafts, then the drawn token, then -1.
 *   num_accepted   [B] int32: k.
 *   p_draft, q_draft  optional [B, γ] float: p_i(x_i), q_i(x_i) for every i
 *                  (0 when T == 0 or the row is flagged).
 *   row_status     optional [B] int32 (SV_ROW_* bits).
 *   workspace      >= sv_chain_workspace_size(desc) bytes (see above).
 */
sv_status sv_verify_chain(const sv_chain_desc* desc,
                          const void* target_logits, const void* draft_logits,
                          const int32_t* d2t, const int32_t* t2d,
                          const int32_t* draft_ids,
                          const float* u_accept, const float* u_resample,
                          int32_t* out_tokens, int32_t* num_accepted,
                          float* p_draft, float* q_draft, int32_t* row_status,
                          void* workspace, size_t workspace_bytes, sv_stream_t stream);

/*
 * sv_verify_chain for callers that cannot allocate device memory (for
 * example code that runs inside another runtime's allocator, or a serving
 * loop that forbids allocations after warm-up).  The pages have no
 * counterpart to this entry point: it is a deployment convenience.
 *
 * Same arguments and results as sv_verify_chain, without the workspace: the
 * scratch is an array of sv_static_scratch_bytes() bytes (16 MiB) built into
 * the library, which every GPU that loads the library keeps until the
 * process exits.  Nothing is allocated and no allocating routine is called.
 *   - A descriptor that needs more scratch than the array holds
 *     (sv_chain_workspace_size(desc) > sv_static_scratch_bytes()) is rejected
 *     with SV_ERR_WORKSPACE_TOO_SMALL before anything runs.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it; make that first call outside any
 *     stream capture.  The cached address belongs to the device's context as
 *     it was then: after cudaDeviceReset on that device the address is stale,
 *     so a process that resets a device must not call this entry point on it
 *     again (restart the process instead).
 *   - An empty batch (desc->batch == 0) is checked like sv_verify_chain
 *     checks it and returns SV_OK without touching the device.
 *   - All calls on a device share the one array, which keeps whatever the
 *     last call left in it.  The verify path needs no zeroed scratch (it
 *     clears its own counters on every call).  Calls that may overlap on the
 *     GPU (different streams, no ordering between them) race on the array:
 *     order them, or use sv_verify_chain with separate workspaces.
 */
sv_status sv_verify_chain_static(const sv_chain_desc* desc,
                                 const void* target_logits, const void* draft_logits,
                                 const int32_t* d2t, const int32_t* t2d,
                                 const int32_t* draft_ids,
                                 const float* u_accept, const float* u_resample,
                                 int32_t* out_tokens, int32_t* num_accepted,
                                 float* p_draft, float* q_draft, int32_t* row_status,
                                 sv_stream_t stream);

/* Size in bytes of the scratch array used by sv_verify_chain_static. */
size_t sv_static_scratch_bytes(void);

typedef struct sv_tree_desc {
  int32_t batch;      /* B >= 0 trees */
  int32_t nodes;      /* N in [1, SV_MAX_TREE_NODES] nodes per tree, node 0 = root */
  int32_t vocab;      /* V in [1, SV_MAX_VOCAB] */
  int32_t max_depth;  /* D in [0, SV_MAX_TREE_DEPTH]: deepest allowed node */
  sv_dtype dtype;
  int64_t row_stride; /* elements between consecutive node rows */
} sv_tree_desc;

/* Workspace bytes for sv_verify_tree (scratch, as for sv_verify_chain).
 * 0 for an invalid descriptor. */
size_t sv_tree_workspace_size(const sv_tree_desc* desc);

/*
 * Greedy verify of B draft token trees ([P2] §5 tree of total_token nodes,
 * depth, top_k; greedy "Match = True").
 *
 * Node 0 is the root (the last committed token; not itself verified).  The
 * logits row of node n predicts the token after n's root path.  A node is
 * accepted when its parent is accepted and its token equals the argmax of
 * the parent's row (lowest id on ties).  The result is the deepest accepted
 * node (lowest node id among equally deep ones) with its root path, plus the
 * bonus token argmax(row of that node).
 *
 *   logits      [B, N] rows of V elements, row b*N+n is node n of tree b.
 *   parents     [B, N] int32: parents[b,0] == -1, 0 <= parents[b,n] < n.
 *   tokens      [B, N] int32: node tokens (tokens[b,0] unused).
 *   accept_len  [B] int32: depth of the accepted node (drafts accepted).
 *   path        [B, D+1] int32: node ids from the root (path[b,0] = 0), -1 padded.
 *   out_tokens  [B, D+1] int32: accepted tokens then the bonus, -1 padded.
 *   row_status  optional [B] int32 (SV_ROW_*).
 */
sv_status sv_verify_tree(const sv_tree_desc* desc, const void* logits,
                         const int32_t* parents, const int32_t* tokens,
                         int32_t* accept_len, int32_t* path, int32_t* out_tokens,
                         int32_t* row_status, void* workspace, size_t workspace_bytes,
                         sv_stream_t stream);

/*
 * The same greedy tree verify, reading only the rows of the accepted
 * frontier ([P2] §5 tree; the accepted nodes of depth d are the only rows
 * that decide depth d+1).  One launch per level, depth 0..D: level d takes
 * the argmax of the rows of the accepted depth-d nodes and keeps their
 * children whose token matches; the walk ends at the first empty level.  It
 * reads (accept_len + 1) rows per tree when sibling tokens are distinct,
 * instead of N.  Arguments, layouts and results are those of
 * sv_verify_tree, with one difference: SV_ROW_EMPTY is reported only for a
 * row the walk reads (rows off the walked path are never read).
 * Workspace: sv_tree_path_workspace_size (scratch, no initialisation).
 */
size_t sv_tree_path_workspace_size(const sv_tree_desc* desc);
sv_status sv_verify_tree_path(const sv_tree_desc* desc, const void* logits,
                              const int32_t* parents, const int32_t* tokens,
                              int32_t* accept_len, int32_t* path, int32_t* out_tokens,
                              int32_t* row_status, void* workspace, size_t workspace_bytes,
                              sv_stream_t stream);

typedef struct sv_tree_sample_desc {
  int32_t batch;             /* B >= 0 trees */
  int32_t nodes;             /* N in [1, SV_MAX_TREE_NODES] nodes per tree, node 0 = root */
  int32_t vocab;             /* V in [1, SV_MAX_VOCAB], shared by target and draft rows */
  int32_t max_depth;         /* D in [0, SV_MAX_TREE_DEPTH] */
  float temperature;         /* T > 0 */
  float top_p;               /* in (0, 1]; 1 = no filtering */
  sv_dtype dtype;            /* of both logits arrays */
  int64_t target_row_stride; /* elements between consecutive node rows (>= V) */
  int64_t draft_row_stride;
} sv_tree_sample_desc;

/* Workspace bytes for sv_verify_tree_sample (scratch, no initialisation);
 * 0 for an invalid descriptor. */
size_t sv_tree_sample_workspace_size(const sv_tree_sample_desc* desc);

/*
 * Speculative-sampling verify of B draft token trees at T > 0 ([P2] §5 tree;
 * [P3] §3.1 accept rule, §6.2 shared T and top_p).  The pages give no rule
 * for several drafts at one position; this call uses sequential per-child
 * rejection with a residual update.  At an accepted node, with
 * p = dist(target row), q = dist(draft row) (softmax of top_p_filter(l / T),
 * as in sv_verify_chain), the residual r starts as p; the node's children
 * are tested in increasing node order: a child with token x is accepted iff
 * u_accept[child] * q(x) < r(x); a rejection replaces r by
 * norm(max(0, r - q)) (when that has no mass -- impossible in exact
 * arithmetic for a token the draft could have drawn -- r is kept and
 * SV_ROW_RESAMPLE_FALLBACK is set).  The first accepted child becomes the
 * node.  When every child is rejected the last token is drawn from r, at a
 * node without children from p, by inverse CDF with u_final (first id whose
 * inclusive prefix exceeds u * total).  The emitted tokens follow the
 * target when each node's children are independent draws from its q.
 *
 *   target_logits [B, N] rows of V elements (row b*N+n: the target at node n).
 *   draft_logits  [B, N] rows of V elements (the draft at node n, which the
 *                 children of n were drawn from; rows of leaves are read only
 *                 by the statistics pass).
 *   parents, tokens [B, N] int32 as for sv_verify_tree.
 *   u_accept      [B, N] float in [0, 1): the accept uniform of each node (n = 0 unused).
 *   u_final       [B] float in [0, 1).
 *   accept_len    [B] int32: depth of the last accepted node.
 *   path          [B, D+1] int32: node ids from the root, -1 padded.
 *   out_tokens    [B, D+1] int32: accepted tokens then the drawn token, -1 padded.
 *   row_status    optional [B] int32 (SV_ROW_*): invalid trees and trees with a
 *                 row of no finite logit emit nothing (accept_len 0, -1s).
 *
 * Launches: the row statistics of all 2*B*N rows, then the walk: a cluster
 * of two thread blocks per tree when 2*B does not exceed the SM count (the
 * two split every residual pass), else one block per tree.
 */
sv_status sv_verify_tree_sample(const sv_tree_sample_desc* desc, const void* target_logits,
                                const void* draft_logits, const int32_t* parents, const int32_t* tokens,
                                const float* u_accept, const float* u_final, int32_t* accept_len,
                                int32_t* path, int32_t* out_tokens, int32_t* row_status,
                                void* workspace, size_t workspace_bytes, sv_stream_t stream);

/*
 * Top-k node expansion for building a draft token tree ([P2] §5: every node
 * grows into its top_k draft tokens): the k ids with the highest logits of
 * each row, in descending logit order, equal logits by lower id (-inf ranks
 * last, by id).  NaN logits are never chosen: a row with fewer than k logits
 * that are not NaN ends in ids -1 and values NaN.  No workspace.
 *
 *   logits   [rows] rows of vocab elements (dtype), stride row_stride (>= vocab).
 *   out_ids  [rows, k] int32.
 *   out_vals optional [rows, k] float: the logits of those ids.
 */
typedef struct sv_topk_desc {
  int32_t rows;        /* R >= 0 */
  int32_t vocab;       /* V in [1, SV_MAX_VOCAB] */
  int32_t k;           /* k in [1, min(V, SV_MAX_TOPK)] */
  sv_dtype dtype;
  int64_t row_stride;
} sv_topk_desc;

sv_status sv_topk(const sv_topk_desc* desc, const void* logits, int32_t* out_ids, float* out_vals,
                  sv_stream_t stream);

/*
 * EAGLE3 scatter of small-vocabulary draft logits into the target
 * vocabulary ([P1] §六 compute_logits): out[r, d2t[j]] = in[r, j] for
 * j < draft_vocab; every other entry of the row is `fill` (normally -INFINITY).
 *
 *   draft_logits [rows] rows of draft_vocab elements, stride in_row_stride.
 *   d2t          [draft_vocab] int32, injective into [0, vocab) (unchecked
 *                here: a duplicate makes the surviving value unspecified,
 *                an out-of-range entry is skipped).
 *   t2d          optional [vocab] int32 inverse map (sv_build_t2d).  With it
 *                the kernel gathers and writes each output element once;
 *                without it, it fills each row and then scatters.
 *   out          [rows] rows of vocab elements (same dtype), stride out_row_stride.
 */
sv_status sv_d2t_scatter(const void* draft_logits, int64_t in_row_stride,
                         const int32_t* d2t, const int32_t* t2d,
                         int32_t rows, int32_t draft_vocab, int32_t vocab,
                         sv_dtype dtype, float fill,
                         void* out, int64_t out_row_stride, sv_stream_t stream);

/*
 * Build t2d, the inverse of d2t ([P1] §六): t2d[d2t[j]] = j, every other
 * target id -1.  `status` (optional, one int32) receives 0 on success, bit 1
 * if a d2t entry is outside [0, vocab), bit 2 if two draft ids map to the
 * same target id (t2d is then unspecified at that id).
 */
sv_status sv_build_t2d(const int32_t* d2t, int32_t draft_vocab, int32_t vocab,
                       int32_t* t2d, int32_t* status, sv_stream_t stream);

typedef struct sv_sample_desc {
  int32_t rows;       /* R >= 0 */
  int32_t vocab;      /* V in [1, SV_MAX_VOCAB] */
  sv_dtype dtype;
  float temperature;  /* >= 0; 0 = argmax (lowest id on ties) */
  float top_p;        /* (0, 1] */
  int64_t row_stride;
} sv_sample_desc;

size_t sv_sample_workspace_size(const sv_sample_desc* desc);

/*
 * Draw one token per row from softmax(top_p_filter(logits / T)) with the
 * uniform u[r] (inverse CDF over ascending ids, as in sv_verify_chain).
 * This is the draft side of [P3] §3.1 / §4.2 (the draft loop's temperature,
 * _apply_top_p, softmax and multinomial), with the randomness supplied.
 *   logits [R] rows of V;  u [R] float in [0,1) (may be NULL when T == 0);
 *   out_tokens [R] int32;  out_prob optional [R] float: probability of the
 *   drawn token (1 for T == 0 is not implied: it is the softmax value).
 */
sv_status sv_sample(const sv_sample_desc* desc, const void* logits, const float* u,
                    int32_t* out_tokens, float* out_prob,
                    void* workspace, size_t workspace_bytes, sv_stream_t stream);

/*
 * The filtered distribution of every row: out_probs[r, j] =
 * softmax(top_p_filter(logits[r] / T))[j], with the same top-p rule and tie
 * order as sv_verify_chain ([P3] §4.2: _apply_top_p, then F.softmax).
 * T must be > 0.  logits [R] rows of V (desc->row_stride); out_probs [R]
 * rows of V float (out_row_stride >= V); workspace as for sv_sample.
 */
sv_status sv_softmax_topp(const sv_sample_desc* desc, const void* logits, float* out_probs,
                          int64_t out_row_stride, void* workspace, size_t workspace_bytes,
                          sv_stream_t stream);

/*
 * Profiling hooks (host-side; they add no device work).
 *
 * sv_set_phase_events: the next call into this library made on the calling
 * host thread records events[0] (cudaEvent_t handles created by the caller)
 * on its stream just before its first kernel launch and events[i] right
 * after its i-th launch, for i < n; the hook is then cleared.  n <= 0 or
 * events == NULL clears it.  Under stream capture the records become graph
 * nodes (cudaEventRecordExternal) that fire on every replay.  This lets a
 * caller time each kernel of a call with CUDA events on the stream the
 * kernels run on.
 *
 * sv_launch_count: kernels launched by this library in this process so far.
 */
void sv_set_phase_events(void* const* events, int32_t n);
uint64_t sv_launch_count(void);

/*
 * Bounds-check flags of the debug build (the same sources compiled with
 * -DSV_DEBUG, as libspec_verify_debug.so).  There, every computed or
 * data-dependent index into a caller buffer or a table (a t2d or d2t entry,
 * a parent id, a query element, a draw's chunk or token, a tree walk) is
 * checked before the access; a failed check skips the access and sets bit
 * SV_DEBUG_INDEX in a device word.  No check traps.  sv_debug_flags waits
 * for the device (cudaDeviceSynchronize), returns the OR of the words and
 * clears them when reset != 0.  ~0u: the words could not be read (a CUDA
 * error).  The release build checks nothing and returns 0.
 */
#define SV_DEBUG_INDEX 1u
uint32_t sv_debug_flags(int32_t reset);

/* Static description of a status code. */
const char* sv_status_string(sv_status status);

/* Library version: major * 10000 + minor * 100 + patch. */
int32_t sv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
