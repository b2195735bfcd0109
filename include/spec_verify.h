/*
 * spec_verify.h -- C ABI of the GB300 (sm_103a) batched draft-token
 * verification library for speculative decoding.
 *
 * The operation is the Leviathan/Chen verification step:
 *   - "Speculative decoding and EAGLE" (aiengineeringfromscratch.com, Phase 10
 *     lesson 25), section "The concept" (K draft tokens, one target pass over
 *     K+1 positions, accept the longest matching prefix, one bonus token when
 *     all K are accepted), section "The exactness rule" (accept x_t if
 *     r < p(x_t)/q(x_t), else draw from (p - q)+ / ||(p - q)+||_1 and stop;
 *     greedy case: accept iff argmax(p) == x_t, else emit argmax(p)) and
 *     section "Tree attention verification" (verify a candidate tree in one
 *     pass, keep the longest accepted branch);
 *   - "Speculative decoding: draft, verify, repeat" (Phase 07 lesson 16),
 *     steps 1-3 (accept_or_reject, residual_dist, bonus token);
 *   - "Speculative Decoding: from idea to SOTA" (mountainai.tech), section 3
 *     (alpha(x) = min(1, p(x)/q(x)); p'(x) = max(0, p(x) - q(x)) / sum).
 *
 * Conventions shared by every entry point:
 *   - All array pointers are DEVICE pointers, row-major and contiguous, with
 *     the vocabulary as the innermost dimension.  The caller owns every buffer;
 *     the library allocates nothing.  Scratch memory ("workspace") is supplied
 *     by the caller, sized by spec_workspace_bytes / spec_tree_workspace_bytes.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     are asynchronous on that stream and never synchronise; results are valid
 *     once the stream has reached the call.  A workspace must not be shared by
 *     calls that may overlap on the GPU.
 *   - Argument errors are detected on the host, before any launch, and return
 *     SPEC_ERR_INVALID_ARG / SPEC_ERR_UNSUPPORTED / SPEC_ERR_WORKSPACE; a
 *     failed launch returns SPEC_ERR_CUDA.  spec_last_error() then describes it.
 *   - Bad data is reported per sequence, never by trapping: num_accepted[b] =
 *     -1 and out_tokens[b, :] = -1 when the sequence has a draft token outside
 *     [0, V) or its verification reads an invalid row (a row with NaN; for
 *     softmax rows also +inf or no finite entry).  num_accepted[b] = -2 means an
 *     internal pipeline wait hit its time limit (every wait in the library is
 *     bounded).
 *   - Vector path: rows whose byte length V * elem_size is a multiple of 16 (and
 *     16-byte aligned base pointers) are streamed with bulk async copies; other
 *     shapes take a scalar path with identical results.
 *   - The vector-path kernels of spec_verify_sample, spec_verify_greedy and
 *     spec_verify_tree_greedy are persistent grids whose CTAs wait on one
 *     another (fixed owner CTAs per sequence, shared work queues), so they are
 *     launched cooperatively: the grid is sized to what the device holds at
 *     once, and where fewer SMs are available than the device reports (an MPS
 *     share, a green context, another cooperative kernel running) the launch
 *     fails with SPEC_ERR_CUDA instead of starting a grid that could stall.
 *     The sampling kernel clears its own control block, so it needs no memset.
 *   - No C++ exception crosses this interface.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SPEC_OK = 0,
  SPEC_ERR_INVALID_ARG = 1, /* NULL pointer, bad size, bad temperature, ... */
  SPEC_ERR_UNSUPPORTED = 2, /* shape beyond a documented limit             */
  SPEC_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed        */
  SPEC_ERR_WORKSPACE = 4    /* workspace missing or too small               */
} spec_status_t;

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype_t;

typedef enum { SPEC_DRAFT_LOGITS = 0, SPEC_DRAFT_PROBS = 1 } spec_draft_kind_t;

/* Limits.  K (draft length) is 0..SPEC_MAX_K; tree node count 1..SPEC_MAX_TREE_NODES. */
#define SPEC_MAX_K 31
#define SPEC_MAX_TREE_NODES 1024

/* Scratch bytes needed by spec_verify_sample / spec_verify_greedy /
 * spec_debug_residual for a batch of B sequences, draft length K, vocabulary
 * V.  Pure host function; 0 for invalid sizes. */
size_t spec_workspace_bytes(int B, int K, int V);

/* Scratch bytes needed by spec_verify_tree_greedy for B sequences of N tree
 * nodes over vocabulary V.  Pure host function; 0 for invalid sizes. */
size_t spec_tree_workspace_bytes(int B, int N, int V);

/* Sampling-mode verification of one speculative step for B sequences.
 *
 *   target_logits [B, K+1, V] (target_dtype): target logits at the K drafted
 *       positions and the one after them.
 *   draft [B, K, V]: draft logits (draft_kind = SPEC_DRAFT_LOGITS, any
 *       spec_dtype_t) or draft probabilities (SPEC_DRAFT_PROBS, SPEC_F32 only,
 *       used exactly as given).  May be NULL when K == 0.
 *   draft_tokens [B, K] int32: the drafted tokens x_t.  May be NULL when K == 0.
 *   uniforms [B, K+1, 2] float32 in [0, 1): uniforms[b,t,0] drives the accept
 *       test at position t, uniforms[b,t,1] the replacement draw at the stopping
 *       position (residual at a rejection, bonus at t == K).
 *   temperature: > 0 and finite; the target and draft logits are both divided
 *       by it before the softmax.  temperature == 0 selects the greedy rule
 *       (identical to spec_verify_greedy; draft and uniforms are then unused).
 *
 * Per sequence: p_t = softmax(target[b,t]/T), q_t = softmax(draft[b,t]/T) (or
 * the given probabilities); for t = 0..K-1 accept x_t iff q_t(x_t) == 0 or
 * uniforms[b,t,0] < p_t(x_t)/q_t(x_t); at the first rejection draw
 * v = smallest index whose running sum of w = max(0, p_t - q_t) exceeds
 * uniforms[b,t,1] * sum(w) (sum(w) == 0 falls back to w = p_t) and stop; if
 * all K are accepted draw the bonus the same way from p_K.
 *
 * Outputs: out_tokens [B, K+1] int32 = the accepted drafts, then the drawn
 * token, then -1 padding; num_accepted [B] int32 = the number of accepted
 * drafts (0..K), or -1 / -2 as described above.
 *
 * Limits: V >= 1; V <= 393216 (SPEC_ERR_UNSUPPORTED beyond). */
spec_status_t spec_verify_sample(const void *target_logits, spec_dtype_t target_dtype,
                                 const void *draft, spec_dtype_t draft_dtype,
                                 spec_draft_kind_t draft_kind, const int32_t *draft_tokens,
                                 const float *uniforms, float temperature, int B, int K, int V,
                                 int32_t *out_tokens, int32_t *num_accepted, void *workspace,
                                 size_t workspace_bytes, void *stream);

/* spec_verify_sample without a caller workspace; it allocates nothing.  The
 * method on the pages has no counterpart: this is an interface variant for
 * callers that cannot hand over device scratch at call time, e.g. a plain C
 * decode loop with no device allocator of its own, or one that must not call
 * cudaMalloc/cudaFree between steps because those synchronise the device.
 *
 * Arguments, semantics, outputs and errors are those of spec_verify_sample.
 * Scratch comes from a fixed 16 MiB (16777216-byte) device array inside the
 * library.  A batch whose spec_workspace_bytes(B, K, V) exceeds that returns
 * SPEC_ERR_UNSUPPORTED (spec_last_error() gives both sizes); B=256, K=5,
 * V=128256 needs 3.4 MB and fits.
 *
 * The first call on each device (with that device current) looks up the
 * array's device address with cudaGetSymbolAddress, which may load the
 * library's device code; make that first call before any stream capture.
 * Later calls on that device reuse the address while its context lives: the
 * first call after the context was re-created (cudaDeviceReset, or a released
 * and re-created primary context) looks the address up again.
 *
 * The array is shared by every call on a device: calls that may overlap on the
 * GPU (different streams, different host threads) race on it and must be
 * serialised by the caller.  Each call clears the part that must start at zero
 * (the kernel's control block and counters) on its own stream before its
 * kernel runs. */
spec_status_t spec_verify_sample_noalloc(const void *target_logits, spec_dtype_t target_dtype,
                                         const void *draft, spec_dtype_t draft_dtype,
                                         spec_draft_kind_t draft_kind,
                                         const int32_t *draft_tokens, const float *uniforms,
                                         float temperature, int B, int K, int V,
                                         int32_t *out_tokens, int32_t *num_accepted, void *stream);

/* Greedy verification ("The exactness rule", greedy case): g_t = argmax of
 * target row t (lowest index on ties, raw logits, no temperature); accept x_t
 * while g_t == x_t; emit g_t at the first mismatch, or g_K when all K match.
 * Shapes and outputs as spec_verify_sample. */
spec_status_t spec_verify_greedy(const void *target_logits, spec_dtype_t target_dtype,
                                 const int32_t *draft_tokens, int B, int K, int V,
                                 int32_t *out_tokens, int32_t *num_accepted, void *workspace,
                                 size_t workspace_bytes, void *stream);

/* Greedy tree verification ("Tree attention verification").
 *
 *   target_logits [B, N, V]: one logit row per tree node; node i's row is the
 *       target's distribution for the token that follows node i.
 *   parents [N] int32 (device): parents[0] = -1 (the root), 0 <= parents[i] < i.
 *   node_tokens [B, N] int32: the token each node proposes (node 0 ignored; a
 *       token outside [0, V) never matches).
 *   max_depth: the tree's depth (longest root-to-node edge count); outputs have
 *       max_depth + 1 columns.
 *
 * Node 0 is accepted; node i is accepted iff its parent is and node_tokens[b,i]
 * == argmax of the parent's row.  The deepest accepted node i* (ties to the
 * smallest index) is kept: out_tokens [B, max_depth+1] = the tokens on the path
 * root -> i* (root excluded), then argmax of i*'s row, then -1 padding;
 * num_accepted [B] = depth(i*); out_path [B, max_depth+1] (optional, may be
 * NULL) = the node ids on that path (root excluded), -1 padded.  A malformed
 * topology or a depth above max_depth gives -1 for every sequence. */
spec_status_t spec_verify_tree_greedy(const void *target_logits, spec_dtype_t target_dtype,
                                      const int32_t *parents, const int32_t *node_tokens, int B,
                                      int N, int V, int max_depth, int32_t *out_tokens,
                                      int32_t *num_accepted, int32_t *out_path, void *workspace,
                                      size_t workspace_bytes, void *stream);

/* Diagnostic twin of spec_verify_sample: runs the same pipeline, but forces
 * sequence `debug_b` to stop at position `debug_t` (0..K; K = the bonus row)
 * and writes the normalised replacement distribution the device computed
 * there, w / sum(w) as float32, to out_row [V] (device), and sum(w) to
 * out_mass [1] (device).  out_tokens / num_accepted receive the pipeline's
 * outputs (sequence debug_b's entry reflects the forced stop). */
spec_status_t spec_debug_residual(const void *target_logits, spec_dtype_t target_dtype,
                                  const void *draft, spec_dtype_t draft_dtype,
                                  spec_draft_kind_t draft_kind, const int32_t *draft_tokens,
                                  const float *uniforms, float temperature, int B, int K, int V,
                                  int debug_b, int debug_t, float *out_row, float *out_mass,
                                  int32_t *out_tokens, int32_t *num_accepted, void *workspace,
                                  size_t workspace_bytes, void *stream);

/* Test hook for the bounded waits (no counterpart on the pages): runs
 * spec_verify_sample with every device-side wait limited to timeout_us
 * microseconds (100..1000000) while the accept scan of sequence stall_b waits
 * for one sweep unit more than the call produces, so that wait runs out.  The
 * call must end with num_accepted[b] = -2 and out_tokens[b, :] = -1 for every
 * b, and leave the context and the workspace usable.  Needs the fused
 * sampling path (T > 0, 16-byte aligned rows); SPEC_ERR_UNSUPPORTED otherwise. */
spec_status_t spec_debug_stall(const void *target_logits, spec_dtype_t target_dtype, const void *draft,
                               spec_dtype_t draft_dtype, spec_draft_kind_t draft_kind, const int32_t *draft_tokens,
                               const float *uniforms, float temperature, int B, int K, int V, int stall_b,
                               unsigned timeout_us, int32_t *out_tokens, int32_t *num_accepted, void *workspace,
                               size_t workspace_bytes, void *stream);

/* Tree attention mask ("Speculative decoding and EAGLE", section "Tree
 * attention verification"; "Speculative Decoding: from idea to SOTA",
 * section 6): when the draft proposes a tree, the target scores all of it in
 * one pass under a mask in which every node attends only to its ancestors and
 * itself.
 *
 *   parents [B, N] int32 (device): one tree per sequence, parents[b, 0] = -1
 *       and 0 <= parents[b, i] < i (breadth-first or any topological order).
 *   masks [B, N, ceil(N/32)] uint32 (device, written): bit j % 32 of word
 *       j / 32 of row i is set iff node j is node i or one of its ancestors.
 *   status [B] int32 (device, written): 0, or -1 when the sequence's parents
 *       break the rule above (its mask is then all zero).
 *
 * Limits: 1 <= N <= 1024. */
spec_status_t spec_tree_mask(const int32_t *parents, int B, int N, uint32_t *masks, int32_t *status,
                             void *stream);

/* Commit on accept for the KV cache ("Speculative decoding: draft, verify,
 * repeat", KV rollback): the verification pass writes the drafts' entries to a
 * scratch buffer; only the accepted ones are appended to the cache, so a
 * rejection leaves the cache at the accepted length.
 *
 *   cache [B, Lmax, entry_bytes] (device, appended to in place).
 *   lengths [B] int32 (device): the cache lengths before the call.
 *   scratch [B, N, entry_bytes] (device): the entries of the verified positions.
 *   path [B, W] int32 (device) or NULL: the scratch slots to append, in order
 *       (e.g. out_path of spec_verify_tree_greedy); NULL means slots 0, 1, ...
 *       (a chain: the first num_accepted drafts).
 *   count [B] int32 (device): entries to append (e.g. num_accepted); a
 *       negative count appends nothing.
 *   new_lengths [B] int32 (device, written): lengths + count; lengths when
 *       count < 0; -1 (nothing appended) when the append would pass Lmax, a
 *       slot is outside [0, N) or count > W with a path.
 *
 * Entries are opaque bytes (call once for keys and once for values, or lay
 * them out together).  new_lengths must not alias lengths. */
spec_status_t spec_kv_commit(void *cache, const int32_t *lengths, const void *scratch, const int32_t *path,
                             const int32_t *count, int B, int Lmax, int N, int W, size_t entry_bytes,
                             int32_t *new_lengths, void *stream);

/* Acceptance statistics of a draft against its target, per drafted position
 * ("Speculative decoding: draft, verify, repeat", step 4: acceptance rate
 * against the divergence between the draft and the verifier; "Speculative
 * Decoding: from idea to SOTA", section 3: x_t is accepted with probability
 * min(1, p/q), so position t is accepted with probability sum_v min(p_t, q_t)).
 *
 *   target_logits [B, K+1, V], draft [B, K, V], draft_kind, temperature: as in
 *       spec_verify_sample (the same buffers may be passed); row K of the
 *       target is not read.  temperature must be > 0.
 *   alpha, kl, tv [B, K] float32 (device, written):
 *       alpha[b,t] = sum_v min(p_t(v), q_t(v)),
 *       kl[b,t]    = KL(q_t || p_t) = sum_{v: q>0} q log(q / p) (natural log),
 *       tv[b,t]    = 1/2 sum_v |p_t(v) - q_t(v)|.
 *   An invalid row pair (a logit row with NaN or +inf or no finite entry; draft
 *   probabilities with NaN or a negative entry) gives NaN in all three; -2 in all
 *   three means an internal wait hit its time limit.
 *
 * Each row pair is read from HBM once.  Draft logits of the target's dtype in
 * rows that 16-byte bulk copies can stream and that exceed 64 KB per pair go
 * through one CTA per SM that reads each pair twice, the second time from L2;
 * every other case through one thread-block cluster per pair that holds it in
 * shared memory.  Limits:
 * V * (target + draft element bytes) <= 1.6 MB, i.e. V <= 409600 for bf16
 * pairs (SPEC_ERR_UNSUPPORTED beyond); 1e-4 <= T. */
spec_status_t spec_row_stats(const void *target_logits, spec_dtype_t target_dtype, const void *draft,
                             spec_dtype_t draft_dtype, spec_draft_kind_t draft_kind, float temperature, int B,
                             int K, int V, float *alpha, float *kl, float *tv, void *stream);

/* Top-k tree drafting ("Speculative decoding and EAGLE", section "Make it": an
 * EAGLE-style drafter builds a candidate tree whose branches are the top-k
 * tokens at each node; exercise 4: the top-3 branches at each depth instead of
 * a chain).  The step that selects the tree's tokens from the draft's logits,
 * without the draft model.
 *
 *   draft_logits [B, N, V] (draft_dtype): one draft row per tree node; row p is
 *       the draft's distribution for the token after node p (rows of leaves are
 *       not read).
 *   parents [N] int32 (device): parents[0] = -1, 0 <= parents[i] < i.
 *   max_children: 1..16, the most children any node may have (a node with
 *       more makes the topology invalid, below).
 *   temperature: > 0; only the log-probabilities depend on it.
 *   node_tokens [B, N] int32 (device, written): the children of node p, in
 *       increasing node index, take the tokens of row p in decreasing logit
 *       order (equal logits: the smaller index first); node 0 gets -1.
 *   node_logq [B, N] float32 (device, written): log q(token) with
 *       q = softmax(row p / T) for each child; 0 for node 0.
 * The children of an invalid row (NaN, +inf, or no finite entry) get -1 and
 * NaN, as do children whose rank is >= V.  A malformed topology, or a node with
 * more than max_children children, gives -1 / NaN for every node.  A row
 * whose copy wait hit its time limit gives its children -2 / NaN.
 * node_tokens and parents can be passed on to spec_tree_mask and
 * spec_verify_tree_greedy.  Limits: N <= 1024. */
spec_status_t spec_tree_draft(const void *draft_logits, spec_dtype_t draft_dtype, const int32_t *parents, int B,
                              int N, int V, int max_children, float temperature, int32_t *node_tokens,
                              float *node_logq, void *stream);

/* Timing hooks for benchmarks: while enabled, each verify call records CUDA
 * events on the call's stream around its kernels (at most max_calls calls are
 * recorded).  spec_profile_end synchronises on the recorded events and returns
 * the summed milliseconds of each part and the number of recorded calls.  For
 * two-kernel paths the parts are the vocabulary sweep and the finishing
 * kernel; the fused sampling path is one kernel, timed as the first part (the
 * second part is then ~0).  Not thread-safe. */
spec_status_t spec_profile_begin(int max_calls);
spec_status_t spec_profile_end(float *sweep_ms, float *finish_ms, int *calls);

/* Human-readable name of a status; description of the most recent failure on
 * the calling thread. */
const char *spec_status_string(spec_status_t status);
const char *spec_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
