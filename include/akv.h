/*
 * akv.h — C ABI of libakv: the AKV hot path (attention over an active KV
 * cache shaped by append / drop / repos) on NVIDIA GB300 (sm_103a).
 *
 * Method: "Cache Engineering for Agents" (arXiv 2610.28577), as restated by
 * the paper review page (sections 3.3-3.4, 4, 4.2, Appendix A.1.1-A.1.2) and
 * by the explainer page (sections 1-4, the system README).
 *
 * Conventions for every entry point:
 *  - The caller owns every buffer.  No entry point allocates device memory;
 *    calls that need scratch take a caller-provided workspace whose size is
 *    returned by the matching *_workspace* query.  Workspaces must be 256-byte
 *    aligned.
 *  - Pointers documented "device" are CUDA device (or managed) pointers;
 *    "host" pointers are read synchronously during the call and may be
 *    reused as soon as the call returns.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and runs asynchronously: a call does not wait for earlier work
 *    on the stream.  Tables planned on the host are copied to the workspace
 *    through pinned host blocks that the library allocates on first use and
 *    keeps for reuse (at most a few, each reused once its copies have
 *    completed; when all are busy the call waits for the oldest).  Arguments
 *    are validated before any
 *    launch: on AKV_ERR_INVALID / AKV_ERR_UNSUPPORTED / AKV_ERR_WORKSPACE
 *    nothing was enqueued.  AKV_ERR_CUDA reports a failed runtime call or
 *    launch.  Kernels that wait on barriers do so with an iteration limit;
 *    when one gives up it sets a bit in the workspace status word (see
 *    akv_workspace_status) instead of hanging or trapping.
 *  - Tensors are token-major and row-major: Q [T, Hq, D], K and V [T, Hkv, D].
 *    Query head h reads KV head h / (Hq / Hkv) (grouped-query attention).
 *  - dtype AKV_F32 or AKV_BF16; arithmetic accumulates in fp32.  D must be
 *    64, Hq % Hkv == 0.  RoPE pairs coordinate i with i + D/2 and turns the
 *    pair by the angle p * rope_base^(-2i/D); scores are scaled by 1/sqrt(D).
 *  - akv_last_error() returns a thread-local message for the last non-OK
 *    status returned on the calling thread.
 */
#ifndef AKV_H_
#define AKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *akv_stream_t; /* same handle as cudaStream_t */

typedef enum {
  AKV_OK = 0,
  AKV_ERR_INVALID = 1,     /* bad argument or op log; nothing enqueued */
  AKV_ERR_CUDA = 2,        /* CUDA runtime call or kernel launch failed */
  AKV_ERR_WORKSPACE = 3,   /* workspace too small or misaligned */
  AKV_ERR_UNSUPPORTED = 4, /* valid request the kernels do not implement */
  AKV_ERR_DEVICE = 5       /* a kernel reported failure via the status word */
} akv_status;

typedef enum { AKV_F32 = 0, AKV_BF16 = 1 } akv_dtype;

/* One request's cache-operation log in operate-after form (paper review page,
 * section 4 and Figure 6; explainer page section 4, system README).
 * All arrays are host memory.
 *   msg_start   [n_msgs + 1] token CSR: message m holds tokens
 *               msg_start[m] .. msg_start[m+1]-1 (logical order), msg_start[0]
 *               = 0, non-decreasing.  Every message is an implicit append.
 *   drop_after, drop_target  [n_drops]: after message drop_after[i] ends, the
 *               KV of message drop_target[i] leaves the active cache
 *               (drop(P), section 3.3).  0 <= drop_target[i] <= drop_after[i]
 *               < n_msgs.  Dropping an already dropped message is a no-op.
 *   repos_after [n_repos]: after that message ends, the survivors are
 *               renumbered 0..r-1 in logical order (repos, section 3.3).
 *               0 <= repos_after[j] < n_msgs; duplicates are a no-op.
 * At one boundary all drops act before the repos. */
typedef struct {
  int32_t n_msgs;
  const int32_t *msg_start;
  int32_t n_drops;
  const int32_t *drop_after;
  const int32_t *drop_target;
  int32_t n_repos;
  const int32_t *repos_after;
} akv_oplog;

typedef struct {
  int32_t Hq, Hkv, D;
  akv_dtype dtype;
  float rope_base;
} akv_shape;

const char *akv_last_error(void);
const char *akv_version(void);

/* ------------------------------------------------------------------------
 * Segment-batch restoration prefill (paper review page section 4.2,
 * Appendix A.1.1, Figure 10): queries are cut at every boundary carrying a
 * drop or repos; each segment attends causally over its own tokens and the
 * still-active KV of earlier segments, so a dropped entry stays visible to
 * the segments before its drop and is hidden from later ones.  Keys are read
 * at the positions of the version current during the query's segment (the
 * temporary per-segment KV versions of A.1.1).  Equivalently, token t attends
 * over the active cache at its append time (sequential replay, section 3.4).
 * ---------------------------------------------------------------------- */

typedef struct akv_plan akv_plan;

/* Plan a batch of n_req requests on the host (validation, segments, key
 * versions, visibility tile lists).  cu_seqlens: host [n_req + 1], request b
 * owns rows cu_seqlens[b] .. cu_seqlens[b+1]-1 of Q/K/V/out and must have
 * cu_seqlens[b+1]-cu_seqlens[b] == ops[b].msg_start[ops[b].n_msgs].
 * logical_idx: host [T] or NULL; when given, row cu_seqlens[b]+i must carry
 * logical index i (rows are in logical order).  On success *plan_out owns a
 * host object released with akv_plan_destroy.  Returns AKV_ERR_INVALID for a
 * bad op log (target later than its boundary, index out of range, ...). */
akv_status akv_plan_create(const akv_shape *shape, int32_t n_req, const int32_t *cu_seqlens,
                           const int32_t *logical_idx, const akv_oplog *ops,
                           akv_plan **plan_out);

/* Plan with shared prefixes (the prefix sharing of the paper review page
 * section 4.2 radix tree, applied inside one batch: a prefix that several
 * requests hold identically is computed once).  share_from, share_len: host
 * [n_req].  share_from[b] = -1: request b shares nothing.  Otherwise
 * request b's first share_len[b] logical rows are the same tokens as the
 * first share_len[b] rows of request a = share_from[b] < b, and are not in
 * the batch: request b owns rows cu_seqlens[b] .. cu_seqlens[b+1]-1, which
 * carry its logical rows share_len[b] .. T_b-1 (cu_seqlens[b+1] -
 * cu_seqlens[b] == T_b - share_len[b], T_b = ops[b].msg_start[n_msgs]), and
 * its rows read the prefix keys from request a's rows.  Conditions
 * (AKV_ERR_INVALID unless noted): share_len[b] is a message boundary common
 * to both requests with the same message lengths before it, and a multiple
 * of 128 (AKV_ERR_UNSUPPORTED otherwise); no drop of either request targets
 * a message of the prefix; request a shares nothing itself. */
akv_status akv_plan_create_shared(const akv_shape *shape, int32_t n_req,
                                  const int32_t *cu_seqlens, const akv_oplog *ops,
                                  const int32_t *share_from, const int32_t *share_len,
                                  akv_plan **plan_out);
void akv_plan_destroy(akv_plan *plan);

typedef struct {
  int64_t T;              /* rows in the batch */
  int64_t n_qtiles;       /* 128-row query tiles (never straddle a request or version) */
  int64_t n_windows;      /* 128-key windows over all tiles */
  int64_t n_full_windows; /* windows that need no in-tile mask */
  int64_t visible_pairs;  /* sum over rows of visible keys (one head) */
  int64_t n_segments;     /* over all requests */
  int32_t max_versions;   /* key versions (1 + repos count) of the largest request */
  int32_t reserved;
  size_t workspace_bytes; /* for akv_segment_attention_run / _visible_counts */
} akv_plan_info;

akv_status akv_plan_get_info(const akv_plan *plan, akv_plan_info *info);

/* Per-row integer tables of the plan (host outputs, each [T], values
 * request-relative): append position, segment, key version, and the first
 * segment that no longer sees the row's key (INT32_MAX if never dropped). */
akv_status akv_plan_tables(const akv_plan *plan, int32_t *tok_pos, int32_t *tok_seg,
                           int32_t *tok_ver, int32_t *drop_seg);

/* Run a planned prefill.  q [T,Hq,D], k/v [T,Hkv,D]: device, raw (not
 * rotated).  out [T,Hq,D] device.  workspace: device, >= workspace_bytes of
 * the plan info.  The plan tables are copied into the workspace by this call
 * (host -> device on `stream`); the plan may be destroyed once it returns. */
akv_status akv_segment_attention_run(const akv_plan *plan, const void *q, const void *k,
                                     const void *v, void *out, void *workspace,
                                     size_t workspace_bytes, akv_stream_t stream);

/* The two halves of a run, for callers that time or overlap them:
 * akv_segment_prepare uploads the plan tables and writes the rotated and
 * permuted key and value copies (the per-segment temporary KV versions of
 * Appendix A.1.1) into the workspace, with, for bf16, the cos/sin of every
 * query row's angles (fp32: the rotated queries); akv_segment_attend then
 * runs the attention over them.  For bf16 the attention kernel rotates each
 * query row as it loads it, so attend reads q (the same raw queries as
 * prepare; ignored for fp32, may be NULL there).  prepare + attend on one
 * stream == run. */
akv_status akv_segment_prepare(const akv_plan *plan, const void *q, const void *k, const void *v,
                               void *workspace, size_t workspace_bytes, akv_stream_t stream);
akv_status akv_segment_attend(const akv_plan *plan, const void *q, void *out, void *workspace,
                              size_t workspace_bytes, akv_stream_t stream);

/* One-shot form: plan, then run.  Same arguments as the two calls above. */
size_t akv_segment_attention_workspace(const akv_shape *shape, int32_t n_req,
                                       const int32_t *cu_seqlens, const akv_oplog *ops);
akv_status akv_segment_attention(const akv_shape *shape, int32_t n_req, const int32_t *cu_seqlens,
                                 const int32_t *logical_idx, const akv_oplog *ops, const void *q,
                                 const void *k, const void *v, void *out, void *workspace,
                                 size_t workspace_bytes, akv_stream_t stream);

/* Visibility as the attention kernels see it: counts[t] (device int32 [T]) =
 * number of keys row t attends over, enumerated through the plan's key
 * windows and the in-tile mask predicate.  Equals the size of the active
 * cache at the row's append time.  Uses the same workspace as a run. */
akv_status akv_segment_visible_counts(const akv_plan *plan, int32_t *counts, void *workspace,
                                      size_t workspace_bytes, akv_stream_t stream);

/* Reads and clears the status word at the start of a workspace used by the
 * calls above (synchronises `stream`).  *code = 0 when no kernel reported a
 * failure; otherwise a bit mask and the call returns AKV_ERR_DEVICE:
 *   1  a barrier wait in a kernel gave up (its outputs are not valid);
 *   2  (bf16) a rotated query or key, or a value, exceeded the fp16 range
 *      of the tensor-core operands (|value| > 65504). */
akv_status akv_workspace_status(void *workspace, akv_stream_t stream, uint32_t *code);

/* ------------------------------------------------------------------------
 * Compaction (drop, section 3.3; active vs logical trajectory, explainer
 * section 1): the active cache right after the drops of boundary `upto`
 * (-1: the last message), as ascending logical indices active_idx[0..n) and
 * their positions active_pos[0..n) in the version current before any repos
 * listed at `upto` (a repos there moves the j-th survivor to position j).
 * T must equal ops->msg_start[ops->n_msgs].  active_idx/active_pos: device
 * int32 [T] (the first *n_active entries are written).  *n_active: host,
 * known when the call returns. */
size_t akv_compact_workspace(const akv_oplog *ops, int32_t T);
akv_status akv_compact(const akv_oplog *ops, int32_t T, int32_t upto, int32_t *active_idx,
                       int32_t *active_pos, int32_t *n_active, void *workspace,
                       size_t workspace_bytes, akv_stream_t stream);

/* ------------------------------------------------------------------------
 * Cache-history tree and drop-aware eviction (paper review page section
 * 4.2: a radix tree whose paths carry the cache-operation history with the
 * tokens -- drop nodes record removed entries, a repos opens a branch of
 * re-numbered positions; eviction frees KV only when no running request
 * uses it, dropped entries before finished requests' entries, tree nodes
 * kept as placeholders, each position version separately; section 3.4 /
 * Figure 5: equal surviving tokens can hold different KV).  Host only: the
 * tree records which KV exists, the caller owns the KV itself.
 *
 * A history is an op log plus token_ids (host int32 [msg_start[n_msgs]],
 * the messages' token ids).  A message node stands for the KV of that
 * message computed after exactly the history on its path; a boundary's
 * drops (as a set) and repos form one operation node.  Storage units: each
 * message node's own KV, and at each repos node a re-rotated copy of every
 * message alive there (the new position version).
 *
 * akv_tree_match: how much of a new request's history is cached.
 *   matched_msgs: leading messages whose node exists (same tokens after the
 *   same history).  A full match continues from the active cache at the end
 *   of the history; a partial one prefills messages matched_msgs.. over the
 *   messages alive when the first of them starts.  Of those needed
 *   messages' tokens: reuse_tokens have a resident copy at the right
 *   positions (copied as is), rotate_tokens (full match only) only at other
 *   positions (converted by key rotation), restore_tokens none (evicted).
 *   prefill_tokens: tokens of the unmatched messages.  kind: RESTORE if any
 *   needed KV was evicted (one segment-batch prefill restores the state),
 *   else PREFILL_SUFFIX for a partial match, else ROTATE if some KV needs
 *   rotation, else REUSE.
 * akv_tree_insert: the request now runs with this history; its whole path
 *   exists and is resident.  The newest copy of each message active at the
 *   end is pinned by the request; every unit on the path is marked dropped
 *   or not by this request's history.  request_id must not be running.
 * akv_tree_finish: the request ended; its pins are released.
 * akv_tree_evict: frees (marks not resident) unpinned units until `tokens`
 *   tokens are freed or none is left: dropped units first, then by the
 *   insert that last held them (oldest first), then by creation order.
 *   *freed: tokens freed.  A unit's pin count is the number of running
 *   requests whose active cache reads that copy: a reference count per
 *   position version.
 * Errors: AKV_ERR_INVALID for NULL arguments, a bad op log or an unknown /
 * duplicate request_id.
 *
 * Pool trees (drop-aware eviction over a page-size-1 KV pool; the system
 * README: drop and repos support page size 1 only).  akv_tree_create_pool
 * makes a tree that also hands out the n_slots token slots of a caller-owned
 * KV pool (the [S, Hkv, D] pools of the decode entry points, S = n_slots):
 *  - a resident unit owns one slot per token; eviction (akv_tree_evict, or
 *    the automatic one below) puts its slots back on the free list;
 *  - akv_tree_insert gives every unit of the history that is not resident
 *    the lowest free slots.  When too few are free it first evicts other
 *    unpinned units in the order above (never a unit of the history being
 *    inserted); if that is not enough it returns AKV_ERR_WORKSPACE and
 *    leaves the request not running, nothing allocated;
 *  - akv_tree_request_writes lists, per token, the slots that request's
 *    insert allocated, with the token's logical index in the history and
 *    its position there: the caller fills each slot with K rotated at that
 *    position and V of that token (akv_append_kv does exactly this) before
 *    anything reads them;
 *  - akv_tree_request_cache lists the request's active cache at the end of
 *    its history in logical order: slot (the kv_indices of a decode),
 *    logical index and position per token.  The listed units are pinned, so
 *    their slots do not move while the request runs;
 *  - akv_tree_reserve gives a running request n more slots (for its decode
 *    appends), evicting if needed; they are freed when it finishes;
 *  - both lists: int32 host arrays of `cap` entries, any of them NULL; all
 *    NULL returns the count in *n only; a cap below the count is
 *    AKV_ERR_INVALID.  Logical indices and positions are those of the
 *    request's own history.
 * On a tree made by akv_tree_create these calls list slot -1 and
 * akv_tree_reserve returns AKV_ERR_INVALID. */
typedef struct akv_tree akv_tree;
typedef enum {
  AKV_TREE_REUSE = 0,
  AKV_TREE_ROTATE = 1,
  AKV_TREE_PREFILL_SUFFIX = 2,
  AKV_TREE_RESTORE = 3
} akv_tree_kind;
typedef struct {
  int32_t kind; /* akv_tree_kind */
  int32_t matched_msgs;
  int64_t reuse_tokens, rotate_tokens, restore_tokens, prefill_tokens;
} akv_tree_match_result;
typedef struct {
  int64_t nodes, running, resident_tokens, pinned_tokens;
} akv_tree_stats_t;
akv_status akv_tree_create(akv_tree **out);
void akv_tree_destroy(akv_tree *tree);
akv_status akv_tree_match(const akv_tree *tree, const akv_oplog *ops, const int32_t *token_ids,
                          akv_tree_match_result *result);
akv_status akv_tree_insert(akv_tree *tree, const akv_oplog *ops, const int32_t *token_ids,
                           int64_t request_id);
akv_status akv_tree_finish(akv_tree *tree, int64_t request_id);
akv_status akv_tree_evict(akv_tree *tree, int64_t tokens, int64_t *freed);
akv_status akv_tree_stats(const akv_tree *tree, akv_tree_stats_t *stats);
akv_status akv_tree_create_pool(int64_t n_slots, akv_tree **out);
akv_status akv_tree_request_writes(const akv_tree *tree, int64_t request_id, int32_t *slots,
                                   int32_t *logical, int32_t *pos, int64_t cap, int64_t *n);
akv_status akv_tree_request_cache(const akv_tree *tree, int64_t request_id, int32_t *slots,
                                  int32_t *logical, int32_t *pos, int64_t cap, int64_t *n);
akv_status akv_tree_reserve(akv_tree *tree, int64_t request_id, int64_t n, int32_t *slots);
akv_status akv_tree_pool_info(const akv_tree *tree, int64_t *pool_slots, int64_t *free_slots);

/* ------------------------------------------------------------------------
 * Repos / position-version conversion (section 3.3, section 4.2 and
 * Appendix A.1.2): for j in 0..r-1, K_out[j] = R(pos_to[j] - pos_from[j]) *
 * K_in[src_idx[j]] and V_out[j] = V_in[src_idx[j]] (values are copied
 * unchanged).  k_in/v_in: device [*, Hkv, D], keys already rotated at
 * pos_from.  src_idx, pos_from: device int32 [r]; pos_to: device int32 [r] or
 * NULL for pos_to[j] = j (the renumbering 0..r-1 of a repos).  k_out/v_out:
 * device [r, Hkv, D]; they must not overlap the inputs. */
akv_status akv_repos_rotate(const akv_shape *shape, int32_t r, const int32_t *src_idx,
                            const int32_t *pos_from, const int32_t *pos_to, const void *k_in,
                            const void *v_in, void *k_out, void *v_out, akv_stream_t stream);

/* Repos at a boundary in one pass (section 3.3 drop + repos, Appendix
 * A.1.2): the result of akv_compact at `upto` followed by akv_repos_rotate
 * with src_idx = active_idx, pos_from = active_pos, pos_to = NULL, without
 * the index lists.  k_in/v_in: device [T, Hkv, D] by logical index, keys
 * rotated at their positions in the version current before a repos at
 * `upto`.  k_out/v_out: device [>= n, Hkv, D], rows 0..n-1 written, K_out[j]
 * rotated at position j; they must not overlap the inputs.  *n_out: host,
 * the survivor count n (known when the call returns; 0 writes nothing).
 * workspace: device, 256-byte aligned, akv_repos_boundary_workspace() bytes
 * (three small per-message tables, uploaded on `stream`). */
size_t akv_repos_boundary_workspace(const akv_oplog *ops, int32_t T);
akv_status akv_repos_boundary(const akv_shape *shape, const akv_oplog *ops, int32_t T,
                              int32_t upto, const void *k_in, const void *v_in, void *k_out,
                              void *v_out, int32_t *n_out, void *workspace,
                              size_t workspace_bytes, akv_stream_t stream);

/* ------------------------------------------------------------------------
 * Decode over the active cache (paper review page section 4 serving flow,
 * "decode reads only the active cache"; system README: drop/repos support
 * page size 1).  Request b's query q[b] (raw [Hq, D]) is rotated at
 * q_pos[b] and attends over pool slots kv_indices[kv_indptr[b] ..
 * kv_indptr[b+1]) of k_pool/v_pool ([S, Hkv, D], keys stored already
 * rotated).  q_pos, kv_indptr ([B+1]), kv_indices: device int32.  max_kv:
 * host, an upper bound on any request's length (sizes the split-KV grid).
 * out [B, Hq, D] device.  A request with no keys gets zeros.
 * Limits: B <= 65535; bf16: max_kv <= 2,048,000 (AKV_ERR_UNSUPPORTED).
 * Work on `stream` (bf16): with 4, 8 or 16 KV heads, and 2 without
 * rotation on read, the attention launch (one CTA per key chunk and request,
 * all KV heads) and the split merge as a programmatic dependent launch;
 * otherwise a memset of B x Hkv merge counters and one launch that also
 * merges. */
size_t akv_decode_workspace(const akv_shape *shape, int32_t B, int32_t max_kv);
akv_status akv_decode_attention(const akv_shape *shape, int32_t B, const void *q,
                                const int32_t *q_pos, const void *k_pool, const void *v_pool,
                                const int32_t *kv_indptr, const int32_t *kv_indices,
                                int32_t max_kv, void *out, void *workspace, size_t workspace_bytes,
                                akv_stream_t stream);

/* Decode with the step's append fused (inside the attention launch):
 * request b's new token -- raw k_new[b] (device [B, Hkv, D]),
 * v_new[b] -- is written into pool slot new_slot[b] (device int32 [B]),
 * its key rotated at q_pos[b] exactly as akv_append_kv would, before the
 * request's keys are read; kv_indices of request b must end with
 * new_slot[b].  Otherwise as akv_decode_attention (same workspace size). */
akv_status akv_decode_attention_append(const akv_shape *shape, int32_t B, const void *q,
                                       const int32_t *q_pos, const void *k_new,
                                       const void *v_new, const int32_t *new_slot, void *k_pool,
                                       void *v_pool, const int32_t *kv_indptr,
                                       const int32_t *kv_indices, int32_t max_kv, void *out,
                                       void *workspace, size_t workspace_bytes,
                                       akv_stream_t stream);

/* Decode with rotation on read (the fused append and in-kernel repos of a
 * serving step; paper review page section 3.3: a key moves between positions
 * by a rotation, values are unchanged).  Same as akv_decode_attention except
 * that k_pool holds keys BEFORE RoPE and kv_pos (device int32, parallel to
 * kv_indices) gives each entry's current position: the kernel rotates each
 * key by R(kv_pos[e]) as it reads it.  A repos then only rewrites kv_pos
 * (e.g. 0..r-1) and the index order; no key is moved or re-rotated.
 * Fused append (optional): k_new, v_new (device [B, Hkv, D], raw) and
 * new_slot (device int32 [B]) are copied into pool slot new_slot[b] before
 * that request's keys are read; request b's index list must then end with
 * new_slot[b] (and its kv_pos entry with q_pos[b]).  Pass all three or none.
 * k_pool/v_pool are written only at those slots.  Workspace: device,
 * 256-byte aligned, akv_decode_rope_workspace() bytes (split-KV partials
 * of 512-key chunks; bf16 adds the merge counters of akv_decode_attention).  bf16: keys are rotated in fp32 and rounded to fp16
 * for the score product, so a rotated key component must stay below 65504
 * in magnitude (a larger one becomes inf); the query keeps ~22 bits as fp16
 * hi + lo parts. */
size_t akv_decode_rope_workspace(const akv_shape *shape, int32_t B, int32_t max_kv);
akv_status akv_decode_attention_rope(const akv_shape *shape, int32_t B, const void *q,
                                     const int32_t *q_pos, const void *k_new, const void *v_new,
                                     const int32_t *new_slot, void *k_pool, void *v_pool,
                                     const int32_t *kv_indptr, const int32_t *kv_indices,
                                     const int32_t *kv_pos, int32_t max_kv, void *out,
                                     void *workspace, size_t workspace_bytes,
                                     akv_stream_t stream);

/* Decode without a workspace.  The paper has no counterpart: this entry
 * point exists for callers that cannot allocate device memory, so cannot
 * pass the workspace akv_decode_attention needs -- for example a plug-in
 * running inside a host framework that owns the whole device memory pool and
 * gives plug-ins no allocation hook, or a request path that must not
 * allocate per call.  Same arguments, semantics and results as
 * akv_decode_attention, minus the workspace: the split-KV partials go to a
 * fixed array in the library's device memory,
 * akv_decode_static_scratch_bytes() bytes (16 MiB) on every GPU where the
 * library's decode module is loaded (see Set-up), held until the process
 * exits.  Nothing is allocated by the call (no cudaMalloc/cudaFree, no allocating library routine).
 *  - Limit: the bytes akv_decode_workspace() returns for the same shape, B
 *    and max_kv (split-KV partials, B * Hq * ceil(max_kv / 1024) * 66 * 4
 *    bytes, plus B * Hkv * 4 bytes of merge counters, each part rounded up
 *    to 256) must fit the array; larger requests return
 *    AKV_ERR_UNSUPPORTED with the sizes in akv_last_error(), before
 *    anything is enqueued.
 *  - Set-up: the array lives in the library module that holds the decode
 *    kernels.  With CUDA's default lazy module loading that module (and
 *    its 16 MiB) is loaded on a device the first time one of the decode
 *    entry points runs there, so the reservation can fail then if the
 *    device is already full; with CUDA_MODULE_LOADING=EAGER it is loaded
 *    with the library.  A call with B = 0 does only this set-up (no launch;
 *    only `shape` is read): a caller that wants the memory reserved up
 *    front makes that call at initialisation, with the device current.
 *    Every call looks the array's address up again (cudaGetSymbolAddress
 *    in the current context, which allocates nothing), so a device reset or
 *    a different context made current between calls does not leave it
 *    writing through a stale address.  Make the first call on a device
 *    before any stream capture.
 *  - Sharing: every call on a device uses the same array.  Calls that
 *    overlap on the GPU (other streams, other host threads) race and corrupt
 *    each other's results; serialise them.  The array keeps the last call's
 *    contents; the call writes every partial it later reads (and, for
 *    head counts other than 2, 4, 8 and 16, first clears the merge
 *    counters with a memset on `stream`). */
akv_status akv_decode_attention_static(const akv_shape *shape, int32_t B, const void *q,
                                       const int32_t *q_pos, const void *k_pool,
                                       const void *v_pool, const int32_t *kv_indptr,
                                       const int32_t *kv_indices, int32_t max_kv, void *out,
                                       akv_stream_t stream);
size_t akv_decode_static_scratch_bytes(void);

/* Debug check of decode index data.  The decode entry points trust
 * kv_indptr / kv_indices (an out-of-range slot would be read from the pool);
 * this call checks them on the device without reading any pool slot:
 * kv_indptr (device int32 [B+1]) starts at 0 and every request's length is
 * in [0, max_kv]; kv_indptr[B] <= n_indices (the entries allocated in
 * kv_indices, device int32); every listed slot is in [0, S) (S = pool rows).
 * Violations are OR-ed into *status (device uint32, which the caller zeroes
 * first): bit 0 (1) the index pointer, bit 1 (2) a slot.  Asynchronous on
 * `stream`; read *status after synchronising.  No counterpart on the pages:
 * the check stands in for a memory checker on data the kernels trust. */
akv_status akv_decode_check_indices(int32_t B, const int32_t *kv_indptr, const int32_t *kv_indices,
                                    int32_t n_indices, int32_t S, int32_t max_kv, uint32_t *status,
                                    akv_stream_t stream);

/* Append (section 3.3): for i in 0..n-1, k_pool[slot[i]] = R(pos[i]) *
 * k_new[i] and v_pool[slot[i]] = v_new[i].  k_new/v_new: device [n, Hkv, D]
 * raw; pos, slot: device int32 [n]; slots must be distinct. */
akv_status akv_append_kv(const akv_shape *shape, int32_t n, const void *k_new, const void *v_new,
                         const int32_t *pos, const int32_t *slot, void *k_pool, void *v_pool,
                         akv_stream_t stream);

/* ------------------------------------------------------------------------
 * Decoder layers of a single-prefill restoration (paper review page section
 * 4.2, Appendix A.1.1, Figure 10): attention is cut into segments, every
 * other layer op (projections, FFN) runs once over the whole batched
 * sequence.  Pre-norm layer: a = RMSNorm(h); q,k,v = a Wq^T, a Wk^T, a Wv^T;
 * h += SegmentAttention(q,k,v) Wo^T; f = RMSNorm(h);
 * h += (silu(f Wg^T) * (f Wu^T)) Wd^T.  The residual stream h is fp32.
 * ---------------------------------------------------------------------- */

/* Y[M,N] (+)= X[M,K] * W[N,K]^T on the tensor cores.  x: device bf16 [M,K];
 * w: device bf16 [N,K] (row n = output feature n); y: device, out_mode 0 =
 * bf16 [M,N] store, 1 = fp32 store, 2 = fp32 y += product.  N % 32 == 0,
 * K % 8 == 0, pointers 16-byte aligned. */
akv_status akv_gemm_bf16(int32_t M, int32_t N, int32_t K, const void *x, const void *w, void *y,
                         int32_t out_mode, akv_stream_t stream);

/* y[r] = x[r] / sqrt(mean(x[r]^2) + eps) * weight (weight NULL = ones).
 * x, y: device [rows, d] of the given dtypes; weight: device fp32 [d]. */
akv_status akv_rmsnorm(int32_t rows, int32_t d, float eps, akv_dtype in_dtype, const void *x,
                       const float *weight, akv_dtype out_dtype, void *y, akv_stream_t stream);

/* out = silu(g) * u element-wise, bf16 [n]; out may equal g. */
akv_status akv_swiglu(int64_t n, const void *g, const void *u, void *out, akv_stream_t stream);

/* Weights of one layer, device bf16, each [out_features][in_features]:
 * wq [Hq*D][d], wk and wv [Hkv*D][d], wo [d][Hq*D], wg and wu [d_ff][d],
 * wd [d][d_ff]. */
typedef struct {
  const void *wq, *wk, *wv, *wo, *wg, *wu, *wd;
} akv_layer_weights;

/* n_layers decoder layers over the planned batch (plan: bf16, its op logs
 * shape every layer's attention the same way), then a final RMSNorm.
 * layers: host array [n_layers]; x: device bf16 [T, d_model] embeddings;
 * out: device fp32 [T, d_model].  workspace >= akv_decoder_workspace();
 * it starts with the status word read by akv_workspace_status. */
size_t akv_decoder_workspace(const akv_plan *plan, int32_t d_model, int32_t d_ff);
akv_status akv_decoder_forward(const akv_plan *plan, int32_t n_layers,
                               const akv_layer_weights *layers, int32_t d_model, int32_t d_ff,
                               float eps, const void *x, float *out, void *workspace,
                               size_t workspace_bytes, akv_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* AKV_H_ */
