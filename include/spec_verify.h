/*
 * spec_verify.h -- C ABI of the GB300 (sm_103a) batched tree speculative-sampling
 * verify library (EAGLE / SpecInfer style).
 *
 * What the operation is (sources cited by page and section):
 *   - p and q are compared after temperature / top-k / top-p / argmax processing
 *     ("LLM speculative decoding: EAGLE", jingming.pro, section 1 note);
 *   - a drafted token x is accepted with probability min(1, p(x)/q(x)); after a
 *     rejection p becomes norm(max(0, p - q)); if every candidate is rejected the
 *     token is resampled from that adjusted distribution, and if every drafted
 *     token along the path is accepted one bonus token is sampled from the next
 *     p (same page, section 2.3 steps 3-5);
 *   - on a draft tree the sampler is applied recursively at every node, trying
 *     the next sibling after a rejection (EAGLE / EAGLE-2 translation,
 *     modelers.csdn.net, sections 1.3.2 and 1.7);
 *   - at temperature 0 the drafted tokens are compared with the target argmax
 *     ("EAGLE close reading", edgeai1.github.io, sections 3 and 5).
 *
 * Conventions shared by every entry point:
 *   - All array arguments are DEVICE pointers owned by the caller, unless stated.
 *     The library allocates nothing and carries no result from one call to the
 *     next.  It does keep small process-wide caches, filled on first use and
 *     never freed: per device, the SM count, whether each kernel's shared-memory
 *     limit has been raised (cudaFuncSetAttribute) and the scratch address of
 *     spec_verify_tree_noalloc; per kernel, its static shared-memory size.  Their
 *     first fill is not synchronised between host threads (make the first call on
 *     a device from one thread); afterwards calls from several threads are safe.
 *     They describe the device and its loaded module: after cudaDeviceReset() in
 *     this process no entry point may be called again (restart the process).
 *   - Every call is asynchronous on `stream` (NULL = the legacy default stream)
 *     and returns before the GPU work finishes; it never synchronises the device.
 *   - The return value is SPEC_OK (0) or a negative SPEC_ERR_* code.  Argument
 *     errors are detected on the host before anything is launched.  Conditions
 *     that depend on device-resident data (a malformed tree, a NaN logit) are
 *     reported per tree in out_status instead.
 *   - Logits are row-major; element (b, n, v) lives at
 *     base + b * batch_stride + n * row_pitch + v (strides in elements).  The base
 *     pointer must be 16-byte aligned and row_pitch * sizeof(elem) and
 *     batch_stride * sizeof(elem) multiples of 16 bytes (batch_stride may be 0:
 *     every tree then reads the same rows).
 *   - Random numbers: Philox4x32-10 (Salmon et al., SC'11) with key
 *     {seed_lo, seed_hi} and counter {node, b, offset_lo, offset_hi}; word 0 is
 *     the accept test of a child node, word 1 the final draw at a node; the
 *     uniform is ((x >> 8) + 1) * 2^-24 in (0, 1].  The same arguments therefore
 *     reproduce the same result bit for bit; callers advance rng_offset per round.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* spec_stream_t;

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;

/* Sampling transforms applied identically to the target row p and the draft row q,
 * in the order temperature -> top-k -> top-p.  Ranking is by raw logit with ties
 * to the lower vocabulary index; top-p keeps the shortest rank-order prefix of the
 * top-k set whose renormalised mass is >= top_p. */
typedef struct {
  float temperature; /* 0: greedy (argmax); > 0: sampling at this temperature */
  int32_t top_k;     /* <= 0 or >= V: off */
  float top_p;       /* >= 1: off; must be > 0 */
  uint32_t flags;    /* SPEC_FLAG_* bits */
} spec_sampling_params;

/* Select the top-k / top-p cut with the full-row radix selection even where the
 * single-pass candidate window would do (both give identical results). */
#define SPEC_FLAG_EXACT_SELECT 1u
/* Self-test of the device-side wait limits (for tests only): the dense row pass
 * withholds the completion of one of its shared-memory copies, so that the bounded
 * wait on it expires (after 20 ms); the affected rows report SPEC_ROW_TIMEOUT and
 * the call still completes. */
#define SPEC_FLAG_TEST_STALL 2u
/* Visited-rows-only schedule (spec_verify_tree and its variants): no dense pass over
 * all B * N rows; the walk computes the statistics (maximum, sum, argmax) of the p
 * and q rows of the nodes it visits, so a step reads about B * (accepted depth + 1)
 * row pairs instead of every row.  Same results.  Ignored by the fused LM-head call,
 * which computes every target row. */
#define SPEC_FLAG_VISITED_ONLY 4u

/* Return codes. */
#define SPEC_OK 0
#define SPEC_ERR_INVALID_ARG (-1)
#define SPEC_ERR_UNSUPPORTED_DTYPE (-2)
#define SPEC_ERR_MISALIGNED (-3)
#define SPEC_ERR_WORKSPACE (-4)
#define SPEC_ERR_CUDA (-5)
#define SPEC_ERR_TOO_LARGE (-6)

/* Per-tree status written to out_status. */
#define SPEC_TREE_OK 0
#define SPEC_ROW_NONFINITE 1 /* a row the walk needed holds NaN or +inf, or is all -inf */
#define SPEC_TREE_INVALID 2  /* parent_idx / draft_tokens malformed, or depth > max_depth */
#define SPEC_ROW_TIMEOUT 3   /* a bounded device-side wait gave up: the row's statistics are
                                not valid (see SPEC_FLAG_TEST_STALL) */

/* Size limits checked on the host. */
#define SPEC_MAX_NODES 4096
#define SPEC_MAX_VOCAB (1 << 21)

/* Statistics of one filtered row (32 bytes).  For a kept token x,
 *   P(x) = exp((z_x - m) / T) / s_f;
 * token x is kept iff key(z_x) > cut_key, or key(z_x) == cut_key and x <= cut_idx,
 * where key() is the order-preserving unsigned image of the fp32 logit
 * (sign bit set -> all bits flipped, else sign bit set; -0 counts as +0).
 * When nothing is truncated (T > 0, top-k and top-p off) every token is kept and
 * the row reports cut_key = 0, cut_idx = V - 1, kept = V. */
typedef struct {
  float m;          /* maximum logit of the row */
  int32_t status;   /* SPEC_TREE_OK, SPEC_ROW_NONFINITE or SPEC_ROW_TIMEOUT */
  double s_f;       /* sum over kept tokens of exp((z - m) / T); 1 at T == 0 */
  uint32_t cut_key; /* key of the last kept token in rank order */
  int32_t cut_idx;  /* vocabulary index of that token */
  int32_t argmax;   /* lowest index of the maximum logit */
  int32_t kept;     /* number of kept tokens */
} spec_row_stats;

/* Work counters of one spec_verify_tree call (algorithmic, not measured bytes). */
typedef struct {
  uint64_t dense_rows;      /* logit rows read by the dense row pass */
  uint64_t dense_bytes;     /* bytes of those rows */
  uint64_t walk_bytes;      /* row bytes read by residual and final-draw passes */
  uint64_t residual_passes; /* rejections that renormalised max(0, p - q) */
  uint64_t final_draws;     /* inverse-CDF draws (corrections and bonus tokens) */
  uint64_t fallback_rows;   /* rows whose cut needed the full-row radix selection */
  uint64_t reserved[2];
} spec_verify_counters;

/* Bytes of device workspace spec_verify_tree needs for B trees of N nodes over a
 * vocabulary of V (the dtype does not change it).  Returns 0 for invalid sizes. */
size_t spec_verify_workspace_size(int32_t B, int32_t N, int32_t V, spec_dtype dtype);

/*
 * Verify B draft trees of N nodes each (node 0 = root, the last accepted prefix
 * token's position; nodes 1..N-1 are drafts).
 *
 * logits_p [B, N, V]: target logits; row n is the target's next-token distribution
 *   after the path root..n.  logits_q [B, N, V]: draft logits; row n is the draft
 *   distribution the children of n were drawn from (siblings share it).  logits_q
 *   may be NULL when temperature == 0 (greedy never reads it).
 * draft_tokens [B, N] int32: token of node n (entry 0 is ignored).
 * parent_idx [B, N] int32: parent of node n; parent_idx[b][0] == -1 and
 *   0 <= parent_idx[b][n] < n for n >= 1.  Trees may differ across b.
 * max_depth: the deepest node of any tree is at most this deep; it sets the
 *   output width W = max_depth + 1.
 * Outputs (device, caller-owned):
 *   out_accept_len [B]: accepted draft tokens (0..depth), -1 for a failed tree;
 *   out_tokens [B, W]: the accepted tokens, then the correction / bonus token,
 *     then -1 padding;
 *   out_accepted_path [B, W]: node 0, then the accepted nodes, then -1 padding;
 *   out_alpha [B, N] (optional, may be NULL): the acceptance probability used for
 *     every tested node, NaN for untested nodes (greedy: 1 accept, 0 reject);
 *   out_status [B] (optional): SPEC_TREE_OK / SPEC_ROW_NONFINITE / SPEC_TREE_INVALID /
 *     SPEC_ROW_TIMEOUT;
 *   out_counters (optional): work counters of this call.
 * workspace: device scratch of at least spec_verify_workspace_size() bytes,
 *   256-byte aligned; its contents are not preserved between calls.
 * Errors: SPEC_ERR_INVALID_ARG (null required pointer, negative or inconsistent
 *   sizes, non-finite or negative temperature, top_p <= 0, unknown flags),
 *   SPEC_ERR_UNSUPPORTED_DTYPE, SPEC_ERR_MISALIGNED, SPEC_ERR_WORKSPACE (too small
 *   or misaligned), SPEC_ERR_TOO_LARGE (N > SPEC_MAX_NODES, V > SPEC_MAX_VOCAB),
 *   SPEC_ERR_CUDA (a launch failed).  B == 0 launches nothing and returns SPEC_OK.
 */
int spec_verify_tree(const void* logits_p, const void* logits_q, spec_dtype dtype, int32_t B,
                     int32_t N, int32_t V, int64_t row_pitch, int64_t batch_stride,
                     const int32_t* draft_tokens, const int32_t* parent_idx, int32_t max_depth,
                     spec_sampling_params params, uint64_t rng_seed, uint64_t rng_offset,
                     int32_t* out_accept_len, int32_t* out_tokens, int32_t* out_accepted_path,
                     float* out_alpha, int32_t* out_status, spec_verify_counters* out_counters,
                     void* workspace, size_t workspace_bytes, spec_stream_t stream);

/* Bytes of the library's own scratch behind spec_verify_tree_noalloc (one copy per
 * device).  With the current workspace layout it holds B * N <= 16376 nodes. */
#define SPEC_STATIC_WORKSPACE_BYTES (1u << 20)

/*
 * spec_verify_tree without a caller workspace and without allocating anything.
 * The method's pages have no counterpart of this call; it exists for callers that
 * must not allocate device memory during a step: cudaMalloc / cudaFree can
 * synchronise the whole device and stall other streams, which a decode loop under
 * a latency budget cannot afford, and a program whose memory pool owns all device
 * memory may forbid allocations it did not make.
 *
 * Arguments, outputs and results are those of spec_verify_tree, minus workspace
 * and workspace_bytes: the scratch is a fixed SPEC_STATIC_WORKSPACE_BYTES array
 * inside this library, one per device, reserved when the library's device code is
 * loaded.  Nothing in it needs to start at zero (the call resets what it reads).
 *
 * Set-up: the first call on a device, with that device current, looks up the
 * scratch's device address (cudaGetSymbolAddress) and caches it; make that first
 * call before any stream capture begins.  Later calls only launch.  The cached
 * address belongs to the device's current context: after cudaDeviceReset() the
 * library's module is loaded anew and the address is stale, so no call may follow
 * a device reset in the same process.
 * Sharing: all calls on one device use the same scratch.  Two calls whose GPU work
 * may overlap (different streams without an ordering event, or concurrent host
 * threads on different streams) race on it and give undefined results; order them
 * on one stream or with events.
 * Errors: as spec_verify_tree; trees too large for the scratch (the workspace that
 * spec_verify_workspace_size reports exceeds SPEC_STATIC_WORKSPACE_BYTES) return
 * SPEC_ERR_TOO_LARGE before anything touches the device; a failed address lookup
 * returns SPEC_ERR_CUDA.
 */
int spec_verify_tree_noalloc(const void* logits_p, const void* logits_q, spec_dtype dtype,
                             int32_t B, int32_t N, int32_t V, int64_t row_pitch,
                             int64_t batch_stride, const int32_t* draft_tokens,
                             const int32_t* parent_idx, int32_t max_depth,
                             spec_sampling_params params, uint64_t rng_seed, uint64_t rng_offset,
                             int32_t* out_accept_len, int32_t* out_tokens,
                             int32_t* out_accepted_path, float* out_alpha, int32_t* out_status,
                             spec_verify_counters* out_counters, spec_stream_t stream);

/* Phases of one verify call, for spec_verify_tree_phases. */
#define SPEC_PHASE_PREPARE 1u /* reset the work counters (when out_counters is requested) */
#define SPEC_PHASE_ROWS 2u    /* dense row pass: statistics of every p row and of the q row
                                 of every node that has a child */
#define SPEC_PHASE_WALK 4u    /* tree checks, the accept walk, residual renormalisation and
                                 the final draw */
#define SPEC_PHASE_ALL 7u

/*
 * spec_verify_tree split into its phases: the phases whose bits are set in
 * `phases` are launched, in the order prepare -> rows -> walk.  Calling it with
 * SPEC_PHASE_PREPARE, then SPEC_PHASE_ROWS, then SPEC_PHASE_WALK on one stream with
 * identical arguments and the same workspace is equivalent to one spec_verify_tree
 * call (which is spec_verify_tree_phases with SPEC_PHASE_ALL); a caller can record
 * events or enqueue other work between the phases.  The workspace carries the state
 * between phases.  Errors as spec_verify_tree; an unknown phase bit or phases == 0
 * is SPEC_ERR_INVALID_ARG.
 */
int spec_verify_tree_phases(uint32_t phases, const void* logits_p, const void* logits_q,
                            spec_dtype dtype, int32_t B, int32_t N, int32_t V, int64_t row_pitch,
                            int64_t batch_stride, const int32_t* draft_tokens,
                            const int32_t* parent_idx, int32_t max_depth,
                            spec_sampling_params params, uint64_t rng_seed, uint64_t rng_offset,
                            int32_t* out_accept_len, int32_t* out_tokens,
                            int32_t* out_accepted_path, float* out_alpha, int32_t* out_status,
                            spec_verify_counters* out_counters, void* workspace,
                            size_t workspace_bytes, spec_stream_t stream);

/* Bytes of device workspace spec_verify_tree_fused_lmhead needs for B trees of N
 * nodes over a vocabulary of V.  Returns 0 for invalid sizes. */
size_t spec_fused_lmhead_workspace_size(int32_t B, int32_t N, int32_t V);

/*
 * Verify with the target logits computed here: p = F W^T, the LM head applied to the
 * feature vector of every tree node (EAGLE obtains the target's next-token
 * distribution of each node from its features this way: "EAGLE close reading",
 * edgeai1.github.io, section 3), on the tensor cores, with the statistics the verify
 * step needs taken from the product before it leaves the chip; then the verify step
 * of spec_verify_tree.
 *
 * features [B*N, d] bf16, row-major (row b*N + n is node n of tree b); lm_head_w
 *   [V, d] bf16, row-major; d a multiple of 8; both 16-byte aligned.
 * logits_q [B, N, V] bf16 draft logits (may be NULL when temperature == 0).
 * out_logits_p [B, N, V] bf16 (device, caller-owned): receives p, rounded to bf16
 *   (the verify step uses these rounded logits).
 * p and q share row_pitch (elements, >= V, row_pitch * 2 a multiple of 16 bytes);
 *   tree b starts at row b * N (batch stride N * row_pitch).
 * All other arguments and outputs as spec_verify_tree; workspace of at least
 * spec_fused_lmhead_workspace_size() bytes, 256-byte aligned.  A device-side wait
 * that gives up marks every tree SPEC_ROW_TIMEOUT.
 * Errors: as spec_verify_tree; SPEC_ERR_MISALIGNED also for d not a multiple of 8.
 */
int spec_verify_tree_fused_lmhead(const void* features, const void* lm_head_w, int32_t d,
                                  const void* logits_q, int32_t B, int32_t N, int32_t V,
                                  int64_t row_pitch, const int32_t* draft_tokens,
                                  const int32_t* parent_idx, int32_t max_depth,
                                  spec_sampling_params params, uint64_t rng_seed,
                                  uint64_t rng_offset, void* out_logits_p,
                                  int32_t* out_accept_len, int32_t* out_tokens,
                                  int32_t* out_accepted_path, float* out_alpha,
                                  int32_t* out_status, spec_verify_counters* out_counters,
                                  void* workspace, size_t workspace_bytes, spec_stream_t stream);

/* Phase of the fused call: the tensor-core LM head and the target rows' statistics
 * (SPEC_PHASE_ROWS then covers the draft rows only). */
#define SPEC_PHASE_LMHEAD 8u
#define SPEC_PHASE_ALL_FUSED 15u

/*
 * spec_verify_tree_fused_lmhead split into its phases, launched in the order
 * prepare -> lmhead -> rows -> walk for the bits set in `phases` (a subset of
 * SPEC_PHASE_ALL_FUSED); calling them one after another on one stream with identical
 * arguments and the same workspace equals one spec_verify_tree_fused_lmhead call.
 * Errors as spec_verify_tree_fused_lmhead; an unknown bit or phases == 0 is
 * SPEC_ERR_INVALID_ARG.
 */
int spec_verify_tree_fused_lmhead_phases(
    uint32_t phases, const void* features, const void* lm_head_w, int32_t d,
    const void* logits_q, int32_t B, int32_t N, int32_t V, int64_t row_pitch,
    const int32_t* draft_tokens, const int32_t* parent_idx, int32_t max_depth,
    spec_sampling_params params, uint64_t rng_seed, uint64_t rng_offset, void* out_logits_p,
    int32_t* out_accept_len, int32_t* out_tokens, int32_t* out_accepted_path, float* out_alpha,
    int32_t* out_status, spec_verify_counters* out_counters, void* workspace,
    size_t workspace_bytes, spec_stream_t stream);

/*
 * The dense row pass alone: filter R rows (row r at logits + r * row_pitch
 * elements) with `params` and write one spec_row_stats per row to out_stats
 * (device, [R]).  Same transforms as spec_verify_tree ("LLM speculative decoding:
 * EAGLE", section 1 note).  Needs no workspace.  Errors as spec_verify_tree.
 */
int spec_filter_rows(const void* logits, spec_dtype dtype, int32_t R, int32_t V,
                     int64_t row_pitch, spec_sampling_params params, spec_row_stats* out_stats,
                     spec_stream_t stream);

/*
 * The Philox4x32-10 words the verify step draws: for i < n, the four 32-bit words
 * of Philox(key = seed, counter = {node_idx[i], b_idx[i], offset_lo, offset_hi})
 * go to out_words[4 i .. 4 i + 3].  b_idx, node_idx, out_words are device arrays.
 */
int spec_philox_words(uint64_t seed, uint64_t offset, const int32_t* b_idx,
                      const int32_t* node_idx, int32_t n, uint32_t* out_words,
                      spec_stream_t stream);

/*
 * Accepted-path commit: after a verify step, keep the cache entries of each tree's
 * accepted path and move them to consecutive positions after the prefix, so the
 * target and draft caches (and the feature cache) continue the accepted sequence
 * ("EAGLE close reading", edgeai1.github.io, section 5: after verification both caches
 * are trimmed to what was accepted).
 *
 * cache: device bytes; the entry of position t of sequence b in plane l (a layer's K
 *   or V, a head, ...) is the row_bytes bytes at
 *   cache + l * plane_stride + b * batch_stride + t * pos_stride (strides in bytes).
 * Node n of tree b sits at position prefix_len[b] + n (node 0, the root, is the last
 *   accepted token); afterwards position prefix_len[b] + k holds node
 *   accepted_path[b][k] for k = 0 .. accept_len[b]; every other position keeps its bytes.
 *   Trees with accept_len < 1 are left as they are.
 * prefix_len [B], accepted_path [B, W], accept_len [B]: device int32 (the verify
 *   outputs); moves whose source or destination is at or beyond n_pos are skipped.
 * The cache, strides and row_bytes must be multiples of 16 bytes; row_bytes <=
 *   pos_stride.  Asynchronous on `stream`; allocates nothing.
 * Errors: SPEC_ERR_INVALID_ARG, SPEC_ERR_MISALIGNED, SPEC_ERR_TOO_LARGE, SPEC_ERR_CUDA.
 */
int spec_commit_accepted_path(void* cache, int32_t B, int32_t n_planes, int32_t n_pos,
                              int64_t plane_stride, int64_t batch_stride, int64_t pos_stride,
                              int64_t row_bytes, const int32_t* prefix_len,
                              const int32_t* accepted_path, const int32_t* accept_len, int32_t W,
                              spec_stream_t stream);

/*
 * Per-request sampling parameters: spec_verify_tree_phases with each tree verified
 * under its own temperature, top-k and top-p (a batch that serves requests with
 * different sampling settings).  temperature [B] (required), top_k [B] and top_p [B]
 * (each may be NULL: off) are DEVICE arrays read by the kernels; tree b is verified
 * exactly as it would be in a spec_verify_tree call with those values, keyed by its
 * own batch index b for the Philox draws.  A tree with temperature 0 takes the greedy
 * argmax chain (its draft rows are not read).  The normalisation is the launch's:
 * top_k <= 0 or >= V is off, top_p >= 1 is off.  A tree whose values are invalid
 * (temperature negative, infinite or NaN; top_p <= 0 or NaN; top_k < 0) gets status
 * SPEC_TREE_INVALID.  logits_q is required.  flags are the launch's SPEC_FLAG_* bits;
 * phases, layouts, workspace, outputs and return codes as spec_verify_tree_phases.
 */
int spec_verify_tree_per_request(uint32_t phases, const void* logits_p, const void* logits_q,
                                 spec_dtype dtype, int32_t B, int32_t N, int32_t V,
                                 int64_t row_pitch, int64_t batch_stride,
                                 const int32_t* draft_tokens, const int32_t* parent_idx,
                                 int32_t max_depth, const float* temperature,
                                 const int32_t* top_k, const float* top_p, uint32_t flags,
                                 uint64_t rng_seed, uint64_t rng_offset, int32_t* out_accept_len,
                                 int32_t* out_tokens, int32_t* out_accepted_path,
                                 float* out_alpha, int32_t* out_status,
                                 spec_verify_counters* out_counters, void* workspace,
                                 size_t workspace_bytes, spec_stream_t stream);

/*
 * Draft-side top-k drafting (EAGLE / EAGLE-2 paper translation, modelers.csdn.net,
 * sections 2.3.1-2.3.2; "LLM speculative decoding: EAGLE", jingming.pro, 4.2.1): for
 * each of R rows of draft logits (a node the draft model expands), the k largest
 * tokens (ties to the lower index, listed in that order) and their confidences, the
 * softmax probability at `temperature` over the whole row.  These are the children
 * (cand_token) and confidences (cand_prob) the dynamic tree below ranks.
 *   logits: device, [R, row_pitch] of dtype, base and row_pitch * sizeof(elem) 16-byte
 *   aligned; out_tokens [R, k] int32, out_probs [R, k] float32, out_status [R] int32
 *   (optional): SPEC_ROW_NONFINITE for a row holding NaN or +inf or all -inf (its
 *   tokens -1 and confidences 0), else SPEC_TREE_OK.
 *   1 <= k <= 32 and k <= V; temperature finite and > 0.
 * Errors: SPEC_ERR_INVALID_ARG, SPEC_ERR_UNSUPPORTED_DTYPE, SPEC_ERR_MISALIGNED,
 * SPEC_ERR_TOO_LARGE (V > SPEC_MAX_VOCAB), SPEC_ERR_CUDA.
 */
int spec_draft_topk(const void* logits, spec_dtype dtype, int32_t R, int32_t V,
                    int64_t row_pitch, int32_t k, float temperature, int32_t* out_tokens,
                    float* out_probs, int32_t* out_status, spec_stream_t stream);

/*
 * Draft LM head + top-k in one call: spec_draft_topk on draft logits formed here,
 * F W^T, from the expanded nodes' draft features F [R, d] (bf16, row-major, device) and
 * the draft LM-head weight W [V, d] (bf16, row-major, device) on the tensor cores.  The
 * bf16 logits go to out_logits [R, logits_pitch] when given (else to the workspace).
 * The children are the k largest of the bf16-rounded logits (ties to the lower index),
 * their confidences the softmax at `temperature` over the row.  1 <= k <= 32, k <= V;
 * d a multiple of 8 and both bases 16-byte aligned (else SPEC_ERR_MISALIGNED).
 * workspace: device, 256-byte aligned, spec_draft_fused_workspace_size(R, V, k) bytes
 * (it holds the logits rows: about 2 R V bytes).
 * Other outputs and errors as spec_draft_topk; a device wait that gave up reports
 * SPEC_ROW_TIMEOUT for every row.
 */
size_t spec_draft_fused_workspace_size(int32_t R, int32_t V, int32_t k);
int spec_draft_topk_fused_lmhead(const void* features, const void* lm_head_w, int32_t d,
                                 int32_t R, int32_t V, int32_t k, float temperature,
                                 void* out_logits, int64_t logits_pitch, int32_t* out_tokens,
                                 float* out_probs, int32_t* out_status, void* workspace,
                                 size_t workspace_bytes, spec_stream_t stream);

/*
 * EAGLE-2 dynamic draft tree (EAGLE / EAGLE-2 paper translation, modelers.csdn.net,
 * sections 2.3.1-2.3.2; "LLM speculative decoding: EAGLE", jingming.pro, 4.2.1).
 * The draft model's candidates of tree b are given in creation order (layer by layer):
 * cand_parent [B, n] (the parent candidate, < its own number, or -1 for a child of
 * the root), cand_token [B, n], cand_prob [B, n] (the draft model's confidence, in
 * [0, 1]).  A candidate's value is the product of the confidences from the root,
 * taken root-first in fp32 (v = v_parent * p, v_root = 1).  All arrays are device
 * arrays; n <= 4096.
 *
 * spec_tree_expand_topk: the expansion step -- the k candidates of [layer_begin,
 *   layer_end) with the largest values (ties to the lower number), into out_idx [B, k]
 *   (-1 where fewer exist).
 * spec_tree_build: the reranking and flattening step -- the m candidates with the
 *   largest values over all layers (a shallower candidate wins a tie, then the lower
 *   number), flattened after the root breadth-first (by depth, then number):
 *   out_tokens [B, m+1] (root_token[b] first), out_parent_idx [B, m+1] (-1 for the
 *   root; the input spec_verify_tree takes), out_position_ids [B, m+1] (depth),
 *   out_src [B, m+1] (candidate number, -1 for the root), out_mask [B, m+1, m+1]
 *   (1 where column j is row i or an ancestor of it: the tree attention mask);
 *   out_status [B] (optional): SPEC_TREE_INVALID for a malformed candidate list (a
 *   parent not before its child, a confidence outside [0, 1] or NaN, a chain deeper
 *   than 64), whose outputs are then -1 (mask 0); SPEC_TREE_OK otherwise.
 *   spec_tree_expand_topk skips malformed candidates.
 * Errors: SPEC_ERR_INVALID_ARG (sizes, null pointers), SPEC_ERR_CUDA.
 */
int spec_tree_expand_topk(const int32_t* cand_parent, const float* cand_prob, int32_t B,
                          int32_t n, int32_t layer_begin, int32_t layer_end, int32_t k,
                          int32_t* out_idx, spec_stream_t stream);
int spec_tree_build(const int32_t* cand_parent, const int32_t* cand_token,
                    const float* cand_prob, const int32_t* root_token, int32_t B, int32_t n,
                    int32_t m, int32_t* out_tokens, int32_t* out_parent_idx,
                    int32_t* out_position_ids, int32_t* out_src, uint8_t* out_mask,
                    int32_t* out_status, spec_stream_t stream);

/*
 * Checked builds.  The library built with -DSPEC_CHECK (build.py's check variant,
 * _build/check/libspecverify_check.so) checks the indices of its dense pass's and
 * walk's buffer accesses on the device; an index out of range sets a bit of that
 * file's error word and is replaced by 0, so the access stays inside its buffer.
 * spec_check_errors writes the dense pass's word to out_words[0] and the walk's to
 * out_words[1] (host memory, 2 words) and clears them; both are 0 when nothing was
 * caught, and always 0 in the regular build.  It waits for the device.  Returns
 * SPEC_OK, SPEC_ERR_INVALID_ARG (NULL out_words) or SPEC_ERR_CUDA.
 * spec_check_build returns 1 in a checked build, else 0.
 */
int spec_check_errors(uint32_t* out_words);
int spec_check_build(void);

/* Static description of a return code (never NULL). */
const char* spec_error_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
