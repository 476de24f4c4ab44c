/*
 * graft.h — C ABI of the Graft hot path on one GPU (sm_103a).
 *
 * Graft (arXiv 2605.20104, "prune then graft" hybrid draft trees for lossless
 * speculative decoding) runs one decode step as:
 *   1. a calibrated confidence check at draft depths 0, 1 and 5 that may stop
 *      the drafter early and split a fixed 60-slot verification budget
 *      between draft and retrieval nodes (8+52, 24+36, 40+20, or 60+0);
 *   2. a retrieval subtree gathered from a GPU-resident continuation matrix
 *      C[V][8] (the 8 most likely successors of every token), expanded from
 *      the current token by an asymmetric template;
 *   3. the hybrid tree flattened into tokens, parent indices, tree positions
 *      and an ancestor mask;
 *   4. greedy verification against the target's logits (longest accepted
 *      path, ties to the lower token id);
 *   5. the online update: every verified position, accepted or rejected,
 *      overwrites C[its token] with the top-8 of its logits row.
 * Around the step: warm-up of the matrix, incremental drafting (checkpoint
 * verdicts as the drafter's layers complete, the retrieval gathered beside
 * the drafter), the ablations without retrieval or with a fixed split,
 * threshold calibration, the coverage-gain diagnostic, and lossless
 * stochastic verification at a temperature.
 * Sources: Hugging Face paper page 2605.20104 (abstract); popular-science
 * article on the paper, section 二 (the three gears: steps 1-5), section 三
 * (superset argument, coverage gain), section 四 (static-tree batched mode),
 * section 五 (ablations), section 六 (warm-up), section 七 (Graft-TAIL).
 *
 * Conventions (all entry points):
 *   - Pointers named d_* are DEVICE pointers owned by the caller; they must
 *     stay valid until the work queued on `stream` has finished.  `stream` is
 *     a cudaStream_t (NULL = legacy default stream).  Each must be aligned to
 *     its element size (GRAFT_EINVAL otherwise); the logits are read with
 *     16-byte loads when the rows start on 16-byte boundaries, with element
 *     loads otherwise.
 *   - Every call is asynchronous and stream-ordered unless stated otherwise.
 *     Argument errors are returned at once and nothing is queued.
 *   - Device-side data errors (token id out of range, NaN logits or
 *     probabilities, malformed trees) set a sticky device error word; the
 *     kernels then keep every access in bounds and finish.  graft_sync()
 *     returns GRAFT_EDEVICE and clears the word.
 *   - The handle owns the continuation matrix and all scratch memory.  A
 *     handle is not thread-safe; queue all its work on one stream at a time.
 *   - Return value: GRAFT_OK (0) or a negative graft_status; the message of
 *     the last failure is available from graft_last_error().
 */
#ifndef GRAFT_H_
#define GRAFT_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct graft_handle graft_handle;

typedef enum {
  GRAFT_OK = 0,
  GRAFT_EINVAL = -1,   /* bad argument; nothing was queued */
  GRAFT_ENOMEM = -2,   /* allocation failed (graft_init; graft_template on the host) */
  GRAFT_ECUDA = -3,    /* a CUDA call failed */
  GRAFT_EDEVICE = -4   /* a kernel flagged bad data (see graft_sync) */
} graft_status;

/* Device error word bits (graft_sync's *out_flags). */
#define GRAFT_ERR_TOKEN 1u   /* a token id outside [0, V) (input or matrix) */
#define GRAFT_ERR_NAN 2u     /* NaN in a logits row or a draft probability */
#define GRAFT_ERR_TREE 4u    /* parent index not before its child, bad position */
#define GRAFT_ERR_TIMEOUT 8u /* a bounded wait inside a kernel expired; that call's results are invalid */

typedef enum {
  GRAFT_MODE_CHECKPOINT = 0, /* article §二: checkpoints at depths 0/1/5 */
  GRAFT_MODE_STATIC = 1,     /* article §四: fixed slots, in-place replacement */
  GRAFT_MODE_TAIL = 2        /* article §七: block draft, tail replaced */
} graft_mode;

typedef enum { GRAFT_F32 = 0, GRAFT_BF16 = 1 } graft_dtype;

typedef struct {
  int32_t vocab;          /* V >= 1 */
  int32_t topk;           /* successors per matrix row; must be 8 */
  int32_t budget;         /* verification slots besides the root (60; 16 for tail); S = budget + 1 <= 64 */
  int32_t max_batch;      /* largest batch passed to assemble / verify_update */
  int32_t mode;           /* graft_mode */
  int32_t logits_dtype;   /* graft_dtype of every logits buffer */
  int32_t ckpt_depth[3];  /* checkpoint draft layers, checked in this order (0, 1, 5) */
  float ckpt_thr[3];      /* fire when the layer's best path confidence < thr (0.30, 0.20, 0.10); in [0, 1] */
  int32_t ckpt_draft[3];  /* draft slots kept when that checkpoint fires (8, 24, 40); retrieval gets the rest */
  int32_t tpl_depth;      /* retrieval template depth (8) */
  int32_t tpl_width;      /* template root width; rank-r node fan-out max(1, width >> r), at most 8 (8) */
  float static_thr;       /* static mode: nodes with path confidence < thr are replaced (0.15); in [0, 1] */
  float tail_thr;         /* tail mode: first block position with confidence < thr starts the tail (0.4); in [0, 1] */
  int32_t max_draft_nodes;/* largest draft tree (<= 256) or block (<= budget) per request */
  int32_t scan_kernel;    /* verify scan: 0 = automatic (cluster per row when every row's
                             cluster fits on the GPU at once and a row's eighth is at most
                             48 KB, else two-pass with unit maxima on
                             16-byte aligned rows, else single-pass), 1 = single-pass with a shared
                             running top-8, 2 = TMA-pipelined (aligned rows of >= 32 KB only),
                             3 = two-pass with unit maxima (pass 2 reads every candidate unit
                             again), 4 = two-pass with unit records (maximum, second largest,
                             position of the maximum: pass 2 reads again only units with two
                             elements at or above its threshold, pass 1 does more work per
                             unit); 3 and 4 take aligned rows only; 5 = cluster per row (one
                             thread-block cluster of 8 CTAs stages each row in shared memory and
                             selects its top-8 on chip, one launch; up to 256 rows whose eighth
                             fits 200 KB, else as 3) */
  int32_t ablation;       /* checkpoint mode only (article §五 ablations; 0 elsewhere):
                             0 = Graft, 1 = confidence pruning without retrieval (the freed
                             slots stay empty), 2 = fixed split (no checkpoints: the top
                             fixed_draft nodes of the whole tree plus budget - fixed_draft
                             retrieval slots, every step) */
  int32_t fixed_draft;    /* draft slots of the fixed split, in [0, budget] (40) */
} graft_config;

/* Fill *cfg with the paper's defaults for `mode` and vocabulary V. */
void graft_default_config(graft_config* cfg, int32_t vocab, int32_t max_batch, int32_t mode,
                          int32_t logits_dtype);

/* Create a handle on the current CUDA device: allocates the continuation
 * matrix (V x 8 int32, every entry -1 = empty), builds the retrieval template
 * and allocates scratch.  Synchronous.  *out receives the handle. */
int graft_init(const graft_config* cfg, graft_handle** out);

/* Free everything the handle owns (synchronises the device first). */
int graft_destroy(graft_handle* h);

/* Warm-up bulk load (article §六): for n = 0..n_rows-1 in order,
 *   C[d_tokens[n]] <- top-8 ids of logits row n  (value descending, id ascending),
 * so the last occurrence of a token wins.  d_logits row n starts at element
 * n * row_stride (row_stride >= V).  Rows whose token recurs later are not read:
 * the last occurrences are listed on the device, the first 4096 of them (on
 * 16-byte aligned rows) take the two-pass scan, any others the single-pass
 * scan.  Queues five or six kernels; no host synchronisation. */
int graft_warmup(graft_handle* h, const int32_t* d_tokens, const void* d_logits, int64_t n_rows,
                 int64_t row_stride, void* stream);

/* Steps 1-3 for `batch` requests (article §二 gears 1-2 and the flatten of
 * gear 3; §四 in static mode; §七 in tail mode).  Inputs per request b:
 *   d_root_tok[b]                     last emitted token (the tree root)
 *   checkpoint / static mode:
 *     d_draft_tok[b][n], d_draft_parent[b][n] (int16, -1 = child of the root,
 *     else an earlier index: BFS order), d_draft_aux[b][n] = the node's draft
 *     probability given its parent, n = draft_nodes
 *   tail mode:
 *     d_draft_tok[b][n] block tokens, d_draft_aux[b][n] per-position
 *     confidences; d_draft_parent is ignored (may be NULL)
 * Outputs per request, S = budget + 1 slots (slot 0 = root):
 *   d_tree_tok[b][S]    token, -1 for a pad slot
 *   d_tree_parent[b][S] parent slot (int8), -1 for the root and pads
 *   d_tree_pos[b][S]    tree position = depth below the root, -1 for pads
 *   d_tree_mask[b][S]   bit j set iff slot j is an ancestor of (or is) the slot
 *   d_info[b][4]        {event, kept draft nodes, realised retrieval nodes, valid slots}
 *                       event = fired depth or -1 (checkpoint), replaced nodes
 *                       (static), tail start t (tail)
 * Reads the matrix as it stands when the kernel runs. */
int graft_assemble(graft_handle* h, int32_t batch, const int32_t* d_root_tok, const int32_t* d_draft_tok,
                   const int16_t* d_draft_parent, const float* d_draft_aux, int32_t draft_nodes,
                   int32_t* d_tree_tok, int8_t* d_tree_parent, int32_t* d_tree_pos, uint64_t* d_tree_mask,
                   int32_t* d_info, void* stream);

/* graft_assemble plus where each slot's token came from:
 *   d_slot_src[b][S]    0 = the root, 1 = a kept draft node, 2 = the matrix
 *                       (a retrieval node; in static mode an in-place
 *                       replacement), -1 = a pad slot
 * so a caller can tell which accepted tokens retrieval contributed (the
 * pages' retrieval hit rate), also in static mode where the replacements do
 * not follow the draft slots.  Same work otherwise; GRAFT_EINVAL for a NULL
 * d_slot_src with batch > 0. */
int graft_assemble_src(graft_handle* h, int32_t batch, const int32_t* d_root_tok, const int32_t* d_draft_tok,
                       const int16_t* d_draft_parent, const float* d_draft_aux, int32_t draft_nodes,
                       int32_t* d_tree_tok, int8_t* d_tree_parent, int32_t* d_tree_pos, uint64_t* d_tree_mask,
                       int32_t* d_info, int8_t* d_slot_src, void* stream);

/* Incremental drafting (article §二 gears 1-2; checkpoint mode only).  The
 * checkpoints exist to stop the drafter early, and the retrieval gather runs
 * beside the drafter instead of after it.  A drafter that expands its tree
 * layer by layer calls, per step:
 *   1. d_event[b] = -1 for every request (caller-owned int32[batch]);
 *   2. after completing layer L (nodes of layers <= L in BFS order, the same
 *      arrays graft_assemble takes, draft_nodes of them per request):
 *      graft_check(..., L, d_event) -- every checkpoint whose layer is <= L is
 *      evaluated in order for requests whose event is still -1; the first
 *      that fires writes its depth.  A request that fired stops growing: its
 *      later layers are not drafted;
 *   3. at any point after its last graft_check, possibly on another stream
 *      while the drafter works on other requests: graft_retrieve(...) gathers
 *      every fired request's retrieval entries from the matrix into
 *      d_retrieved[b][budget] (template order, -1 = not realised);
 *   4. graft_assemble_staged(...) with the final tree: the same outputs as
 *      graft_assemble on that tree (checkpoints are not re-evaluated, entries
 *      are not gathered again), at the cost of the flatten alone.
 * The matrix must not change between steps 3 and 4 (graft_verify_update and
 * graft_warmup write it).  Under the fixed-split ablation graft_check does
 * nothing and graft_retrieve gathers budget - fixed_draft entries for every
 * request.  All three are asynchronous on `stream`; argument errors return
 * GRAFT_EINVAL at once (also in static and tail modes).  An event that is not
 * a checkpoint depth counts as no firing and sets GRAFT_ERR_TREE. */
int graft_check(graft_handle* h, int32_t batch, const int16_t* d_draft_parent, const float* d_draft_prob,
                int32_t draft_nodes, int32_t layer, int32_t* d_event, void* stream);
int graft_retrieve(graft_handle* h, int32_t batch, const int32_t* d_root_tok, const int32_t* d_event,
                   int32_t* d_retrieved, void* stream);

int graft_assemble_staged(graft_handle* h, int32_t batch, const int32_t* d_root_tok, const int32_t* d_draft_tok,
                          const int16_t* d_draft_parent, const float* d_draft_prob, int32_t draft_nodes,
                          const int32_t* d_event, const int32_t* d_retrieved, int32_t* d_tree_tok,
                          int8_t* d_tree_parent, int32_t* d_tree_pos, uint64_t* d_tree_mask, int32_t* d_info,
                          void* stream);

/* The retrieval template (article §二, second gear: rank paths below the
 * anchor; the rank-r successor of a node has max(1, width >> r) children of
 * its own, the anchor min(8, width); depth <= `depth`; entries in increasing
 * (rank sum, depth, rank path) order).  Host only, no handle, no GPU: writes
 * the first min(len, template size) entries -- the template graft_init builds
 * from tpl_depth / tpl_width, of which a split with R retrieval slots uses
 * the first R -- as parent_out[j] (index of the parent entry, -1 = the
 * anchor), rank_out[j] (the matrix column the entry gathers, 0..7) and
 * depth_out[j] (1 = a child of the anchor).  Entry j is d_retrieved[b][j] of
 * graft_retrieve.  The caller owns the three arrays (len int32 each; they may
 * be null when len is 0).  Returns the number of entries written, or
 * GRAFT_EINVAL for depth outside [1, 16], width outside [1, 64], len outside
 * [0, 65536] or a null array. */
int graft_template(int32_t depth, int32_t width, int32_t len, int32_t* parent_out, int32_t* rank_out,
                   int32_t* depth_out);

/* Threshold calibration (article §二: the checkpoint thresholds are set from
 * the distribution of path confidences seen during warm-up).
 * graft_confidence: d_best[b][k] = best path confidence of request b's draft
 *   nodes at checkpoint layer ckpt_depth[k] (-1 when that layer is empty);
 *   checkpoint and static modes.  Asynchronous on `stream`.
 * graft_calibrate_thresholds (host only, no handle): thr_out[k] = the
 *   nearest-rank `quantile` (in (0, 1]) of the non-negative best[i][k],
 *   i < n_rows: the smallest sample value with at least that fraction of the
 *   sample at or below it.  GRAFT_EINVAL if a checkpoint has no sample.
 * graft_set_thresholds: replace the handle's ckpt_thr (each in [0, 1]); later
 *   calls use them. */
int graft_confidence(graft_handle* h, int32_t batch, const int16_t* d_draft_parent, const float* d_draft_prob,
                     int32_t draft_nodes, float* d_best, void* stream);
int graft_calibrate_thresholds(const float* best, int32_t n_rows, double quantile, float* thr_out);
int graft_set_thresholds(graft_handle* h, const float* thr);

/* Coverage gain of the retrieval graft (article §三), a diagnostic; checkpoint
 * and tail modes.  For request b, with the tree and info record graft_assemble
 * wrote and the target's logits of that tree (as graft_verify_update takes
 * them): every retrieved slot whose parent is a kept slot (the root, or the
 * last kept block token) carries a boundary candidate, new unless a kept draft
 * child of the same parent has the same token; d_gain[b] = the sum over the
 * new candidates of softmax(parent's row)[token], in fp32.  Reads one logits
 * row per boundary parent.  Asynchronous on `stream`. */
int graft_coverage(graft_handle* h, int32_t batch, const int32_t* d_tree_tok, const int8_t* d_tree_parent,
                   const int32_t* d_info, const void* d_logits, int64_t row_stride, float* d_gain, void* stream);

/* Steps 4-5 (article §二 gear 3, §三): one pass over the logits of every
 * valid slot (the two-pass scan re-reads the few 512-byte pieces of a row
 * that can hold its largest values; for small steps each row is staged in
 * the shared memory of a thread-block cluster and read once) computes its
 * top-8 (element 0 = the greedy argmax), then
 *   accepted(i)  <=> every non-root node j on the root->i path has
 *                    tok[j] == argmax(row of parent(j));
 *   winner       =  the accepted slot of greatest position (ties: lower slot);
 *   d_accept_len[b] = position of the winner;
 *   d_out_tokens[b][S] = the winner's path tokens after the root, then the
 *                        bonus token argmax(row of winner), then -1s;
 * and every valid slot overwrites C[its token] with its top-8 (the last
 * writer in (request, slot) order wins).  Pad slots (tok < 0) are not read;
 * a request without a valid root (all its slots pads) gets d_accept_len 0
 * and d_out_tokens all -1.
 * The tree arrays are those written by graft_assemble (or equivalent ones).
 * d_logits row (b, i) starts at element (b*S + i) * row_stride (row_stride >= V). */
int graft_verify_update(graft_handle* h, int32_t batch, const int32_t* d_tree_tok, const int8_t* d_tree_parent,
                        const int32_t* d_tree_pos, const uint64_t* d_tree_mask, const void* d_logits,
                        int64_t row_stride, int32_t* d_accept_len, int32_t* d_out_tokens, void* stream);

/* Stochastic variant of graft_verify_update (article §二 third gear: the
 * output distribution equals sampling from the target at `temperature`).
 * The top-8 of every valid row and the matrix update are those of
 * graft_verify_update; acceptance instead walks the tree from the root: at
 * node n with p = softmax(row_n / temperature), n's children are tested in
 * slot order, child c accepted when d_u_accept[b][c] * rem < p(token of c),
 * rem being the mass of the tokens not yet rejected at n (a repeated token
 * has none left); acceptance descends into c.  When every child of n is
 * rejected, or n is a leaf, the final token is the first v (in id order)
 * whose cumulative mass among the unrejected tokens exceeds
 * d_u_resid[b] * their total.  Every emitted token is so distributed exactly
 * as the target's p, whatever the candidates.
 *   d_u_accept  DEVICE float [batch][S], uniforms in [0, 1), one per slot
 *   d_u_resid   DEVICE float [batch], uniforms in [0, 1)
 *   d_accept_len[b] = accepted path length; d_out_tokens[b] = path tokens,
 *   then the final token, then -1s.  Probabilities are computed in fp32.
 * Asynchronous; GRAFT_EINVAL for a temperature that is not finite and > 0,
 * or whose inverse is not finite (below about 3e-39). */
int graft_verify_update_sample(graft_handle* h, int32_t batch, const int32_t* d_tree_tok, const int8_t* d_tree_parent,
                               const int32_t* d_tree_pos, const uint64_t* d_tree_mask, const void* d_logits,
                               int64_t row_stride, float temperature, const float* d_u_accept,
                               const float* d_u_resid, int32_t* d_accept_len, int32_t* d_out_tokens, void* stream);

/* Allocation-free variant of graft_verify_update.  It has no counterpart in
 * the paper: it is an integration entry point for callers that cannot call
 * cudaMalloc, such as an engine that records its decode step into a CUDA
 * graph (allocation is not allowed while a stream is being captured) or one
 * whose device memory is fully pre-planned by its own arena or by another
 * runtime's caching allocator.  Those callers cannot create a graft_handle,
 * so this call takes the continuation matrix as a caller buffer and runs the
 * single-pass scan and finishing kernels (graft_verify_update's path for
 * unaligned rows; same results) on fixed scratch memory compiled into the
 * library.
 *   vocab, logits_dtype      as in graft_config
 *   batch, slots             requests and slots per request (S); batch * slots
 *                            must be <= GRAFT_NOALLOC_MAX_ROWS, slots <= 64
 *   d_tree_*, d_logits, row_stride, d_accept_len, d_out_tokens
 *                            as in graft_verify_update
 *   d_matrix                 DEVICE [vocab][8] int32 continuation matrix, read
 *                            and updated in place (-1 = empty entry)
 *   d_err_flags              DEVICE uint32 word the kernels OR GRAFT_ERR_* bits
 *                            into; the caller zeroes and reads it
 * The scratch is a fixed GRAFT_NOALLOC_BYTES device array: every GPU that
 * loads the library holds it until the process exits, and all calls share it,
 * so calls that overlap on the GPU (for example on two streams at once) race.
 * Nothing is carried from one call to the next.  The first call on a device
 * looks up the array's device address (cudaGetSymbolAddress, no allocation);
 * make that first call before any stream capture.  The address is tied to
 * the device's context: the first call after cudaDeviceReset (or after the
 * primary context was released and made again) looks it up anew, so make
 * that call outside a capture too.  The current device must be the device of
 * `stream` and of every d_* buffer.  Asynchronous; returns GRAFT_EINVAL for
 * bad arguments, sizes beyond the limit or a stream of another device
 * (nothing queued), GRAFT_ECUDA if a CUDA call fails. */
#define GRAFT_NOALLOC_MAX_ROWS 2048
#define GRAFT_NOALLOC_BYTES (GRAFT_NOALLOC_MAX_ROWS * (16 * 8 * 8 + 4 + 8 * 4))
int graft_verify_update_noalloc(int32_t vocab, int32_t logits_dtype, int32_t batch, int32_t slots,
                                const int32_t* d_tree_tok, const int8_t* d_tree_parent, const int32_t* d_tree_pos,
                                const uint64_t* d_tree_mask, const void* d_logits, int64_t row_stride,
                                int32_t* d_matrix, int32_t* d_accept_len, int32_t* d_out_tokens,
                                uint32_t* d_err_flags, void* stream);

/* Copy the continuation matrix (V x 8 int32, row-major) to / from HOST memory.
 * Synchronous with respect to `stream`. */
int graft_get_matrix(graft_handle* h, int32_t* host_out, void* stream);
int graft_set_matrix(graft_handle* h, const int32_t* host_in, void* stream);

/* Device pointer to the continuation matrix (V x 8 int32), owned by the handle. */
int32_t* graft_matrix_device_ptr(graft_handle* h);

/* Synchronise `stream`, read and clear the device error word.  *out_flags
 * (may be NULL) receives the GRAFT_ERR_* bits.  Returns GRAFT_EDEVICE if any
 * bit was set. */
int graft_sync(graft_handle* h, void* stream, uint32_t* out_flags);

/* Message of the last failed call on this handle ("" if none). */
const char* graft_last_error(const graft_handle* h);

/* Kernel timing (tracing).  Every call that queues work is also wrapped in an
 * NVTX range named after it (graft_verify_update, ...), visible to profilers
 * that record NVTX.  When enabled, every kernel this handle launches
 * is bracketed by two CUDA events recorded on the call's stream (a few
 * hundred nanoseconds each).  graft_profile_read synchronises the device and
 * writes, for the kernels of the most recent calls since the last read (at
 * most `max` of them), their names (static strings) and durations in
 * milliseconds; it returns the number written and forgets them. */
int graft_profile_enable(graft_handle* h, int32_t on);
int graft_profile_read(graft_handle* h, const char** names, float* ms, int32_t max);

/* Number of kernel launches the last graft_assemble / graft_verify_update /
 * graft_warmup call queued. */
int32_t graft_last_launch_count(const graft_handle* h);

/* Failure detection: the kernels that stage logits with bulk copies (the
 * TMA-pipelined verify scan, scan_kernel 2, the cluster-per-row verify,
 * scan_kernel 5 or the automatic choice for small steps, and the stochastic
 * walk of graft_verify_update_sample on aligned rows) bound every
 * mbarrier wait by a number of polls; on expiry they set GRAFT_ERR_TIMEOUT in
 * the handle's error word, stop issuing copies, wait (for about a second at
 * most) for the copies they have in flight, and finish, leaving the handle
 * usable; the step's outputs are then invalid.  This call sets that limit for later calls on the handle
 * (polls = 0 restores the default of 2^22 polls), so a test can make the
 * waits run out on purpose.  It has no counterpart in the paper. */
int graft_set_wait_limit(graft_handle* h, uint32_t polls);

#ifdef __cplusplus
}
#endif
#endif /* GRAFT_H_ */
