/*
 * sfi.h -- C ABI of libsfi, the GB300 (sm_103a) decode-attention hot path of
 * Slow-Fast Inference (SFI), with the Vegas-style aggregated selection.
 *
 * Method sources (web-page summaries, cited by page title and section):
 *  - "Slow-Fast Inference: Training-Free Inference Acceleration via
 *    Within-Sentence Support Stability" (gist.science 2603.12038; Italian,
 *    Portuguese and Korean pages), sections "Slow-Fast paradigm" (fast and
 *    slow steps), "Selector" (evidence, prior, reverse-KL fusion and its
 *    closed form s = (1-lambda) f + lambda r, Top-K) and "System design".
 *  - "Vegas: self-speculative decoding with verification-guided sparse
 *    attention" (gist.science 2602.07223, Italian page), sections 2.A
 *    (aggregated attention-logit selection) and 2.B (Collect-2-Query).
 *
 * Conventions shared by every call
 *  - Ownership: the caller owns every buffer and the stream.  Calls other
 *    than sfi_ctx_create allocate nothing; scratch comes from a caller-owned
 *    device workspace whose size the matching *_workspace_size call returns.
 *    A workspace must be zero-filled (cudaMemsetAsync) before its first use;
 *    every call that returns SFI_OK and whose device status (sfi_read_status)
 *    stays 0 leaves it ready for the next call.  After a nonzero device
 *    status, zero-fill it again: its work and merge counters may be left
 *    mid-count.  Calls that share one workspace must not overlap on the GPU.
 *  - Asynchrony: every call only enqueues kernels on `stream` (a
 *    cudaStream_t; NULL is the legacy default stream) and returns.
 *  - Errors: arguments are validated on the host before anything is
 *    launched; on failure nothing is enqueued and the status names the
 *    problem, with a message from sfi_last_error() (thread-local).  Kernels
 *    never trap: anomalies they detect (a length beyond the capacity, an
 *    index outside the eligible range, a pipeline wait that timed out) set
 *    bits of a status word in the workspace, read with sfi_read_status.
 *  - Data types: q, k and v share one type (SFI_F32 or SFI_BF16).  Outputs
 *    (attention output, evidence, key norms, fused scores, logit sums) are
 *    fp32; positions are int32.  All arithmetic accumulates in fp32.
 *  - Shapes: B sequences, H_q query heads, H_kv KV heads (H_kv divides H_q;
 *    query head h reads KV head h / (H_q / H_kv)), head_dim d in {64, 128}.
 *  - KV cache layout (per layer): sequence b's block starts kv_offset[b]
 *    elements into k (and v) and is [H_kv][kv_cap[b]][d] row-major, so row i
 *    of KV head g is at k + kv_offset[b] + (g * kv_cap[b] + i) * d.  Rows must
 *    start on 16-byte boundaries (d * element size is a multiple of 16 and
 *    kv_offset[b] * element size is too).
 *  - n_b = len[b] is the cache length of sequence b including the current
 *    token; positions 0..n_b-1 are valid.
 *  - Per-position outputs (f, knorm, s, logit sums) of sequence b and KV head
 *    g are rows of length max_len at (b * H_kv + g) * max_len; entries at or
 *    past n_b are left untouched.
 *  - Capacity limits (SFI_ERR_CAPACITY beyond them): batch <= 1024;
 *    batch * n_kv_heads <= 4096; for every call that selects (sfi_select,
 *    sfi_select_refined, a decode context) max_len <= 327680 positions per
 *    row.  Further per-call limits are stated with the call.
 */
#ifndef SFI_H_
#define SFI_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SFI_OK = 0,
  SFI_ERR_INVALID_ARG = 1, /* null pointer, bad size, inconsistent shape */
  SFI_ERR_UNSUPPORTED = 2, /* dtype, head_dim or group size not built */
  SFI_ERR_CAPACITY = 3,    /* a size beyond a documented limit */
  SFI_ERR_WORKSPACE = 4,   /* workspace null or smaller than required */
  SFI_ERR_CUDA = 5         /* a CUDA runtime call failed */
} sfi_status;

typedef enum { SFI_F32 = 0, SFI_BF16 = 1 } sfi_dtype;

/* Device status bits (sfi_read_status). */
#define SFI_DEV_LEN_OVER_CAP   0x1u  /* len[b] > kv_cap[b] or len[b] > max_len */
#define SFI_DEV_BAD_INDEX      0x2u  /* a selected position outside [0, n_b) */
#define SFI_DEV_WAIT_TIMEOUT   0x4u  /* a pipeline wait gave up */
#define SFI_DEV_ITEMS_OVERFLOW 0x8u  /* more work items than the workspace holds */
#define SFI_DEV_REFINE         0x10u /* a refinement met an inconsistent candidate list */

typedef void* sfi_stream; /* a cudaStream_t */

/* Batch and cache geometry of one layer.  Device pointers: kv_offset, kv_cap,
 * len.  max_len (host) bounds every len[b]; it sizes grids, workspaces and
 * the per-position output rows. */
typedef struct {
  int32_t batch;
  int32_t n_q_heads;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t dtype; /* sfi_dtype */
  int32_t max_len;
  const int64_t* kv_offset; /* device [B], elements */
  const int32_t* kv_cap;    /* device [B], positions per KV head */
  const int32_t* len;       /* device [B], n_b including the current token */
} sfi_layout;

/* Selection and managed-state parameters (SFI pages, "Slow-Fast paradigm":
 * sink tokens, a recent window of about 256 tokens, selected memory). */
typedef enum {
  SFI_SELECT_FUSED = 0,         /* SFI: s = (1-lambda) f + lambda r per (b, KV head) */
  SFI_SELECT_LOGIT_SUM_SEQ = 1, /* Vegas: top-k of the logit sum over all heads, one set per b */
  SFI_SELECT_LOGIT_SUM_HEAD = 2 /* Vegas grouped per KV head: top-k of each KV head's logit sum */
} sfi_select_mode;

typedef struct {
  int32_t n_sink; /* sinks: positions [0, n_sink) */
  int32_t window; /* recent window: [max(n_sink, n - window), n), holds the current token */
  int32_t k;      /* selected positions per (sequence, KV head); idx rows have stride k */
  float lambda;   /* weight of the prior in the fusion, in [0, 1] */
  int32_t mode;   /* sfi_select_mode */
} sfi_params;

/* ---------------------------------------------------------------- errors */

/* Message of the last failed call on this thread ("" if none). */
const char* sfi_last_error(void);

/* Copy the workspace's device status word to *status_host (synchronises
 * `stream`) and clear it.  Returns SFI_ERR_CUDA if the copy fails. */
sfi_status sfi_read_status(void* ws, uint32_t* status_host, sfi_stream stream);

/* Number of streaming multiprocessors of the current device (host query). */
int32_t sfi_device_sm_count(void);

/* Failure detection (no counterpart on the pages): every attention and
 * verify launch gives each consumer warp's wait for a stage of cache rows a
 * limit in SM clocks, and every selector launch each wait of its chunk CTAs
 * for one another.  A wait that runs out sets SFI_DEV_WAIT_TIMEOUT; an
 * attention CTA then skips the arithmetic of the stages it still holds,
 * takes no further work and returns, a selector CTA goes on without waiting
 * (every access stays in bounds).  The call's output is then not
 * meaningful; zero-fill the workspace before reusing it.  `cycles` applies to every later launch from
 * any thread of the process; 0 restores the default of 4e9 clocks (about 2 s).
 * SFI_ERR_INVALID_ARG for cycles < 0. */
sfi_status sfi_set_wait_limit(int64_t cycles);

/* ---------------------------------------------------------------- slow step */

/* Slow step (SFI pages, "Slow-Fast paradigm", slow steps: dense attention
 * over the whole accessible history, whose logits are the evidence; "Selector":
 * the evidence distribution f and the cache statistics).
 *
 * For every sequence b, query head h (KV head g) and position i < n_b:
 *   l_{h,i} = q_h . k_{g,i} / sqrt(d),  p_h = softmax_i(l_h),
 *   out[b][h] = sum_i p_{h,i} v_{g,i}                     (dense GQA output)
 *   f[b][g][i] = (1/G) sum_{h in group g} p_{h,i}          (if f_out != NULL)
 *   knorm[b][g][i] = ||k_{g,i}||_2                         (if knorm_out != NULL)
 * q: [B][H_q][d] (dtype); out: [B][H_q][d] fp32.  With f_out and knorm_out
 * both NULL this is the plain dense decode baseline (no evidence traffic).
 * Kernels: a split-K flash-decode pass over the cache with a fused merge of
 * the splits, then (for f) a pass over the stored logits. */
size_t sfi_slow_attn_workspace_size(const sfi_layout* layout);
sfi_status sfi_slow_attn(const sfi_layout* layout, const void* q, const void* k, const void* v,
                         float* out, float* f_out, float* knorm_out,
                         void* ws, size_t ws_bytes, sfi_stream stream);

/* ---------------------------------------------------------------- selector */

/* Selector (SFI ko page, section 2.B: s = argmin_s (1-lambda) KL(f||s) +
 * lambda KL(r||s) = (1-lambda) f + lambda r, then Top-K).
 *
 * SFI_SELECT_FUSED, per (b, g): E = [n_sink, max(n_sink, n_b - window));
 *   r_i = knorm_i / sum_{j in E} knorm_j on E, 0 elsewhere;
 *   s_i = (1-lambda) f_i + lambda r_i for i < n_b (written to s_out if not NULL);
 *   idx_out[b][g][0..count) = the count = min(k, |E|) positions of E with the
 *   largest s, ties to the lower position, in ascending order.
 *   `evidence` is f ([B][H_kv][max_len]); `knorm` the key norms.
 * SFI_SELECT_LOGIT_SUM_SEQ (Vegas, sections 2.A and 2.B), per b:
 *   `evidence` holds per-KV-head logit sums (sfi_verify_attn); L_i = sum_g of
 *   them; P = [0, n_b - window) with n_sink = 0 (window = the verify rows);
 *   the top min(k, |P|) positions of L (ties to the lower position, ascending)
 *   are written to every KV head's row idx_out[b][g]; knorm is unused and
 *   lambda must be 0; s_out (if not NULL) receives L in row g = 0.
 * SFI_SELECT_LOGIT_SUM_HEAD (Vegas, section 2.A with the head set of one KV
 *   head), per (b, g): the top min(k, |P|) positions of P by that KV head's
 *   logit sum evidence[b][g][i] (same order and tie rule, its own set per KV
 *   head); knorm is unused, lambda and n_sink must be 0; s_out receives the
 *   ranked values.
 * idx_out: [B][H_kv][k] int32; count_out: [B][H_kv] int32 (device).
 * One launch; the CTAs that share a selecting unit wait for one another at
 * up to five barriers, and the launch cuts units into several CTAs only when
 * all its CTAs can be resident at once, so a concurrent launch on another
 * stream can delay it but not block it (each wait has the limit of
 * sfi_set_wait_limit). */
size_t sfi_select_workspace_size(const sfi_layout* layout, const sfi_params* params);
sfi_status sfi_select(const sfi_layout* layout, const sfi_params* params,
                      const float* evidence, const float* knorm,
                      int32_t* idx_out, int32_t* count_out, float* s_out,
                      void* ws, size_t ws_bytes, sfi_stream stream);

/* Selector refinements (SFI it/pt/ko pages, section "Selector": Soft-NMS
 * against neighbouring, correlated tokens within one head; cross-head
 * exclusivity against a token chosen again by another head).  The pages give
 * no formula; this is the builder's reading:
 *  - exclusivity: the KV heads of a sequence select in index order; head g
 *    ranks s_i * exp(-excl_beta * c_i), where c_i counts the heads g' < g
 *    whose selection holds i (excl_beta = 0: off);
 *  - Soft-NMS: greedy Gaussian Soft-NMS (Bodla et al., ICCV 2017) with
 *    position i as the box [i - rho, i + rho], rho = nms_radius: repeatedly
 *    take the position of E with the largest current score (ties to the
 *    lower position) and multiply the score of every remaining position j
 *    with |i - j| <= 2 rho by exp(-IoU(i, j)^2 / nms_sigma), IoU(d) =
 *    (2 rho + 1 - d) / (2 rho + 1 + d); the first min(k, |E|) positions
 *    taken are the selection (nms_radius = 0: plain Top-K).
 * sfi_select_refined computes s exactly as sfi_select in SFI_SELECT_FUSED mode
 * (the only mode it takes) and writes each (b, g)'s selection to idx_out in
 * ascending order, count_out = min(k, |E|).  Limits: nms_radius <= 8; with
 * nms_radius > 0, min(max_len, (k - 1)(4 nms_radius + 1) + 1) <= 98304 (else
 * SFI_ERR_CAPACITY).  With excl_beta > 0 the KV heads run one after another
 * (two launches each).  The workspace (sfi_select_refined_workspace_size,
 * 0 for invalid arguments) follows the shared rules; the call clears the part
 * it needs cleared itself. */
typedef struct {
  int32_t nms_radius; /* rho >= 0 */
  float nms_sigma;    /* sigma > 0 of the Gaussian decay (read when nms_radius > 0) */
  float excl_beta;    /* beta >= 0 */
} sfi_refine;

size_t sfi_select_refined_workspace_size(const sfi_layout* layout, const sfi_params* params,
                                         const sfi_refine* refine);
sfi_status sfi_select_refined(const sfi_layout* layout, const sfi_params* params,
                              const sfi_refine* refine, const float* f, const float* knorm,
                              int32_t* idx_out, int32_t* count_out, float* s_out,
                              void* ws, size_t ws_bytes, sfi_stream stream);

/* ---------------------------------------------------------------- fast step */

/* Fast step (SFI pages, "Slow-Fast paradigm", fast steps: attention over the
 * managed sparse state only -- sinks, recent window, selected memory).
 *
 * For every (b, g) the row set is [0, min(n_sink, n_b)) + idx[b][g][0..count[b][g])
 * + [max(n_sink, n_b - window), n_b); each query head of group g attends to
 * those rows with softmax attention (scale 1/sqrt(d)).  The selected positions
 * must lie in [n_sink, n_b - window) (disjoint from sinks and window); a
 * position outside [0, n_b) is replaced by position 0 and flagged
 * SFI_DEV_BAD_INDEX (the call's output is then not meaningful).  Rows are
 * gathered from the cache with 16-byte asynchronous copies. */
size_t sfi_fast_attn_workspace_size(const sfi_layout* layout, const sfi_params* params);
sfi_status sfi_fast_attn(const sfi_layout* layout, const sfi_params* params,
                         const void* q, const void* k, const void* v,
                         const int32_t* idx, const int32_t* count, float* out,
                         void* ws, size_t ws_bytes, sfi_stream stream);

/* ---------------------------------------------------------------- Vegas verify */

/* Verification attention with collected logit sums (Vegas, gist.science
 * 2602.07223: section 2 "Verification phase" -- dense attention with the
 * gamma + 1 rows of the draft chain; section 2.A -- the selected prefix set
 * maximises the attention logits summed over the collected rows and all
 * query heads; section 2.B "Collect-2-Query" -- collect only the first draft
 * row and the bonus row).
 *
 * n_b = len[b] includes the n_rows chain tokens; the prefix is
 * P = [0, n_b - n_rows).  Row t (0 <= t < n_rows) of sequence b sits at
 * position n_b - n_rows + t and attends to [0, n_b - n_rows + t]:
 *   out[b][t][h] = softmax-weighted sum of v over those positions (fp32).
 * If logitsum_out is not NULL, for every KV head g and prefix position i:
 *   logitsum_out[b][g][i] = sum over t in collect_rows, h in group g of
 *                           q_{t,h} . k_{g,i} / sqrt(d)      (natural units);
 * summing those rows over g gives the aggregated logits the selector's
 * SFI_SELECT_LOGIT_SUM_SEQ mode ranks (with window = n_rows, n_sink = 0);
 * SFI_SELECT_LOGIT_SUM_HEAD ranks each KV head's row on its own.
 * collect_rows = {0, n_rows - 1} is Collect-2; every row (0 .. n_rows - 1)
 * is the un-reduced aggregation of section 2.A.
 * q: [B][n_rows][H_q][d] bf16; out: [B][n_rows][H_q][d] fp32;
 * collect_rows: host array of n_collect distinct rows.
 * Limits (SFI_ERR_UNSUPPORTED beyond them): bf16 only; n_rows <= 8;
 * n_rows * G <= 32.  The workspace is sized by
 * sfi_verify_attn_workspace_size (it holds n_rows * G partial rows per
 * work item). */
size_t sfi_verify_attn_workspace_size(const sfi_layout* layout, int32_t n_rows);
sfi_status sfi_verify_attn(const sfi_layout* layout, int32_t n_rows, const int32_t* collect_rows,
                           int32_t n_collect, const void* q, const void* k, const void* v,
                           float* out, float* logitsum_out, void* ws, size_t ws_bytes,
                           sfi_stream stream);

/* Fast step that allocates nothing and takes no workspace.  The pages have
 * no counterpart to this call; it exists for callers that may not allocate
 * device memory on the path that runs the step -- for example a plug-in
 * interface that hands over only inputs and outputs, or a serving loop that
 * promised to allocate nothing after start-up because cudaMalloc can
 * synchronise the whole device.  It computes exactly what sfi_fast_attn
 * computes (same arguments and layout, minus the workspace).
 *  - Scratch: a fixed 16 MiB device array inside the library, kept by every
 *    GPU that loads the library until the process exits.  It holds the
 *    status word, one counter per (sequence, KV head) and the split partial
 *    results of head_dim + 2 floats per query head and work piece.  Each
 *    (sequence, KV head) is cut into at most 64 work pieces, and into no more
 *    than the array holds for all of them.  Geometries whose B * H_kv units
 *    do not fit even one piece each, or whose n_sink + k + window rows would
 *    need more than 64 pieces per unit, are rejected with SFI_ERR_CAPACITY
 *    and a message giving the sizes.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress); make that first call before capturing a stream
 *    into a CUDA graph.
 *  - Each call clears the status word and counters with cudaMemsetAsync on
 *    `stream` and calls no allocating routine.
 *  - All calls share the one array: calls that overlap on the GPU (other
 *    streams, other threads) race on it and must be serialised by the caller.
 *    The device status word of this call is not readable through
 *    sfi_read_status (there is no workspace). */
sfi_status sfi_fast_attn_noalloc(const sfi_layout* layout, const sfi_params* params,
                                 const void* q, const void* k, const void* v,
                                 const int32_t* idx, const int32_t* count, float* out,
                                 sfi_stream stream);

/* ---------------------------------------------------------------- decode driver */

typedef struct sfi_ctx sfi_ctx;

typedef struct {
  int32_t batch, n_q_heads, n_kv_heads, head_dim, dtype;
  int32_t max_len;  /* bound on every len[b] over the context's life */
  int32_t n_layers; /* each layer keeps its own selection */
  sfi_params params;
  int32_t budget;   /* fast steps allowed between refreshes; 0 = unlimited */
  /* != 0: overlap each layer's selector with the next layer's attention (SFI
   * pages, "System design": selection runs asynchronously beside decoding).
   * The selector then runs on a high-priority stream of the context, with a
   * second set of evidence buffers; the caller's stream joins it at the last
   * layer of each step.  0: the selector runs on the caller's stream. */
  int32_t async_select;
  /* Selector refinements applied at every refresh (reading and limits as for
   * sfi_select_refined); all zero: plain Top-K.  With excl_beta > 0 a
   * refreshing layer runs its KV heads' selections one after another. */
  sfi_refine refine;
} sfi_ctx_desc;

/* Create a decode context: allocates (with cudaMalloc, once) each layer's
 * selection buffers and key-norm store, and the shared evidence/workspace
 * buffers (two sets when async_select != 0; with a refinement each set adds
 * its candidate lists and exclusivity counts), and with async_select its
 * stream and events.
 * The key norms (the prior's cache statistic) of every (layer, sequence, KV
 * head) are kept across steps: a refresh computes only the norms of cache
 * rows appended since that layer's last refresh, since a cache row never
 * changes once written.  If a sequence's cache rows are replaced (a new
 * request in its batch slot, a rewritten cache), call sfi_ctx_reset. */
sfi_status sfi_ctx_create(const sfi_ctx_desc* desc, sfi_ctx** ctx_out);
sfi_status sfi_ctx_destroy(sfi_ctx* ctx);

/* One decode step of one layer (SFI pages, "Slow-Fast paradigm": a slow step
 * at a semantic boundary or when the reuse budget is exhausted, a fast step
 * otherwise).  At layer 0 the step's decision is taken per sequence from
 * is_boundary_host[b] (host, [B]): slow if at a boundary, if the sequence has
 * no selection yet, or if budget > 0 and it has run `budget` fast steps since
 * its last slow step; all layers of the step reuse that decision.  The layer
 * then runs one mixed launch (dense rows for slow sequences, managed-state
 * rows for fast ones); for slow sequences it also computes f and the key
 * norms and refreshes the layer's selection.  is_boundary_host is read only
 * when layer == 0.  q: [B][H_q][d]; out: [B][H_q][d] fp32.
 * With async_select, the selector of a layer below the last may still run
 * after the caller's stream has passed this call; the step of the last layer
 * orders every selector before later work on `stream`, and
 * sfi_ctx_selection / sfi_ctx_read_status order themselves after them.  The
 * layout's device arrays need stay valid only until this call's attention
 * has run (the selector reads a copy of len). */
sfi_status sfi_decode_step(sfi_ctx* ctx, int32_t layer, const uint8_t* is_boundary_host,
                           const sfi_layout* layout, const void* q, const void* k,
                           const void* v, float* out, sfi_stream stream);

/* Host-only schedule step used by sfi_decode_step (no GPU work), exposed so
 * a caller can plan ahead: for each b, slow_out[b] = is_boundary[b] ||
 * !have_sel[b] || (budget > 0 && since[b] >= budget); then have_sel[b] = 1
 * and since[b] = 0 for slow sequences, since[b] += 1 for fast ones.  All
 * arrays are host [B]. */
sfi_status sfi_schedule(int32_t batch, int32_t budget, const uint8_t* is_boundary,
                        uint8_t* have_sel, int32_t* since, uint8_t* slow_out);

/* Forget the schedule state (every sequence starts again without a
 * selection, so its next step is slow) and the stored key norms, and
 * zero-fill the context's workspace, clearing its device status.  Synchronous: waits for the
 * device (cudaMemset), so no decode step of this context may be in flight
 * on another thread. */
sfi_status sfi_ctx_reset(sfi_ctx* ctx);

/* Device-time profiling of sfi_decode_step (off by default).  enable != 0
 * (re)starts recording: every later decode step records CUDA events around
 * its attention launch and around its evidence + selector launches.
 * sfi_ctx_profile_read waits for the recorded events and returns the summed
 * device milliseconds and launch counts since the last enable.  enable == 0
 * stops recording. */
sfi_status sfi_ctx_profile(sfi_ctx* ctx, int32_t enable);
sfi_status sfi_ctx_profile_read(sfi_ctx* ctx, double* attn_ms, int64_t* attn_launches,
                                double* select_ms, int64_t* select_launches);

/* OR of the device status words of the context's workspaces (the bits
 * SFI_DEV_*), cleared; waits for `stream` after ordering it behind every
 * selector enqueued so far.  Returns SFI_ERR_CUDA if a copy fails. */
sfi_status sfi_ctx_read_status(sfi_ctx* ctx, uint32_t* status_host, sfi_stream stream);

/* The current step's decision (host [B], 1 = slow). */
sfi_status sfi_ctx_slow_mask(const sfi_ctx* ctx, uint8_t* slow_host);

/* Copy a layer's current selection into caller device buffers idx_out
 * ([B][H_kv][k] int32) and count_out ([B][H_kv] int32), enqueued on stream
 * behind every selector enqueued so far. */
sfi_status sfi_ctx_selection(const sfi_ctx* ctx, int32_t layer, int32_t* idx_out,
                             int32_t* count_out, sfi_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* SFI_H_ */
