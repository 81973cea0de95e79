/*
 * upf.h -- C ABI of libupf: UniPrefill's per-full-attention-layer token
 * selection on one NVIDIA GB300 (sm_103a).
 *
 * Source of the method: the article "中国科学院与腾讯微信合作解决AI排队等待问题"
 * (m.youleyou.com/wenzhang/2886770, a reprint of a 163.com piece on UniPrefill,
 * arXiv:2605.06221).  Its section 二 (two) gives the three steps (tail-query
 * importance estimation; top-p block filtering with sink/tail exemption;
 * cross-layer propagation of the drop), its section 三 (three) the system side
 * (fused GPU kernels with online normalisation, a binary keep mask, no CPU round
 * trip; batch metadata rewritten after a drop; a drop-history record of layer id
 * and kept count).
 *
 * Conventions shared by every call
 * --------------------------------
 * - All pointers named *_dev or documented "device" point to device memory of
 *   the context's GPU; "host" pointers to host memory.  The caller owns every
 *   buffer.  The library allocates nothing but its context (upf_create) and
 *   never touches the caller's allocator.
 * - Compute calls are asynchronous on the caller's `stream` (a cudaStream_t
 *   passed as void*; NULL = the legacy default stream).  Argument errors are
 *   detected on the host before anything is launched and returned at once;
 *   nothing is written in that case.
 * - Errors found on the device (non-finite scores, a full drop history, an
 *   inconsistent cu_seqlens_dev) set a status word in the context; the call that
 *   launched the work still returns UPF_OK.  upf_sync_status() waits for the
 *   stream and returns (then clears) that status.  One context must not be used
 *   by two streams at the same time.
 * - upf_last_error() returns a thread-local message for the last failure.
 *
 * Packed varlen batch (continuous batching, section 三): R requests are packed
 * back to back into one token stream of T = cu_seqlens[R] tokens; request r
 * owns packed tokens [cu_seqlens[r], cu_seqlens[r+1]).  L_r = its length
 * (0 allowed).  Tail ("questioner") rows of request r are its last
 * n_eff = min(n_tail, L_r) tokens (section 二, first step).
 */
#ifndef UPF_H
#define UPF_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define UPF_VERSION 1

typedef enum upf_status {
  UPF_OK = 0,
  UPF_ERR_INVALID_ARG = 1,   /* bad pointer, size, alignment or descriptor */
  UPF_ERR_UNSUPPORTED = 2,   /* valid but outside what the kernels support */
  UPF_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed */
  UPF_ERR_CAPACITY = 4,      /* drop history full (device-detected) */
  UPF_ERR_NONFINITE = 5,     /* NaN/Inf score reached the selection (device-detected) */
  UPF_ERR_TIMEOUT = 6        /* a bounded device wait expired (device-detected) */
} upf_status;

/* Opaque per-device context: a small device status word and cached device
 * properties.  Created for one device; every call must run with that device's
 * memory. */
typedef struct upf_ctx upf_ctx;

/* Batch descriptor (section 三: continuous batching; GQA head layout).
 * cu_seqlens_dev:  device int32 [num_reqs+1], cu[0] = 0, non-decreasing.
 * cu_seqlens_host: host copy of the same values (used to size grids and the
 *                  workspace; the device copy is re-checked on the GPU, and a
 *                  disagreement is reported through the status word as
 *                  UPF_ERR_INVALID_ARG).  upf_select_tokens on the tensor-core
 *                  path with at most 64 requests addresses the batch through
 *                  the host copy (its descriptor travels in the kernel
 *                  parameters); otherwise the device copy, once checked,
 *                  drives the kernels and a rejected one makes them do no work.
 * num_q_heads, num_kv_heads: H_q and H_kv, H_q % H_kv == 0.
 * head_dim: d, one of 64, 128, 256.
 * kv_of_q: host int32 [H_q] giving the kv head each q head reads, every kv head
 *          used by exactly H_q/H_kv q heads; NULL = contiguous groups
 *          (q head h reads kv head h / (H_q/H_kv)). */
typedef struct upf_batch {
  int32_t num_reqs;
  const int32_t* cu_seqlens_dev;
  const int32_t* cu_seqlens_host;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  const int32_t* kv_of_q;
} upf_batch;

/* Hyper-parameters (section 二; defaults from section 二 and section 五):
 * n_tail = 128 questioners, block = G = 64 tokens, top_p = 0.99,
 * sink_keep = tail_keep = 128 exempt tokens at each end.
 * softmax_scale <= 0 selects 1/sqrt(head_dim). */
typedef struct upf_params {
  int32_t n_tail;
  int32_t block;
  int32_t sink_keep;
  int32_t tail_keep;
  float top_p;
  float softmax_scale;
} upf_params;

/* Outputs of the compaction (section 二, third step; section 三, metadata and
 * drop history).  Row buffers hold at most T rows; only the first total_kept
 * rows are written.  Pointer pairs marked "nullable pair" may both be NULL.
 * row_bytes:      bytes of one hidden-state row (multiple of 16; e.g. 2*hidden
 *                 for bf16), both hidden pointers 16-byte aligned.
 * hidden_in/out:  [T, row_bytes] / [T, row_bytes] (nullable pair).
 * pos_in/out:     int64 [T] position ids (nullable pair).
 * slot_in/out:    int64 [T] KV-cache slot ids (nullable pair).
 *                 These six may be device memory or host memory the device
 *                 reads and writes directly (page-locked host memory under
 *                 unified addressing, or any host memory where the device has
 *                 pageable-memory access): the gather then moves only the kept
 *                 rows across the host link.  Other host pointers are
 *                 rejected with UPF_ERR_INVALID_ARG.
 * kept_index:     device int32 [T]: packed input index of each kept row (nullable).
 * cu_seqlens_out: device int32 [R+1]: packed offsets of the compacted batch.
 * total_kept:     device int32 [1]: cu_seqlens_out[R].
 * layer_id:       recorded in the drop history.
 * history:        device int32 [R, history_cap, 2]: record i of request r is
 *                 (layer id, kept tokens) at history[(r*cap + i)*2 + {0,1}].
 * history_len:    device int32 [R]: records per request; each call appends one
 *                 record to every request.  If any request already holds
 *                 history_cap records, no record is written and the status
 *                 word becomes UPF_ERR_CAPACITY.  history/history_len may both
 *                 be NULL (no record). */
typedef struct upf_compact_io {
  int64_t row_bytes;
  const void* hidden_in;
  void* hidden_out;
  const int64_t* pos_in;
  int64_t* pos_out;
  const int64_t* slot_in;
  int64_t* slot_out;
  int32_t* kept_index;
  int32_t* cu_seqlens_out;
  int32_t* total_kept;
  int32_t layer_id;
  int32_t history_cap;
  int32_t* history;
  int32_t* history_len;
} upf_compact_io;

/* Library version (UPF_VERSION). */
int upf_version(void);

/* Fill *p with the article's defaults (n=128, G=64, p=0.99, 128/128, scale 1/sqrt(d)). */
void upf_default_params(upf_params* p);

/* Human-readable name of a status code (static string). */
const char* upf_status_name(upf_status s);

/* Thread-local message describing the last failed call on this thread ("" if none). */
const char* upf_last_error(void);

/* Create a context on `device` (allocates a few bytes of device memory for the
 * status word).  *out receives the context.  Errors: INVALID_ARG (out NULL or
 * bad device), CUDA. */
upf_status upf_create(upf_ctx** out, int device);

/* Destroy a context (waits for nothing; the caller must have synchronised). */
upf_status upf_destroy(upf_ctx* ctx);

/* Wait for `stream`, return the device status word set by earlier calls on it
 * (UPF_OK if none) and reset it. */
upf_status upf_sync_status(upf_ctx* ctx, void* stream);

/* Bytes of device workspace that upf_score/upf_select/upf_compact/
 * upf_select_tokens need for this batch and these parameters (the same size
 * serves all four).  Returns 0 and sets the last error if the arguments are
 * invalid.  The workspace is scratch: its contents on entry do not matter and
 * on exit are unspecified; it must be 256-byte aligned. */
size_t upf_workspace_bytes(const upf_batch* batch, const upf_params* params);

/* Work split of the two scoring passes for this batch (inspection and tests;
 * no GPU needed): keys per split of pass 1 and pass 2, the number of work
 * items of each pass, and the CTAs that run one item of each pass (1, or 2
 * for a CTA pair sharing M = 256 MMAs; the passes may differ, and then pass 2
 * runs one query chunk per two of pass 1).  Any output may be NULL.  The
 * tensor-core passes run one CTA per SM, so the split is chosen by the
 * estimated time of the items over the device's 152 SMs (76 pairs).  Errors:
 * as upf_workspace_bytes. */
upf_status upf_plan_info(const upf_batch* batch, const upf_params* params, int32_t* key_split1, int32_t* key_split2,
                         int64_t* items1, int64_t* items2, int32_t* ctas_per_item1, int32_t* ctas_per_item2);

/* Tail-query importance of every token (section 二, first step; section 三,
 * scores + online normalisation):
 *   s_k = 1/(H_q * n_eff) * sum_h sum_{j : t_j >= k} softmax_j(k),
 * softmax_j over keys 0..t_j of scale * (q_{h,j} . k_{g(h),k}), per request.
 * q: device bf16, token t head h at q + t*q_row_stride + h*head_dim (only the
 *    tail rows are read); q_row_stride >= H_q*d elements, a multiple of 8.
 * k: device bf16, token t kv head g at k + t*k_row_stride + g*head_dim;
 *    k_row_stride >= H_kv*d, a multiple of 8.  q and k 16-byte aligned.
 * scores: device float32 [T].
 * ws / ws_bytes: workspace of at least upf_workspace_bytes() bytes.
 * q and k may point at a range of heads inside wider rows (the row strides
 * stay those of the full rows): a tensor-parallel rank scores its own heads
 * this way, normalised over the heads it was given (section 三, multi-GPU:
 * the ranks' scores are then summed before the decision).
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
upf_status upf_score(upf_ctx* ctx, const upf_batch* batch, const upf_params* params,
                     const void* q, int64_t q_row_stride, const void* k, int64_t k_row_stride,
                     float* scores, void* ws, size_t ws_bytes, void* stream);

/* upf_score for one tensor-parallel rank (section 三, multi-GPU: every GPU
 * scores the heads it holds and the per-GPU scores are summed before the
 * keep decision).  `batch` describes this rank's heads only (num_q_heads and
 * num_kv_heads of the slice, q and k pointing at the slice inside wider rows
 * as for upf_score); the scores are normalised by num_q_heads_total, the
 * q-head count over all ranks:
 *   s_k = 1/(num_q_heads_total * n_eff) * sum_{h of this rank} sum_j softmax_j(k),
 * so the element-wise sum of the ranks' scores is upf_score's result over
 * all heads (a plain sum all-reduce, no rescaling).  With num_q_heads_total =
 * num_q_heads it is upf_score.  Errors: as upf_score; INVALID_ARG if
 * num_q_heads_total < num_q_heads. */
upf_status upf_score_shard(upf_ctx* ctx, const upf_batch* batch, const upf_params* params,
                           int32_t num_q_heads_total, const void* q, int64_t q_row_stride, const void* k,
                           int64_t k_row_stride, float* scores, void* ws, size_t ws_bytes, void* stream);

/* Block pooling, top-p selection, exemption and the binary keep mask (section
 * 二, second step and exemption paragraph; section 三, binary mask).  Per
 * request: block means b_i over blocks [iG, min((i+1)G, L)); rank blocks by
 * b, highest first, ties to the lower index; keep the shortest prefix whose
 * running sum reaches top_p * (sum of all b); OR in every block that overlaps
 * the first sink_keep or the last tail_keep tokens; expand to tokens.
 * scores:       device float32 [T] (e.g. from upf_score).
 * block_scores: device float32 [sum_r ceil(L_r/G)] block means, request-major
 *               (nullable: then kept in the workspace).
 * keep_bits:    device uint32 [ceil(T/32)]: bit (t % 32) of word t/32 is 1 iff
 *               packed token t is kept.  Bits past T are 0.
 * kept_count:   device int32 [R]: kept tokens per request.
 * A request with more than 16384 blocks is UNSUPPORTED.  Scores are importances
 * (probabilities): a NaN, infinite or negative block score sets
 * UPF_ERR_NONFINITE in the status word and keeps that whole request.
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
upf_status upf_select(upf_ctx* ctx, const upf_batch* batch, const upf_params* params,
                      const float* scores, float* block_scores, uint32_t* keep_bits,
                      int32_t* kept_count, void* ws, size_t ws_bytes, void* stream);

/* Compaction of kept tokens and the drop-history append (section 二, third
 * step: later layers see only kept tokens, the dropped ones stay frozen in the
 * untouched inputs; section 三: positions/slot metadata follow the drop, and
 * (layer id, kept count) is recorded).  Out of place and order preserving:
 * kept token t (in packed order) becomes output row (number of kept tokens
 * before t).  keep_bits: device uint32 [ceil(T/32)] as produced by upf_select
 * (bits past T must be 0).  Only batch->num_reqs and the cu_seqlens pointers
 * of `batch` are used.  Errors: INVALID_ARG, CUDA. */
upf_status upf_compact(upf_ctx* ctx, const upf_batch* batch, const uint32_t* keep_bits,
                       const upf_compact_io* io, void* ws, size_t ws_bytes, void* stream);

/* The whole per-layer path in one call: upf_score, upf_select and upf_compact
 * on the same stream, sharing one workspace.  scores and block_scores are
 * nullable (then kept in the workspace).  Errors: as the three calls. */
upf_status upf_select_tokens(upf_ctx* ctx, const upf_batch* batch, const upf_params* params,
                             const void* q, int64_t q_row_stride, const void* k, int64_t k_row_stride,
                             float* scores, float* block_scores, uint32_t* keep_bits, int32_t* kept_count,
                             const upf_compact_io* io, void* ws, size_t ws_bytes, void* stream);

/* Revival of frozen tokens (section 二, third step: the hidden states of
 * dropped tokens are frozen and carried forward so they can be revived).
 * Writes the rows a compacted batch produced back to their token positions
 * in the full-length buffer: full[kept_index[o]] = rows[o] for o < *total_kept;
 * rows of dropped tokens in `full` keep their frozen contents.
 * kept_index, total_kept: device int32 [T] / [1] as written by upf_compact.
 * rows: device [>= total_kept, row_bytes]; full: device [T, row_bytes] with
 * T = batch cu_seqlens_host[R]; row_bytes a positive multiple of 16, both
 * pointers 16-byte aligned.  Indices outside [0, T) are skipped.
 * Errors: INVALID_ARG, CUDA. */
upf_status upf_revive(upf_ctx* ctx, const upf_batch* batch, const int32_t* kept_index, const int32_t* total_kept,
                      const void* rows, int64_t row_bytes, void* full, void* stream);

/* KV entries each request's layer `layer_id` holds (section 三, last
 * paragraph: decode reads the drop-history bill to know how many KV entries
 * each layer wrote).  A drop at full-attention layer l keeps c tokens for that
 * layer and every later one until the next drop, so kv_len[r] = c of the
 * latest record of request r whose layer id <= layer_id (records are appended
 * in layer order), or the prompt length L_r if there is none.
 * history, history_len, history_cap: as in upf_compact_io (device).
 * kv_len: device int32 [R].  Errors: INVALID_ARG, CUDA. */
upf_status upf_history_kv_len(upf_ctx* ctx, const upf_batch* batch, const int32_t* history,
                              const int32_t* history_len, int32_t history_cap, int32_t layer_id, int32_t* kv_len,
                              void* stream);

/* No-allocation variant of upf_select.  The article has no counterpart: this
 * is an integration entry point for callers that cannot allocate device
 * memory -- a serving engine that reserves nearly all GPU memory for its own
 * pools at start-up and gives libraries no allocation hook, or a plugin that
 * runs inside such an engine and may not bypass its allocator.  It needs no
 * context and no workspace: the scratch of the select kernels (the batch
 * descriptor and, if block_scores is NULL, the block means) lives in one
 * fixed-size device array compiled into the library, about 270 KiB, which
 * every GPU that loads the library holds until the process exits.
 * It runs on the caller's current device and stream.
 * Same inputs, outputs and results as upf_select.  Limits: at most
 * UPF_NOALLOC_MAX_REQS requests and UPF_NOALLOC_MAX_BLOCKS blocks in total
 * (and 16384 per request); larger batches return UPF_ERR_UNSUPPORTED.
 * status_dev: device int32 [1] (nullable) that receives device-detected
 * errors (first error wins; the caller clears it); when NULL such errors go to
 * a status word inside the array and are not reported.  Pass status_dev:
 * without it a failed call cannot be told from a good one.  What the outputs
 * then hold: a request with a NaN, infinite or negative block score keeps all
 * its tokens (as in upf_select); if cu_seqlens_dev disagrees with
 * cu_seqlens_host, the device descriptor is zeroed, so every keep bit is 0
 * and every kept_count is 0 -- the sink and tail tokens included.
 * The array is shared by every call and keeps the last call's contents; each
 * call rewrites what it reads.  Calls whose GPU work overlaps (different
 * streams or host threads) race on it: serialise them.  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress) with that
 * device current; make that first call before any stream capture begins.
 * It calls no cudaMalloc, cudaFree or other allocating routine.  Errors:
 * INVALID_ARG, UNSUPPORTED, CUDA (message in upf_last_error()). */
#define UPF_NOALLOC_MAX_REQS 1024
#define UPF_NOALLOC_MAX_BLOCKS 65536
upf_status upf_select_noalloc(const upf_batch* batch, const upf_params* params, const float* scores,
                              float* block_scores, uint32_t* keep_bits, int32_t* kept_count,
                              int32_t* status_dev, void* stream);

/* Failure detection (not a step of the article's method).  Every wait
 * inside the tensor-core scoring kernels is bounded; when one expires the
 * kernel records UPF_ERR_TIMEOUT in the status word, stops issuing work,
 * waits for its outstanding copies and MMAs, frees its tensor memory and
 * returns, so the context stays usable.  This sets the limit of the pipeline
 * waits (a role waiting for another role's data), in SM clock cycles, for
 * later calls on `ctx`; 0 restores the default (4e9 cycles, about 2 s).  The
 * waits that wind a kernel down always keep the default.  A very small limit
 * makes a pipeline wait expire on purpose: that is how the timeout path is
 * tested.  Errors: INVALID_ARG (ctx NULL, cycles < 0). */
upf_status upf_set_wait_limit(upf_ctx* ctx, int64_t cycles);

/* Tracing (per-stage device timing).  Stages, in launch order:
 * 0 describe (batch descriptor; upf_select_tokens launches none for batches
 * whose descriptor travels in the kernel parameters), 1 score pass 1, 2 score
 * pass 2, 3 finalize / block means, 4 select, 5 compact count, 6 compact
 * index, 7 compact gather. */
#define UPF_NUM_STAGES 8

/* Name of stage i (static string; "" if out of range). */
const char* upf_stage_name(int32_t stage);

/* on != 0: every later launch made through this context is bracketed by two
 * CUDA events on the caller's stream (events come from a pool the context owns).
 * Launch counting is always on. */
upf_status upf_profile_enable(upf_ctx* ctx, int32_t on);

/* Wait for the recorded events and return, per stage (n_stages entries, at most
 * UPF_NUM_STAGES), the launches made and the summed device milliseconds (0
 * while profiling is off) since the previous read; both are then reset.
 * launches and ms may be NULL. */
upf_status upf_profile_read(upf_ctx* ctx, int32_t* launches, double* ms, int32_t n_stages);

#ifdef __cplusplus
}
#endif

#endif /* UPF_H */
