/*
 * tnd_attn.h — C ABI of the TND FlashAttention forward and score-gradient
 * library for NVIDIA B300 (sm_103a).
 *
 * The operation is the one described on the Ascend CANN pages
 * "aclnnFlashAttentionUnpaddingScoreGrad" (function description: forward
 * Y = Dropout(Softmax(Mask(scale * Q K^T)), keep_prob) V and the backward
 * dV = P^T dY, dQ = dS K * scale, dK = dS^T Q * scale) and
 * "aclnnFlashAttentionUnpaddingScoreGradV5" (function description: the
 * attention sink, m = max(sink, max S), denominator sum exp(S - m) +
 * exp(sink - m), and its gradient dSink).  dS is P o (z dP - rowsum(dY o O))
 * with z the dropout multiplier (keep-bit / keepProb).
 *
 * Conventions shared by every call
 * --------------------------------
 * Layout "TND" ([UnpadGrad] parameters section, inputLayout): rows of all
 * sequences packed back to back.
 *   query, dq                      : [Tq,  Nq,  D]  row-major
 *   key, dk                        : [Tkv, Nkv, D]  row-major
 *   dy, attention_out / attention_in : [Tq,  Nq,  Dv] row-major
 *   value, dv                      : [Tkv, Nkv, Dv] row-major
 *   D = head_dim, Dv = value_head_dim ([UnpadGrad] constraints: qD == kD >=
 *   vD, so 1 <= Dv <= D; scale_value is used as given).  The tensor-core
 *   kernels take Dv == D; other calls run on the CUDA-core kernels.
 *   softmax_max, softmax_sum                    : fp32 [Tq, Nq, 8]; the 8
 *       values of a row are equal copies (the pages fix the [T,N,8] shape
 *       without saying what the 8 lanes hold).  The forward writes all 8,
 *       the gradient reads lane 0.  max is in natural-log units over the
 *       scaled, masked logits; sum is taken before dropout; both include the
 *       sink when one is given.  A row with no kept key and no sink has
 *       max = -inf, sum = 0 and a zero output row.
 *   drop_mask: uint8 packed keep-bits ([UnpadGrad] parameters,
 *       dropMaskOptional, (sum_b sum_n Sq*Skv)/8 bytes).  Bit of
 *       (sequence b, q-head h, q-row i, kv-row j) is at flat index
 *       base_b + (h*Sq_b + i)*Skv_b + j, base_b = sum_{b'<b} Nq*Sq_b'*Skv_b';
 *       byte = index >> 3, bit = index & 7 (least significant first); 1 keeps.
 *       May be NULL when keep_prob == 1 (then it is ignored).
 *   sink, dsink: fp32 [Nq] ([UnpadGradV5] constraints: one value per head).
 * All element tensors share one dtype ([UnpadGrad] constraints: query, key,
 * value, dy dtypes must agree).  Every device pointer must be 16-byte aligned.
 *
 * cu_seqlens_q / cu_seqlens_kv: HOST arrays of batch+1 int64 cumulative
 * offsets (0 = cu[0] <= cu[1] <= ... <= cu[batch] = T).  They carry
 * actualSeqQLen / actualSeqKvLen ([UnpadGrad] parameters: the S of each
 * batch entry).  A sequence may be empty.
 *
 * sparse_mode ([UnpadGrad] parameters, sparseMode; i, j are the row and
 * column within sequence b):
 *   0  without atten_mask: no mask, pre_tokens / next_tokens ignored;
 *      with atten_mask: keep where the matrix is 0 and
 *      -pre_tokens <= j - i <= next_tokens (pre_tokens + next_tokens >= 0)
 *   1  keep where the matrix is 0 (atten_mask required)
 *   2  lower triangle from the top-left vertex:      keep j <= i
 *   3  lower triangle from the bottom-right vertex:  keep j <= i + Skv - Sq
 *   4  band: keep -pre_tokens <= j - i <= next_tokens (needs Sq_b == Skv_b
 *      for every sequence and pre_tokens + next_tokens >= 0)
 *   6  prefix: keep j <= i + Skv - Sq or j < prefix[b] (prefix required;
 *      batch <= 1024; 0 <= prefix[b] <= Skv_b)
 *   5, 7, 8 (padded full matrix, external split) return TND_ERR_UNSUPPORTED.
 *   Modes 2, 3, 4 and 6 are computed from indices: the pages' compressed
 *   matrices for them only restate these rules, so an atten_mask passed with
 *   them is not read.
 * atten_mask ([UnpadGrad] parameters, attenMaskOptional): device uint8 (or
 *   bool) [S1Max, S2Max] row-major, S1Max = max_b Sq_b, S2Max = max_b Skv_b;
 *   one matrix for every sequence and head, indexed by (i, j); nonzero
 *   masks, 0 keeps.  Read only by modes 0 and 1.
 * prefix ([UnpadGrad] parameters, prefixOptional): HOST array of batch int64
 *   values N_b, read only by mode 6 (NULL otherwise).
 * A row that keeps no key (and has no sink) gets max = -inf, sum = 0 and a
 * zero output row; its gradient rows are zero.
 * pse ([UnpadGrad] parameters, pseShiftOptional; [ScoreV2] parameters,
 *   pseType): device tensor in the element dtype, [pse_batch, Nq, 1024,
 *   S2Max] row-major with pse_batch = B (one per sequence) or 1 (shared).
 *   It holds the last 1024 rows of each sequence's [Sq, Skv] bias (the
 *   pages' alibi compression, ori_pse[:, :, -1024:, :]): row i of a sequence
 *   is stored row i - (Sq - 1024), so a sequence shorter than 1024 uses the
 *   bottom Sq rows; a row above the stored ones (i < Sq - 1024) is read along
 *   its diagonal from stored row 0, column j + (Sq - 1024 - i), which is
 *   exact for a bias that depends on i - j only (alibi).  pse_type 1 adds it
 *   before the scale (scale * (QK^T + pse), the grad page's formula), 0 after
 *   it (scale * QK^T + pse).  pse_type 2 and 3 generate the pse inside
 *   ([ScoreV2] parameters: realShiftOptional is then FLOAT32 [B, N] or [N]):
 *   pse is a device fp32 array of slopes [pse_batch, Nq] (pse_batch = B or 1)
 *   and the bias, added after the scale, is -slope * |i - j| (2) or
 *   -slope * sqrt(|i - j|) (3); the pages do not print the generator, this
 *   is the alibi reading of their table.  With a pse, sparse_mode must be 2
 *   or 3 and Sq_b == Skv_b for every sequence (the pages' alibi constraint),
 *   else TND_ERR_UNSUPPORTED.  NULL = no pse (pse_batch and pse_type
 *   ignored); a pse_type outside 0..3 is TND_ERR_INVALID.
 *   dpseOut is a reserved output on the pages and is not produced.
 * GQA: Nq % Nkv == 0; query head h uses key/value head h / (Nq/Nkv).
 *
 * Two phases, as on the pages ([UnpadGrad] function prototype section): a
 * *_workspace_size call validates every argument and returns the device
 * workspace the run call needs; the run call validates again, enqueues the
 * work on `stream` (a cudaStream_t; NULL = legacy default stream) and returns
 * without waiting.  The caller owns every buffer, including the workspace
 * (at least 256-byte aligned; cudaMalloc memory is).  The library allocates
 * no device memory.  Argument errors are reported before any device work is
 * enqueued and leave every output untouched.  Outputs are fully overwritten
 * on success, zero where nothing contributes.  Results are bitwise
 * deterministic run to run unless TND_OPT_DETERMINISTIC is switched off.
 * Calls on one workspace must not overlap in time.
 */
#ifndef TND_ATTN_H
#define TND_ATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes.  NULLPTR / INVALID mirror the pages' ACLNN_ERR_PARAM_NULLPTR
 * (161001) and ACLNN_ERR_PARAM_INVALID (161002) ([ScoreV2] return values). */
typedef enum tnd_status {
    TND_OK = 0,
    TND_ERR_NULLPTR = 1,        /* a required pointer is NULL                          */
    TND_ERR_INVALID = 2,        /* dtype, shape, scalar or alignment outside the pages' limits */
    TND_ERR_UNSUPPORTED = 3,    /* allowed by the pages but not implemented here       */
    TND_ERR_WORKSPACE = 4,      /* workspace NULL, misaligned or smaller than required */
    TND_ERR_CUDA = 5,           /* a CUDA runtime call failed                          */
    TND_ERR_DEVICE_TIMEOUT = 6, /* a bounded device-side wait expired                  */
    TND_ERR_DEVICE_CHECK = 7    /* a device-side consistency check failed              */
} tnd_status;

typedef enum tnd_dtype { TND_F16 = 0, TND_BF16 = 1, TND_F32 = 2 } tnd_dtype;

/*
 * Forward workspace size ([UnpadGrad]/[ScoreV2] function prototype: first
 * phase).  Checks all shape / scalar arguments ([UnpadGrad] and
 * [UnpadGradV5] constraints: T in [1, 1M], N in [1, 256], D in [1, 768],
 * Dv in [1, D],
 * B in [1, 20000], keep_prob in (0, 1], headNum == Nq, Nq % Nkv == 0) and
 * the sparse_mode rules above.  has_drop_mask / has_atten_mask / has_sink
 * say whether the run call will pass those inputs; prefix is the host
 * prefix array (mode 6).  Writes the byte count to *workspace_size.
 */
tnd_status tnd_attn_fwd_workspace_size(
    tnd_dtype dtype, int64_t batch, const int64_t *cu_seqlens_q, const int64_t *cu_seqlens_kv,
    const int64_t *prefix, int64_t head_num, int64_t kv_head_num, int64_t head_dim,
    int64_t value_head_dim, double scale_value, double keep_prob, int64_t pre_tokens,
    int64_t next_tokens, int64_t sparse_mode, int has_drop_mask, int has_atten_mask, int has_sink,
    uint64_t *workspace_size);

/*
 * Forward ([ScoreV2] function description and parameters): writes
 * attention_out [Tq,Nq,Dv] (dtype), softmax_max and softmax_sum [Tq,Nq,8]
 * (fp32).  pse, drop_mask, atten_mask, sink and prefix may be NULL where the
 * conventions above allow it; the pse checks are made here (the workspace
 * size does not depend on it).
 */
tnd_status tnd_attn_fwd(
    const void *query, const void *key, const void *value, const void *pse, int64_t pse_batch,
    int64_t pse_type, const uint8_t *drop_mask, const uint8_t *atten_mask, const float *sink,
    tnd_dtype dtype, int64_t batch,
    const int64_t *cu_seqlens_q, const int64_t *cu_seqlens_kv, const int64_t *prefix,
    int64_t head_num, int64_t kv_head_num, int64_t head_dim, int64_t value_head_dim,
    double scale_value, double keep_prob, int64_t pre_tokens, int64_t next_tokens,
    int64_t sparse_mode, void *attention_out, float *softmax_max, float *softmax_sum,
    void *workspace, uint64_t workspace_size, void *stream);

/* Gradient workspace size (first phase of [UnpadGrad]); same arguments and
 * checks as the forward's. */
tnd_status tnd_attn_grad_workspace_size(
    tnd_dtype dtype, int64_t batch, const int64_t *cu_seqlens_q, const int64_t *cu_seqlens_kv,
    const int64_t *prefix, int64_t head_num, int64_t kv_head_num, int64_t head_dim,
    int64_t value_head_dim, double scale_value, double keep_prob, int64_t pre_tokens,
    int64_t next_tokens, int64_t sparse_mode, int has_drop_mask, int has_atten_mask, int has_sink,
    uint64_t *workspace_size);

/*
 * Score-gradient ([UnpadGrad] second phase; inputs and outputs as in its
 * parameters section, plus sinkInOptional / dSink of [UnpadGradV5]).
 * Inputs: query, key, value, dy; softmax_max, softmax_sum and attention_in
 * as written by tnd_attn_fwd; drop_mask (NULL when keep_prob == 1);
 * pse, atten_mask and prefix as for the forward (the same ones it was given);
 * sink (NULL = no sink).  Outputs: dq [Tq,Nq,D], dk [Tkv,Nkv,D], dv [Tkv,Nkv,Dv]
 * (dtype; dk and dv are summed over the Nq/Nkv query heads of each kv
 * head), dsink [Nq] fp32 (required when sink is given, ignored otherwise).
 */
tnd_status tnd_attn_grad(
    const void *query, const void *key, const void *value, const void *dy, const void *pse,
    int64_t pse_batch, int64_t pse_type, const uint8_t *drop_mask, const uint8_t *atten_mask,
    const float *softmax_max,
    const float *softmax_sum, const void *attention_in, const float *sink, tnd_dtype dtype,
    int64_t batch, const int64_t *cu_seqlens_q, const int64_t *cu_seqlens_kv,
    const int64_t *prefix, int64_t head_num, int64_t kv_head_num, int64_t head_dim,
    int64_t value_head_dim, double scale_value, double keep_prob, int64_t pre_tokens,
    int64_t next_tokens, int64_t sparse_mode, void *dq, void *dk, void *dv, float *dsink,
    void *workspace, uint64_t workspace_size, void *stream);

/*
 * Waits for `stream`, then reports the device-side status of the last
 * forward / gradient enqueued on this workspace: TND_OK,
 * TND_ERR_DEVICE_TIMEOUT (a bounded wait expired; the outputs of that call
 * are not valid) or TND_ERR_DEVICE_CHECK.  TND_ERR_CUDA if the stream
 * reports an error.  The status is cleared by the next run call.
 */
tnd_status tnd_attn_device_status(const void *workspace, uint64_t workspace_size, void *stream);

/* Static, human-readable text for a status code. */
const char *tnd_status_string(tnd_status status);

/*
 * Library options (process-wide; set them before enqueueing work).
 *   TND_OPT_GRAD_PATH: 0 = automatic (tensor-core kernel where it applies),
 *                      1 = always the CUDA-core kernels.
 *   TND_OPT_WAIT_LIMIT_MS: upper bound of every device-side wait (default 2000).
 *   TND_OPT_PROFILE: 1 = record CUDA events around each kernel of every call
 *                    (read with tnd_attn_profile_read), 0 = off (default).
 *   TND_OPT_TEST_SKIP_LOAD: test hook for the bounded waits ([UnpadGrad]
 *                    constraints: a wait that cannot finish must end in a
 *                    timeout error, not a hang).  1 = the tensor-core
 *                    gradient's first CTA never loads its first K tile, so
 *                    the wait for it expires and the call reports
 *                    TND_ERR_DEVICE_TIMEOUT through tnd_attn_device_status
 *                    (its outputs are then invalid); 0 = off (default).
 *   TND_OPT_DETERMINISTIC: deterministic computing ([UnpadGradV5]
 *                    constraints: the gradient is non-deterministic unless
 *                    deterministic computing is switched on).  1 (default) =
 *                    the tensor-core gradient adds the dQ contributions of
 *                    every (q block, head) in a fixed order, so repeated
 *                    calls give bitwise identical results; 0 = they are
 *                    added in arrival order (same tolerance against the
 *                    exact result, rounding order varies from call to call).
 *                    The forward and the CUDA-core kernels are deterministic
 *                    either way.
 */
typedef enum tnd_option {
    TND_OPT_GRAD_PATH = 0,
    TND_OPT_WAIT_LIMIT_MS = 1,
    TND_OPT_PROFILE = 2,
    TND_OPT_TEST_SKIP_LOAD = 3,
    TND_OPT_DETERMINISTIC = 4
} tnd_option;
tnd_status tnd_attn_set_option(tnd_option option, int64_t value);

/*
 * Per-kernel device time recorded since the last reset (TND_OPT_PROFILE on).
 * Waits for the recorded events.  For up to `capacity` kernel kinds writes
 * the kind's name (static string), its total milliseconds and its launch
 * count; returns the number of kinds in *count.  reset != 0 clears the record
 * after reading.  The record keeps the last 4096 launches.
 */
tnd_status tnd_attn_profile_read(const char **names, double *total_ms, int64_t *launches,
                                 int capacity, int *count, int reset);

/*
 * Host-side view of the gradient plan (for tests of the schedule; no device
 * work).  For the problem described by the arguments writes up to
 * `capacity` work units as 5 int64 each (sequence b, kv head g, kv block j,
 * first q block, end q block) in the order the tensor-core kernel takes
 * them, the unit count to *n_units and the number of (q-row, kv-row)
 * pairs the index rule keeps, summed over sequences and query heads, to
 * *kept_pairs (the attention-mask matrix is not seen here: with one, the
 * count is of the pairs its band admits).  Blocks are 128 kv rows and 128
 * q rows.
 */
tnd_status tnd_attn_grad_plan(
    int64_t batch, const int64_t *cu_seqlens_q, const int64_t *cu_seqlens_kv,
    const int64_t *prefix, int64_t head_num, int64_t kv_head_num, int64_t pre_tokens,
    int64_t next_tokens, int64_t sparse_mode, int has_atten_mask, int64_t *units,
    int64_t capacity, int64_t *n_units, int64_t *kept_pairs);

/*
 * Gradient without a caller-provided workspace.  The pages have no
 * counterpart: their operator always takes a workspace the caller allocates.
 *
 * For callers that cannot allocate device memory, for instance a plug-in
 * that only receives buffers from its host framework's allocator, or a
 * process that reserved all device memory at start-up.  Arguments and
 * results are those of tnd_attn_grad without `workspace` / `workspace_size`,
 * `pse`, `atten_mask`, `prefix` and `value_head_dim` (value and dy have
 * head_dim columns; sparse_mode 1 and 6 return TND_ERR_NULLPTR);
 * the caller still passes every input and output.
 *
 * The workspace is a fixed device array inside this library of
 * TND_STATIC_WS_BYTES bytes, held on every GPU that loads the library until
 * the process exits.  A problem whose tnd_attn_grad_workspace_size exceeds
 * it returns TND_ERR_WORKSPACE before any device work.  No call allocates
 * memory (no cudaMalloc / cudaFree, no pinned host staging, no allocating
 * library routine); the plan is copied from pageable host memory, so the
 * call may wait for earlier work on `stream` before it returns.  The first
 * call on each device looks the array's device address up (with that device
 * current) and keeps it, looking it up again if the device's context changes
 * (cudaDeviceReset); make that first call before any stream capture.  Every
 * call shares the one array and it keeps the last call's contents: each
 * call rewrites the parts that must start at zero (status words, dQ chain
 * counters) on its stream before its kernels run, so calls in sequence are
 * independent, but calls that overlap on the GPU (other streams, other host
 * threads) race on it and give wrong results.  Device-side errors of these
 * calls are read with tnd_attn_grad_static_ws_status.
 */
#define TND_STATIC_WS_BYTES (32ull << 20)
tnd_status tnd_attn_grad_static_ws(
    const void *query, const void *key, const void *value, const void *dy,
    const uint8_t *drop_mask, const float *softmax_max, const float *softmax_sum,
    const void *attention_in, const float *sink, tnd_dtype dtype, int64_t batch,
    const int64_t *cu_seqlens_q, const int64_t *cu_seqlens_kv, int64_t head_num,
    int64_t kv_head_num, int64_t head_dim, double scale_value, double keep_prob,
    int64_t pre_tokens, int64_t next_tokens, int64_t sparse_mode, void *dq, void *dk, void *dv,
    float *dsink, void *stream);

/*
 * tnd_attn_device_status for the fixed workspace of tnd_attn_grad_static_ws
 * on the current device: waits for `stream`, then returns TND_OK,
 * TND_ERR_DEVICE_TIMEOUT or TND_ERR_DEVICE_CHECK for the last such call.
 */
tnd_status tnd_attn_grad_static_ws_status(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* TND_ATTN_H */
