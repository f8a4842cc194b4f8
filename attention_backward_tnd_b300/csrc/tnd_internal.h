// Internal declarations shared by the host API and the kernels of the TND
// attention library.  Nothing here is part of the public C ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <utility>

#include "../../include/tnd_attn.h"

namespace tnd {

// Rows per block of the tensor-core gradient: kv block (UMMA M) and q block.
constexpr int kKvBlock = 128;
constexpr int kQBlock = 128;
// Rows per block of the CUDA-core kernels.
constexpr int kSimtRows = 32;

// Offsets into the status area at the start of every workspace.
constexpr int kStatusWord = 0;     // first device error code (0 = none)
constexpr int kStatusDetail = 1;   // where it happened (kernel-specific)
constexpr int kWorkCounter = 2;    // next unit of the persistent kernel
constexpr size_t kStatusBytes = 256;

// One sequence of the packed batch, as the kernels see it.
struct SeqDesc {
    int64_t tq;         // first query row (token index) of the sequence
    int64_t tk;         // first key/value row
    int32_t sq;         // query rows
    int32_t skv;        // key/value rows
    int64_t mask_base;  // flat keep-bit index of (h=0, i=0, j=0)
    int32_t qblk0;      // global index of its first 128-row q block
    int32_t nqblk;      // number of 128-row q blocks
    int32_t prefix;     // prefixOptional N_b (sparseMode 6; 0 otherwise)
    int32_t pad;
};

// Index rules of the masks, after mapping the pages' sparseMode (and the
// attention-mask matrix) onto them.
enum MaskRule : int32_t {
    kRuleAll = 0,      // every (i, j)
    kRuleTopLeft = 2,  // j <= i
    kRuleCausal = 3,   // j <= i + Skv - Sq
    kRuleBand = 4,     // -pre <= j - i <= next
    kRulePrefix = 6,   // j <= i + Skv - Sq or j < N_b
};

// Mask description: an index rule, plus (sparseMode 0 with a matrix, and 1)
// the attention-mask matrix, which further drops the (i, j) it marks.
struct MaskSpec {
    int32_t mode;              // MaskRule
    int64_t pre;
    int64_t next;
    const uint8_t *amask;      // [S1Max][S2Max] bytes, nonzero masks (NULL = none)
    int64_t amask_cols;        // S2Max
    const uint64_t *keep_q;    // packed keep bits of the matrix, row i: bit j (forward)
    const uint64_t *keep_kv;   // transposed, row j: bit i (gradient)
    int32_t words_q;           // 64-bit words per row of keep_q (even)
    int32_t words_kv;          // 64-bit words per row of keep_kv (even)
};

// Key range [lo, hi] of the index rule for query row i (empty when lo > hi);
// prefix_n is the sequence's N_b.  Rows of every rule keep one contiguous
// range whose ends never decrease with i, which the schedules rely on (the
// prefix rule's two parts both start at column 0).
__host__ __device__ inline void key_range(const MaskSpec &m, int64_t sq, int64_t skv, int64_t prefix_n,
                                          int64_t i, int64_t &lo, int64_t &hi)
{
    lo = 0;
    hi = skv - 1;
    if (m.mode == kRuleTopLeft) {
        hi = hi < i ? hi : i;
    } else if (m.mode == kRuleCausal) {
        const int64_t e = i + skv - sq;
        hi = hi < e ? hi : e;
    } else if (m.mode == kRuleBand) {
        const int64_t a = i - m.pre, e = i + m.next;
        lo = lo > a ? lo : a;
        hi = hi < e ? hi : e;
    } else if (m.mode == kRulePrefix) {
        int64_t e = i + skv - sq;
        e = e > prefix_n - 1 ? e : prefix_n - 1;
        hi = hi < e ? hi : e;
    }
}

// Whether the attention-mask matrix keeps in-sequence (i, j) (true without one).
__host__ __device__ inline bool matrix_keeps(const MaskSpec &m, int64_t i, int64_t j)
{
    return m.amask == nullptr || m.amask[i * m.amask_cols + j] == 0;
}

// pseShiftOptional.  pseType 0 / 1: for each sequence (or for all, when
// batch is 1) and query head, the last 1024 rows of the sequence's [Sq, Skv]
// bias, stored as [batch][Nq][1024][cols] in the element dtype.  Row i of a
// sequence is stored row i - (Sq - 1024); a row above the stored ones is read
// along its diagonal from stored row 0, column j + (Sq - 1024 - i).
// pseType 2 / 3 ("aclnnFlashAttentionScoreV2", parameters: generated inside
// from FLOAT32 [B, N] or [N]): one fp32 slope per (sequence or all, head),
// the bias being the alibi -slope |i - j| (2) or -slope sqrt(|i - j|) (3).
struct PseSpec {
    const void *ptr;   // NULL = no pse
    int32_t batch;     // 1 or B
    int32_t type;      // pseType 1: s = scale*(qk + pse); 0, 2, 3: s = scale*qk + pse
    int64_t cols;      // S2Max (stored types)
};

__host__ __device__ inline bool pse_generated(const PseSpec &ps) { return ps.type >= 2; }

// slope of (sequence b, head h) of a generated pse
__device__ __forceinline__ float pse_slope(const PseSpec &ps, int32_t nq, int64_t b, int64_t h)
{
    return reinterpret_cast<const float *>(ps.ptr)[(ps.batch == 1 ? 0 : b) * nq + h];
}

// the generated bias at distance |i - j|
__device__ __forceinline__ float pse_alibi(int32_t type, float slope, int64_t i, int64_t j)
{
    const float dist = (float)(i > j ? i - j : j - i);
    return -slope * (type == 2 ? dist : sqrtf(dist));
}

__host__ __device__ inline int64_t pse_index(const PseSpec &ps, int32_t nq, int64_t b, int64_t h, int64_t sq,
                                             int64_t i, int64_t j)
{
    int64_t r = i - (sq - 1024), c = j;
    if (r < 0) {
        c = j - r;
        r = 0;
    }
    const int64_t bb = ps.batch == 1 ? 0 : b;
    return ((bb * nq + h) * 1024 + r) * ps.cols + c;
}

// Work unit of the tensor-core gradient: kv block j of kv head g of
// sequence b, visiting q blocks [qb_lo, qb_hi) for each of the group's heads.
struct GradUnit {
    int32_t b, g, j, qb_lo, qb_hi, pad0, pad1, pad2;
};

// Contributors of one global q block: kv blocks [jlo, jhi] (jlo = -1: none).
struct QBlockInfo {
    int32_t jlo, jhi;
};

// Per-row vectors of the gradient (lse2, D, sink terms) are stored blocked:
// one 128-float vector per (global 128-row q block, query head), rows past the
// sequence end padded (lse2 = +inf, D = 0, sink term = 0).  Index of row i of
// sequence sd, head h:
__host__ __device__ inline int64_t row_vec_index(const SeqDesc &sd, int32_t nq, int32_t h, int64_t i)
{
    return ((int64_t)(sd.qblk0 + (int32_t)(i / kQBlock)) * nq + h) * kQBlock + (i % kQBlock);
}

// Everything a gradient launch needs to know (device pointers into the
// caller's buffers and the workspace).
struct GradArgs {
    const void *q, *k, *v, *dy, *o;
    const uint8_t *drop_mask;
    int64_t mask_bytes;       // size of drop_mask in bytes
    const float *smax, *ssum, *sink;
    void *dq, *dk, *dv;
    float *dsink;
    int dtype;
    int32_t batch, nq, nkv, d, group;
    int32_t vd;               // head dim of value, dy, the output and dV (<= d)
    int64_t tq, tkv;
    float scale, keep_prob, inv_keep;
    MaskSpec mask;
    PseSpec pse;
    int has_drop, has_sink;
    // workspace regions
    uint32_t *status;
    const SeqDesc *seqs;
    const int2 *q_items;      // (b, first row) per 32-row q block
    int32_t n_q_items;
    const int2 *kv_items;     // (b, first row) per 32-row kv block
    int32_t n_kv_items;
    const int2 *qblk_rows;    // (b, first row) per global 64-row q block
    int32_t n_qblk;
    float *lse2;              // blocked [q block][Nq][64]: m*log2(e) + log2(l)  (+inf if l == 0)
    float *drow;              // blocked: rowsum(dY o O)
    float *sinkrow;           // blocked: -p_sink * D  (sink only)
    // tensor-core path
    const GradUnit *units;
    int32_t n_units;
    const QBlockInfo *qblk;   // [n_qblk]
    int32_t *flags;           // [n_qblk][Nq] dQ chain counters (completed contributions)
    float *dqacc;             // [Tq][Nq][D] fp32 partial sums
    int64_t wait_limit_cycles;
    int32_t num_sms;
    int32_t test_flags;       // bit 0: CTA 0 skips its first K load (bounded-wait test)
    int32_t deterministic;    // 1: dQ contributions added in chain order; 0: in arrival order
};

struct FwdArgs {
    const void *q, *k, *v;
    const uint8_t *drop_mask;
    const float *sink;
    void *o;
    float *smax, *ssum;
    int dtype;
    int32_t batch, nq, nkv, d, group;
    int32_t vd;               // head dim of value, dy, the output and dV (<= d)
    int64_t tq, tkv;
    float scale, keep_prob, inv_keep;
    MaskSpec mask;
    PseSpec pse;
    int has_drop, has_sink;
    uint32_t *status;
    const SeqDesc *seqs;
    const int2 *q_items;
    int32_t n_q_items;
    // tensor-core forward
    int64_t mask_bytes;
    const QBlockInfo *qblk;   // kv block range of every 128-row q block
    const int2 *qblk_rows;    // (b, first row) per q block
    const int2 *fwd_units;    // (q block, head), longest kv range first
    int32_t n_fwd_units;
    int64_t wait_limit_cycles;
    int32_t num_sms;
};

// Launches `kernel` as a programmatic dependent of the previous kernel on
// stream s: it may be scheduled before that kernel finishes and must call
// griddepcontrol.wait before reading what that kernel wrote.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Kernel launchers (each returns the CUDA error of its launch).
// Packs the [rows][cols] attention-mask bytes into keep bits: keep_q (row i,
// bit j) and / or keep_kv (row j, bit i), whichever is non-NULL; bits past
// the matrix are 0.
cudaError_t launch_amask_pack(const uint8_t *amask, int64_t rows, int64_t cols, uint64_t *keep_q, int32_t words_q,
                              uint64_t *keep_kv, int32_t words_kv, cudaStream_t s);
cudaError_t launch_fwd_simt(const FwdArgs &a, cudaStream_t s);
// Tensor-core forward (bf16/fp16, D = 64 or 128); false where it does not apply.
bool fwd_tc_supported(int dtype, int d);
cudaError_t launch_fwd_tc(const FwdArgs &a, cudaStream_t s);
// Gradient prepass: the blocked per-row vectors; with tc_state also zeroes
// the dQ chain counters.
cudaError_t launch_prepass(const GradArgs &a, bool tc_state, cudaStream_t s);
cudaError_t launch_grad_dkdv_simt(const GradArgs &a, cudaStream_t s);
cudaError_t launch_grad_dq_simt(const GradArgs &a, cudaStream_t s);
cudaError_t launch_sink_reduce(const GradArgs &a, cudaStream_t s);
// Tensor-core gradient (bf16/fp16, D = 64 or 128); false where it does not apply.
bool grad_tc_supported(int dtype, int d);
cudaError_t launch_grad_tc(const GradArgs &a, cudaStream_t s);
// dQ = scale * accumulated partial sums, in the output dtype; zero for q
// blocks that no kv block reaches (tensor-core path).
cudaError_t launch_dq_finalize(const GradArgs &a, cudaStream_t s);

// The gradient call behind tnd_attn_grad.  pinned_upload = false copies the
// plan from pageable host memory and allocates nothing (the library's pinned
// staging slots are allocated on first use).
tnd_status grad_run(const void *q, const void *k, const void *v, const void *dy, const void *pse, int64_t pse_batch,
                    int64_t pse_type, const uint8_t *drop_mask, const uint8_t *atten_mask, const float *smax,
                    const float *ssum, const void *o,
                    const float *sink, tnd_dtype dtype, int64_t batch, const int64_t *cuq, const int64_t *cukv,
                    const int64_t *prefix, int64_t nq, int64_t nkv, int64_t d, int64_t vd,
                    double scale, double keep, int64_t pre, int64_t next, int64_t mode, void *dq, void *dk, void *dv,
                    float *dsink, void *ws, uint64_t ws_size, void *stream, bool pinned_upload);

}  // namespace tnd
