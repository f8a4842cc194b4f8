// CUDA-core kernels of the TND attention library: the forward, the gradient
// prepass (rowsum(dY o O), log2-sum-exp, sink terms), a dK/dV kernel, a dQ
// kernel and the dSink reduction.  They serve every dtype (fp32 included),
// every head dim up to 768 and a value head dim below the query / key one
// ("aclnnFlashAttentionUnpaddingScoreGrad", constraints: qD == kD >= vD; Q, K,
// dQ, dK have D columns, V, dY, O, dV have Dv); the tensor-core gradient
// replaces the dK/dV and dQ kernels for bf16/fp16 at D = Dv = 64 and 128.
//
// Formulas: "aclnnFlashAttentionUnpaddingScoreGrad", function description
// (forward Y = Dropout(Softmax(Mask(scale Q K^T)), keep_prob) V; backward
// dV = P^T dY, dQ = dS K * scale, dK = dS^T Q * scale) and
// "aclnnFlashAttentionUnpaddingScoreGradV5", function description (sink:
// m = max(sink, max S), denominator adds exp(sink - m); dSink).
//
// Thread layout of the row kernels: 128 threads = 32 rows x 4 lanes; lane c4
// of a row owns columns c4, c4+4, c4+8, ...; a dot product of two rows is four
// partial sums combined with two shuffles.  Exponentials are base 2 on
// logits pre-multiplied by scale*log2(e).
#include "tnd_device.cuh"

#include <cmath>

namespace tnd {
namespace {

constexpr int R = kSimtRows;  // rows per block
constexpr int kThreads = 128;

// Union [ulo, uhi] of the kept key ranges of the rows held by the block
// (empty: ulo > uhi).  Every thread passes its row's range.
__device__ __forceinline__ void block_union(int64_t lo, int64_t hi, int64_t &ulo, int64_t &uhi)
{
    __shared__ long long s_lo[kThreads / 32], s_hi[kThreads / 32];
    long long a = (lo <= hi) ? lo : LLONG_MAX, b = (lo <= hi) ? hi : LLONG_MIN;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a = min(a, __shfl_xor_sync(0xffffffffu, a, o));
        b = max(b, __shfl_xor_sync(0xffffffffu, b, o));
    }
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        s_lo[w] = a;
        s_hi[w] = b;
    }
    __syncthreads();
    a = s_lo[0];
    b = s_hi[0];
#pragma unroll
    for (int i = 1; i < kThreads / 32; ++i) {
        a = min(a, s_lo[i]);
        b = max(b, s_hi[i]);
    }
    __syncthreads();
    ulo = a;
    uhi = b;
}

// pse term of (sequence b, head h, row i, column j) in the log2 units of the
// scores (pseType 1 is scaled like QK^T, the others are added after the
// scale; 2 and 3 are generated from the head's slope).
template <typename T>
__device__ __forceinline__ float pse_term(const PseSpec &ps, int32_t nq, float C, int64_t b, int64_t h, int64_t sq,
                                          int64_t i, int64_t j)
{
    if (pse_generated(ps)) return pse_alibi(ps.type, pse_slope(ps, nq, b, h), i, j) * kLog2e;
    const T *pp = (const T *)ps.ptr;
    return Elem<T>::load(pp + pse_index(ps, nq, b, h, sq, i, j)) * (ps.type == 1 ? C : kLog2e);
}

__device__ __forceinline__ float quad_sum(float x)
{
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    return x;
}

// Cooperative load of rows [r0, r0+R) of a [rows, nheads, D] tensor (head hh)
// into smem as fp32 [R][DMAX]; rows at or past `limit` and columns at or past
// D read as 0 (the row kernels multiply whole DMAX-wide rows).
template <typename T, int DMAX>
__device__ __forceinline__ void load_tile(float *dst, const T *src, int64_t row_base, int64_t r0,
                                          int64_t limit, int nheads, int hh, int D, float mul)
{
    for (int e = threadIdx.x; e < R * DMAX; e += kThreads) {
        const int rr = e / DMAX, cc = e - rr * DMAX;
        const int64_t row = r0 + rr;
        float x = 0.0f;
        if (row < limit && cc < D) x = Elem<T>::load(src + ((row_base + row) * nheads + hh) * (int64_t)D + cc) * mul;
        dst[e] = x;
    }
}

// ---------------------------------------------------------------------------
// forward: one block per (32 query rows, query head)
// ---------------------------------------------------------------------------
template <typename T, int DMAX>
__global__ void __launch_bounds__(kThreads) fwd_simt_kernel(FwdArgs a)
{
    constexpr int DP = DMAX / 4;
    extern __shared__ float smem[];
    float *Ks = smem, *Vs = smem + R * DMAX;
    const int2 it = a.q_items[blockIdx.x];
    const SeqDesc sd = a.seqs[it.x];
    const int h = blockIdx.y, g = h / a.group, D = a.d, Dv = a.vd;
    const int r = threadIdx.x >> 2, c4 = threadIdx.x & 3;
    const int64_t i = (int64_t)it.y + r;
    const bool row_ok = i < sd.sq;
    const T *Q = (const T *)a.q, *K = (const T *)a.k, *V = (const T *)a.v;
    const float C = a.scale * kLog2e;

    float qreg[DP], acc[DP];
#pragma unroll
    for (int k = 0; k < DP; ++k) {
        const int col = c4 + 4 * k;
        qreg[k] = (row_ok && col < D) ? Elem<T>::load(Q + ((sd.tq + i) * a.nq + h) * (int64_t)D + col) * C : 0.0f;
        acc[k] = 0.0f;
    }
    float m = -INFINITY, l = 0.0f;
    if (a.has_sink) {
        m = a.sink[h] * kLog2e;
        l = 1.0f;
    }
    int64_t lo = 1, hi = 0;
    if (row_ok) key_range(a.mask, sd.sq, sd.skv, sd.prefix, i, lo, hi);
    int64_t ulo, uhi;
    block_union(lo, hi, ulo, uhi);

    for (int64_t kt = (ulo <= uhi) ? (ulo / R) * R : 1; kt <= uhi; kt += R) {
        __syncthreads();
        load_tile<T, DMAX>(Ks, K, sd.tk, kt, sd.skv, a.nkv, g, D, 1.0f);
        load_tile<T, DMAX>(Vs, V, sd.tk, kt, sd.skv, a.nkv, g, Dv, 1.0f);
        __syncthreads();
        for (int c = 0; c < R; ++c) {
            const int64_t j = kt + c;
            float s = 0.0f;
#pragma unroll
            for (int k = 0; k < DP; ++k) s += qreg[k] * Ks[c * DMAX + c4 + 4 * k];
            s = quad_sum(s);
            if (j >= lo && j <= hi && matrix_keeps(a.mask, i, j)) {
                if (a.pse.ptr) s += pse_term<T>(a.pse, a.nq, C, it.x, h, sd.sq, i, j);
                const float mn = fmaxf(m, s);
                const float corr = ex2(m - mn);
                const float p = ex2(s - mn);
                const float z = a.has_drop ? drop_z(a.drop_mask, sd.mask_base, h, i, j, sd.sq, sd.skv, a.inv_keep) : 1.0f;
                const float pz = p * z;
                l = l * corr + p;
#pragma unroll
                for (int k = 0; k < DP; ++k) acc[k] = acc[k] * corr + pz * Vs[c * DMAX + c4 + 4 * k];
                m = mn;
            }
        }
    }
    if (!row_ok) return;
    const float inv = l > 0.0f ? 1.0f / l : 0.0f;
    T *O = (T *)a.o;
#pragma unroll
    for (int k = 0; k < DP; ++k) {
        const int col = c4 + 4 * k;
        if (col < Dv) Elem<T>::store(O + ((sd.tq + i) * a.nq + h) * (int64_t)Dv + col, acc[k] * inv);
    }
    const float mnat = (m == -INFINITY) ? -INFINITY : m * kLn2;
    const int64_t rbase = ((sd.tq + i) * a.nq + h) * 8;
    for (int e = c4; e < 8; e += 4) {
        a.smax[rbase + e] = mnat;
        a.ssum[rbase + e] = l;
    }
}

// ---------------------------------------------------------------------------
// gradient prepass: writes the blocked per-row vectors (padded rows
// included), one block per (128-row q block, head), heads in x so that
// blocks running together read neighbouring pieces of the same rows (q
// blocks, at most 1M / 128 + B, fit y).  Eight lanes share a
// row and read dY and O with 16-byte loads when the row length allows it
// (D * sizeof(T) a multiple of 16, at most 256 bytes).  With tc_state it
// also zeroes the dQ chain counters of the tensor-core gradient.
// ---------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ float dot16(const uint4 &x, const uint4 &y)
{
    const T *a = reinterpret_cast<const T *>(&x);
    const T *b = reinterpret_cast<const T *>(&y);
    float s = 0.0f;
#pragma unroll
    for (int e = 0; e < (int)(16 / sizeof(T)); ++e) s += Elem<T>::load(a + e) * Elem<T>::load(b + e);
    return s;
}

template <typename T>
__global__ void __launch_bounds__(256) prepass_kernel(GradArgs a, int tc_state)
{
    // block (q block qg, head h): 128 rows, 32 groups of 8 lanes, 4 rows per
    // group with all their loads issued before the sums
    const int h = blockIdx.x, qg = blockIdx.y;   // heads of a q block side by side: adjacent rows
    const int lane = threadIdx.x & 31, sub = lane & 7, grp = threadIdx.x >> 3;
    const int2 qr = a.qblk_rows[qg];
    const SeqDesc sd = a.seqs[qr.x];
    const T *dY = (const T *)a.dy, *O = (const T *)a.o;
    const int Dv = a.vd;                                    // dY and O rows
    const bool vec = ((Dv * (int)sizeof(T)) & 15) == 0 && Dv * (int)sizeof(T) <= 256;
    const int chunks = Dv * (int)sizeof(T) / 16;            // 16-byte chunks per row (at most 16)
    // the forward's max and sum of the group's rows, requested with dY and O
    // (one lane per row reads them)
    float mv[4], lv[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int64_t i = (int64_t)qr.y + grp + 32 * k;
        const int64_t r = (sd.tq + i) * a.nq + h;
        const bool rd = sub == 0 && i < sd.sq;
        mv[k] = rd ? __ldg(a.smax + r * 8) : 0.0f;
        lv[k] = rd ? __ldg(a.ssum + r * 8) : 0.0f;
    }
    float dot[4];
    if (vec) {
        uint4 y[4][2], o[4][2];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t i = (int64_t)qr.y + grp + 32 * k;
            const int64_t r = (sd.tq + i) * a.nq + h;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int c = sub + 8 * e;
                const bool ld = i < sd.sq && c < chunks;
                y[k][e] = ld ? __ldg(reinterpret_cast<const uint4 *>(dY + r * Dv) + c) : make_uint4(0, 0, 0, 0);
                o[k][e] = ld ? __ldg(reinterpret_cast<const uint4 *>(O + r * Dv) + c) : make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) dot[k] = dot16<T>(y[k][0], o[k][0]) + dot16<T>(y[k][1], o[k][1]);
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t i = (int64_t)qr.y + grp + 32 * k;
            const int64_t r = (sd.tq + i) * a.nq + h;
            dot[k] = 0.0f;
            if (i < sd.sq)
                for (int c = sub; c < Dv; c += 8) dot[k] += Elem<T>::load(dY + r * Dv + c) * Elem<T>::load(O + r * Dv + c);
        }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float d = dot[k];
        d += __shfl_xor_sync(0xffffffffu, d, 1);
        d += __shfl_xor_sync(0xffffffffu, d, 2);
        d += __shfl_xor_sync(0xffffffffu, d, 4);
        const int rr = grp + 32 * k;
        const int64_t i = (int64_t)qr.y + rr;
        const int64_t w = ((int64_t)qg * a.nq + h) * kQBlock + rr;   // blocked vector index
        if (sub != 0) continue;
        if (i >= sd.sq) {
            a.drow[w] = 0.0f;
            a.lse2[w] = INFINITY;
            if (a.has_sink) a.sinkrow[w] = 0.0f;
        } else {
            const float m = mv[k], l = lv[k];
            const bool live = l > 0.0f;
            a.drow[w] = d;
            a.lse2[w] = live ? m * kLog2e + lg2(l) : INFINITY;
            if (a.has_sink) a.sinkrow[w] = live ? -ex2((a.sink[h] - m) * kLog2e) / l * d : 0.0f;
        }
    }
    if (tc_state && threadIdx.x == 0) a.flags[(int64_t)qg * a.nq + h] = 0;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");   // the gradient kernel may be scheduled
}

// ---------------------------------------------------------------------------
// dK, dV: one block per (32 kv rows, kv head)
// ---------------------------------------------------------------------------
template <typename T, int DMAX>
__global__ void __launch_bounds__(kThreads) grad_dkdv_simt_kernel(GradArgs a)
{
    constexpr int DP = DMAX / 4;
    extern __shared__ float smem[];
    float *Qs = smem, *dYs = smem + R * DMAX;
    float *lses = dYs + R * DMAX, *Ds = lses + R;
    const int2 it = a.kv_items[blockIdx.x];
    const SeqDesc sd = a.seqs[it.x];
    const int g = blockIdx.y, D = a.d, Dv = a.vd;
    const int r = threadIdx.x >> 2, c4 = threadIdx.x & 3;
    const int64_t j = (int64_t)it.y + r;
    const bool row_ok = j < sd.skv;
    const T *Q = (const T *)a.q, *K = (const T *)a.k, *V = (const T *)a.v, *dY = (const T *)a.dy;
    const float C = a.scale * kLog2e;

    float kreg[DP], vreg[DP], adk[DP], adv[DP];
#pragma unroll
    for (int k = 0; k < DP; ++k) {
        const int col = c4 + 4 * k;
        const int64_t row = (sd.tk + j) * a.nkv + g;
        kreg[k] = (row_ok && col < D) ? Elem<T>::load(K + row * D + col) * C : 0.0f;
        vreg[k] = (row_ok && col < Dv) ? Elem<T>::load(V + row * Dv + col) : 0.0f;
        adk[k] = 0.0f;
        adv[k] = 0.0f;
    }
    const int64_t j0 = it.y, j1 = min((int64_t)it.y + R, (int64_t)sd.skv) - 1;
    const int lane = threadIdx.x & 31;

    for (int h = g * a.group; h < (g + 1) * a.group; ++h) {
        for (int64_t qt = 0; qt < sd.sq; qt += R) {
            // does any row of this q tile keep a key of [j0, j1]?
            int64_t lo = 1, hi = 0;
            if (qt + lane < sd.sq) key_range(a.mask, sd.sq, sd.skv, sd.prefix, qt + lane, lo, hi);
            const bool hit = (lo <= hi) && (hi >= j0) && (lo <= j1);
            if (!__syncthreads_or(hit)) continue;
            load_tile<T, DMAX>(Qs, Q, sd.tq, qt, sd.sq, a.nq, h, D, 1.0f);
            load_tile<T, DMAX>(dYs, dY, sd.tq, qt, sd.sq, a.nq, h, Dv, 1.0f);
            if (threadIdx.x < R) {
                const int64_t i = qt + threadIdx.x;
                const bool ok = i < sd.sq;
                lses[threadIdx.x] = ok ? a.lse2[row_vec_index(sd, a.nq, h, i)] : INFINITY;
                Ds[threadIdx.x] = ok ? a.drow[row_vec_index(sd, a.nq, h, i)] : 0.0f;
            }
            __syncthreads();
            for (int rr = 0; rr < R; ++rr) {
                const int64_t i = qt + rr;
                float s = 0.0f, dp = 0.0f;
#pragma unroll
                for (int k = 0; k < DP; ++k) {
                    s += Qs[rr * DMAX + c4 + 4 * k] * kreg[k];
                    dp += dYs[rr * DMAX + c4 + 4 * k] * vreg[k];
                }
                s = quad_sum(s);
                dp = quad_sum(dp);
                int64_t rlo = 1, rhi = 0;
                if (i < sd.sq) key_range(a.mask, sd.sq, sd.skv, sd.prefix, i, rlo, rhi);
                if (row_ok && j >= rlo && j <= rhi && matrix_keeps(a.mask, i, j)) {
                    if (a.pse.ptr) s += pse_term<T>(a.pse, a.nq, C, it.x, h, sd.sq, i, j);
                    const float p = ex2(s - lses[rr]);
                    const float z = a.has_drop ? drop_z(a.drop_mask, sd.mask_base, h, i, j, sd.sq, sd.skv, a.inv_keep) : 1.0f;
                    const float pz = p * z;
                    const float ds = p * (z * dp - Ds[rr]);
#pragma unroll
                    for (int k = 0; k < DP; ++k) {
                        adv[k] += pz * dYs[rr * DMAX + c4 + 4 * k];
                        adk[k] += ds * Qs[rr * DMAX + c4 + 4 * k];
                    }
                }
            }
            __syncthreads();
        }
    }
    if (!row_ok) return;
    T *dK = (T *)a.dk, *dV = (T *)a.dv;
#pragma unroll
    for (int k = 0; k < DP; ++k) {
        const int col = c4 + 4 * k;
        const int64_t row = (sd.tk + j) * a.nkv + g;
        if (col < D) Elem<T>::store(dK + row * D + col, adk[k] * a.scale);
        if (col < Dv) Elem<T>::store(dV + row * Dv + col, adv[k]);
    }
}

// ---------------------------------------------------------------------------
// dQ: one block per (32 query rows, query head)
// ---------------------------------------------------------------------------
template <typename T, int DMAX>
__global__ void __launch_bounds__(kThreads) grad_dq_simt_kernel(GradArgs a)
{
    constexpr int DP = DMAX / 4;
    extern __shared__ float smem[];
    float *Ks = smem, *Vs = smem + R * DMAX;
    const int2 it = a.q_items[blockIdx.x];
    const SeqDesc sd = a.seqs[it.x];
    const int h = blockIdx.y, g = h / a.group, D = a.d, Dv = a.vd;
    const int r = threadIdx.x >> 2, c4 = threadIdx.x & 3;
    const int64_t i = (int64_t)it.y + r;
    const bool row_ok = i < sd.sq;
    const T *Q = (const T *)a.q, *K = (const T *)a.k, *V = (const T *)a.v, *dY = (const T *)a.dy;
    const float C = a.scale * kLog2e;

    float qreg[DP], dyreg[DP], acc[DP];
#pragma unroll
    for (int k = 0; k < DP; ++k) {
        const int col = c4 + 4 * k;
        const int64_t row = (sd.tq + i) * a.nq + h;
        qreg[k] = (row_ok && col < D) ? Elem<T>::load(Q + row * D + col) * C : 0.0f;
        dyreg[k] = (row_ok && col < Dv) ? Elem<T>::load(dY + row * Dv + col) : 0.0f;
        acc[k] = 0.0f;
    }
    const float lse = row_ok ? a.lse2[row_vec_index(sd, a.nq, h, i)] : INFINITY;
    const float Di = row_ok ? a.drow[row_vec_index(sd, a.nq, h, i)] : 0.0f;
    int64_t lo = 1, hi = 0;
    if (row_ok) key_range(a.mask, sd.sq, sd.skv, sd.prefix, i, lo, hi);
    int64_t ulo, uhi;
    block_union(lo, hi, ulo, uhi);

    for (int64_t kt = (ulo <= uhi) ? (ulo / R) * R : 1; kt <= uhi; kt += R) {
        __syncthreads();
        load_tile<T, DMAX>(Ks, K, sd.tk, kt, sd.skv, a.nkv, g, D, 1.0f);
        load_tile<T, DMAX>(Vs, V, sd.tk, kt, sd.skv, a.nkv, g, Dv, 1.0f);
        __syncthreads();
        for (int c = 0; c < R; ++c) {
            const int64_t j = kt + c;
            float s = 0.0f, dp = 0.0f;
#pragma unroll
            for (int k = 0; k < DP; ++k) {
                s += qreg[k] * Ks[c * DMAX + c4 + 4 * k];
                dp += dyreg[k] * Vs[c * DMAX + c4 + 4 * k];
            }
            s = quad_sum(s);
            dp = quad_sum(dp);
            if (j >= lo && j <= hi && matrix_keeps(a.mask, i, j)) {
                if (a.pse.ptr) s += pse_term<T>(a.pse, a.nq, C, it.x, h, sd.sq, i, j);
                const float p = ex2(s - lse);
                const float z = a.has_drop ? drop_z(a.drop_mask, sd.mask_base, h, i, j, sd.sq, sd.skv, a.inv_keep) : 1.0f;
                const float ds = p * (z * dp - Di);
#pragma unroll
                for (int k = 0; k < DP; ++k) acc[k] += ds * Ks[c * DMAX + c4 + 4 * k];
            }
        }
    }
    if (!row_ok) return;
    T *dQ = (T *)a.dq;
#pragma unroll
    for (int k = 0; k < DP; ++k) {
        const int col = c4 + 4 * k;
        if (col < D) Elem<T>::store(dQ + ((sd.tq + i) * a.nq + h) * (int64_t)D + col, acc[k] * a.scale);
    }
}

// ---------------------------------------------------------------------------
// dSink_h = sum over all query rows of the head of -p_sink * D (fixed order;
// padded rows hold 0)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) sink_reduce_kernel(GradArgs a)
{
    __shared__ float part[256];
    const int h = blockIdx.x;
    float acc = 0.0f;
    const int64_t n = (int64_t)a.n_qblk * kQBlock;
    for (int64_t e = threadIdx.x; e < n; e += 256) {
        const int64_t qg = e / kQBlock;
        acc += a.sinkrow[(qg * a.nq + h) * kQBlock + (e - qg * kQBlock)];
    }
    part[threadIdx.x] = acc;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if (threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) a.dsink[h] = part[0];
}

template <template <typename, int> class Launch, typename... Args>
cudaError_t dispatch(int dtype, int d, Args &&...args)
{
    if (dtype == TND_BF16) {
        if (d <= 64) return Launch<__nv_bfloat16, 64>::run(args...);
        if (d <= 128) return Launch<__nv_bfloat16, 128>::run(args...);
        if (d <= 256) return Launch<__nv_bfloat16, 256>::run(args...);
        return Launch<__nv_bfloat16, 768>::run(args...);
    }
    if (dtype == TND_F16) {
        if (d <= 64) return Launch<__half, 64>::run(args...);
        if (d <= 128) return Launch<__half, 128>::run(args...);
        if (d <= 256) return Launch<__half, 256>::run(args...);
        return Launch<__half, 768>::run(args...);
    }
    if (d <= 64) return Launch<float, 64>::run(args...);
    if (d <= 128) return Launch<float, 128>::run(args...);
    if (d <= 256) return Launch<float, 256>::run(args...);
    return Launch<float, 768>::run(args...);
}

// ---------------------------------------------------------------------------
// attention-mask matrix -> keep bits, for the tensor-core kernels
// ---------------------------------------------------------------------------
// One block per 64 x 64 tile of the [rows][cols] byte matrix: the tile is
// staged in shared memory as keep flags (matrix value 0), then each warp
// turns tile rows (keep_q: row i, bit j) or tile columns (keep_kv: row j,
// bit i) into 64-bit words, two ballots per word.  Tiles past the matrix
// write zero words, so every word of the padded rows is defined.
__global__ void __launch_bounds__(256) amask_pack_kernel(const uint8_t *amask, int64_t rows, int64_t cols,
                                                         uint64_t *keep_q, int32_t words_q, uint64_t *keep_kv,
                                                         int32_t words_kv)
{
    __shared__ uint8_t tile[64][65];
    const int64_t r0 = (int64_t)blockIdx.y * 64, c0 = (int64_t)blockIdx.x * 64;
    for (int e = threadIdx.x; e < 64 * 64; e += blockDim.x) {
        const int r = e >> 6, c = e & 63;
        const int64_t gr = r0 + r, gc = c0 + c;
        tile[r][c] = (gr < rows && gc < cols) ? (uint8_t)(__ldg(amask + gr * cols + gc) == 0) : (uint8_t)0;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (keep_q) {
        for (int r = warp; r < 64; r += 8) {
            const uint32_t lo = __ballot_sync(0xffffffffu, tile[r][lane]);
            const uint32_t hi = __ballot_sync(0xffffffffu, tile[r][32 + lane]);
            if (lane == 0 && r0 + r < rows) keep_q[(r0 + r) * words_q + blockIdx.x] = ((uint64_t)hi << 32) | lo;
        }
    }
    if (keep_kv) {
        for (int c = warp; c < 64; c += 8) {
            const uint32_t lo = __ballot_sync(0xffffffffu, tile[lane][c]);
            const uint32_t hi = __ballot_sync(0xffffffffu, tile[32 + lane][c]);
            if (lane == 0 && c0 + c < cols) keep_kv[(c0 + c) * words_kv + blockIdx.y] = ((uint64_t)hi << 32) | lo;
        }
    }
}

template <typename T, int DMAX> struct FwdLaunch {
    static cudaError_t run(const FwdArgs &a, cudaStream_t s)
    {
        if (a.n_q_items == 0) return cudaSuccess;
        const size_t smem = 2 * R * DMAX * sizeof(float);
        cudaError_t e = cudaFuncSetAttribute(fwd_simt_kernel<T, DMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        fwd_simt_kernel<T, DMAX><<<dim3(a.n_q_items, a.nq), kThreads, smem, s>>>(a);
        return cudaGetLastError();
    }
};

template <typename T, int DMAX> struct DkdvLaunch {
    static cudaError_t run(const GradArgs &a, cudaStream_t s)
    {
        if (a.n_kv_items == 0) return cudaSuccess;
        const size_t smem = (2 * R * DMAX + 2 * R) * sizeof(float);
        cudaError_t e = cudaFuncSetAttribute(grad_dkdv_simt_kernel<T, DMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        grad_dkdv_simt_kernel<T, DMAX><<<dim3(a.n_kv_items, a.nkv), kThreads, smem, s>>>(a);
        return cudaGetLastError();
    }
};

template <typename T, int DMAX> struct DqLaunch {
    static cudaError_t run(const GradArgs &a, cudaStream_t s)
    {
        if (a.n_q_items == 0) return cudaSuccess;
        const size_t smem = 2 * R * DMAX * sizeof(float);
        cudaError_t e = cudaFuncSetAttribute(grad_dq_simt_kernel<T, DMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        grad_dq_simt_kernel<T, DMAX><<<dim3(a.n_q_items, a.nq), kThreads, smem, s>>>(a);
        return cudaGetLastError();
    }
};

template <typename T, int DMAX> struct PrepassLaunch {
    static cudaError_t run(const GradArgs &a, bool tc_state, cudaStream_t s)
    {
        if (a.n_qblk == 0) return cudaSuccess;
        const dim3 grid((unsigned)a.nq, (unsigned)a.n_qblk);
        prepass_kernel<T><<<grid, 256, 0, s>>>(a, tc_state ? 1 : 0);
        return cudaGetLastError();
    }
};

}  // namespace

cudaError_t launch_fwd_simt(const FwdArgs &a, cudaStream_t s) { return dispatch<FwdLaunch>(a.dtype, a.d, a, s); }
cudaError_t launch_grad_dkdv_simt(const GradArgs &a, cudaStream_t s) { return dispatch<DkdvLaunch>(a.dtype, a.d, a, s); }
cudaError_t launch_grad_dq_simt(const GradArgs &a, cudaStream_t s) { return dispatch<DqLaunch>(a.dtype, a.d, a, s); }

cudaError_t launch_prepass(const GradArgs &a, bool tc_state, cudaStream_t s)
{
    return dispatch<PrepassLaunch>(a.dtype, a.d, a, tc_state, s);
}

cudaError_t launch_amask_pack(const uint8_t *amask, int64_t rows, int64_t cols, uint64_t *keep_q, int32_t words_q,
                              uint64_t *keep_kv, int32_t words_kv, cudaStream_t s)
{
    // grid: one block per 64 x 64 tile, rows and columns rounded up to 128
    const int64_t gx = 2 * ((cols + 127) / 128), gy = 2 * ((rows + 127) / 128);
    if (rows < 1 || cols < 1 || gy > 65535 || gx > INT32_MAX) return cudaErrorInvalidValue;
    if ((keep_q && words_q != gx) || (keep_kv && words_kv != gy)) return cudaErrorInvalidValue;
    amask_pack_kernel<<<dim3((unsigned)gx, (unsigned)gy), 256, 0, s>>>(amask, rows, cols, keep_q, words_q, keep_kv,
                                                                        words_kv);
    return cudaGetLastError();
}

cudaError_t launch_sink_reduce(const GradArgs &a, cudaStream_t s)
{
    if (!a.has_sink || a.nq == 0) return cudaSuccess;
    sink_reduce_kernel<<<a.nq, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace tnd
