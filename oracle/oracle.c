/*
 * fp64 CPU oracle for the TND FlashAttention forward and score-gradient.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
 * CPU-baseline leg of the benchmark load this library.  It shares no code,
 * header, table or helper with the CUDA library and is never on its path.
 *
 * Sources (Ascend CANN operator pages):
 *   [UnpadGrad]   "aclnnFlashAttentionUnpaddingScoreGrad"   (zh, 8.3.RC1alpha002)
 *   [UnpadGradV5] "aclnnFlashAttentionUnpaddingScoreGradV5" (en)
 *   [ScoreV2]     "aclnnFlashAttentionScoreV2"              (zh, news repost)
 *
 * What is computed, per sequence b, query head h (kv head g = h / (Nq/Nkv)),
 * query row i and key row j of that sequence:
 *   s_ij  = scale * <Q_i, K_j>                                [UnpadGrad, function
 *           description: S = Mask((QK^T + pse)/sqrt(d)); scaleValue stands for
 *           1/sqrt(d), parameters section]
 *           with a pse: scale * (<Q_i, K_j> + pse_ij) (pseType 1, the grad
 *           page's formula) or scale * <Q_i, K_j> + pse_ij (pseType 0)
 *           [ScoreV2, parameters: pseType 0 multiplies then adds, 1 adds then
 *           multiplies]
 *   kept_ij from sparseMode / preTokens / nextTokens          [UnpadGrad, parameters:
 *           sparseMode]
 *   m_i   = max over kept s_ij (and the sink logit if given)  [UnpadGradV5, function
 *           description: m = max(sink, max(S))]
 *   l_i   = sum over kept exp(s_ij - m_i) (+ exp(sink - m_i)) [UnpadGradV5, the
 *           Attention formula's denominator]
 *   p_ij  = exp(s_ij - m_i) / l_i  (0 if not kept or l_i = 0)
 *   z_ij  = keep-bit / keepProb    (1 without dropout)        [UnpadGrad, function
 *           description: P = Dropout(Softmax(S), keep_prob); parameters:
 *           dropMaskOptional size (sum_b sum_n Sq*Skv)/8, keepProb = share of 1s]
 *   O_i   = sum_j p_ij z_ij V_j                                [UnpadGrad: Y = P V]
 * and the gradient:
 *   dP_ij = <dY_i, V_j>,   D_i = <dY_i, O_i>
 *   dS_ij = p_ij (z_ij dP_ij - D_i)
 *   dV_j  = sum_{h in g} sum_i p_ij z_ij dY_i                  [UnpadGrad: dV = P^T dY]
 *   dQ_i  = scale * sum_j dS_ij K_j                            [UnpadGrad: dQ = dS K / sqrt(d)]
 *   dK_j  = scale * sum_{h in g} sum_i dS_ij Q_i               [UnpadGrad: dK = dS^T Q / sqrt(d)]
 *   dSink_h = - sum_b sum_i (exp(sink_h - m_i) / l_i) D_i      [UnpadGradV5: dSink =
 *           reduce(-P * dP * SimpleSoftmax(sink, x_max, x_sum)), with
 *           sum_j P_ij dP_ij read as D_i]
 *
 * Readings taken where the pages are silent (all listed in the design notes):
 *   - dS is the derivative of the stated forward: with P the pre-dropout softmax
 *     and dropout applied as P*z, d(sum dY*O)/ds_ij = p_ij (z_ij dP_ij - D_i).
 *   - sparseMode 3 keeps j <= i + (Skv - Sq) (lower triangle anchored at the
 *     bottom-right vertex); mode 2 keeps j <= i (top-left vertex); mode 4 keeps
 *     -preTokens <= j - i <= nextTokens; mode 0 without an attention-mask
 *     tensor keeps everything and ignores preTokens/nextTokens.
 *   - attenMaskOptional [UnpadGrad, parameters; ScoreV2, parameters: 1 masks,
 *     0 keeps] is one [S1Max, S2Max] matrix (the longest query and key
 *     sequence) shared by every sequence and head, indexed by the in-sequence
 *     row i and column j.  Mode 1 keeps where it is 0; mode 0 with the matrix
 *     keeps where it is 0 and inside the preTokens/nextTokens band (the
 *     parameters section: the part between preTokens and nextTokens is
 *     computed); modes 2, 3, 4 and 6 take the pages' compressed matrices,
 *     which only restate their index rules, so the matrix is not read there.
 *   - mode 6 (prefix) keeps j <= i + (Skv - Sq) (the bottom-right lower
 *     triangle, the upper part of the compressed matrix) or j < N_b, the
 *     sequence's prefixOptional value (the lower part: the first N_b columns
 *     kept for every row).
 *   - keep-bit of (b, h, i, j) sits at flat index
 *     base_b + (h*Sq_b + i)*Skv_b + j, base_b = sum_{b'<b} Nq*Sq_b'*Skv_b',
 *     byte = index >> 3, bit = index & 7 (least significant bit first).
 *   - a row with no kept key and no sink has m = -inf, l = 0, O = 0 and
 *     contributes nothing to the gradient.
 *   - pseShiftOptional [UnpadGrad, parameters: shape [B,N,H,S] or [1,N,H,S],
 *     H = 1024; alibi needs a lower triangle and Sq = Skv; UnpadGradV5,
 *     constraints: alibi_compress = ori_pse[:, :, -1024:, :]] holds, per
 *     sequence (or for all, when its first dimension is 1) and query head,
 *     the last 1024 rows of the [Sq, Skv] bias: row i of the sequence is
 *     stored row i - (Sq - 1024) (so a sequence shorter than 1024 sits at the
 *     bottom of the 1024 rows), and a row above the stored ones (i < Sq - 1024)
 *     is read along its diagonal from stored row 0, column j + (Sq - 1024 - i),
 *     which reproduces a bias that depends only on i - j (alibi).  dpseOut is
 *     a reserved output on the pages and is not computed.
 *   - pseType 2 / 3 [ScoreV2, parameters]: the pse is generated inside from
 *     one fp32 slope per (sequence or all, head), [B, N] or [N]; the pages do
 *     not print the generator.  Reading: the alibi bias -slope |i - j| (2) and
 *     -slope sqrt(|i - j|) (3, the table's extra sqrt), added after the scale
 *     (both "multiply, then add").
 *   - head dims [UnpadGrad, constraints: qD == kD >= vD]: query, key, dQ and
 *     dK have D columns; value, dy, the attention output and dV have Dv <= D
 *     (Dv = D when not given).  <Q_i, K_j> runs over D, <dY_i, V_j> and
 *     <dY_i, O_i> over Dv; scaleValue is used as given.
 *
 * Everything is plain fp64 loops over rows; the selection fields of
 * ora_problem (head range, first row per sequence) only narrow loop bounds so
 * that tests can evaluate part of a large problem.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct ora_problem {
    int64_t B;
    const int64_t *cu_q;    /* B+1 cumulative query offsets, cu_q[0] = 0        */
    const int64_t *cu_kv;   /* B+1 cumulative key/value offsets                 */
    int64_t Nq, Nkv, D;
    double scale;           /* scaleValue                                       */
    double keep_prob;       /* keepProb in (0, 1]                               */
    int64_t pre_tokens, next_tokens, sparse_mode;
    const uint8_t *drop_mask; /* packed keep-bits, NULL = no dropout            */
    const double *sink;       /* [Nq] sink logits, NULL = no sink               */
    /* selection: heads [h_lo, h_hi) and rows i >= row_lo[b] (NULL = all rows) */
    int64_t h_lo, h_hi;
    const int64_t *row_lo;
    /* attenMaskOptional [mask_rows][mask_cols], nonzero masks (NULL = none);
     * prefixOptional [B] (NULL = none) */
    const uint8_t *atten_mask;
    int64_t mask_rows, mask_cols;
    const int64_t *prefix;
    /* pseShiftOptional [pse_batch][Nq][1024][pse_cols] (NULL = none) and pseType */
    const double *pse;
    int64_t pse_batch, pse_cols, pse_type;
    /* head dim of value, dy, attention out and dv (0 = D); query and key use D */
    int64_t Dv;
} ora_problem;

/* sparseMode predicate; [UnpadGrad, parameters: sparseMode]. */
int ora_keep(int64_t mode, int64_t pre, int64_t next, int64_t sq, int64_t skv,
             int64_t i, int64_t j)
{
    switch (mode) {
    case 0: return 1;                                  /* no attenMask: keep all */
    case 2: return j <= i;                             /* leftUpCausal           */
    case 3: return j <= i + (skv - sq);                /* rightDownCausal        */
    case 4: return (j - i >= -pre) && (j - i <= next); /* band                   */
    default: return 0;
    }
}

/* Whether (b, i, j) is kept: the sparseMode rule with the attention-mask
 * matrix and the prefix where the mode uses them [UnpadGrad, parameters:
 * sparseMode, attenMaskOptional, prefixOptional]. */
int ora_keep_at(const ora_problem *p, int64_t b, int64_t sq, int64_t skv, int64_t i, int64_t j)
{
    const int64_t mode = p->sparse_mode;
    const int masked = p->atten_mask != NULL && p->atten_mask[i * p->mask_cols + j] != 0;
    switch (mode) {
    case 0:
        if (p->atten_mask == NULL) return 1;
        return !masked && (j - i >= -p->pre_tokens) && (j - i <= p->next_tokens);
    case 1: return !masked;
    case 6: return j <= i + (skv - sq) || j < p->prefix[b];
    default: return ora_keep(mode, p->pre_tokens, p->next_tokens, sq, skv, i, j);
    }
}

/* pse of (b, h, i, j).  pseType 0 / 1: from the stored last 1024 rows of the
 * sequence's bias [UnpadGrad, parameters: pseShiftOptional; UnpadGradV5,
 * constraints: alibi compression]; rows above the stored ones along their
 * diagonal.  pseType 2 / 3: generated from the fp32 slope of (b, h) [ScoreV2,
 * parameters: realShiftOptional is FLOAT32 [B, N] or [N] for them; the pseType
 * table: generated inside, multiply then add (3: then sqrt)], read as the alibi
 * bias -slope |i - j| (2) and -slope sqrt(|i - j|) (3). */
double ora_pse_at(const ora_problem *p, int64_t b, int64_t h, int64_t sq, int64_t i, int64_t j)
{
    const int64_t bb = p->pse_batch == 1 ? 0 : b;
    if (p->pse_type == 2 || p->pse_type == 3) {
        const double slope = p->pse[bb * p->Nq + h];
        const double dist = (double)(i > j ? i - j : j - i);
        return -slope * (p->pse_type == 2 ? dist : sqrt(dist));
    }
    int64_t r = i - (sq - 1024), c = j;
    if (r < 0) {
        c = j - r;
        r = 0;
    }
    return p->pse[((bb * p->Nq + h) * 1024 + r) * p->pse_cols + c];
}

/* the logit s_ij from <Q_i, K_j> [UnpadGrad: (QK^T + pse)/sqrt(d); ScoreV2: pseType 1
 * adds then multiplies, every other type multiplies then adds] */
static double logit(const ora_problem *p, double qk, int64_t b, int64_t h, int64_t sq, int64_t i, int64_t j)
{
    if (p->pse == NULL) return p->scale * qk;
    const double pse = ora_pse_at(p, b, h, sq, i, j);
    return p->pse_type == 1 ? p->scale * (qk + pse) : p->scale * qk + pse;
}

/* first flat keep-bit index of sequence b */
int64_t ora_mask_base(const ora_problem *p, int64_t b)
{
    int64_t base = 0;
    for (int64_t bb = 0; bb < b; ++bb) {
        base += p->Nq * (p->cu_q[bb + 1] - p->cu_q[bb]) * (p->cu_kv[bb + 1] - p->cu_kv[bb]);
    }
    return base;
}

int ora_keep_bit(const uint8_t *mask, int64_t index)
{
    return (mask[index >> 3] >> (index & 7)) & 1;
}

/* z_ij: dropout multiplier of one (b, h, i, j) */
static double drop_z(const ora_problem *p, int64_t base, int64_t h, int64_t i, int64_t j,
                     int64_t sq, int64_t skv)
{
    if (p->drop_mask == NULL || p->keep_prob >= 1.0) return 1.0;
    int64_t index = base + (h * sq + i) * skv + j;
    return ora_keep_bit(p->drop_mask, index) ? 1.0 / p->keep_prob : 0.0;
}

static double dot(const double *a, const double *b, int64_t n)
{
    double acc = 0.0;
    for (int64_t d = 0; d < n; ++d) acc += a[d] * b[d];
    return acc;
}

/* vD [UnpadGrad, constraints: qD == kD >= vD] */
static int64_t value_dim(const ora_problem *p) { return p->Dv > 0 ? p->Dv : p->D; }

static int row_selected(const ora_problem *p, int64_t b, int64_t i)
{
    return p->row_lo == NULL || i >= p->row_lo[b];
}

/* scores s_ij of row (b, h, i) into s[0..skv), kept flags into kept[] */
static void row_scores(const ora_problem *p, const double *q, const double *k,
                       int64_t b, int64_t h, int64_t i, double *s, unsigned char *kept)
{
    const int64_t G = p->Nq / p->Nkv, g = h / G, D = p->D;
    const int64_t tq = p->cu_q[b], tk = p->cu_kv[b];
    const int64_t sq = p->cu_q[b + 1] - tq, skv = p->cu_kv[b + 1] - tk;
    const double *qi = q + ((tq + i) * p->Nq + h) * D;
    for (int64_t j = 0; j < skv; ++j) {
        kept[j] = (unsigned char)ora_keep_at(p, b, sq, skv, i, j);
        s[j] = kept[j] ? logit(p, dot(qi, k + ((tk + j) * p->Nkv + g) * D, D), b, h, sq, i, j) : 0.0;
    }
}

/* m_i and l_i of one row from its scores; [UnpadGradV5] sink formulas */
static void row_max_sum(const ora_problem *p, int64_t h, const double *s, const unsigned char *kept,
                        int64_t skv, double *m_out, double *l_out)
{
    double m = -INFINITY;
    for (int64_t j = 0; j < skv; ++j)
        if (kept[j] && s[j] > m) m = s[j];
    if (p->sink && p->sink[h] > m) m = p->sink[h];
    double l = 0.0;
    if (m > -INFINITY) {
        for (int64_t j = 0; j < skv; ++j)
            if (kept[j]) l += exp(s[j] - m);
        if (p->sink) l += exp(p->sink[h] - m);
    }
    *m_out = m;
    *l_out = l;
}

static int64_t max_skv(const ora_problem *p)
{
    int64_t mx = 1;
    for (int64_t b = 0; b < p->B; ++b) {
        int64_t s = p->cu_kv[b + 1] - p->cu_kv[b];
        if (s > mx) mx = s;
    }
    return mx;
}

/* (b, h, i) of flat query-row index r over all sequences and heads; -1 if none */
static int row_of(const ora_problem *p, int64_t r, int64_t *b_out, int64_t *h_out, int64_t *i_out)
{
    const int64_t t = r / p->Nq, h = r % p->Nq;
    for (int64_t b = 0; b < p->B; ++b) {
        if (t >= p->cu_q[b] && t < p->cu_q[b + 1]) {
            *b_out = b;
            *h_out = h;
            *i_out = t - p->cu_q[b];
            return 0;
        }
    }
    return -1;
}

/*
 * Forward: out [Tq][Nq][Dv], smax / ssum [Tq][Nq] (natural-log units).
 * [UnpadGrad] Y = Dropout(Softmax(Mask(scale QK^T)), keep_prob) V, with the
 * forward's max and sum as described for softmaxMax / softmaxSum [ScoreV2].
 * Every query row is independent; rows run in parallel.
 */
int ora_fwd(const ora_problem *p, const double *q, const double *k, const double *v,
            double *out, double *smax, double *ssum)
{
    const int64_t Dv = value_dim(p), G = p->Nq / p->Nkv;
    const int64_t nrows = p->cu_q[p->B] * p->Nq, skvmax = max_skv(p);
    int err = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * skvmax);
        unsigned char *kept = (unsigned char *)malloc(skvmax);
        if (!s || !kept) err = 1;
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < nrows; ++r) {
            int64_t b, h, i;
            if (!s || !kept || row_of(p, r, &b, &h, &i)) continue;
            if (h < p->h_lo || h >= p->h_hi || !row_selected(p, b, i)) continue;
            const int64_t g = h / G, tq = p->cu_q[b], tk = p->cu_kv[b];
            const int64_t sq = p->cu_q[b + 1] - tq, skv = p->cu_kv[b + 1] - tk;
            const int64_t base = ora_mask_base(p, b);
            double m, l;
            row_scores(p, q, k, b, h, i, s, kept);
            row_max_sum(p, h, s, kept, skv, &m, &l);
            double *o = out + r * Dv;
            for (int64_t d = 0; d < Dv; ++d) o[d] = 0.0;
            if (l > 0.0) {
                for (int64_t j = 0; j < skv; ++j) {
                    if (!kept[j]) continue;
                    const double w = exp(s[j] - m) / l * drop_z(p, base, h, i, j, sq, skv);
                    const double *vj = v + ((tk + j) * p->Nkv + g) * Dv;
                    for (int64_t d = 0; d < Dv; ++d) o[d] += w * vj[d];
                }
            }
            smax[r] = m;
            ssum[r] = l;
        }
        free(s);
        free(kept);
    }
    return err;
}

/* dS_ij of one (b, h, i, j) from the row's statistics; 0 if not kept */
static double grad_ds(const ora_problem *p, const double *q, const double *k, const double *v,
                      const double *dy, double m, double l, double Di, int64_t b, int64_t base,
                      int64_t h, int64_t i, int64_t j, double *pz_out)
{
    const int64_t G = p->Nq / p->Nkv, g = h / G, D = p->D, Dv = value_dim(p);
    const int64_t tq = p->cu_q[b], tk = p->cu_kv[b];
    const int64_t sq = p->cu_q[b + 1] - tq, skv = p->cu_kv[b + 1] - tk;
    *pz_out = 0.0;
    if (!ora_keep_at(p, b, sq, skv, i, j) || !(l > 0.0)) return 0.0;
    const int64_t r = (tq + i) * p->Nq + h;
    const double *kj = k + ((tk + j) * p->Nkv + g) * D, *vj = v + ((tk + j) * p->Nkv + g) * Dv;
    const double s = logit(p, dot(q + r * D, kj, D), b, h, sq, i, j);
    const double pij = exp(s - m) / l;
    const double z = drop_z(p, base, h, i, j, sq, skv);
    const double dP = dot(dy + r * Dv, vj, Dv);
    *pz_out = pij * z;
    return pij * (z * dP - Di);
}

/*
 * Gradient from the forward's out / smax / ssum (as the grad operator consumes
 * attentionIn, softmaxMax and softmaxSum [UnpadGrad, parameters]).
 * dq like q, dk like k, dv like v; dsink [Nq] (may be NULL without a sink).
 * ds_dense (may be NULL): dS at the flat keep-bit index of every (b,h,i,j).
 * Only selected heads / rows are written; dk / dv of every kv row of every
 * selected kv group are overwritten (they sum over the selected rows only).
 * Three passes, each over independent outputs: D_i per query row, dQ per
 * query row, dK / dV per key row.
 */
int ora_grad(const ora_problem *p, const double *q, const double *k, const double *v,
             const double *dy, const double *out, const double *smax, const double *ssum,
             double *dq, double *dk, double *dv, double *dsink, double *ds_dense)
{
    const int64_t D = p->D, Dv = value_dim(p), G = p->Nq / p->Nkv;
    const int64_t nrows = p->cu_q[p->B] * p->Nq, nkvrows = p->cu_kv[p->B] * p->Nkv;
    double *Drow = (double *)calloc((size_t)(nrows > 0 ? nrows : 1), sizeof(double));
    if (!Drow) return 1;
    /* D_i = <dY_i, O_i> */
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < nrows; ++r) Drow[r] = dot(dy + r * Dv, out + r * Dv, Dv);
    /* dQ_i = scale * sum_j dS_ij K_j */
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t b, h, i;
        if (row_of(p, r, &b, &h, &i)) continue;
        if (h < p->h_lo || h >= p->h_hi || !row_selected(p, b, i)) continue;
        const int64_t g = h / G, tk = p->cu_kv[b], skv = p->cu_kv[b + 1] - tk;
        const int64_t sq = p->cu_q[b + 1] - p->cu_q[b];
        const int64_t base = ora_mask_base(p, b);
        double *dqi = dq + r * D;
        for (int64_t d = 0; d < D; ++d) dqi[d] = 0.0;
        for (int64_t j = 0; j < skv; ++j) {
            double pz;
            const double dS = grad_ds(p, q, k, v, dy, smax[r], ssum[r], Drow[r], b, base, h, i, j, &pz);
            if (dS == 0.0) continue;
            const double *kj = k + ((tk + j) * p->Nkv + g) * D;
            for (int64_t d = 0; d < D; ++d) dqi[d] += p->scale * dS * kj[d];
            if (ds_dense) ds_dense[base + (h * sq + i) * skv + j] = dS;
        }
    }
    /* dK_j = scale * sum_{h in g} sum_i dS_ij Q_i,  dV_j = sum_{h in g} sum_i p_ij z_ij dY_i */
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t kr = 0; kr < nkvrows; ++kr) {
        const int64_t t = kr / p->Nkv, g = kr % p->Nkv;
        if ((g + 1) * G <= p->h_lo || g * G >= p->h_hi) continue;
        int64_t b = 0;
        while (b < p->B && !(t >= p->cu_kv[b] && t < p->cu_kv[b + 1])) ++b;
        if (b >= p->B) continue;
        const int64_t j = t - p->cu_kv[b], tq = p->cu_q[b], sq = p->cu_q[b + 1] - tq;
        const int64_t base = ora_mask_base(p, b);
        double *dkj = dk + kr * D, *dvj = dv + kr * Dv;
        for (int64_t d = 0; d < D; ++d) dkj[d] = 0.0;
        for (int64_t d = 0; d < Dv; ++d) dvj[d] = 0.0;
        for (int64_t h = g * G; h < (g + 1) * G; ++h) {
            if (h < p->h_lo || h >= p->h_hi) continue;
            for (int64_t i = p->row_lo ? p->row_lo[b] : 0; i < sq; ++i) {
                if (!row_selected(p, b, i)) continue;
                const int64_t r = (tq + i) * p->Nq + h;
                double pz;
                const double dS = grad_ds(p, q, k, v, dy, smax[r], ssum[r], Drow[r], b, base, h, i, j, &pz);
                const double *qi = q + r * D, *dyi = dy + r * Dv;
                for (int64_t d = 0; d < D; ++d) dkj[d] += p->scale * dS * qi[d];
                for (int64_t d = 0; d < Dv; ++d) dvj[d] += pz * dyi[d];
            }
        }
    }
    /* dSink_h = -sum_i exp(sink_h - m_i) / l_i * D_i, summed in row order */
    if (dsink) {
        for (int64_t h = p->h_lo; h < p->h_hi; ++h) dsink[h] = 0.0;
        if (p->sink) {
            for (int64_t r = 0; r < nrows; ++r) {
                int64_t b, h, i;
                if (row_of(p, r, &b, &h, &i)) continue;
                if (h < p->h_lo || h >= p->h_hi || !row_selected(p, b, i)) continue;
                if (ssum[r] > 0.0) dsink[h] -= exp(p->sink[h] - smax[r]) / ssum[r] * Drow[r];
            }
        }
    }
    free(Drow);
    return 0;
}
