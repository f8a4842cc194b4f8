// Host side of the C ABI declared in include/tnd_attn.h: argument checks
// (the first phase of the pages' two-phase interface, "function prototype"
// and "constraints" sections of aclnnFlashAttentionUnpaddingScoreGrad /
// ...GradV5), the per-call plan (sequence table, work lists, tensor-core
// units), the workspace layout and the kernel launches.
#include "tnd_internal.h"

#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstring>
#include <memory>
#include <mutex>
#include <vector>

namespace tnd {
namespace {

// ---------------------------------------------------------------------------
// process-wide options and the kernel-time record
// ---------------------------------------------------------------------------
struct Options {
    int grad_path = 0;
    int64_t wait_limit_ms = 2000;
    int profile = 0;
    int test_skip_load = 0;
    int deterministic = 1;
};
Options g_opt;
std::mutex g_mu;

struct ProfEntry {
    int kind;
    cudaEvent_t start, stop;
};
const char *kKindNames[] = {"fwd_simt",         "grad_prepass", "grad_dkdv_simt", "grad_dq_simt", "grad_sink_reduce",
                            "grad_tc_main",     "grad_dq_finalize", "fwd_tc",     "atten_mask_pack"};
constexpr int kNumKinds = sizeof(kKindNames) / sizeof(kKindNames[0]);
enum Kind { K_FWD = 0, K_PREPASS, K_DKDV, K_DQ, K_SINK, K_TC, K_FIN, K_FWD_TC, K_PACK };
std::vector<ProfEntry> g_prof;
std::vector<cudaEvent_t> g_event_pool;
constexpr size_t kProfCap = 4096;

cudaEvent_t take_event()
{
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

// Runs `launch` on stream s, bracketed by events when profiling is on.
template <typename F>
cudaError_t timed(int kind, cudaStream_t s, F &&launch)
{
    if (!g_opt.profile) return launch();
    std::lock_guard<std::mutex> lk(g_mu);
    cudaEvent_t a = take_event(), b = take_event();
    if (!a || !b) return launch();
    cudaEventRecord(a, s);
    cudaError_t e = launch();
    cudaEventRecord(b, s);
    if (g_prof.size() >= kProfCap) {
        cudaEventSynchronize(g_prof.front().stop);
        g_event_pool.push_back(g_prof.front().start);
        g_event_pool.push_back(g_prof.front().stop);
        g_prof.erase(g_prof.begin());
    }
    g_prof.push_back({kind, a, b});
    return e;
}

// ---------------------------------------------------------------------------
// validation
// ---------------------------------------------------------------------------
struct Problem {
    int dtype = 0;
    int64_t batch = 0;
    const int64_t *cuq = nullptr, *cukv = nullptr;
    int64_t nq = 0, nkv = 0, d = 0;
    int64_t dv = 0;                    // value / dy / output head dim (qD == kD >= vD)
    double scale = 0, keep = 1;
    int64_t pre = 0, next = 0, mode = 0;
    bool has_drop = false, has_sink = false;
    bool has_amask = false;            // the attention-mask matrix is read (sparseMode 0 / 1)
    const int64_t *prefix = nullptr;   // prefixOptional (sparseMode 6)
    int64_t tq = 0, tkv = 0;
    int64_t s1max = 0, s2max = 0;      // longest query / key sequence: the matrix is [S1Max][S2Max]
};

constexpr int64_t kMaxTokens = int64_t(1) << 20;  // T in [1, 1M]
constexpr int64_t kMaxHeads = 256;                // N in [1, 256]
constexpr int64_t kMaxHeadDim = 768;              // D in [1, 768] (V5 page)
constexpr int64_t kMaxBatch = 20000;              // B in [1, 20000] (V5 page)
constexpr int64_t kMaxBatchPrefix = 1024;         // B in [1, 1K] with prefixOptional
constexpr int64_t kTokenClamp = int64_t(1) << 40; // |preTokens|, |nextTokens| beyond any T act alike
constexpr int64_t kSimtMaxHeadDim = 768;          // the CUDA-core kernels (instances up to D = 64, 128, 256, 768)

// Argument checks of the first phase ([UnpadGrad] parameters and constraints:
// sparseMode, attenMaskOptional, prefixOptional).  Modes 0 (with the matrix)
// and 1 read the attention-mask matrix; modes 2, 3, 4 and 6 are index rules
// (the pages' compressed matrices for them restate those rules, so a matrix
// passed with them is not read); mode 6 reads prefix; 5, 7 and 8 are not
// implemented.
tnd_status validate(int dtype, int64_t batch, const int64_t *cuq, const int64_t *cukv, const int64_t *prefix,
                    int64_t nq, int64_t nkv, int64_t d, int64_t vd, double scale, double keep, int64_t pre,
                    int64_t next, int64_t mode, bool has_drop, bool has_amask, bool has_sink, Problem &p)
{
    if (!cuq || !cukv) return TND_ERR_NULLPTR;
    if (keep < 1.0 && !has_drop) return TND_ERR_NULLPTR;  // dropMask needed when keepProb < 1
    if (mode == 1 && !has_amask) return TND_ERR_NULLPTR;  // the full matrix is the mask
    if (mode == 6 && !prefix) return TND_ERR_NULLPTR;
    if (dtype != TND_F16 && dtype != TND_BF16 && dtype != TND_F32) return TND_ERR_INVALID;
    if (batch < 1 || batch > kMaxBatch) return TND_ERR_INVALID;
    if (cuq[0] != 0 || cukv[0] != 0) return TND_ERR_INVALID;
    for (int64_t b = 0; b < batch; ++b) {
        if (cuq[b + 1] < cuq[b] || cukv[b + 1] < cukv[b]) return TND_ERR_INVALID;
    }
    p.tq = cuq[batch];
    p.tkv = cukv[batch];
    if (p.tq < 1 || p.tq > kMaxTokens || p.tkv < 1 || p.tkv > kMaxTokens) return TND_ERR_INVALID;
    if (nq < 1 || nq > kMaxHeads || nkv < 1 || nkv > kMaxHeads || nq % nkv != 0) return TND_ERR_INVALID;
    if (d < 1 || d > kMaxHeadDim) return TND_ERR_INVALID;
    if (vd < 1 || vd > d) return TND_ERR_INVALID;         // qD == kD >= vD
    if (!(keep > 0.0 && keep <= 1.0)) return TND_ERR_INVALID;
    if (!std::isfinite(scale)) return TND_ERR_INVALID;
    if (mode < 0 || mode > 8) return TND_ERR_INVALID;
    pre = std::max(-kTokenClamp, std::min(pre, kTokenClamp));
    next = std::max(-kTokenClamp, std::min(next, kTokenClamp));
    const bool band = mode == 4 || (mode == 0 && has_amask);
    if (band && pre + next < 0) return TND_ERR_INVALID;  // band needs an intersection
    if (mode == 5 || mode >= 7) return TND_ERR_UNSUPPORTED;
    if (mode == 4) {
        for (int64_t b = 0; b < batch; ++b) {
            if (cuq[b + 1] - cuq[b] != cukv[b + 1] - cukv[b]) return TND_ERR_UNSUPPORTED;
        }
    }
    if (mode == 6) {
        if (batch > kMaxBatchPrefix) return TND_ERR_INVALID;
        for (int64_t b = 0; b < batch; ++b) {
            if (prefix[b] < 0 || prefix[b] > cukv[b + 1] - cukv[b]) return TND_ERR_INVALID;
        }
    }
    if (d > kSimtMaxHeadDim) return TND_ERR_UNSUPPORTED;
    p.dtype = dtype;
    p.batch = batch;
    p.cuq = cuq;
    p.cukv = cukv;
    p.nq = nq;
    p.nkv = nkv;
    p.d = d;
    p.dv = vd;
    p.scale = scale;
    p.keep = keep;
    p.pre = pre;
    p.next = next;
    p.mode = mode;
    p.has_drop = has_drop && keep < 1.0;
    p.has_sink = has_sink;
    p.has_amask = has_amask && (mode == 0 || mode == 1);
    p.prefix = mode == 6 ? prefix : nullptr;
    for (int64_t b = 0; b < batch; ++b) {
        p.s1max = std::max(p.s1max, cuq[b + 1] - cuq[b]);
        p.s2max = std::max(p.s2max, cukv[b + 1] - cukv[b]);
    }
    return TND_OK;
}

// pseShiftOptional checks ([UnpadGrad] parameters: shape [B or 1, N, 1024, S];
// alibi needs a lower-triangle mask and Sq = Skv; [ScoreV2] parameters:
// pseType 0 / 1 take the given pse, 2 / 3 generate it inside from fp32 slopes
// [B, N] or [N], only for Sq = Skv).
tnd_status check_pse(const Problem &p, const void *pse, int64_t pse_batch, int64_t pse_type)
{
    if (!pse) return TND_OK;
    if (pse_type < 0 || pse_type > 3) return TND_ERR_INVALID;
    if (pse_batch != 1 && pse_batch != p.batch) return TND_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(pse) & 15u) != 0) return TND_ERR_INVALID;
    if (p.mode != 2 && p.mode != 3) return TND_ERR_UNSUPPORTED;
    for (int64_t b = 0; b < p.batch; ++b) {
        if (p.cuq[b + 1] - p.cuq[b] != p.cukv[b + 1] - p.cukv[b]) return TND_ERR_UNSUPPORTED;
    }
    return TND_OK;
}

PseSpec pse_of(const Problem &p, const void *pse, int64_t pse_batch, int64_t pse_type)
{
    PseSpec ps{};
    ps.ptr = pse;
    ps.batch = (int32_t)pse_batch;
    ps.type = (int32_t)pse_type;
    ps.cols = p.s2max;
    return ps;
}

// The index rule of the problem's sparseMode (the matrix pointers are filled
// in by the run calls).
MaskSpec mask_of(const Problem &p)
{
    MaskSpec m{};
    switch (p.mode) {
    case 0: m.mode = p.has_amask ? kRuleBand : kRuleAll; break;
    case 1: m.mode = kRuleAll; break;
    case 2: m.mode = kRuleTopLeft; break;
    case 3: m.mode = kRuleCausal; break;
    case 4: m.mode = kRuleBand; break;
    default: m.mode = kRulePrefix; break;
    }
    m.pre = p.pre;
    m.next = p.next;
    return m;
}

// 64-bit words per row of the packed matrix: rows of keep_q cover S2Max
// columns, rows of keep_kv S1Max rows, rounded up to 128 bits.
int32_t words_q_of(const Problem &p) { return (int32_t)(2 * ((p.s2max + 127) / 128)); }
int32_t words_kv_of(const Problem &p) { return (int32_t)(2 * ((p.s1max + 127) / 128)); }

int64_t mask_bits_total(const Problem &p)
{
    int64_t n = 0;
    for (int64_t b = 0; b < p.batch; ++b) n += p.nq * (p.cuq[b + 1] - p.cuq[b]) * (p.cukv[b + 1] - p.cukv[b]);
    return n;
}

bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---------------------------------------------------------------------------
// plan: sequence table, CUDA-core work lists and tensor-core units
// ---------------------------------------------------------------------------
struct Plan {
    std::vector<SeqDesc> seqs;
    std::vector<int2> q_items, kv_items;
    std::vector<GradUnit> units;
    std::vector<QBlockInfo> qblk;
    std::vector<int2> qblk_rows;  // (b, first row) of every 128-row q block, in global order
    std::vector<int2> fwd_units;  // tensor-core forward: (q block, head), longest kv range first
    int64_t kept_pairs = 0;       // summed over sequences and query heads
    std::vector<unsigned char> image;  // status words + plan arrays, as copied to the workspace
};

// L2 share (bytes) for the q-side tiles of the gradient units that run together.
constexpr int64_t kL2GroupBytes = int64_t(48) << 20;

// Union of the kept key ranges of query rows [r0, r1) (empty: lo > hi).
void rows_union(const MaskSpec &m, int64_t sq, int64_t skv, int64_t prefix_n, int64_t r0, int64_t r1,
                int64_t &ulo, int64_t &uhi)
{
    ulo = INT64_MAX;
    uhi = INT64_MIN;
    for (int64_t i = r0; i < r1; ++i) {
        int64_t lo, hi;
        key_range(m, sq, skv, prefix_n, i, lo, hi);
        if (lo > hi) continue;
        ulo = std::min(ulo, lo);
        uhi = std::max(uhi, hi);
    }
}

void build_plan(const Problem &p, bool with_units, Plan &pl)
{
    const MaskSpec m = mask_of(p);
    const int64_t G = p.nq / p.nkv;
    pl.seqs.resize(p.batch);
    int64_t base = 0, qblk0 = 0;
    struct GroupWork {
        int64_t work;
        int32_t b;
    };
    std::vector<GroupWork> gw;
    std::vector<std::vector<GradUnit>> seq_units(p.batch);
    for (int64_t b = 0; b < p.batch; ++b) {
        const int64_t sq = p.cuq[b + 1] - p.cuq[b], skv = p.cukv[b + 1] - p.cukv[b];
        SeqDesc &sd = pl.seqs[b];
        sd.tq = p.cuq[b];
        sd.tk = p.cukv[b];
        sd.sq = (int32_t)sq;
        sd.skv = (int32_t)skv;
        sd.mask_base = base;
        sd.qblk0 = (int32_t)qblk0;
        sd.nqblk = (int32_t)((sq + kQBlock - 1) / kQBlock);
        sd.prefix = p.prefix ? (int32_t)p.prefix[b] : 0;
        base += p.nq * sq * skv;
        qblk0 += sd.nqblk;
        for (int64_t r = 0; r < sq; r += kSimtRows) pl.q_items.push_back(make_int2((int)b, (int)r));
        for (int64_t r = 0; r < skv; r += kSimtRows) pl.kv_items.push_back(make_int2((int)b, (int)r));
        for (int64_t r = 0; r < sq; r += kQBlock) pl.qblk_rows.push_back(make_int2((int)b, (int)r));
        for (int64_t i = 0; i < sq; ++i) {
            int64_t lo, hi;
            key_range(m, sq, skv, sd.prefix, i, lo, hi);
            if (hi >= lo) pl.kept_pairs += (hi - lo + 1) * p.nq;
        }
        if (!with_units) continue;
        const int64_t nkb = (skv + kKvBlock - 1) / kKvBlock;
        std::vector<int32_t> ilo(nkb, INT32_MAX), ihi(nkb, -1);
        for (int64_t qb = 0; qb < sd.nqblk; ++qb) {
            int64_t ulo, uhi;
            rows_union(m, sq, skv, sd.prefix, qb * kQBlock, std::min<int64_t>(sq, (qb + 1) * kQBlock), ulo, uhi);
            QBlockInfo qi;
            if (ulo > uhi) {
                qi.jlo = qi.jhi = -1;
            } else {
                qi.jlo = (int32_t)(ulo / kKvBlock);
                qi.jhi = (int32_t)(uhi / kKvBlock);
                for (int64_t j = qi.jlo; j <= qi.jhi; ++j) {
                    ilo[j] = std::min<int32_t>(ilo[j], (int32_t)qb);
                    ihi[j] = std::max<int32_t>(ihi[j], (int32_t)qb);
                }
            }
            pl.qblk.push_back(qi);
        }
        int64_t work = 0;
        // kv blocks in descending order: the dQ chain of a q block runs from
        // its highest contributing kv block down to its lowest.
        for (int64_t j = nkb - 1; j >= 0; --j) {
            GradUnit u{};
            u.b = (int32_t)b;
            u.j = (int32_t)j;
            u.qb_lo = ihi[j] < 0 ? 0 : ilo[j];
            u.qb_hi = ihi[j] < 0 ? 0 : ihi[j] + 1;
            work += u.qb_hi - u.qb_lo + 1;
            seq_units[b].push_back(u);
        }
        gw.push_back({work, (int32_t)b});
    }
    if (!with_units) return;
    // forward units: every (q block, head), q blocks with the longest kv
    // range first (heads of a q block together)
    {
        std::vector<int> order(pl.qblk.size());
        for (size_t q = 0; q < order.size(); ++q) order[q] = (int)q;
        auto span = [&](int q) { return pl.qblk[q].jlo < 0 ? 0 : pl.qblk[q].jhi - pl.qblk[q].jlo + 1; };
        std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return span(x) > span(y); });
        for (int q : order)
            for (int64_t h = 0; h < p.nq; ++h) pl.fwd_units.push_back(make_int2(q, (int)h));
    }
    // Gradient units: sequences with the most work first.  Within a
    // sequence the kv heads go in groups, and a group's kv blocks in
    // descending order (every kv head's chain is dispatched in chain order,
    // so no unit ever waits on one not yet handed out) with the group's heads
    // of a block together: under a causal mask the low kv blocks carry the
    // most tiles, and interleaving heads makes the last units of a group
    // similar in size.  A group holds as many kv heads as keep the q-side
    // tiles its units sweep (Q, dY and the fp32 dQ accumulator of every q
    // block of the group's query heads) within kL2GroupBytes, so the units
    // running together re-read those tiles from L2 rather than from HBM.
    std::stable_sort(gw.begin(), gw.end(), [](const GroupWork &x, const GroupWork &y) { return x.work > y.work; });
    const int64_t tile_bytes = (int64_t)kQBlock * p.d * (2 + 2 + 4);   // Q, dY (16-bit) and fp32 dQ rows
    for (const GroupWork &w : gw) {
        const int64_t per_head = G * (int64_t)pl.seqs[w.b].nqblk * tile_bytes;
        const int64_t hg = std::max<int64_t>(1, std::min<int64_t>(p.nkv, kL2GroupBytes / std::max<int64_t>(1, per_head)));
        for (int64_t g0 = 0; g0 < p.nkv; g0 += hg) {
            for (GradUnit u : seq_units[w.b]) {
                for (int64_t g = g0; g < std::min(p.nkv, g0 + hg); ++g) {
                    u.g = (int32_t)g;
                    pl.units.push_back(u);
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// workspace layout
// ---------------------------------------------------------------------------
struct Layout {
    size_t seqs = 0, q_items = 0, kv_items = 0, units = 0, qblk = 0, qblk_rows = 0, fwd_units = 0;  // offsets of the
    size_t plan_end = 0;                                                                // copied plan
    size_t flags = 0, lse2 = 0, drow = 0, sinkrow = 0, dqacc = 0, keep_bits = 0, total = 0;
};

// Offsets of the copied plan (status words first); the rest of the layout
// follows plan_end.
void plan_offsets(const Plan &pl, Layout &L, size_t &off)
{
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = round_up(off + bytes, 256);
        return o;
    };
    L.seqs = take(pl.seqs.size() * sizeof(SeqDesc));
    L.q_items = take(pl.q_items.size() * sizeof(int2));
    L.kv_items = take(pl.kv_items.size() * sizeof(int2));
    L.units = take(pl.units.size() * sizeof(GradUnit));
    L.qblk = take(pl.qblk.size() * sizeof(QBlockInfo));
    L.qblk_rows = take(pl.qblk_rows.size() * sizeof(int2));
    L.fwd_units = take(pl.fwd_units.size() * sizeof(int2));
    L.plan_end = off;
}

Layout layout_for(const Problem &p, const Plan &pl, bool grad, bool tc)
{
    Layout L;
    size_t off = kStatusBytes;
    plan_offsets(pl, L, off);
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = round_up(off + bytes, 256);
        return o;
    };
    if (grad) {
        const size_t vec = pl.qblk_rows.size() * (size_t)p.nq * kQBlock;  // blocked per-row vectors
        L.flags = take(tc ? pl.qblk.size() * (size_t)p.nq * sizeof(int32_t) : 0);
        L.lse2 = take(vec * sizeof(float));
        L.drow = take(vec * sizeof(float));
        L.sinkrow = take(p.has_sink ? vec * sizeof(float) : 0);
        L.dqacc = take(tc ? (size_t)p.tq * (size_t)p.nq * (size_t)p.d * sizeof(float) : 0);
    }
    // packed attention-mask matrix for the tensor-core kernels (forward:
    // rows of q, gradient: rows of kv)
    if (tc && p.has_amask)
        L.keep_bits = take(grad ? (size_t)p.s2max * words_kv_of(p) * sizeof(uint64_t)
                                : (size_t)p.s1max * words_q_of(p) * sizeof(uint64_t));
    L.total = off;
    return L;
}

// Host image of the workspace's first plan_end bytes: zeroed status words,
// then the plan arrays at their offsets.
void build_image(Plan &pl)
{
    Layout L;
    size_t off = kStatusBytes;
    plan_offsets(pl, L, off);
    pl.image.assign(L.plan_end, 0);
    auto put = [&](size_t o, const void *src, size_t bytes) {
        if (bytes) std::memcpy(pl.image.data() + o, src, bytes);
    };
    put(L.seqs, pl.seqs.data(), pl.seqs.size() * sizeof(SeqDesc));
    put(L.q_items, pl.q_items.data(), pl.q_items.size() * sizeof(int2));
    put(L.kv_items, pl.kv_items.data(), pl.kv_items.size() * sizeof(int2));
    put(L.units, pl.units.data(), pl.units.size() * sizeof(GradUnit));
    put(L.qblk, pl.qblk.data(), pl.qblk.size() * sizeof(QBlockInfo));
    put(L.qblk_rows, pl.qblk_rows.data(), pl.qblk_rows.size() * sizeof(int2));
    put(L.fwd_units, pl.fwd_units.data(), pl.fwd_units.size() * sizeof(int2));
}

// Plans depend only on the sequence table, head counts and the mask; calls
// that repeat a problem (every training step of a fixed batch) reuse the
// plan instead of rebuilding it.  Small LRU, shared by all threads.
struct PlanKey {
    int64_t batch, nq, nkv, d, mode, pre, next;
    bool with_units, has_amask;
    std::vector<int64_t> cuq, cukv, prefix;
    bool operator==(const PlanKey &o) const
    {
        return batch == o.batch && nq == o.nq && nkv == o.nkv && d == o.d && mode == o.mode && pre == o.pre &&
               next == o.next &&
               with_units == o.with_units && has_amask == o.has_amask && cuq == o.cuq && cukv == o.cukv &&
               prefix == o.prefix;
    }
};
constexpr size_t kPlanCacheSize = 8;
std::vector<std::pair<PlanKey, std::shared_ptr<const Plan>>> g_plan_cache;  // most recent last
std::mutex g_plan_mu;

std::shared_ptr<const Plan> get_plan(const Problem &p, bool with_units)
{
    PlanKey key{p.batch, p.nq, p.nkv, p.d, p.mode, p.pre, p.next, with_units, p.has_amask,
                std::vector<int64_t>(p.cuq, p.cuq + p.batch + 1), std::vector<int64_t>(p.cukv, p.cukv + p.batch + 1),
                p.prefix ? std::vector<int64_t>(p.prefix, p.prefix + p.batch) : std::vector<int64_t>()};
    {
        std::lock_guard<std::mutex> lk(g_plan_mu);
        for (size_t i = g_plan_cache.size(); i-- > 0;) {
            if (g_plan_cache[i].first == key) {
                auto hit = g_plan_cache[i];
                g_plan_cache.erase(g_plan_cache.begin() + (long)i);
                g_plan_cache.push_back(hit);
                return hit.second;
            }
        }
    }
    auto pl = std::make_shared<Plan>();
    build_plan(p, with_units, *pl);
    build_image(*pl);
    std::lock_guard<std::mutex> lk(g_plan_mu);
    if (g_plan_cache.size() >= kPlanCacheSize) g_plan_cache.erase(g_plan_cache.begin());
    g_plan_cache.emplace_back(std::move(key), pl);
    return pl;
}

// Clock rate and SM count of the current device, queried once per device
// (the clock-rate query costs hundreds of microseconds on some drivers).
struct DeviceInfo {
    int clock_khz = 0, num_sms = 0;
};
DeviceInfo device_info()
{
    constexpr int kMaxDev = 64;
    static DeviceInfo cache[kMaxDev];
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) dev = -1;
    if (dev >= 0) {
        std::lock_guard<std::mutex> lk(mu);
        if (cache[dev].num_sms > 0) return cache[dev];
    }
    DeviceInfo di;
    if (dev >= 0) {
        cudaDeviceGetAttribute(&di.clock_khz, cudaDevAttrClockRate, dev);
        cudaDeviceGetAttribute(&di.num_sms, cudaDevAttrMultiProcessorCount, dev);
    }
    if (di.clock_khz <= 0) di.clock_khz = 2000000;
    if (di.num_sms <= 0) di.num_sms = 148;
    if (dev >= 0) {
        std::lock_guard<std::mutex> lk(mu);
        cache[dev] = di;
    }
    return di;
}

// The tensor-core kernels take equal head dims only.
bool tc_grad_layout(const Problem &p) { return grad_tc_supported(p.dtype, (int)p.d) && p.dv == p.d; }
bool tc_fwd_layout(const Problem &p) { return fwd_tc_supported(p.dtype, (int)p.d) && p.dv == p.d; }
bool use_tc(const Problem &p) { return g_opt.grad_path == 0 && tc_grad_layout(p); }
bool use_fwd_tc(const Problem &p) { return g_opt.grad_path == 0 && tc_fwd_layout(p); }

// Pinned host staging of plan uploads.  A copy from pageable host memory may
// make the runtime wait for the stream before it starts, so a run call would
// block its caller until earlier work on the stream has drained.  Each device
// gets a ring of pinned slots; a slot is refilled only once the event recorded
// after its previous copy has completed, which with kStageSlots slots is
// normally long past.  Slots grow (rarely) by reallocation.
constexpr int kStageSlots = 8;
constexpr int kStageDevices = 64;
struct StageSlot {
    void *host = nullptr;
    size_t cap = 0;
    cudaEvent_t done = nullptr;
};
struct StageRing {
    std::mutex mu;
    StageSlot slot[kStageSlots];
    unsigned next = 0;
};
StageRing g_stage[kStageDevices];

// Enqueues a copy of `bytes` host bytes to device address `dst` on stream s
// without waiting for the stream.  Falls back to a plain copy when pinned
// memory cannot be had.
cudaError_t staged_copy(void *dst, const void *src, size_t bytes, cudaStream_t s)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kStageDevices)
        return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, s);
    StageRing &r = g_stage[dev];
    std::lock_guard<std::mutex> lk(r.mu);
    StageSlot &sl = r.slot[r.next++ % kStageSlots];
    if (!sl.done && cudaEventCreateWithFlags(&sl.done, cudaEventDisableTiming) != cudaSuccess) {
        sl.done = nullptr;
        return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, s);
    }
    if (cudaEventSynchronize(sl.done) != cudaSuccess) return cudaErrorUnknown;
    if (sl.cap < bytes) {
        if (sl.host) cudaFreeHost(sl.host);
        sl.host = nullptr;
        sl.cap = 0;
        size_t cap = 64 << 10;
        while (cap < bytes) cap *= 2;
        if (cudaHostAlloc(&sl.host, cap, cudaHostAllocPortable) != cudaSuccess) {
            sl.host = nullptr;
            cudaGetLastError();
            return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, s);
        }
        sl.cap = cap;
    }
    std::memcpy(sl.host, src, bytes);
    cudaError_t e = cudaMemcpyAsync(dst, sl.host, bytes, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return e;
    return cudaEventRecord(sl.done, s);
}

// Copies the plan image (zeroed status words, then the plan arrays) into the
// workspace.  `pinned` selects the staged copy; without it the copy reads the
// plan's own (pageable) image and nothing is allocated.  The dQ chain
// counters are zeroed by the prepass kernel.
tnd_status upload_plan(const Plan &pl, void *ws, cudaStream_t s, bool pinned = true)
{
    const cudaError_t ce = pinned ? staged_copy(ws, pl.image.data(), pl.image.size(), s)
                                  : cudaMemcpyAsync(ws, pl.image.data(), pl.image.size(), cudaMemcpyHostToDevice, s);
    return ce == cudaSuccess ? TND_OK : TND_ERR_CUDA;
}

template <typename A>
void fill_common(A &a, const Problem &p, const Plan &pl, const Layout &L, void *ws)
{
    char *w = (char *)ws;
    a.dtype = p.dtype;
    a.batch = (int32_t)p.batch;
    a.nq = (int32_t)p.nq;
    a.nkv = (int32_t)p.nkv;
    a.d = (int32_t)p.d;
    a.vd = (int32_t)p.dv;
    a.group = (int32_t)(p.nq / p.nkv);
    a.tq = p.tq;
    a.tkv = p.tkv;
    a.scale = (float)p.scale;
    a.keep_prob = (float)p.keep;
    a.inv_keep = (float)(1.0 / p.keep);
    a.mask = mask_of(p);
    a.has_drop = p.has_drop;
    a.has_sink = p.has_sink;
    a.status = (uint32_t *)w;
    a.seqs = (const SeqDesc *)(w + L.seqs);
    a.q_items = (const int2 *)(w + L.q_items);
    a.n_q_items = (int32_t)pl.q_items.size();
}

#ifdef TND_HOST_STATS
// Diagnostic build only: host microseconds per phase of tnd_attn_grad.
double g_host_us[8];
struct HostClock {
    std::chrono::steady_clock::time_point t = std::chrono::steady_clock::now();
    void lap(int i)
    {
        const auto n = std::chrono::steady_clock::now();
        g_host_us[i] += std::chrono::duration<double, std::micro>(n - t).count();
        t = n;
    }
};
#define HOST_LAP(i) hc.lap(i)
#else
struct HostClock {};
#define HOST_LAP(i) ((void)0)
#endif

}  // namespace
}  // namespace tnd

using namespace tnd;

#ifdef TND_HOST_STATS
extern "C" void tnd_debug_host_stats(double *out, int reset)
{
    for (int i = 0; i < 8; ++i) {
        out[i] = g_host_us[i];
        if (reset) g_host_us[i] = 0.0;
    }
}
#endif

extern "C" {

const char *tnd_status_string(tnd_status s)
{
    switch (s) {
    case TND_OK: return "ok";
    case TND_ERR_NULLPTR: return "a required pointer argument is NULL";
    case TND_ERR_INVALID: return "an argument is outside the supported dtype, shape, scalar or alignment limits";
    case TND_ERR_UNSUPPORTED: return "the argument combination is valid but not implemented by this library";
    case TND_ERR_WORKSPACE: return "the workspace is NULL, misaligned or smaller than required";
    case TND_ERR_CUDA: return "a CUDA runtime call failed";
    case TND_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait expired; outputs of that call are invalid";
    case TND_ERR_DEVICE_CHECK: return "a device-side consistency check failed";
    }
    return "unknown status";
}

tnd_status tnd_attn_set_option(tnd_option option, int64_t value)
{
    std::lock_guard<std::mutex> lk(g_mu);
    switch (option) {
    case TND_OPT_GRAD_PATH:
        if (value != 0 && value != 1) return TND_ERR_INVALID;
        g_opt.grad_path = (int)value;
        return TND_OK;
    case TND_OPT_WAIT_LIMIT_MS:
        if (value < 1 || value > 600000) return TND_ERR_INVALID;
        g_opt.wait_limit_ms = value;
        return TND_OK;
    case TND_OPT_PROFILE:
        if (value != 0 && value != 1) return TND_ERR_INVALID;
        g_opt.profile = (int)value;
        return TND_OK;
    case TND_OPT_TEST_SKIP_LOAD:
        if (value != 0 && value != 1) return TND_ERR_INVALID;
        g_opt.test_skip_load = (int)value;
        return TND_OK;
    case TND_OPT_DETERMINISTIC:
        if (value != 0 && value != 1) return TND_ERR_INVALID;
        g_opt.deterministic = (int)value;
        return TND_OK;
    }
    return TND_ERR_INVALID;
}

tnd_status tnd_attn_profile_read(const char **names, double *total_ms, int64_t *launches, int capacity,
                                 int *count, int reset)
{
    if (!count) return TND_ERR_NULLPTR;
    std::lock_guard<std::mutex> lk(g_mu);
    double ms[kNumKinds] = {0};
    int64_t n[kNumKinds] = {0};
    for (const ProfEntry &e : g_prof) {
        if (cudaEventSynchronize(e.stop) != cudaSuccess) return TND_ERR_CUDA;
        float t = 0.0f;
        if (cudaEventElapsedTime(&t, e.start, e.stop) != cudaSuccess) return TND_ERR_CUDA;
        ms[e.kind] += t;
        n[e.kind] += 1;
    }
    for (int k = 0; k < kNumKinds && k < capacity; ++k) {
        if (names) names[k] = kKindNames[k];
        if (total_ms) total_ms[k] = ms[k];
        if (launches) launches[k] = n[k];
    }
    *count = kNumKinds;
    if (reset) {
        for (const ProfEntry &e : g_prof) {
            g_event_pool.push_back(e.start);
            g_event_pool.push_back(e.stop);
        }
        g_prof.clear();
    }
    return TND_OK;
}

tnd_status tnd_attn_fwd_workspace_size(tnd_dtype dtype, int64_t batch, const int64_t *cuq, const int64_t *cukv,
                                       const int64_t *prefix, int64_t nq, int64_t nkv, int64_t d, int64_t vd,
                                       double scale, double keep, int64_t pre, int64_t next, int64_t mode,
                                       int has_drop, int has_amask, int has_sink, uint64_t *ws_size)
{
    if (!ws_size) return TND_ERR_NULLPTR;
    Problem p;
    tnd_status st = validate(dtype, batch, cuq, cukv, prefix, nq, nkv, d, vd, scale, keep, pre, next, mode,
                             has_drop != 0, has_amask != 0, has_sink != 0, p);
    if (st != TND_OK) return st;
    const bool tc_layout = tc_fwd_layout(p);
    auto plp = get_plan(p, tc_layout);
    *ws_size = layout_for(p, *plp, false, tc_layout).total;
    return TND_OK;
}

tnd_status tnd_attn_fwd(const void *q, const void *k, const void *v, const void *pse, int64_t pse_batch,
                        int64_t pse_type, const uint8_t *drop_mask, const uint8_t *atten_mask, const float *sink,
                        tnd_dtype dtype, int64_t batch, const int64_t *cuq, const int64_t *cukv,
                        const int64_t *prefix, int64_t nq, int64_t nkv, int64_t d, int64_t vd, double scale,
                        double keep, int64_t pre, int64_t next, int64_t mode, void *out, float *smax, float *ssum,
                        void *ws, uint64_t ws_size, void *stream)
{
    if (!q || !k || !v || !out || !smax || !ssum) return TND_ERR_NULLPTR;
    Problem p;
    tnd_status st = validate(dtype, batch, cuq, cukv, prefix, nq, nkv, d, vd, scale, keep, pre, next, mode,
                             drop_mask != nullptr, atten_mask != nullptr, sink != nullptr, p);
    if (st != TND_OK) return st;
    st = check_pse(p, pse, pse_batch, pse_type);
    if (st != TND_OK) return st;
    for (const void *ptr : {q, k, v, (const void *)out, (const void *)smax, (const void *)ssum})
        if (!aligned16(ptr)) return TND_ERR_INVALID;
    const bool tc_layout = tc_fwd_layout(p);
    auto plp = get_plan(p, tc_layout);
    const Plan &pl = *plp;
    const Layout L = layout_for(p, pl, false, tc_layout);
    if (!ws || ws_size < L.total || (reinterpret_cast<uintptr_t>(ws) & 255u)) return TND_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    st = upload_plan(pl, ws, s);
    if (st != TND_OK) return st;
    FwdArgs a{};
    fill_common(a, p, pl, L, ws);
    char *w = (char *)ws;
    a.q = q;
    a.k = k;
    a.v = v;
    a.drop_mask = p.has_drop ? drop_mask : nullptr;
    a.sink = sink;
    a.o = out;
    a.smax = smax;
    a.ssum = ssum;
    a.mask_bytes = (mask_bits_total(p) + 7) / 8;
    a.pse = pse_of(p, pse, pse_batch, pse_type);
    a.qblk = (const QBlockInfo *)(w + L.qblk);
    a.qblk_rows = (const int2 *)(w + L.qblk_rows);
    a.fwd_units = (const int2 *)(w + L.fwd_units);
    a.n_fwd_units = (int32_t)pl.fwd_units.size();
    {
        const DeviceInfo di = device_info();
        a.wait_limit_cycles = g_opt.wait_limit_ms * (int64_t)di.clock_khz;
        a.num_sms = di.num_sms;
    }
    const bool tc = tc_layout && use_fwd_tc(p);
    if (p.has_amask) {
        a.mask.amask = atten_mask;
        a.mask.amask_cols = p.s2max;
        if (tc) {
            a.mask.keep_q = (const uint64_t *)(w + L.keep_bits);
            a.mask.words_q = words_q_of(p);
            if (timed(K_PACK, s, [&] {
                    return launch_amask_pack(atten_mask, p.s1max, p.s2max, (uint64_t *)(w + L.keep_bits),
                                             a.mask.words_q, nullptr, 0, s);
                }) != cudaSuccess)
                return TND_ERR_CUDA;
        }
    }
    if (tc) {
        if (timed(K_FWD_TC, s, [&] { return launch_fwd_tc(a, s); }) != cudaSuccess) return TND_ERR_CUDA;
    } else {
        if (timed(K_FWD, s, [&] { return launch_fwd_simt(a, s); }) != cudaSuccess) return TND_ERR_CUDA;
    }
    return TND_OK;
}

tnd_status tnd_attn_grad_workspace_size(tnd_dtype dtype, int64_t batch, const int64_t *cuq, const int64_t *cukv,
                                        const int64_t *prefix, int64_t nq, int64_t nkv, int64_t d, int64_t vd,
                                        double scale, double keep, int64_t pre, int64_t next, int64_t mode,
                                        int has_drop, int has_amask, int has_sink, uint64_t *ws_size)
{
    if (!ws_size) return TND_ERR_NULLPTR;
    Problem p;
    tnd_status st = validate(dtype, batch, cuq, cukv, prefix, nq, nkv, d, vd, scale, keep, pre, next, mode,
                             has_drop != 0, has_amask != 0, has_sink != 0, p);
    if (st != TND_OK) return st;
    const bool tc = tc_grad_layout(p);
    auto plp = get_plan(p, tc);
    *ws_size = layout_for(p, *plp, true, tc).total;
    return TND_OK;
}

}  // extern "C"

namespace tnd {

tnd_status grad_run(const void *q, const void *k, const void *v, const void *dy, const void *pse, int64_t pse_batch,
                    int64_t pse_type, const uint8_t *drop_mask, const uint8_t *atten_mask, const float *smax,
                    const float *ssum, const void *o, const float *sink, tnd_dtype dtype, int64_t batch,
                    const int64_t *cuq, const int64_t *cukv, const int64_t *prefix, int64_t nq, int64_t nkv,
                    int64_t d, int64_t vd, double scale, double keep, int64_t pre, int64_t next, int64_t mode,
                    void *dq, void *dk, void *dv, float *dsink, void *ws, uint64_t ws_size, void *stream,
                    bool pinned_upload)
{
    if (!q || !k || !v || !dy || !smax || !ssum || !o || !dq || !dk || !dv) return TND_ERR_NULLPTR;
    if (sink && !dsink) return TND_ERR_NULLPTR;
    HostClock hc;
    (void)hc;
    Problem p;
    tnd_status st = validate(dtype, batch, cuq, cukv, prefix, nq, nkv, d, vd, scale, keep, pre, next, mode,
                             drop_mask != nullptr, atten_mask != nullptr, sink != nullptr, p);
    if (st != TND_OK) return st;
    st = check_pse(p, pse, pse_batch, pse_type);
    if (st != TND_OK) return st;
    for (const void *ptr : {q, k, v, dy, (const void *)smax, (const void *)ssum, o, (const void *)dq,
                            (const void *)dk, (const void *)dv})
        if (!aligned16(ptr)) return TND_ERR_INVALID;
    HOST_LAP(0);
    const bool tc_layout = tc_grad_layout(p);
    const bool tc = use_tc(p);
    auto plp = get_plan(p, tc_layout);
    const Plan &pl = *plp;
    const Layout L = layout_for(p, pl, true, tc_layout);
    if (!ws || ws_size < L.total || (reinterpret_cast<uintptr_t>(ws) & 255u)) return TND_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    HOST_LAP(1);
    st = upload_plan(pl, ws, s, pinned_upload);
    if (st != TND_OK) return st;
    HOST_LAP(2);
    GradArgs a{};
    fill_common(a, p, pl, L, ws);
    char *w = (char *)ws;
    a.q = q;
    a.k = k;
    a.v = v;
    a.dy = dy;
    a.o = o;
    a.drop_mask = p.has_drop ? drop_mask : nullptr;
    a.smax = smax;
    a.ssum = ssum;
    a.sink = sink;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.dsink = dsink;
    a.kv_items = (const int2 *)(w + L.kv_items);
    a.n_kv_items = (int32_t)pl.kv_items.size();
    a.lse2 = (float *)(w + L.lse2);
    a.drow = (float *)(w + L.drow);
    a.sinkrow = p.has_sink ? (float *)(w + L.sinkrow) : nullptr;
    a.units = (const GradUnit *)(w + L.units);
    a.n_units = (int32_t)pl.units.size();
    a.qblk = (const QBlockInfo *)(w + L.qblk);
    a.qblk_rows = (const int2 *)(w + L.qblk_rows);
    a.n_qblk = (int32_t)pl.qblk_rows.size();
    a.flags = (int32_t *)(w + L.flags);
    a.dqacc = tc_layout ? (float *)(w + L.dqacc) : nullptr;
    a.mask_bytes = (mask_bits_total(p) + 7) / 8;
    a.pse = pse_of(p, pse, pse_batch, pse_type);
    {
        const DeviceInfo di = device_info();
        a.wait_limit_cycles = g_opt.wait_limit_ms * (int64_t)di.clock_khz;
        a.num_sms = di.num_sms;
        a.test_flags = g_opt.test_skip_load ? 1 : 0;
        a.deterministic = g_opt.deterministic;
    }
    if (p.has_amask) {
        a.mask.amask = atten_mask;
        a.mask.amask_cols = p.s2max;
        if (tc) {
            a.mask.keep_kv = (const uint64_t *)(w + L.keep_bits);
            a.mask.words_kv = words_kv_of(p);
            if (timed(K_PACK, s, [&] {
                    return launch_amask_pack(atten_mask, p.s1max, p.s2max, nullptr, 0, (uint64_t *)(w + L.keep_bits),
                                             a.mask.words_kv, s);
                }) != cudaSuccess)
                return TND_ERR_CUDA;
        }
    }
    HOST_LAP(3);
    if (timed(K_PREPASS, s, [&] { return launch_prepass(a, tc, s); }) != cudaSuccess) return TND_ERR_CUDA;
    HOST_LAP(4);
    if (tc) {
        if (timed(K_TC, s, [&] { return launch_grad_tc(a, s); }) != cudaSuccess) return TND_ERR_CUDA;
        HOST_LAP(5);
        if (timed(K_FIN, s, [&] { return launch_dq_finalize(a, s); }) != cudaSuccess) return TND_ERR_CUDA;
        HOST_LAP(6);
    } else {
        if (timed(K_DKDV, s, [&] { return launch_grad_dkdv_simt(a, s); }) != cudaSuccess) return TND_ERR_CUDA;
        if (timed(K_DQ, s, [&] { return launch_grad_dq_simt(a, s); }) != cudaSuccess) return TND_ERR_CUDA;
    }
    if (p.has_sink) {
        if (timed(K_SINK, s, [&] { return launch_sink_reduce(a, s); }) != cudaSuccess) return TND_ERR_CUDA;
    }
    return TND_OK;
}

}  // namespace tnd

extern "C" {

tnd_status tnd_attn_grad(const void *q, const void *k, const void *v, const void *dy, const void *pse,
                         int64_t pse_batch, int64_t pse_type, const uint8_t *drop_mask, const uint8_t *atten_mask,
                         const float *smax, const float *ssum, const void *o, const float *sink, tnd_dtype dtype,
                         int64_t batch, const int64_t *cuq, const int64_t *cukv, const int64_t *prefix, int64_t nq,
                         int64_t nkv, int64_t d, int64_t vd, double scale, double keep, int64_t pre, int64_t next,
                         int64_t mode, void *dq, void *dk, void *dv, float *dsink, void *ws, uint64_t ws_size,
                         void *stream)
{
    return grad_run(q, k, v, dy, pse, pse_batch, pse_type, drop_mask, atten_mask, smax, ssum, o, sink, dtype, batch,
                    cuq, cukv, prefix, nq, nkv, d, vd, scale, keep, pre, next, mode, dq, dk, dv, dsink, ws, ws_size,
                    stream, true);
}

tnd_status tnd_attn_device_status(const void *ws, uint64_t ws_size, void *stream)
{
    if (!ws) return TND_ERR_NULLPTR;
    if (ws_size < kStatusBytes) return TND_ERR_WORKSPACE;
    uint32_t words[4] = {0, 0, 0, 0};
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemcpyAsync(words, ws, sizeof(words), cudaMemcpyDeviceToHost, s) != cudaSuccess) return TND_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return TND_ERR_CUDA;
    if (words[kStatusWord] == 0) return TND_OK;
    if (words[kStatusWord] == (uint32_t)TND_ERR_DEVICE_TIMEOUT) return TND_ERR_DEVICE_TIMEOUT;
    return TND_ERR_DEVICE_CHECK;
}

tnd_status tnd_attn_grad_plan(int64_t batch, const int64_t *cuq, const int64_t *cukv, const int64_t *prefix,
                              int64_t nq, int64_t nkv, int64_t pre, int64_t next, int64_t mode, int has_amask,
                              int64_t *units, int64_t capacity, int64_t *n_units, int64_t *kept_pairs)
{
    if (!n_units || !kept_pairs) return TND_ERR_NULLPTR;
    Problem p;
    tnd_status st = validate(TND_BF16, batch, cuq, cukv, prefix, nq, nkv, 128, 128, 1.0, 1.0, pre, next, mode, false,
                             has_amask != 0, false, p);
    if (st != TND_OK) return st;
    Plan pl;
    build_plan(p, true, pl);
    *n_units = (int64_t)pl.units.size();
    *kept_pairs = pl.kept_pairs;
    if (units) {
        for (int64_t u = 0; u < (int64_t)pl.units.size() && u < capacity; ++u) {
            const GradUnit &g = pl.units[u];
            units[5 * u + 0] = g.b;
            units[5 * u + 1] = g.g;
            units[5 * u + 2] = g.j;
            units[5 * u + 3] = g.qb_lo;
            units[5 * u + 4] = g.qb_hi;
        }
    }
    return TND_OK;
}

}  // extern "C"
