// Tensor-core (tcgen05) forward for bf16 / fp16 at D = 64 or 128 on sm_103a.
//
// Computes, per sequence b, query head h and 128-row q block i
// ("aclnnFlashAttentionUnpaddingScoreGrad", function description: forward
// Y = Dropout(Softmax(Mask(scale Q K^T)), keep_prob) V; "...ScoreGradV5",
// function description: the sink enters the max and the denominator;
// "aclnnFlashAttentionScoreV2", parameters: attentionOut, softmaxMax,
// softmaxSum):
//     for every kv block j that some row of block i sees:
//         S   = Q_i K_j^T                    (UMMA, smem x smem -> TMEM)
//         P   = exp2(S * scale*log2e - m)    (online, m the running row max)
//         O  += (P o keep) V_j               (UMMA, A = P from TMEM)
//     O *= 1 / (l keepProb); softmaxMax = m (natural log units),
//     softmaxSum = l, 8 copies.
// The running max is updated lazily: a row's O and l are rescaled (in TMEM)
// only when its block max exceeds the max in use by more than 2^8, so P
// stays below 256; the emitted max and sum are those of the true row max.
//
// Warp roles (320 threads, one CTA per SM, persistent over (q block, head)
// units taken in plan order, longest kv range first):
//   warp 0      TMA producer: Q per unit (two stages, so the next unit's Q
//               loads while one runs); K, V per kv block (two stages)
//   warp 1      TMEM allocator and single-thread UMMA issuer
//   warps 2-9   softmax warps: thread = TMEM lane = q row, two warps per lane
//               quarter, each on 64 of a block's 128 kv columns (they trade
//               block maxima and, at a unit's end, sums); O out at unit end,
//               half of its columns each
// TMEM: O (HD columns), two S buffers of 128 columns (S(j) in buffer j % 2,
// then P packed in place, each 32-column chunk in its own first 16 columns,
// until O += P V has read it).
// Every wait is bounded; on expiry the kernel records TND_ERR_DEVICE_TIMEOUT
// in the workspace status word and winds down instead of hanging.
#include "ptx_sm103.cuh"
#include "tnd_device.cuh"

#include <cudaTypedefs.h>

namespace tnd {
namespace {

using namespace ptx;

constexpr int BN = kKvBlock;             // 128 kv rows (UMMA N of S, K of O += P V)
constexpr int kThreads = 320;
constexpr int NS = 2;                    // K / V stages
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TM_O = 0, TM_S = 256; // S buffers at 256 and 384
constexpr uint32_t kColBlk = 128 * 128;  // one 64-element column block of 128 rows (16 KB)
constexpr float kRescaleLog2 = 8.0f;     // lazy rescale threshold (log2 units)

template <int HD>
struct FGeo {
    static constexpr uint32_t NCB = HD / 64;
    static constexpr uint32_t kTile = 128 * HD * 2;       // Q, K or V tile
    static constexpr uint32_t OFF_Q = 0;                   // 2 stages (a unit's Q in stage ku % 2)
    static constexpr uint32_t OFF_K = OFF_Q + 2 * kTile;   // NS stages
    static constexpr uint32_t OFF_V = OFF_K + NS * kTile;  // NS stages
    static constexpr uint32_t OFF_BAR = OFF_V + NS * kTile;
    static constexpr uint32_t kNumBars = 32;   // >= F_NUM_BARS
    static constexpr uint32_t OFF_MISC = OFF_BAR + kNumBars * 8;
    static constexpr uint32_t OFF_XCH = OFF_MISC + 64;     // softmax halves' exchange, 2 x [2][128] fp32
    static constexpr uint32_t kSmemBytes = OFF_XCH + 2 * 2 * 128 * 4;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
};

enum : int {
    F_Q_FULL = 0,               // [2]  count 1 + tx (stage ku % 2)
    F_Q_EMPTY = 2,              // [2]  count 1 (commit after the unit's last UMMA)
    F_K_FULL = 4,               // [NS] count 1 + tx
    F_K_EMPTY = F_K_FULL + NS,  // [NS] count 1 (commit after S)
    F_V_FULL = F_K_EMPTY + NS,  // [NS] count 1 + tx
    F_V_EMPTY = F_V_FULL + NS,  // [NS] count 1 (commit after O += P V)
    F_S_FULL = F_V_EMPTY + NS,  // [2]  count 1 (commit)
    F_P_READY = F_S_FULL + 2,   // [2]  count 256
    F_PV_DONE = F_P_READY + 2,  // [2]  count 1 (commit after O += P V: P read, O current)
    F_O_FULL = F_PV_DONE + 2,   //      count 1 (commit after the unit's last O += P V)
    F_O_FREE = F_O_FULL + 1,    //      count 256 (O read out)
    F_UNIT_FULL = F_O_FREE + 1, // [2]  count 1
    F_UNIT_EMPTY = F_UNIT_FULL + 2,  // [2] count 9 (MMA + 8 softmax warps)
    F_DRAIN = F_UNIT_EMPTY + 2,      //     count 1
    F_XCH = F_DRAIN + 1,             // [4] count 64 (the two softmax warps of a lane quarter)
    F_NUM_BARS = F_XCH + 4
};
static_assert(F_NUM_BARS <= 32, "barrier slots");
constexpr uint32_t MISC_TMEM = 0, MISC_RING = 1, MISC_ABORT = 3;

struct FSmem {
    uint8_t *base;
    uint32_t off_bar, off_misc;
    __device__ uint64_t *bar(int i) const { return reinterpret_cast<uint64_t *>(base + off_bar) + i; }
    __device__ uint32_t *misc() const { return reinterpret_cast<uint32_t *>(base + off_misc); }
    __device__ volatile int *abort_flag() const { return reinterpret_cast<volatile int *>(misc() + MISC_ABORT); }
};

__device__ __forceinline__ bool fwait(const FSmem &sm, int bar, uint32_t k, const FwdArgs &a)
{
    const long long t0 = clock64();
    while (!mbar_try_wait(sm.bar(bar), k & 1u)) {
        if (*sm.abort_flag()) return false;
        if (clock64() - t0 > a.wait_limit_cycles) {
            set_status(a.status, TND_ERR_DEVICE_TIMEOUT, (k << 12) | ((threadIdx.x >> 5) << 6) | (uint32_t)bar);
            *sm.abort_flag() = 1;
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ bool fwait_warp(const FSmem &sm, int bar, uint32_t k, const FwdArgs &a)
{
    const bool ok = fwait(sm, bar, k, a);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void fdrain(const FSmem &sm, int bar, uint32_t k, const FwdArgs &a)
{
    const long long t0 = clock64();
    while (!mbar_try_wait(sm.bar(bar), k & 1u) && clock64() - t0 < a.wait_limit_cycles) {
    }
}

__device__ __forceinline__ uint64_t fdesc_at(uint64_t d, uint32_t off) { return d + (uint64_t)(off >> 4); }

template <bool BF16>
__device__ __forceinline__ uint32_t fpack2(float lo, float hi)
{
    return BF16 ? pack_bf16(lo, hi) : pack_f16(lo, hi);
}

struct FUnit {
    int qg, h, jlo, n;   // global q block, head, first kv block, kv blocks (0: no key)
    int b;               // sequence
    SeqDesc sd;
    int64_t q0;          // first q row of the block within its sequence
};

__device__ __forceinline__ FUnit funit(const FwdArgs &a, int u)
{
    const int2 fu = a.fwd_units[u];
    FUnit U;
    U.qg = fu.x;
    U.h = fu.y;
    const QBlockInfo qi = a.qblk[fu.x];
    const int2 qr = a.qblk_rows[fu.x];
    U.sd = a.seqs[qr.x];
    U.b = qr.x;
    U.q0 = qr.y;
    U.jlo = qi.jlo;
    U.n = qi.jlo < 0 ? 0 : qi.jhi - qi.jlo + 1;
    return U;
}

// Keep-bits of row i over kv columns j0 .. j0 + 127 (128 consecutive bits of
// the packed mask), as four 32-bit words.
__device__ __forceinline__ void fetch_keep128(const FwdArgs &a, const SeqDesc &sd, int h, int64_t i, int64_t j0,
                                              uint32_t (&w)[5], uint32_t &sh)
{
#pragma unroll
    for (int e = 0; e < 5; ++e) w[e] = 0u;
    sh = 0u;
    if (i >= sd.sq) return;
    const int64_t p = sd.mask_base + ((int64_t)h * sd.sq + i) * sd.skv + j0;
    if ((reinterpret_cast<uintptr_t>(a.drop_mask) & 3) == 0) {
        const uint32_t *m32 = reinterpret_cast<const uint32_t *>(a.drop_mask);
        const int64_t wi = p >> 5;
        sh = (uint32_t)(p & 31);
#pragma unroll
        for (int e = 0; e < 5; ++e) {
            if ((wi + e + 1) * 4 <= a.mask_bytes) {
                w[e] = __ldg(m32 + wi + e);
            } else {
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const int64_t bi = (wi + e) * 4 + b;
                    w[e] |= (uint32_t)((bi < a.mask_bytes) ? a.drop_mask[bi] : 0) << (8 * b);
                }
            }
        }
    } else {
        // unaligned mask: bytes
        const int64_t b0 = p >> 3;
        sh = (uint32_t)(p & 7);
#pragma unroll
        for (int e = 0; e < 17; ++e) {
            const int64_t bi = b0 + e;
            const uint32_t byte = (bi < a.mask_bytes) ? a.drop_mask[bi] : 0u;
            if (e < 16) w[e >> 2] |= byte << (8 * (e & 3));
            else w[4] = byte;
        }
    }
}

// TMEM column of the packed P for kv columns 16 kk .. 16 kk + 15 within an S
// buffer: each 32-column chunk of S holds its own 32 P values, packed two per
// column, in its first 16 columns
__device__ __forceinline__ uint32_t fpk_col(int kk) { return (uint32_t)((kk >> 1) * 32 + (kk & 1) * 8); }

// pse terms (log2 units of C * S) of row i over kv columns jc .. jc + 31, 0
// outside the sequence (those columns are masked anyway)
template <bool BF16>
__device__ __forceinline__ void fpse_chunk(const FwdArgs &a, const FUnit &U, int64_t i, bool row_ok, int64_t jc,
                                           float C, float (&t)[32])
{
    using Elt = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
    if (pse_generated(a.pse)) {
        const float slope = pse_slope(a.pse, a.nq, U.b, U.h);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
            const int64_t j = jc + c;
            t[c] = (row_ok && j < U.sd.skv) ? pse_alibi(a.pse.type, slope, i, j) * kLog2e : 0.0f;
        }
        return;
    }
    const Elt *pp = reinterpret_cast<const Elt *>(a.pse.ptr);
    const float mul = a.pse.type == 1 ? C : kLog2e;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
        const int64_t j = jc + c;
        float x = 0.0f;
        if (row_ok && j < U.sd.skv) {
            const Elt e = pp[pse_index(a.pse, a.nq, U.b, U.h, U.sd.sq, i, j)];
            if constexpr (BF16) x = __bfloat162float(e);
            else x = __half2float(e);
        }
        t[c] = x * mul;
    }
}

// PSE = true adds pseShiftOptional to the scores: pass 1 writes C S + pse term
// back into the S buffer, which pass 2 then reads as is.
template <bool BF16, int HD, bool PSE>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ FwdArgs a, const __grid_constant__ CUtensorMap tmQ,
                  const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV)
{
    using G_ = FGeo<HD>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0) set_status(a.status, TND_ERR_DEVICE_CHECK, 0x401u);
        return;
    }
    FSmem sm;
    sm.base = smem_raw;
    sm.off_bar = G_::OFF_BAR;
    sm.off_misc = G_::OFF_MISC;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    using Out = typename std::conditional<BF16, __nv_bfloat16, __half>::type;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(sm.bar(F_Q_FULL + i), 1);
            mbar_init(sm.bar(F_Q_EMPTY + i), 1);
        }
        for (int i = 0; i < NS; ++i) {
            mbar_init(sm.bar(F_K_FULL + i), 1);
            mbar_init(sm.bar(F_K_EMPTY + i), 1);
            mbar_init(sm.bar(F_V_FULL + i), 1);
            mbar_init(sm.bar(F_V_EMPTY + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(sm.bar(F_S_FULL + i), 1);
            mbar_init(sm.bar(F_P_READY + i), 256);
            mbar_init(sm.bar(F_PV_DONE + i), 1);
            mbar_init(sm.bar(F_UNIT_FULL + i), 1);
            mbar_init(sm.bar(F_UNIT_EMPTY + i), 9);
        }
        mbar_init(sm.bar(F_O_FULL), 1);
        mbar_init(sm.bar(F_O_FREE), 256);
        mbar_init(sm.bar(F_DRAIN), 1);
        for (int q = 0; q < 4; ++q) mbar_init(sm.bar(F_XCH + q), 64);
        *sm.abort_flag() = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(sm.misc() + MISC_TMEM, kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm.misc() + MISC_TMEM);
    uint32_t armed[2 + 2 * NS] = {};   // producer: phases armed per load barrier (Q; K stages; V stages)

    if (warp == 0) {
        // ================================================================ producer
        uint32_t ui = 0, ku = 0, kb = 0;
        int *counter = reinterpret_cast<int *>(a.status + kWorkCounter);
        bool ok = true;
        while (ok) {
            int u = 0;
            if (lane == 0) u = atomicAdd(counter, 1);
            u = __shfl_sync(0xffffffffu, u, 0);
            const uint32_t slot = ui & 1u;
            if (ui >= 2 && !fwait_warp(sm, F_UNIT_EMPTY + slot, (ui >> 1) - 1, a)) break;
            if (lane == 0) {
                *reinterpret_cast<volatile int *>(sm.misc() + MISC_RING + slot) = (u < a.n_fwd_units) ? u : -1;
                mbar_arrive(sm.bar(F_UNIT_FULL + slot));
            }
            ++ui;
            if (u >= a.n_fwd_units) break;
            const FUnit U = funit(a, u);
            if (U.n == 0) continue;
            // Q of this unit in stage ku % 2, free once unit ku - 2 is done: it
            // loads while the previous unit still runs
            const uint32_t qs = ku & 1u;
            if (ku >= 2 && !fwait_warp(sm, F_Q_EMPTY + qs, (ku >> 1) - 1, a)) break;
            if (lane == 0) {
                uint64_t *qb = sm.bar(F_Q_FULL + qs);
                mbar_arrive_expect_tx(qb, G_::kTile);
                const int z = (int)(U.sd.tq + U.q0);
                for (uint32_t cb = 0; cb < G_::NCB; ++cb)
                    tma_load_3d(sm.base + G_::OFF_Q + qs * G_::kTile + cb * kColBlk, &tmQ, qb, 64 * cb, U.h, z);
            }
            ++armed[qs];
            const int g = U.h / a.group;
            for (int t = 0; t < U.n; ++t, ++kb) {
                const uint32_t s = kb % NS, k = kb / NS;
                const int z = (int)(U.sd.tk + (int64_t)(U.jlo + t) * BN);
                if (k >= 1 && !fwait_warp(sm, F_K_EMPTY + s, k - 1, a)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    uint64_t *fb = sm.bar(F_K_FULL + s);
                    mbar_arrive_expect_tx(fb, G_::kTile);
                    for (uint32_t cb = 0; cb < G_::NCB; ++cb)
                        tma_load_3d(sm.base + G_::OFF_K + s * G_::kTile + cb * kColBlk, &tmK, fb, 64 * cb, g, z);
                }
                ++armed[2 + s];
                if (k >= 1 && !fwait_warp(sm, F_V_EMPTY + s, k - 1, a)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    uint64_t *fb = sm.bar(F_V_FULL + s);
                    mbar_arrive_expect_tx(fb, G_::kTile);
                    for (uint32_t cb = 0; cb < G_::NCB; ++cb)
                        tma_load_3d(sm.base + G_::OFF_V + s * G_::kTile + cb * kColBlk, &tmV, fb, 64 * cb, g, z);
                }
                ++armed[2 + NS + s];
            }
            ++ku;
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            const uint32_t idS = instr_desc_f16(BF16, 128, BN, false, false);   // S = Q K^T
            const uint32_t idO = instr_desc_f16(BF16, 128, HD, false, true);    // O += P V (A in TMEM)
            const uint32_t sbase = smem_u32(sm.base);
            const uint64_t dQ = smem_desc_sw128(sbase + G_::OFF_Q, 16, 1024);
            const uint64_t dK0 = smem_desc_sw128(sbase + G_::OFF_K, 16, 1024);
            const uint64_t dV0 = smem_desc_sw128(sbase + G_::OFF_V, kColBlk, 1024);
            constexpr int KS = HD / 16;
            uint32_t ui = 0, ku = 0, gb = 0;
            bool ok = true;
            // S(g) = Q K(g)^T into S buffer g % 2, once O += P V of block g - 2 has
            // read P out of it
            auto issue_s = [&](uint32_t g, bool first) -> bool {
                const uint32_t s = g % NS, b = g & 1u;
                if (first && !fwait(sm, F_Q_FULL + (ku & 1u), ku >> 1, a)) return false;
                if (g >= 2 && !fwait(sm, F_PV_DONE + b, (g >> 1) - 1, a)) return false;
                if (!fwait(sm, F_K_FULL + s, g / NS, a)) return false;
                tc_fence_after();
                const uint64_t dk = fdesc_at(dK0, s * G_::kTile);
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    const uint32_t off = (kk >> 2) * kColBlk + (kk & 3) * 32;
                    mma_ss(tmem + TM_S + 128 * b, fdesc_at(dQ, (ku & 1u) * G_::kTile + off), fdesc_at(dk, off), idS,
                           kk > 0);
                }
                mma_commit(sm.bar(F_S_FULL + b));
                mma_commit(sm.bar(F_K_EMPTY + s));
                return true;
            };
            while (ok) {
                const uint32_t slot = ui & 1u;
                if (!fwait(sm, F_UNIT_FULL + slot, ui >> 1, a)) break;
                const int u = *reinterpret_cast<volatile int *>(sm.misc() + MISC_RING + slot);
                mbar_arrive(sm.bar(F_UNIT_EMPTY + slot));
                ++ui;
                if (u < 0) break;
                const FUnit U = funit(a, u);
                if (U.n == 0) continue;
                const uint32_t g0 = gb, g_end = gb + (uint32_t)U.n;
                if (!issue_s(g0, true) || (g0 + 1 < g_end && !issue_s(g0 + 1, false))) break;
                for (uint32_t g = g0; g < g_end; ++g) {
                    const uint32_t s = g % NS, b = g & 1u;
                    if (g == g0 && ku >= 1 && !fwait(sm, F_O_FREE, ku - 1, a)) {
                        ok = false;
                        break;
                    }
                    if (!fwait(sm, F_P_READY + b, g >> 1, a) || !fwait(sm, F_V_FULL + s, g / NS, a)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // O += P V: A = P (TMEM, packed: K slice kk at column 8 kk), B = V MN-major
                    const uint64_t dv = fdesc_at(dV0, s * G_::kTile);
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        mma_ts(tmem + TM_O, tmem + TM_S + 128 * b + fpk_col(kk), fdesc_at(dv, kk * 2048), idO,
                               (g > g0 || kk > 0));
                    mma_commit(sm.bar(F_PV_DONE + b));
                    mma_commit(sm.bar(F_V_EMPTY + s));
                    if (g + 2 < g_end && !issue_s(g + 2, false)) {
                        ok = false;
                        break;
                    }
                }
                if (!ok) break;
                mma_commit(sm.bar(F_O_FULL));
                mma_commit(sm.bar(F_Q_EMPTY + (ku & 1u)));
                gb = g_end;
                ++ku;
            }
            mma_commit(sm.bar(F_DRAIN));
            const long long t0 = clock64();
            while (!mbar_try_wait(sm.bar(F_DRAIN), 0) && clock64() - t0 < a.wait_limit_cycles) {
            }
        }
        __syncwarp();
    } else {
        // ================================================================ softmax warps
        // Two warps per TMEM lane quarter: warps 2-5 take kv columns 0-63 of
        // a block, warps 6-9 columns 64-127 (thread = q row).  The two halves
        // of a row trade their block maxima (and, at a unit's end, their sums)
        // through shared memory under a 64-thread named barrier per quarter.
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const int row = quarter * 32 + lane;                 // q row within the block = TMEM lane
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const float C = a.scale * kLog2e;
        // exchange k of a quarter goes through slot k % 2 ([2 halves][128 rows])
        // and completion k of the quarter's barrier (64 arrivals); exchange
        // k + 2 rewrites the slot only after both halves have passed k + 1,
        // so after both have read k
        float *xch = reinterpret_cast<float *>(sm.base + G_::OFF_XCH);
        uint32_t xk = 0;
        auto trade = [&](float mine, float &other) -> bool {
            float *slot = xch + (xk & 1u) * 256;
            slot[half * 128 + row] = mine;
            mbar_arrive(sm.bar(F_XCH + quarter));
            const bool okw = fwait_warp(sm, F_XCH + quarter, xk, a);
            other = slot[(half ^ 1) * 128 + row];
            ++xk;
            return okw;
        };
        Out *O = reinterpret_cast<Out *>(a.o);
        uint32_t ui = 0, ku = 0, gb = 0;
        bool ok = true;
        while (ok) {
            const uint32_t slot = ui & 1u;
            if (!fwait_warp(sm, F_UNIT_FULL + slot, ui >> 1, a)) break;
            const int u = *reinterpret_cast<volatile int *>(sm.misc() + MISC_RING + slot);
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.bar(F_UNIT_EMPTY + slot));
            ++ui;
            if (u < 0) break;
            const FUnit U = funit(a, u);
            const int64_t i = U.q0 + row;                     // q row in the sequence
            const bool row_ok = i < U.sd.sq;
            int64_t lo = 1, hi = 0;                           // kept key range of the row
            if (row_ok) key_range(a.mask, U.sd.sq, U.sd.skv, U.sd.prefix, i, lo, hi);
            // running state (log2 units): m_use = max in use, m_true = row max;
            // l is this half's share of the row sum (the sink counts in half 0)
            float m_use = -INFINITY, m_true = -INFINITY, l = 0.0f;
            if (a.has_sink && row_ok) {
                m_use = m_true = a.sink[U.h] * kLog2e;
                l = half == 0 ? 1.0f : 0.0f;
            }
            for (int t = 0; t < U.n; ++t) {
                const uint32_t g = gb + t, b = g & 1u;
                const int64_t j0 = (int64_t)(U.jlo + t) * BN;
                const int64_t jh = j0 + 64 * half;            // this half's first column
                uint32_t kw[5], ksh = 0;
                if (a.has_drop) fetch_keep128(a, U.sd, U.h, i, j0, kw, ksh);
                // attention-mask matrix bits of this half's 64 columns (all kept without one)
                uint2 am = make_uint2(~0u, ~0u);
                if (a.mask.keep_q != nullptr) {
                    am = row_ok ? __ldg(reinterpret_cast<const uint2 *>(a.mask.keep_q + i * a.mask.words_q + (jh >> 6)))
                                : make_uint2(0u, 0u);
                }
                if (!fwait_warp(sm, F_S_FULL + b, g >> 1, a)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t s_addr = tmem + lane_addr + TM_S + 128 * b + 64 * half;
                // keep bits of the half's two 32-column chunks: the range [lo, hi]
                // relative to jh, and the matrix
                uint32_t km[2];
                {
                    const int64_t clo = max(lo - jh, (int64_t)0), chi = min(hi - jh, (int64_t)63);
                    const uint32_t amw[2] = {am.x, am.y};
#pragma unroll
                    for (int ch = 0; ch < 2; ++ch) {
                        const int64_t l0 = clo - 32 * ch, h0 = chi - 32 * ch;
                        km[ch] = (l0 > 31 || h0 < 0 || l0 > h0)
                                     ? 0u
                                     : (~0u << (l0 < 0 ? 0 : (int)l0)) & (~0u >> (31 - (h0 > 31 ? 31 : (int)h0)));
                        km[ch] &= amw[ch];
                    }
                }
                // pass 1: block max over the half's kept columns, then the row's
                float bmax = -INFINITY;
                const float cs = PSE ? 1.0f : C;      // with a pse, the S buffer holds C S + pse term
#pragma unroll
                for (int ch = 0; ch < 2; ++ch) {
                    uint32_t raw[32];
                    tmem_ld32(s_addr + 32 * ch, raw);
                    if constexpr (PSE) {
                        float t[32];
                        fpse_chunk<BF16>(a, U, i, row_ok, jh + 32 * ch, C, t);
#pragma unroll
                        for (int c = 0; c < 32; ++c) raw[c] = __float_as_uint(fmaf(__uint_as_float(raw[c]), C, t[c]));
                        tmem_st32(s_addr + 32 * ch, raw);
                    }
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        if ((km[ch] >> c) & 1u) bmax = fmaxf(bmax, __uint_as_float(raw[c]) * cs);
                    }
                }
                {
                    float other;
                    if (!trade(bmax, other)) {
                        ok = false;
                        break;
                    }
                    bmax = fmaxf(bmax, other);
                }
                // lazy rescale: only when the max in use falls more than 2^8 behind
                m_true = fmaxf(m_true, bmax);
                float alpha = 1.0f;
                bool rescale_o = false;
                if (bmax > m_use + kRescaleLog2 || (m_use == -INFINITY && bmax > -INFINITY)) {
                    if (m_use > -INFINITY) {
                        alpha = ex2(m_use - bmax);
                        rescale_o = t > 0;
                    }
                    l *= alpha;
                    m_use = bmax;
                }
                if (__any_sync(0xffffffffu, rescale_o)) {
                    // O must hold every earlier block's P V before it is scaled
                    // (each half scales its HD / 2 columns)
                    if (!fwait_warp(sm, F_PV_DONE + (b ^ 1u), (g - 1) >> 1, a)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int ch = 0; ch < HD / 64; ++ch) {
                        uint32_t raw[32];
                        const uint32_t oa = tmem + lane_addr + TM_O + (HD / 2) * half + 32 * ch;
                        tmem_ld32(oa, raw);
#pragma unroll
                        for (int c = 0; c < 32; ++c) raw[c] = __float_as_uint(__uint_as_float(raw[c]) * alpha);
                        tmem_st32(oa, raw);
                    }
                }
                // pass 2: P = exp2(s C - m_use) on kept columns; l += P; Pd = P z
                // packed into the first 16 columns of its own 32-column chunk
                const float mneg = (m_use == -INFINITY) ? 0.0f : -m_use;
                // keep-bit words of this half's 64 columns (selected, not indexed,
                // so kw stays in registers)
                const uint32_t kwh[3] = {half ? kw[2] : kw[0], half ? kw[3] : kw[1], half ? kw[4] : kw[2]};
#pragma unroll
                for (int ch = 0; ch < 2; ++ch) {
                    uint32_t raw[32];
                    tmem_ld32(s_addr + 32 * ch, raw);
                    uint32_t zw = 0xffffffffu;
                    if (a.has_drop) zw = __funnelshift_r(kwh[ch], kwh[ch + 1], ksh);
                    float p[32];
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const bool kept = (km[ch] >> c) & 1u;
                        p[c] = kept ? ex2(fmaf(__uint_as_float(raw[c]), cs, mneg)) : 0.0f;
                        l += p[c];
                    }
                    uint32_t pk[16];
                    if (a.has_drop) {
                        // keep-bit only: 1 / keepProb is applied to O in fp32 at the end,
                        // so the packed operand carries no rounded scale factor
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            const float p0 = ((zw >> (2 * c)) & 1u) ? p[2 * c] : 0.0f;
                            const float p1 = ((zw >> (2 * c + 1)) & 1u) ? p[2 * c + 1] : 0.0f;
                            pk[c] = fpack2<BF16>(p0, p1);
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < 16; ++c) pk[c] = fpack2<BF16>(p[2 * c], p[2 * c + 1]);
                    }
                    tmem_st16(s_addr + 32 * ch, pk);   // over this chunk's already read S columns
                }
                tc_fence_before();
                mbar_arrive(sm.bar(F_P_READY + b));
            }
            if (!ok) break;
            // ---- unit end: O / l, max and sum of the true row max (8 copies)
            {
                float other;                                  // the row's sum: both halves
                if (!trade(l, other)) break;
                l += other;
            }
            float m_out = m_true, l_out = l;
            if (m_true > -INFINITY && m_use > -INFINITY) l_out = l * ex2(m_use - m_true);
            const float inv = (l > 0.0f ? 1.0f / l : 0.0f) * (a.has_drop ? a.inv_keep : 1.0f);
            const int64_t r = (U.sd.tq + i) * a.nq + U.h;
            if (U.n > 0) {
                if (!fwait_warp(sm, F_O_FULL, ku, a)) break;
                tc_fence_after();
#pragma unroll
                for (int ch = 0; ch < HD / 64; ++ch) {
                    uint32_t raw[32];
                    const int col = (HD / 2) * half + 32 * ch;
                    tmem_ld32(tmem + lane_addr + TM_O + col, raw);
                    if (row_ok) {
                        Out *dst = O + r * HD + col;
#pragma unroll
                        for (int c = 0; c < 32; c += 8) {
                            uint4 pkt;
                            pkt.x = fpack2<BF16>(__uint_as_float(raw[c]) * inv, __uint_as_float(raw[c + 1]) * inv);
                            pkt.y = fpack2<BF16>(__uint_as_float(raw[c + 2]) * inv, __uint_as_float(raw[c + 3]) * inv);
                            pkt.z = fpack2<BF16>(__uint_as_float(raw[c + 4]) * inv, __uint_as_float(raw[c + 5]) * inv);
                            pkt.w = fpack2<BF16>(__uint_as_float(raw[c + 6]) * inv, __uint_as_float(raw[c + 7]) * inv);
                            *reinterpret_cast<uint4 *>(dst + c) = pkt;
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(sm.bar(F_O_FREE));
                ++ku;
            } else if (row_ok) {
                Out *dst = O + r * HD + (HD / 2) * half;
                for (int c = 0; c < HD / 2; c += 8) *reinterpret_cast<uint4 *>(dst + c) = make_uint4(0, 0, 0, 0);
            }
            if (row_ok && half == 0) {
                const float mn = (m_out == -INFINITY) ? -INFINITY : m_out * kLn2;
                const float4 mv = make_float4(mn, mn, mn, mn), lv = make_float4(l_out, l_out, l_out, l_out);
                float4 *pm = reinterpret_cast<float4 *>(a.smax + r * 8);
                float4 *pl = reinterpret_cast<float4 *>(a.ssum + r * 8);
                pm[0] = mv;
                pm[1] = mv;
                pl[0] = lv;
                pl[1] = lv;
            }
            gb += U.n;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    // after an abort, TMA loads nobody waited for may still be in flight
    if (warp == 0 && lane == 0 && *sm.abort_flag()) {
        if (armed[0]) fdrain(sm, F_Q_FULL, armed[0] - 1, a);
        if (armed[1]) fdrain(sm, F_Q_FULL + 1, armed[1] - 1, a);
#pragma unroll
        for (int s = 0; s < NS; ++s) {
            if (armed[2 + s]) fdrain(sm, F_K_FULL + s, armed[2 + s] - 1, a);
            if (armed[2 + NS + s]) fdrain(sm, F_V_FULL + s, armed[2 + NS + s] - 1, a);
        }
    }
}

PFN_cuTensorMapEncodeTiled_v12000 fencode()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool done = false;
    if (!done) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        done = true;
    }
    return fn;
}

bool fmap(CUtensorMap *m, const void *ptr, int64_t rows, int64_t heads, int hd, bool bf16)
{
    auto fn = fencode();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)hd, (cuuint64_t)heads, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)hd * 2, (cuuint64_t)(heads * hd * 2)};
    cuuint32_t box[3] = {64, 1, 128};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
              const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool BF16, int HD, bool PSE>
cudaError_t flaunch(const FwdArgs &a, cudaStream_t s)
{
    CUtensorMap mq, mk, mv;
    if (!fmap(&mq, a.q, a.tq, a.nq, HD, BF16) || !fmap(&mk, a.k, a.tkv, a.nkv, HD, BF16) ||
        !fmap(&mv, a.v, a.tkv, a.nkv, HD, BF16))
        return cudaErrorInvalidValue;
    const int grid = std::min<int>(a.num_sms, a.n_fwd_units);
    constexpr uint32_t smem = FGeo<HD>::kSmemBytes;
    cudaError_t e =
        cudaFuncSetAttribute(fwd_tc_kernel<BF16, HD, PSE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    fwd_tc_kernel<BF16, HD, PSE><<<grid, kThreads, smem, s>>>(a, mq, mk, mv);
    return cudaGetLastError();
}

}  // namespace

bool fwd_tc_supported(int dtype, int d) { return (dtype == TND_BF16 || dtype == TND_F16) && (d == 64 || d == 128); }

cudaError_t launch_fwd_tc(const FwdArgs &a, cudaStream_t s)
{
    if (a.n_fwd_units == 0) return cudaSuccess;
    const bool bf16 = a.dtype == TND_BF16;
    if (a.pse.ptr) {
        if (a.d == 128) return bf16 ? flaunch<true, 128, true>(a, s) : flaunch<false, 128, true>(a, s);
        if (a.d == 64) return bf16 ? flaunch<true, 64, true>(a, s) : flaunch<false, 64, true>(a, s);
        return cudaErrorInvalidValue;
    }
    if (a.d == 128) return bf16 ? flaunch<true, 128, false>(a, s) : flaunch<false, 128, false>(a, s);
    if (a.d == 64) return bf16 ? flaunch<true, 64, false>(a, s) : flaunch<false, 64, false>(a, s);
    return cudaErrorInvalidValue;
}

}  // namespace tnd
