// Tensor-core (tcgen05) score-gradient for bf16 / fp16 at D = 128 on sm_103a.
//
// Computes, per sequence b, kv head g, 128-row kv block j and every query
// head h of the group with every 64-row q block i that sees block j
// ("aclnnFlashAttentionUnpaddingScoreGrad", function description):
//     S^T   = K_j Q_i^T                      (UMMA, smem x smem -> TMEM)
//     dP^T  = V_j dY_i^T                     (UMMA, smem x smem -> TMEM)
//     P^T   = exp2(S^T * scale*log2e - lse2_i) masked, Pd^T = P^T o z
//     dS^T  = P^T o (z dP^T - D_i)           (CUDA cores, from TMEM)
//     dV_j += Pd^T dY_i                      (UMMA, A = Pd^T from TMEM)
//     dK_j += dS^T Q_i                       (UMMA, A = dS^T from TMEM)
//     dQ_i^T = K_j^T dS^T                    (UMMA, smem x smem -> TMEM)
// dK_j (x scale) and dV_j leave TMEM once per unit.  The dQ tile of every
// (q block, head) is added into an fp32 accumulator by TMA bulk stores /
// reductions issued in a fixed order (highest contributing kv block first,
// each contributor waiting for its predecessor's counter), and
// dq_finalize_kernel writes dQ = scale * accumulator in the output dtype.
// No atomic operation touches data, so results are bitwise deterministic.
//
// Warp roles (352 threads, one CTA per SM, persistent over work units taken
// in plan order from a counter):
//   warp 0      TMA producer: K (double-buffered) and V (single) per unit,
//               Q / dY and the tile's lse2 / D vectors per tile, dropout
//               keep-bits staged in shared memory
//   warp 1      TMEM allocator and single-thread UMMA issuer
//   warps 2-5   softmax-gradient warps: thread = TMEM lane = kv row
//   warps 6-9   epilogue: dQ^T tile TMEM -> shared staging (thread = feature),
//               dK / dV TMEM -> global (thread = kv row) at unit end
//   warp 10     dQ writer: orders and issues the accumulator updates
// Every wait is bounded; on expiry the kernel records TND_ERR_DEVICE_TIMEOUT
// in the workspace status word and winds down instead of hanging.
#include "ptx_sm103.cuh"
#include "tnd_device.cuh"

#include <cudaTypedefs.h>
#include <mutex>

namespace tnd {
namespace {

using namespace ptx;

constexpr int HD = 128;                 // head dim
constexpr int BC = kKvBlock;            // 128 kv rows per block (UMMA M)
constexpr int BR = kQBlock;             // 64 q rows per block (UMMA N of S^T, dP^T, dQ^T)
constexpr int NSTAGE = 2;               // Q / dY ring depth
constexpr int kThreads = 352;
constexpr int kEpilogueWarp0 = 6;       // warps 6-9
constexpr int kWriterWarp = 10;
constexpr uint32_t kTmemCols = 512;

// TMEM columns
constexpr uint32_t TM_DV = 0, TM_DK = 128, TM_S0 = 256, TM_DP = 384, TM_DQ = 448;

// shared memory layout (offsets from a 1024-byte aligned base)
constexpr uint32_t kKvTile = BC * HD * 2;     // 32768: two 64-column blocks of 128 rows x 128 B
constexpr uint32_t kKvColBlk = BC * 128;      // 16384
constexpr uint32_t kQTile = BR * HD * 2;      // 16384: two 64-column blocks of 64 rows x 128 B
constexpr uint32_t kQColBlk = BR * 128;       // 8192
constexpr uint32_t kStgBytes = BR * HD * 4;   // 32768: dQ tile, fp32 [64 rows][128 features]
constexpr uint32_t kVecBytes = 2 * BR * 4;    // per stage: lse2[64], D[64]
constexpr uint32_t OFF_K = 0;                                 // 2 buffers
constexpr uint32_t OFF_V = OFF_K + 2 * kKvTile;               // 1 buffer
constexpr uint32_t OFF_Q = OFF_V + kKvTile;
constexpr uint32_t OFF_DY = OFF_Q + NSTAGE * kQTile;
constexpr uint32_t OFF_DS = OFF_DY + NSTAGE * kQTile;         // dS^T: 128 kv rows x 64 q (128 B)
constexpr uint32_t OFF_STG = OFF_DS + BC * 128;
constexpr uint32_t OFF_VEC = OFF_STG + kStgBytes;
constexpr uint32_t OFF_BITS = OFF_VEC + NSTAGE * kVecBytes;   // per stage: [64 rows][4 words]
constexpr uint32_t OFF_BAR = OFF_BITS + NSTAGE * BR * 4 * 4;
constexpr uint32_t kNumBars = 32;
constexpr uint32_t OFF_MISC = OFF_BAR + kNumBars * 8;
constexpr uint32_t kSmemUsed = OFF_MISC + 64;
// The whole 227 KB opt-in: one CTA per SM either way, and every operand
// descriptor's reach (tile base + strides) stays inside the allocation.
constexpr uint32_t kSmemBytes = 232448;
static_assert(kSmemUsed + 1024 <= kSmemBytes, "shared memory budget");
static_assert(OFF_STG % 1024 == 0 && OFF_DS % 1024 == 0 && OFF_VEC % 16 == 0, "alignment");

// mbarrier indices
enum : int {
    B_K_FULL = 0,      // [2]  count 1 + tx
    B_K_EMPTY = 2,     // [2]  count 1 (commit)
    B_V_FULL = 4,      //      count 1 + tx
    B_V_EMPTY = 5,     //      count 1 (commit after the unit's last dP)
    B_Q_FULL = 6,      // [2]  count 32 + tx
    B_Q_EMPTY = 8,     // [2]  count 1 (commit)
    B_S_FULL = 10,     // [2]  count 1 (commit)
    B_P_READY = 12,    // [2]  count 128
    B_S_FREE = 14,     // [2]  count 1 (commit)
    B_DP_FULL = 16,    //      count 1 (commit)
    B_DS_READY = 17,   //      count 128
    B_DK_DONE = 18,    //      count 1 (commit)
    B_DQ_FULL = 19,    //      count 1 (commit); also: dS smem of that tile consumed
    B_DQ_FREE = 20,    //      count 128
    B_ACC_FULL = 21,   //      count 1 (commit)
    B_ACC_FREE = 22,   //      count 128
    B_UNIT_FULL = 23,  // [2]  count 1
    B_UNIT_EMPTY = 25, // [2]  count 10 (MMA + 4 softmax + 4 epilogue warps + writer)
    B_DRAIN = 27,      //      count 1 (commit)
    B_STG_FULL = 28,   //      count 128
    B_STG_FREE = 29,   //      count 1
};

// misc words
constexpr uint32_t MISC_TMEM = 0, MISC_RING = 1, MISC_ABORT = 3;

struct Smem {
    uint8_t *base;
    __device__ uint64_t *bar(int i) const { return reinterpret_cast<uint64_t *>(base + OFF_BAR) + i; }
    __device__ uint32_t *misc() const { return reinterpret_cast<uint32_t *>(base + OFF_MISC); }
    __device__ volatile int *abort_flag() const { return reinterpret_cast<volatile int *>(misc() + MISC_ABORT); }
};

// Wait for completion `k` (0-based) of barrier `bar`, bounded.
__device__ __forceinline__ bool wait_k(const Smem &sm, int bar, uint32_t k, const GradArgs &a)
{
    uint64_t *b = sm.bar(bar);
    const uint32_t parity = k & 1u;
    if (mbar_try_wait(b, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(b, parity)) return true;
        if (*sm.abort_flag()) return false;
        if (clock64() - t0 > a.wait_limit_cycles) {
            set_status(a.status, TND_ERR_DEVICE_TIMEOUT, 0x100u + (uint32_t)bar);
            *sm.abort_flag() = 1;
            return false;
        }
    }
}

// Warp-uniform variant: every lane polls, all lanes agree on the outcome.
__device__ __forceinline__ bool wait_warp(const Smem &sm, int bar, uint32_t k, const GradArgs &a)
{
    const bool ok = wait_k(sm, bar, k, a);
    return __all_sync(0xffffffffu, ok);
}

// Bounded wait that ignores the abort flag (drains in-flight async copies).
__device__ __forceinline__ void drain_k(const Smem &sm, int bar, uint32_t k, const GradArgs &a)
{
    const long long t0 = clock64();
    while (!mbar_try_wait(sm.bar(bar), k & 1u) && clock64() - t0 < a.wait_limit_cycles) {
    }
}

struct UnitInfo {
    int b, g, jb, qb_lo, ntiles;
    SeqDesc sd;
};

__device__ __forceinline__ UnitInfo unit_info(const GradArgs &a, int u)
{
    const GradUnit gu = a.units[u];
    UnitInfo ui;
    ui.b = gu.b;
    ui.g = gu.g;
    ui.jb = gu.j;
    ui.qb_lo = gu.qb_lo;
    ui.ntiles = (gu.qb_hi - gu.qb_lo) * a.group;
    ui.sd = a.seqs[gu.b];
    return ui;
}

// Reads the unit index published in ring slot `ui % 2` (-1 = no more work).
__device__ __forceinline__ bool read_unit(const Smem &sm, uint32_t ui, const GradArgs &a, int &u, bool elect)
{
    const uint32_t slot = ui & 1u;
    if (!wait_warp(sm, B_UNIT_FULL + slot, ui >> 1, a)) return false;
    u = *reinterpret_cast<volatile int *>(sm.misc() + MISC_RING + slot);
    __syncwarp();
    if (elect) mbar_arrive(sm.bar(B_UNIT_EMPTY + slot));
    return true;
}

// Single-thread variant.
__device__ __forceinline__ bool read_unit1(const Smem &sm, uint32_t ui, const GradArgs &a, int &u)
{
    const uint32_t slot = ui & 1u;
    if (!wait_k(sm, B_UNIT_FULL + slot, ui >> 1, a)) return false;
    u = *reinterpret_cast<volatile int *>(sm.misc() + MISC_RING + slot);
    mbar_arrive(sm.bar(B_UNIT_EMPTY + slot));
    return true;
}

// Columns [c_lo, c_hi] of the q block (rows q0 + c) that keep kv row jj.
__device__ __forceinline__ uint64_t keep_columns(const GradArgs &a, const SeqDesc &sd, int64_t q0, int64_t jj)
{
    if (jj >= sd.skv) return 0ull;
    int64_t lo = 0, hi = BR - 1;
    const int64_t rows = (int64_t)sd.sq - q0;           // valid rows in the block
    if (rows - 1 < hi) hi = rows - 1;
    const MaskSpec &m = a.mask;
    if (m.mode == 2) {
        lo = max(lo, jj - q0);
    } else if (m.mode == 3) {
        lo = max(lo, jj - ((int64_t)sd.skv - sd.sq) - q0);
    } else if (m.mode == 4) {
        lo = max(lo, jj - m.next - q0);
        hi = min(hi, jj + m.pre - q0);
    }
    if (lo > hi) return 0ull;
    return (~0ull << lo) & (~0ull >> (63 - hi));
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    return BF16 ? pack_bf16(lo, hi) : pack_f16(lo, hi);
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    grad_tc_kernel(const __grid_constant__ GradArgs a, const __grid_constant__ CUtensorMap tmQ,
                   const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ CUtensorMap tmDY, const __grid_constant__ CUtensorMap tmDQ)
{
    extern __shared__ uint8_t smem_raw[];
    Smem sm;
    sm.base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = a.group;
    using Out = typename std::conditional<BF16, __nv_bfloat16, __half>::type;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(sm.bar(B_K_FULL + i), 1);
            mbar_init(sm.bar(B_K_EMPTY + i), 1);
            mbar_init(sm.bar(B_Q_FULL + i), 32);
            mbar_init(sm.bar(B_Q_EMPTY + i), 1);
            mbar_init(sm.bar(B_S_FULL + i), 1);
            mbar_init(sm.bar(B_P_READY + i), 128);
            mbar_init(sm.bar(B_S_FREE + i), 1);
            mbar_init(sm.bar(B_UNIT_FULL + i), 1);
            mbar_init(sm.bar(B_UNIT_EMPTY + i), 10);
        }
        mbar_init(sm.bar(B_V_FULL), 1);
        mbar_init(sm.bar(B_V_EMPTY), 1);
        mbar_init(sm.bar(B_DP_FULL), 1);
        mbar_init(sm.bar(B_DS_READY), 128);
        mbar_init(sm.bar(B_DK_DONE), 1);
        mbar_init(sm.bar(B_DQ_FULL), 1);
        mbar_init(sm.bar(B_DQ_FREE), 128);
        mbar_init(sm.bar(B_ACC_FULL), 1);
        mbar_init(sm.bar(B_ACC_FREE), 128);
        mbar_init(sm.bar(B_DRAIN), 1);
        mbar_init(sm.bar(B_STG_FULL), 128);
        mbar_init(sm.bar(B_STG_FREE), 1);
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
        prefetch_tmap(&tmDY);
        prefetch_tmap(&tmDQ);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm.misc() + MISC_TMEM);

    if (warp == 0) {
        // ================================================================ producer
        uint32_t ui = 0, ku = 0, gt = 0;
        int *counter = reinterpret_cast<int *>(a.status + kWorkCounter);
        while (true) {
            int u = 0;
            if (lane == 0) u = atomicAdd(counter, 1);
            u = __shfl_sync(0xffffffffu, u, 0);
            const uint32_t slot = ui & 1u;
            if (ui >= 2 && !wait_warp(sm, B_UNIT_EMPTY + slot, (ui >> 1) - 1, a)) break;
            if (lane == 0) {
                *reinterpret_cast<volatile int *>(sm.misc() + MISC_RING + slot) = (u < a.n_units) ? u : -1;
                mbar_arrive(sm.bar(B_UNIT_FULL + slot));
            }
            ++ui;
            if (u >= a.n_units) break;
            const UnitInfo U = unit_info(a, u);
            if (U.ntiles == 0) continue;
            const int z_kv = (int)(U.sd.tk + (int64_t)U.jb * BC);
            const uint32_t kb = ku & 1u;
            if (ku >= 2 && !wait_warp(sm, B_K_EMPTY + kb, (ku >> 1) - 1, a)) break;
            if (lane == 0) {
                uint64_t *fb = sm.bar(B_K_FULL + kb);
                mbar_arrive_expect_tx(fb, kKvTile);
                uint8_t *kt = sm.base + OFF_K + kb * kKvTile;
                tma_load_3d(kt, &tmK, fb, 0, U.g, z_kv);
                tma_load_3d(kt + kKvColBlk, &tmK, fb, 64, U.g, z_kv);
            }
            bool ok = true;
            for (int t = 0; t < U.ntiles; ++t, ++gt) {
                const int qb = U.qb_lo + t / G, h = U.g * G + t % G;
                const uint32_t s = gt % NSTAGE, k = gt / NSTAGE;
                if (k >= 1 && !wait_warp(sm, B_Q_EMPTY + s, k - 1, a)) {
                    ok = false;
                    break;
                }
                const int64_t q0 = (int64_t)qb * BR;
                if (a.has_drop) {
                    uint32_t *bits = reinterpret_cast<uint32_t *>(sm.base + OFF_BITS + s * BR * 16);
                    for (int w = lane; w < BR * 4; w += 32) {
                        const int r = w >> 2, wi = w & 3;
                        const int64_t ii = q0 + r;
                        uint32_t word = 0;
                        if (ii < U.sd.sq) {
                            const int64_t pos = U.sd.mask_base + ((int64_t)h * U.sd.sq + ii) * U.sd.skv +
                                                (int64_t)U.jb * BC + 32 * wi;
                            const int64_t byte0 = pos >> 3;
                            const int sh = (int)(pos & 7);
                            uint64_t acc = 0;
#pragma unroll
                            for (int bb = 0; bb < 5; ++bb) {
                                const int64_t bi = byte0 + bb;
                                const uint64_t v = (bi < a.mask_bytes) ? (uint64_t)a.drop_mask[bi] : 0ull;
                                acc |= v << (8 * bb);
                            }
                            word = (uint32_t)(acc >> sh);
                        }
                        bits[w] = word;
                    }
                }
                __syncwarp();
                uint64_t *fb = sm.bar(B_Q_FULL + s);
                if (lane == 0) {
                    mbar_arrive_expect_tx(fb, 2 * kQTile + kVecBytes);
                    const int z = (int)(U.sd.tq + q0);
                    uint8_t *qt = sm.base + OFF_Q + s * kQTile, *dyt = sm.base + OFF_DY + s * kQTile;
                    tma_load_3d(qt, &tmQ, fb, 0, h, z);
                    tma_load_3d(qt + kQColBlk, &tmQ, fb, 64, h, z);
                    tma_load_3d(dyt, &tmDY, fb, 0, h, z);
                    tma_load_3d(dyt + kQColBlk, &tmDY, fb, 64, h, z);
                    const int64_t vidx = ((int64_t)(U.sd.qblk0 + qb) * a.nq + h) * BR;
                    uint8_t *vec = sm.base + OFF_VEC + s * kVecBytes;
                    bulk_g2s(vec, a.lse2 + vidx, BR * 4, fb);
                    bulk_g2s(vec + BR * 4, a.drow + vidx, BR * 4, fb);
                } else {
                    mbar_arrive(fb);
                }
                if (t == 0) {
                    // V after the unit's first Q / dY tile: its buffer frees when the
                    // previous unit's last dP^T completes
                    if (ku >= 1 && !wait_warp(sm, B_V_EMPTY, ku - 1, a)) {
                        ok = false;
                        ++gt;
                        break;
                    }
                    if (lane == 0) {
                        uint64_t *vb = sm.bar(B_V_FULL);
                        mbar_arrive_expect_tx(vb, kKvTile);
                        uint8_t *vt = sm.base + OFF_V;
                        tma_load_3d(vt, &tmV, vb, 0, U.g, z_kv);
                        tma_load_3d(vt + kKvColBlk, &tmV, vb, 64, U.g, z_kv);
                    }
                }
            }
            ++ku;
            if (!ok) break;
        }
        // outstanding TMA writes must land before the CTA can leave.  K loads
        // were issued for units [0, ku), V loads for the same units except
        // possibly the last one if the wait before it failed: draining a phase
        // that never started only costs the bounded wait.
        if (*sm.abort_flag() && lane == 0) {
            for (uint32_t s = 0; s < NSTAGE && s < gt; ++s) {
                const uint32_t last = ((gt - 1 - s) / NSTAGE) * NSTAGE + s;  // last tile that used stage s
                drain_k(sm, B_Q_FULL + s, last / NSTAGE, a);
            }
            for (uint32_t kb = 0; kb < 2 && kb < ku; ++kb) {
                const uint32_t last = ((ku - 1 - kb) / 2) * 2 + kb;
                drain_k(sm, B_K_FULL + kb, last / 2, a);
            }
            if (ku >= 1) drain_k(sm, B_V_FULL, ku - 1, a);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            const uint32_t idS = instr_desc_f16(BF16, 128, BR, false, false);    // S^T, dP^T
            const uint32_t idKV = instr_desc_f16(BF16, 128, HD, false, true);    // dV, dK (A in TMEM)
            const uint32_t idQ = instr_desc_f16(BF16, 128, BR, true, true);      // dQ^T
            const uint32_t sbase = smem_u32(sm.base);
            const uint32_t vaddr = sbase + OFF_V;
            uint32_t ui = 0, ku = 0, gt = 0;
            bool ok = true;
            while (ok) {
                int u;
                if (!read_unit1(sm, ui, a, u)) break;
                ++ui;
                if (u < 0) break;
                const UnitInfo U = unit_info(a, u);
                if (U.ntiles == 0) continue;
                const uint32_t kb = ku & 1u;
                if (!wait_k(sm, B_K_FULL + kb, ku >> 1, a)) break;
                tc_fence_after();
                const uint32_t kaddr = sbase + OFF_K + kb * kKvTile;
                const uint32_t g_end = gt + (uint32_t)U.ntiles;
                // S^T(t) = K Q(t)^T, K-major both
                auto issue_s = [&](uint32_t g_t) -> bool {
                    const uint32_t s = g_t % NSTAGE, b = g_t & 1u;
                    if (!wait_k(sm, B_Q_FULL + s, g_t / NSTAGE, a)) return false;
                    if (g_t >= 2 && !wait_k(sm, B_S_FREE + b, (g_t >> 1) - 1, a)) return false;
                    tc_fence_after();
                    const uint32_t qaddr = sbase + OFF_Q + s * kQTile;
#pragma unroll
                    for (int kk = 0; kk < HD / 16; ++kk) {
                        const uint32_t cb = kk >> 2, off = (kk & 3) * 32;
                        mma_ss(tmem + TM_S0 + b * 64, smem_desc_sw128(kaddr + cb * kKvColBlk + off, 16, 1024),
                               smem_desc_sw128(qaddr + cb * kQColBlk + off, 16, 1024), idS, kk > 0);
                    }
                    mma_commit(sm.bar(B_S_FULL + b));
                    return true;
                };
                // dP^T(t) = V dY(t)^T, once dK(t-1) has consumed dS^T(t-1) from TMEM
                auto issue_dp = [&](uint32_t g_t) -> bool {
                    const uint32_t s = g_t % NSTAGE;
                    if (g_t >= 1 && !wait_k(sm, B_DK_DONE, g_t - 1, a)) return false;
                    tc_fence_after();
                    const uint32_t dyaddr = sbase + OFF_DY + s * kQTile;
#pragma unroll
                    for (int kk = 0; kk < HD / 16; ++kk) {
                        const uint32_t cb = kk >> 2, off = (kk & 3) * 32;
                        mma_ss(tmem + TM_DP, smem_desc_sw128(vaddr + cb * kKvColBlk + off, 16, 1024),
                               smem_desc_sw128(dyaddr + cb * kQColBlk + off, 16, 1024), idS, kk > 0);
                    }
                    mma_commit(sm.bar(B_DP_FULL));
                    if (g_t + 1 == g_end) mma_commit(sm.bar(B_V_EMPTY));   // last reader of V
                    return true;
                };
                if (!issue_s(gt)) break;
                if (!wait_k(sm, B_V_FULL, ku, a)) break;
                if (!issue_dp(gt)) break;
                for (int t = 0; t < U.ntiles; ++t) {
                    const uint32_t g_t = gt + t, s = g_t % NSTAGE, b = g_t & 1u;
                    if (t + 1 < U.ntiles && !issue_s(g_t + 1)) {
                        ok = false;
                        break;
                    }
                    if (t == 0 && ku >= 1 && !wait_k(sm, B_ACC_FREE, ku - 1, a)) {
                        ok = false;
                        break;
                    }
                    // dV += Pd^T dY(t): A = Pd^T (TMEM, 32 packed columns), B = dY MN-major (N = 128)
                    if (!wait_k(sm, B_P_READY + b, g_t >> 1, a)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t qaddr = sbase + OFF_Q + s * kQTile, dyaddr = sbase + OFF_DY + s * kQTile;
#pragma unroll
                    for (int kk = 0; kk < BR / 16; ++kk) {
                        mma_ts(tmem + TM_DV, tmem + TM_S0 + b * 64 + kk * 8,
                               smem_desc_sw128(dyaddr + kk * 2048, kQColBlk, 1024), idKV, (t > 0 || kk > 0));
                    }
                    mma_commit(sm.bar(B_S_FREE + b));
                    // dK += dS^T Q(t): A = dS^T (TMEM), B = Q MN-major
                    if (!wait_k(sm, B_DS_READY, g_t, a)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < BR / 16; ++kk) {
                        mma_ts(tmem + TM_DK, tmem + TM_DP + kk * 8,
                               smem_desc_sw128(qaddr + kk * 2048, kQColBlk, 1024), idKV, (t > 0 || kk > 0));
                    }
                    mma_commit(sm.bar(B_Q_EMPTY + s));
                    mma_commit(sm.bar(B_DK_DONE));
                    // dP^T of the next tile ahead of this tile's dQ^T: the softmax
                    // warps get it one GEMM earlier
                    if (t + 1 < U.ntiles && !issue_dp(g_t + 1)) {
                        ok = false;
                        break;
                    }
                    // dQ^T(t) = K^T dS^T: A = K MN-major (M = 128 features), B = dS^T MN-major (N = 64)
                    if (g_t >= 1 && !wait_k(sm, B_DQ_FREE, g_t - 1, a)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < BC / 16; ++kk) {
                        mma_ss(tmem + TM_DQ, smem_desc_sw128(kaddr + kk * 2048, kKvColBlk, 1024),
                               smem_desc_sw128(sbase + OFF_DS + kk * 2048, kQColBlk, 1024), idQ, kk > 0);
                    }
                    mma_commit(sm.bar(B_DQ_FULL));
                }
                if (!ok) break;
                mma_commit(sm.bar(B_ACC_FULL));
                mma_commit(sm.bar(B_K_EMPTY + kb));
                gt += U.ntiles;
                ++ku;
            }
            // every issued UMMA must finish before TMEM is released
            mma_commit(sm.bar(B_DRAIN));
            const long long t0 = clock64();
            while (!mbar_try_wait(sm.bar(B_DRAIN), 0) && clock64() - t0 < a.wait_limit_cycles) {
            }
        }
        __syncwarp();
    } else if (warp < kEpilogueWarp0) {
        // ================================================================ softmax gradient
        const int quarter = warp & 3;
        const int jl = quarter * 32 + lane;                 // kv row within the block = TMEM lane
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const float C = a.scale * kLog2e;
        uint32_t ui = 0, gt = 0;
        while (true) {
            int u;
            if (!read_unit(sm, ui, a, u, lane == 0)) break;
            ++ui;
            if (u < 0) break;
            const UnitInfo U = unit_info(a, u);
            bool ok = true;
            for (int t = 0; t < U.ntiles; ++t, ++gt) {
                const int qb = U.qb_lo + t / G;
                const uint32_t s = gt % NSTAGE, b = gt & 1u;
                const int64_t q0 = (int64_t)qb * BR;
                const int64_t jj = (int64_t)U.jb * BC + jl;
                const uint64_t keep = keep_columns(a, U.sd, q0, jj);
                const bool full = __all_sync(0xffffffffu, keep == ~0ull);
                if (!wait_warp(sm, B_Q_FULL + s, gt / NSTAGE, a) || !wait_warp(sm, B_S_FULL + b, gt >> 1, a)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float *lse = reinterpret_cast<const float *>(sm.base + OFF_VEC + s * kVecBytes);
                const float *dvec = lse + BR;
                uint64_t zbits = ~0ull;
                if (a.has_drop) {
                    const uint32_t *bits = reinterpret_cast<const uint32_t *>(sm.base + OFF_BITS + s * BR * 16);
                    zbits = 0;
#pragma unroll 8
                    for (int c = 0; c < BR; ++c) zbits |= (uint64_t)((bits[c * 4 + quarter] >> lane) & 1u) << c;
                }
                // ---- phase 1: P^T from S^T, Pd^T = P^T o z into TMEM
                float p[BR];
                uint32_t raw[32];
                const uint32_t s_addr = tmem + lane_addr + TM_S0 + b * 64;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    tmem_ld32(s_addr + half * 32, raw);
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        p[half * 32 + c] = ex2(fmaf(__uint_as_float(raw[c]), C, -lse[half * 32 + c]));
                    }
                }
                if (!full) {
#pragma unroll
                    for (int c = 0; c < BR; ++c) p[c] = ((keep >> c) & 1ull) ? p[c] : 0.0f;
                }
                uint32_t pk[32];
                if (a.has_drop) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const float z0 = ((zbits >> (2 * c)) & 1ull) ? a.inv_keep : 0.0f;
                        const float z1 = ((zbits >> (2 * c + 1)) & 1ull) ? a.inv_keep : 0.0f;
                        pk[c] = pack2<BF16>(p[2 * c] * z0, p[2 * c + 1] * z1);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 32; ++c) pk[c] = pack2<BF16>(p[2 * c], p[2 * c + 1]);
                }
                tmem_st32(s_addr, pk);
                tc_fence_before();
                mbar_arrive(sm.bar(B_P_READY + b));
                // ---- phase 2: dS^T = P^T o (z dP^T - D) into TMEM and shared memory
                if (!wait_warp(sm, B_DP_FULL, gt, a)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t dp_addr = tmem + lane_addr + TM_DP;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    tmem_ld32(dp_addr + half * 32, raw);
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        const int c0 = half * 32 + c;
                        float dp0 = __uint_as_float(raw[c]), dp1 = __uint_as_float(raw[c + 1]);
                        if (a.has_drop) {
                            dp0 = ((zbits >> c0) & 1ull) ? dp0 * a.inv_keep : 0.0f;
                            dp1 = ((zbits >> (c0 + 1)) & 1ull) ? dp1 * a.inv_keep : 0.0f;
                        }
                        pk[(half * 32 + c) >> 1] = pack2<BF16>(p[c0] * (dp0 - dvec[c0]), p[c0 + 1] * (dp1 - dvec[c0 + 1]));
                    }
                }
                tmem_st32(dp_addr, pk);
                // the previous tile's dQ^T GEMM must have read the dS^T buffer
                if (gt >= 1 && !wait_warp(sm, B_DQ_FULL, gt - 1, a)) {
                    ok = false;
                    break;
                }
                {
                    uint8_t *row = sm.base + OFF_DS + jl * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint4 v = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                        *reinterpret_cast<uint4 *>(row + ((c ^ (jl & 7)) << 4)) = v;
                    }
                }
                fence_async_smem();
                tc_fence_before();
                mbar_arrive(sm.bar(B_DS_READY));
            }
            if (!ok) break;
        }
    } else if (warp < kWriterWarp) {
        // ================================================================ epilogue
        const int quarter = warp & 3;
        const int ln = quarter * 32 + lane;                 // TMEM lane: feature d (dQ^T) or kv row (dK/dV)
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        Out *dK = reinterpret_cast<Out *>(a.dk);
        Out *dV = reinterpret_cast<Out *>(a.dv);
        float *stg = reinterpret_cast<float *>(sm.base + OFF_STG) + ln;
        uint32_t ui = 0, ku = 0, gt = 0;
        while (true) {
            int u;
            if (!read_unit(sm, ui, a, u, lane == 0)) break;
            ++ui;
            if (u < 0) break;
            const UnitInfo U = unit_info(a, u);
            const int64_t jj = (int64_t)U.jb * BC + ln;
            const bool row_ok = jj < U.sd.skv;
            const int64_t kv_off = ((U.sd.tk + jj) * a.nkv + U.g) * (int64_t)HD;
            if (U.ntiles == 0) {
                if (row_ok) {
                    for (int c = 0; c < HD; c += 8) {
                        *reinterpret_cast<uint4 *>(dK + kv_off + c) = make_uint4(0, 0, 0, 0);
                        *reinterpret_cast<uint4 *>(dV + kv_off + c) = make_uint4(0, 0, 0, 0);
                    }
                }
                continue;
            }
            bool ok = true;
            for (int t = 0; t < U.ntiles; ++t, ++gt) {
                if (!wait_warp(sm, B_DQ_FULL, gt, a)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t v[BR];
                tmem_ld32(tmem + lane_addr + TM_DQ, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
                tmem_ld32(tmem + lane_addr + TM_DQ + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
                tc_fence_before();
                mbar_arrive(sm.bar(B_DQ_FREE));
                // staging [64 q rows][128 features] fp32, free once the writer's
                // previous bulk operation has read it
                if (gt >= 1 && !wait_warp(sm, B_STG_FREE, gt - 1, a)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int c = 0; c < BR; ++c) stg[c * HD] = __uint_as_float(v[c]);
                fence_async_smem();
                mbar_arrive(sm.bar(B_STG_FULL));
            }
            if (!ok) break;
            // unit epilogue: dV, dK (x scale) out of TMEM
            if (!wait_warp(sm, B_ACC_FULL, ku, a)) break;
            tc_fence_after();
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                const uint32_t col0 = which == 0 ? TM_DV : TM_DK;
                const float mul = which == 0 ? 1.0f : a.scale;
                Out *dst = (which == 0 ? dV : dK) + kv_off;
#pragma unroll
                for (int chunk = 0; chunk < HD / 32; ++chunk) {
                    uint32_t raw[32];
                    tmem_ld32(tmem + lane_addr + col0 + chunk * 32, raw);
                    if (row_ok) {
#pragma unroll
                        for (int c = 0; c < 32; c += 8) {
                            uint4 pkt;
                            pkt.x = pack2<BF16>(__uint_as_float(raw[c]) * mul, __uint_as_float(raw[c + 1]) * mul);
                            pkt.y = pack2<BF16>(__uint_as_float(raw[c + 2]) * mul, __uint_as_float(raw[c + 3]) * mul);
                            pkt.z = pack2<BF16>(__uint_as_float(raw[c + 4]) * mul, __uint_as_float(raw[c + 5]) * mul);
                            pkt.w = pack2<BF16>(__uint_as_float(raw[c + 6]) * mul, __uint_as_float(raw[c + 7]) * mul);
                            *reinterpret_cast<uint4 *>(dst + chunk * 32 + c) = pkt;
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(sm.bar(B_ACC_FREE));
            ++ku;
        }
    } else {
        // ================================================================ dQ writer
        // Adds each staged dQ^T tile into the fp32 accumulator of its (q block,
        // head): the first contributor stores, later ones add, each after the
        // previous contributor's counter says its update has completed.  A
        // counter is released one tile late (when the next bulk group is in
        // flight), but never held while this thread waits on another counter.
        if (lane == 0) {
            uint32_t ui = 0, gt = 0;
            int *pend_flag = nullptr;
            int pend_val = 0;
            auto release_pending = [&](bool all) {
                if (!pend_flag) return;
                if (all) bulk_wait0();
                else bulk_wait1();
                fence_async_global();
                st_release_gpu(pend_flag, pend_val);
                pend_flag = nullptr;
            };
            bool ok = true;
            while (ok) {
                int u;
                if (!read_unit1(sm, ui, a, u)) break;
                ++ui;
                if (u < 0) break;
                const UnitInfo U = unit_info(a, u);
                for (int t = 0; t < U.ntiles; ++t, ++gt) {
                    const int qb = U.qb_lo + t / G, h = U.g * G + t % G;
                    const int qg = U.sd.qblk0 + qb;
                    const QBlockInfo qi = a.qblk[qg];
                    int *flag = a.flags + (int64_t)qg * a.nq + h;
                    const int64_t q0 = (int64_t)qb * BR;
                    const int rows = (int)min((int64_t)BR, (int64_t)U.sd.sq - q0);
                    const int pos = qi.jhi - U.jb;
                    if (!wait_k(sm, B_STG_FULL, gt, a)) {
                        ok = false;
                        break;
                    }
                    if (pos > 0) {
                        if (ld_acquire_gpu(flag) < pos) {
                            release_pending(true);
                            const long long t0 = clock64();
                            while (ld_acquire_gpu(flag) < pos) {
                                if (*sm.abort_flag()) {
                                    ok = false;
                                    break;
                                }
                                if (clock64() - t0 > a.wait_limit_cycles) {
                                    set_status(a.status, TND_ERR_DEVICE_TIMEOUT, 0x200u);
                                    *sm.abort_flag() = 1;
                                    ok = false;
                                    break;
                                }
                                __nanosleep(32);
                            }
                            if (!ok) break;
                        }
                        fence_async_global();
                    }
                    const uint8_t *stg = sm.base + OFF_STG;
                    const int z = (int)(U.sd.tq + q0);
                    if (rows == BR) {
                        if (pos == 0) tma_store_3d(&tmDQ, stg, 0, h, z);
                        else tma_reduce_add_3d(&tmDQ, stg, 0, h, z);
                    } else {
                        // ragged last block of a sequence: only its own rows
                        for (int r = 0; r < rows; ++r) {
                            float *dst = a.dqacc + ((int64_t)(z + r) * a.nq + h) * HD;
                            if (pos == 0) bulk_s2g(dst, stg + r * HD * 4, HD * 4);
                            else bulk_reduce_add_f32(dst, stg + r * HD * 4, HD * 4);
                        }
                    }
                    bulk_commit();
                    bulk_wait_read0();
                    mbar_arrive(sm.bar(B_STG_FREE));
                    release_pending(false);
                    pend_flag = flag;
                    pend_val = pos + 1;
                }
            }
            release_pending(true);
            bulk_wait0();
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// dQ = scale * accumulator in the output dtype, one (q block, head) per
// iteration; q blocks no kv block reaches get zeros.
template <typename Out>
__global__ void __launch_bounds__(256) dq_finalize_kernel(GradArgs a)
{
    Out *dQ = reinterpret_cast<Out *>(a.dq);
    const int64_t n = (int64_t)a.n_qblk * a.nq;
    for (int64_t w = blockIdx.x; w < n; w += gridDim.x) {
        const int qg = (int)(w / a.nq), h = (int)(w - (int64_t)qg * a.nq);
        const int2 qr = a.qblk_rows[qg];
        const SeqDesc sd = a.seqs[qr.x];
        const int rows = min(BR, sd.sq - qr.y);
        const bool covered = a.qblk[qg].jlo >= 0;
        for (int e = threadIdx.x; e < rows * (HD / 4); e += blockDim.x) {
            const int r = e / (HD / 4), c4 = e - r * (HD / 4);
            const int64_t off = ((sd.tq + qr.y + r) * a.nq + h) * (int64_t)HD + c4 * 4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (covered) v = __ldcs(reinterpret_cast<const float4 *>(a.dqacc + off));
            uint2 pk;
            if (std::is_same<Out, __nv_bfloat16>::value) {
                pk.x = pack_bf16(v.x * a.scale, v.y * a.scale);
                pk.y = pack_bf16(v.z * a.scale, v.w * a.scale);
            } else {
                pk.x = pack_f16(v.x * a.scale, v.y * a.scale);
                pk.y = pack_f16(v.z * a.scale, v.w * a.scale);
            }
            *reinterpret_cast<uint2 *>(dQ + off) = pk;
        }
    }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// [rows, heads, 128] tensor of 16-bit elements, boxes of 64 features x 1 head x `box_rows` rows
bool make_map(CUtensorMap *m, const void *ptr, int64_t rows, int64_t heads, int box_rows, bool bf16)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)HD, (cuuint64_t)heads, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)HD * 2, (cuuint64_t)(heads * HD * 2)};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                    const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// dQ accumulator [rows, heads, 128] fp32, boxes of 128 features x 1 head x 64 rows (no swizzle)
bool make_acc_map(CUtensorMap *m, const float *ptr, int64_t rows, int64_t heads)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)HD, (cuuint64_t)heads, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)HD * 4, (cuuint64_t)(heads * HD * 4)};
    cuuint32_t box[3] = {HD, 1, BR};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

bool grad_tc_supported(int dtype, int d) { return (dtype == TND_BF16 || dtype == TND_F16) && d == HD; }

cudaError_t launch_grad_tc(const GradArgs &a, cudaStream_t s)
{
    if (a.n_units == 0) return cudaSuccess;
    const bool bf16 = a.dtype == TND_BF16;
    CUtensorMap mq, mk, mv, mdy, mdq;
    if (!make_map(&mq, a.q, a.tq, a.nq, BR, bf16) || !make_map(&mk, a.k, a.tkv, a.nkv, BC, bf16) ||
        !make_map(&mv, a.v, a.tkv, a.nkv, BC, bf16) || !make_map(&mdy, a.dy, a.tq, a.nq, BR, bf16) ||
        !make_acc_map(&mdq, a.dqacc, a.tq, a.nq))
        return cudaErrorInvalidValue;
    const int grid = std::min<int>(a.num_sms, a.n_units);
    cudaError_t e;
    if (bf16) {
        e = cudaFuncSetAttribute(grad_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        grad_tc_kernel<true><<<grid, kThreads, kSmemBytes, s>>>(a, mq, mk, mv, mdy, mdq);
    } else {
        e = cudaFuncSetAttribute(grad_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        grad_tc_kernel<false><<<grid, kThreads, kSmemBytes, s>>>(a, mq, mk, mv, mdy, mdq);
    }
    return cudaGetLastError();
}

cudaError_t launch_dq_finalize(const GradArgs &a, cudaStream_t s)
{
    const int64_t n = (int64_t)a.n_qblk * a.nq;
    if (n == 0) return cudaSuccess;
    const int grid = (int)std::min<int64_t>(n, (int64_t)a.num_sms * 8);
    if (a.dtype == TND_BF16) dq_finalize_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(a);
    else dq_finalize_kernel<__half><<<grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace tnd
