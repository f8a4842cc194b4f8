// Tensor-core (tcgen05) score-gradient for bf16 / fp16 at D = 64 or 128 on
// sm_103a.
//
// Computes, per sequence b, kv head g, 128-row kv block j and every query
// head h of the group with every 128-row q block i that sees block j
// ("aclnnFlashAttentionUnpaddingScoreGrad", function description):
//     S^T   = K_j Q_i^T                      (UMMA, smem x smem -> TMEM)
//     dP^T  = V_j dY_i^T                     (UMMA, smem x smem -> TMEM)
//     P^T   = exp2(S^T * scale*log2e - lse2_i) masked, Pd^T = P^T o z
//     dS^T  = P^T o (z dP^T - D_i)           (CUDA cores, TMEM -> shared memory)
//     dV_j += Pd^T dY_i                      (UMMA, A = Pd^T from TMEM)
//     dK_j += dS^T Q_i                       (UMMA, smem x smem)
//     dQ_i^T = K_j^T dS^T                    (UMMA, smem x smem -> TMEM)
// dK_j (x scale) and dV_j leave TMEM once per unit.  The dQ tile of every
// (q block, head) is combined across its contributing kv blocks in a fixed
// order, highest kv block first: the compute warps stage each tile's dQ^T in
// shared memory (in the tile's own Q and dY stages, whose UMMA readers are
// done by then), and a writer warp stores it into an fp32 accumulator with
// TMA (first contributor) or adds it with TMA bulk reduce-adds (later ones),
// each only after its predecessor's counter says that update is complete.
// dq_finalize_kernel then writes dQ = scale * accumulator in the output
// dtype.  The adds are read-modify-writes in global memory, but their order
// is fixed, so results are bitwise deterministic.  With the library's
// deterministic option off (the non-deterministic default of the
// "aclnnFlashAttentionUnpaddingScoreGradV5" constraints), a
// later contributor waits only for the first one's store and adds in
// arrival order: the same sum, rounded in a run-dependent order.
//
// Tiles are 128 kv rows x 128 q rows, so S^T, dP^T and dQ^T are N = 128
// UMMAs.  TMEM (512 columns): dV, dK accumulators; S^T (then Pd^T packed
// in place until dV has read it; the compute warps keep P^T in registers
// for dS^T); dP^T (then, once the compute warps have read it, the tile's
// dQ^T).  dS^T goes to its own shared-memory
// buffer, the A operand of dK and the B operand of dQ^T.  The UMMA issue
// order per tile t is [P^T(t) ready] dV(t), [dS^T(t) ready] dK(t), dQ^T(t),
// S^T(t+1), [dQ^T(t) read out] dP^T(t+1); the compute warps take P^T(t),
// dS^T(t), then the epilogue of t (dQ^T out of TMEM), so S^T(t+1) runs
// under that epilogue and dP^T(t+1) under P^T(t+1).
//
// Warp roles (352 threads, one CTA per SM, persistent over work units taken
// in plan order from a counter):
//   warp 0      TMA producer: K, V per unit; Q (+ lse2 / D vectors) and dY
//               per tile (two stages each)
//   warp 1      TMEM allocator and UMMA issuer (the warp runs the issue code
//               together; one elected lane issues)
//   warps 2-9   compute warps, two per TMEM lane quarter, each on 64 of the
//               tile's 128 q columns.  Per tile: P^T (thread = kv row),
//               dS^T, then the tile's epilogue (dQ^T out of TMEM, thread =
//               feature, into shared-memory staging; dK, dV at unit end)
//   warp 10     dQ writer: chain order, TMA store / reduce-add of the staged
//               tile, counter release
// Every wait is bounded; on expiry the kernel records TND_ERR_DEVICE_TIMEOUT
// in the workspace status word and winds down instead of hanging.
#include "ptx_sm103.cuh"
#include "tnd_device.cuh"

#include <cudaTypedefs.h>
#include <mutex>

namespace tnd {
namespace {

using namespace ptx;

constexpr int BC = kKvBlock;            // 128 kv rows per block (UMMA M)
constexpr int BR = kQBlock;             // 128 q rows per block (UMMA N of S^T, dP^T, dQ^T)
constexpr int kThreads = 352;
constexpr int kComputeWarp0 = 2;        // warps 2-9 (two per TMEM lane quarter)
constexpr int kComputeThreads = 256;
constexpr int kWriterWarp = 10;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TM_S = 256, TM_DP = 384;   // S^T / P^T; dP^T / dQ^T
constexpr uint32_t kColBlk = 128 * 128;       // one 64-element column block of 128 rows (16 KB)

// Shared-memory layout for head dim HD (offsets from a 1024-byte aligned
// base).  Tiles are stored as 64-element column blocks of 128 rows x 128 B
// with the 128-byte swizzle, the layout TMA writes and UMMA reads.
template <int HD>
struct Geo {
    static constexpr uint32_t NCB = HD / 64;              // column blocks per row
    static constexpr uint32_t kKvTile = BC * HD * 2;      // K or V tile
    static constexpr uint32_t kQTile = BR * HD * 2;       // Q or dY tile
    static constexpr uint32_t kDsBytes = BC * BR * 2;     // dS^T, 128 kv rows x 128 q
    static constexpr uint32_t kVecBytes = 2 * BR * 4;     // lse2[128], D[128]
    static constexpr uint32_t OFF_K = 0;
    static constexpr uint32_t OFF_V = OFF_K + kKvTile;
    static constexpr uint32_t OFF_Q = OFF_V + kKvTile;    // 2 stages
    static constexpr uint32_t OFF_DY = OFF_Q + 2 * kQTile;  // 2 stages
    static constexpr uint32_t OFF_DS = OFF_DY + 2 * kQTile;
    static constexpr uint32_t OFF_VEC = OFF_DS + kDsBytes;  // 2 stages
    static constexpr uint32_t OFF_BAR = OFF_VEC + 2 * kVecBytes;
    static constexpr uint32_t kNumBars = 30;
    static constexpr uint32_t OFF_MISC = OFF_BAR + kNumBars * 8;
    static constexpr uint32_t kSmemBytes = OFF_MISC + 64;
    // For HD = 64 the dQ^T UMMA has M = 128 and its A operand's second
    // column block reads the 16 KB after K (the V tile): rows 64-127 of that
    // dQ^T are never read.
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(OFF_DS % 1024 == 0 && OFF_Q % 1024 == 0 && OFF_DY % 1024 == 0 && OFF_VEC % 16 == 0, "align");
};

// mbarrier indices.  Every per-tile barrier with a single buffer is awaited
// by roles that can never lag more than one completion behind (each
// producer of a completion t+1 waits, directly or through a chain of
// hand-offs, on the waiter having passed completion t).
enum : int {
    B_K_FULL = 0,      //      count 1 + tx
    B_K_EMPTY = 1,     //      count 1 (commit after the unit's last dQ^T)
    B_V_FULL = 2,      //      count 1 + tx
    B_V_EMPTY = 3,     //      count 1 (commit after the unit's last dP^T)
    B_Q_FULL = 4,      // [2]  count 1 + tx (Q tile + lse2 / D vectors, stage t % 2)
    B_Q_EMPTY = 6,     // [2]  count 2 (commit after dK; the writer, once the dQ^T staged
                       //      in this stage has been read)
    B_DY_FULL = 8,     // [2]  count 1 + tx
    B_DY_EMPTY = 10,   // [2]  count 2 (commit after dV and dP^T; the writer, once the dQ^T
                       //      staged in this stage has been read)
    B_S_FULL = 12,     //      count 1 (commit)
    B_P_READY = 13,    // [2]  count 128 (per softmax half: q columns 0-63, 64-127)
    B_PV_DONE = 15,    //      count 1 (commit after dV: P^T consumed, S buffer free)
    B_DP_FULL = 16,    //      count 1 (commit)
    B_DS_READY = 17,   //      count 256
    B_DQ_FULL = 18,    //      count 1 (commit after dQ^T; dK and dQ^T have read dS)
    B_DQ_FREE = 19,    //      count 256 (dQ^T read out of TMEM)
    B_ACC_FULL = 20,   //      count 1 (commit after the unit's last tile)
    B_ACC_FREE = 21,   //      count 256 (dK / dV read out)
    B_UNIT_FULL = 22,  // [2]  count 1
    B_UNIT_EMPTY = 24, // [2]  count 10 (MMA + 8 compute warps + writer)
    B_DRAIN = 26,      //      count 1 (commit)
    B_STG_FULL = 27,   // [2]  count 256 (dQ^T of a tile of stage t % 2 staged)
};

// misc words
constexpr uint32_t MISC_TMEM = 0, MISC_RING = 1, MISC_ABORT = 3;

#ifdef TND_TRACE
// Diagnostic build only: a clock-stamped event log of the first kTraceCtas
// CTAs, one ring per warp (lane 0 records): {clock64, (event << 24) | tile}.
// The event count lives in a register of the recording thread (`n`), so an
// event costs two fire-and-forget stores and no global round trip.
constexpr int kTraceCtas = 2, kTraceLen = 8192;
__device__ unsigned long long g_trace[kTraceCtas][11][kTraceLen][2];
__device__ unsigned int g_trace_n[kTraceCtas][11];
__device__ unsigned long long g_cta_span[1024][2];
__device__ __forceinline__ void trace(uint32_t &n, uint32_t ev, uint32_t k)
{
    if ((threadIdx.x & 31) != 0 || blockIdx.x >= kTraceCtas) return;
    const int w = threadIdx.x >> 5;
    const unsigned i = n++;
    if (i < (unsigned)kTraceLen) {
        ulonglong2 rec = make_ulonglong2((unsigned long long)clock64(), ((unsigned long long)ev << 24) | (k & 0xffffffu));
        *reinterpret_cast<ulonglong2 *>(&g_trace[blockIdx.x][w][i][0]) = rec;
    }
}
__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
#define TRACE(ev, k) trace(trace_n, (ev), (k))
#else
#define TRACE(ev, k) ((void)0)
#endif
// trace events
enum : uint32_t {
    EV_UNIT = 1, EV_W_QFULL, EV_W_DYFULL, EV_W_KFULL, EV_W_VFULL, EV_W_PVDONE, EV_W_DQFREE, EV_W_ACCFREE,
    EV_W_P0, EV_W_P1, EV_W_DS, EV_I_S, EV_I_DP, EV_I_DV, EV_I_DK, EV_I_DQ,                  // MMA issuer
    EV_C_SFULL = 20, EV_C_PDONE, EV_C_DPFULL, EV_C_DSDONE, EV_C_DQFULL, EV_C_DQFREE, EV_C_CHAIN, EV_C_EPIDONE,
    EV_C_UNITOUT,                                                                             // compute warps
    EV_L_Q = 40, EV_L_DY, EV_L_K, EV_L_V,                                                     // producer
    EV_W_STG = 50, EV_W_CHAIN, EV_W_ISSUED, EV_W_READ, EV_W_WRITTEN,                          // dQ writer
};

struct Smem {
    uint8_t *base;
    uint32_t off_bar, off_misc;
    __device__ uint64_t *bar(int i) const { return reinterpret_cast<uint64_t *>(base + off_bar) + i; }
    __device__ uint32_t *misc() const { return reinterpret_cast<uint32_t *>(base + off_misc); }
    __device__ volatile int *abort_flag() const { return reinterpret_cast<volatile int *>(misc() + MISC_ABORT); }
};

// Wait for completion `k` (0-based) of barrier `bar`, bounded.
__device__ __forceinline__ bool wait_k(const Smem &sm, int bar, uint32_t k, const GradArgs &a)
{
    uint64_t *b = sm.bar(bar);
    const uint32_t parity = k & 1u;
    const long long t0 = clock64();
    while (!mbar_try_wait(b, parity)) {
        if (*sm.abort_flag()) return false;
        if (clock64() - t0 > a.wait_limit_cycles) {
            // detail: completion index, warp, barrier
            set_status(a.status, TND_ERR_DEVICE_TIMEOUT, (k << 12) | ((threadIdx.x >> 5) << 6) | (uint32_t)bar);
            *sm.abort_flag() = 1;
            return false;
        }
    }
    return true;
}

// Non-suspending phase test: mbarrier.test_wait reacts to the phase flip
// without the resume delay of a suspended try_wait.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Polling variant for a whole converged warp (the UMMA issuer): every lane
// tests the phase and the warp leaves together, as soon as any lane has seen
// it complete (the barrier cannot move a further phase before this warp acts).
__device__ __forceinline__ bool wait_uni(const Smem &sm, int bar, uint32_t k, const GradArgs &a)
{
    uint64_t *b = sm.bar(bar);
    const uint32_t parity = k & 1u;
    const long long t0 = clock64();
    while (!__any_sync(0xffffffffu, mbar_test_wait(b, parity))) {
        if (__any_sync(0xffffffffu, *sm.abort_flag() != 0)) return false;
        if (__any_sync(0xffffffffu, clock64() - t0 > a.wait_limit_cycles)) {
            if ((threadIdx.x & 31) == 0) {
                set_status(a.status, TND_ERR_DEVICE_TIMEOUT, (k << 12) | ((threadIdx.x >> 5) << 6) | (uint32_t)bar);
                *sm.abort_flag() = 1;
            }
            __syncwarp();
            return false;
        }
    }
    return true;
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
__device__ __forceinline__ bool read_unit(const Smem &sm, uint32_t ui, const GradArgs &a, int &u)
{
    const uint32_t slot = ui & 1u;
    if (!wait_warp(sm, B_UNIT_FULL + slot, ui >> 1, a)) return false;
    u = *reinterpret_cast<volatile int *>(sm.misc() + MISC_RING + slot);
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(sm.bar(B_UNIT_EMPTY + slot));
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

// The 64 q rows starting at q row qc0 (a multiple of 64) that keep kv row
// jj, as a bit mask: the index rule gives a range [c_lo, c_hi] of them, the
// attention-mask matrix (when there is one) the bits of that row.
__device__ __forceinline__ uint64_t keep_columns(const GradArgs &a, const SeqDesc &sd, int64_t qc0, int64_t jj)
{
    if (jj >= sd.skv) return 0ull;
    int64_t lo = 0, hi = 63;
    const int64_t rows = (int64_t)sd.sq - qc0;           // valid rows from qc0 on
    if (rows - 1 < hi) hi = rows - 1;
    const MaskSpec &m = a.mask;
    if (m.mode == kRuleTopLeft) {
        lo = max(lo, jj - qc0);
    } else if (m.mode == kRuleCausal || (m.mode == kRulePrefix && jj >= sd.prefix)) {
        lo = max(lo, jj - ((int64_t)sd.skv - sd.sq) - qc0);
    } else if (m.mode == kRuleBand) {
        lo = max(lo, jj - m.next - qc0);
        hi = min(hi, jj + m.pre - qc0);
    }
    if (lo > hi) return 0ull;
    const uint64_t range = (~0ull << lo) & (~0ull >> (63 - hi));
    if (m.keep_kv == nullptr) return range;
    return range & __ldg(m.keep_kv + jj * m.words_kv + (qc0 >> 6));
}

// Dropout keep-bits of the tile, for one softmax warp: kv rows
// j0 .. j0 + 31 (one per lane) of q rows qc0 .. qc0 + 63.  The bits of one q
// row over those 32 kv rows are 32 consecutive bits of the packed mask
// (little-endian in each byte): lane L fetches them for q rows qc0 + L and
// qc0 + 32 + L (two aligned 32-bit words each, or bytes when the mask is not
// 4-byte aligned), and a warp transpose hands lane r the bit of kv row j0 + r
// for all 64 q rows.
struct KeepWin {
    uint32_t w[2][2];
    uint32_t sh[2];
};

__device__ __forceinline__ void keep_fetch(const GradArgs &a, const SeqDesc &sd, int h, int64_t qc0, int64_t j0,
                                           int lane, KeepWin &kw)
{
    const bool aligned = (reinterpret_cast<uintptr_t>(a.drop_mask) & 3) == 0;
    const uint32_t *m32 = reinterpret_cast<const uint32_t *>(a.drop_mask);
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int64_t i = qc0 + lane + 32 * rr;
        kw.w[rr][0] = kw.w[rr][1] = 0u;
        kw.sh[rr] = 0u;
        if (i >= sd.sq || j0 >= sd.skv) continue;
        const int64_t p = sd.mask_base + ((int64_t)h * sd.sq + i) * sd.skv + j0;   // first bit
        if (aligned) {
            const int64_t wi = p >> 5;
            kw.sh[rr] = (uint32_t)(p & 31);
            // the last word may reach past the mask's end: its bytes beyond
            // mask_bytes are read byte by byte
            if ((wi + 2) * 4 <= a.mask_bytes) {
                kw.w[rr][0] = __ldg(m32 + wi);
                kw.w[rr][1] = __ldg(m32 + wi + 1);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int64_t bi = wi * 4 + e;
                    const uint32_t byte = (bi < a.mask_bytes) ? a.drop_mask[bi] : 0u;
                    kw.w[rr][e >> 2] |= byte << (8 * (e & 3));
                }
            }
        } else {
            const int64_t b0 = p >> 3;
            kw.sh[rr] = (uint32_t)(p & 7);
#pragma unroll
            for (int e = 0; e < 5; ++e) {
                const int64_t bi = b0 + e;
                const uint32_t byte = (bi < a.mask_bytes) ? a.drop_mask[bi] : 0u;
                if (e < 4) kw.w[rr][0] |= byte << (8 * e);
                else kw.w[rr][1] = byte;
            }
        }
    }
}

// bit c of the result = keep-bit of (q row qc0 + c, kv row j0 + lane)
__device__ __forceinline__ uint64_t keep_transpose(const KeepWin &kw, int lane)
{
    const uint32_t win0 = __funnelshift_r(kw.w[0][0], kw.w[0][1], kw.sh[0]);
    const uint32_t win1 = __funnelshift_r(kw.w[1][0], kw.w[1][1], kw.sh[1]);
    uint32_t z0 = 0, z1 = 0;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
        z0 |= ((__shfl_sync(0xffffffffu, win0, c) >> lane) & 1u) << c;
        z1 |= ((__shfl_sync(0xffffffffu, win1, c) >> lane) & 1u) << c;
    }
    return (uint64_t)z0 | ((uint64_t)z1 << 32);
}

// Shared-memory descriptors are built once per buffer; adding (byte offset
// >> 4) to one moves its start address (the 14-bit field never overflows:
// every address is below 256 KB).
__device__ __forceinline__ uint64_t desc_at(uint64_t base_desc, uint32_t byte_off)
{
    return base_desc + (uint64_t)(byte_off >> 4);
}

// TMEM column of the k-th 16-row K slice of packed Pd^T.  The softmax
// replaces each 32-column chunk of S^T (q columns 32c .. 32c + 31) by 16
// columns of packed Pd^T followed by 16 columns of packed fp16 P^T, so slice
// kk (q columns 16kk .. 16kk + 15) sits at 32 (kk / 2) + 8 (kk % 2).
__device__ __forceinline__ uint32_t pk_col(int kk) { return (uint32_t)((kk >> 1) * 32 + (kk & 1) * 8); }

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    return BF16 ? pack_bf16(lo, hi) : pack_f16(lo, hi);
}

// pse terms (in the log2 units of C * S^T) of q rows qc .. qc + 31 for kv row
// jj of head h, 0 outside the sequence (those columns are masked anyway)
template <bool BF16>
__device__ __forceinline__ void pse_chunk(const GradArgs &a, const UnitInfo &U, int h, int64_t qc, int64_t jj, float C,
                                          float (&t)[32])
{
    using Elt = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
    if (pse_generated(a.pse)) {
        const float slope = pse_slope(a.pse, a.nq, U.b, h);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
            const int64_t i = qc + c;
            t[c] = (i < U.sd.sq && jj < U.sd.skv) ? pse_alibi(a.pse.type, slope, i, jj) * kLog2e : 0.0f;
        }
        return;
    }
    const Elt *pp = reinterpret_cast<const Elt *>(a.pse.ptr);
    const float mul = a.pse.type == 1 ? C : kLog2e;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
        const int64_t i = qc + c;
        float x = 0.0f;
        if (i < U.sd.sq && jj < U.sd.skv) {
            const Elt e = pp[pse_index(a.pse, a.nq, U.b, h, U.sd.sq, i, jj)];
            if constexpr (BF16) x = __bfloat162float(e);
            else x = __half2float(e);
        }
        t[c] = x * mul;
    }
}

// DROP = false: the kernel carries no dropout code, which keeps the compute
// warps' loop small; DROP = true applies the keep-bits when the call has them.
// PSE = true adds pseShiftOptional to the recomputed scores.
template <bool BF16, int HD, bool DROP, bool PSE>
__global__ void __launch_bounds__(kThreads, 1)
    grad_tc_kernel(const __grid_constant__ GradArgs a, const __grid_constant__ CUtensorMap tmQ,
                   const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ CUtensorMap tmDY, const __grid_constant__ CUtensorMap tmDQ)
{
    using G_ = Geo<HD>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the swizzled operand tiles need a 1024-byte aligned base; the layout
    // fills the whole allocation, so there is no room to realign
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0) set_status(a.status, TND_ERR_DEVICE_CHECK, 0x400u);
        return;
    }
    Smem sm;
    sm.base = smem_raw;
    sm.off_bar = G_::OFF_BAR;
    sm.off_misc = G_::OFF_MISC;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = a.group;
    using Out = typename std::conditional<BF16, __nv_bfloat16, __half>::type;

    if (threadIdx.x == 0) {
        mbar_init(sm.bar(B_K_FULL), 1);
        mbar_init(sm.bar(B_K_EMPTY), 1);
        mbar_init(sm.bar(B_V_FULL), 1);
        mbar_init(sm.bar(B_V_EMPTY), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(sm.bar(B_Q_FULL + i), 1);
            mbar_init(sm.bar(B_Q_EMPTY + i), 2);
            mbar_init(sm.bar(B_DY_FULL + i), 1);
            mbar_init(sm.bar(B_DY_EMPTY + i), 2);
            mbar_init(sm.bar(B_P_READY + i), 128);
            mbar_init(sm.bar(B_UNIT_FULL + i), 1);
            mbar_init(sm.bar(B_UNIT_EMPTY + i), 10);
        }
        mbar_init(sm.bar(B_S_FULL), 1);
        mbar_init(sm.bar(B_PV_DONE), 1);
        mbar_init(sm.bar(B_DP_FULL), 1);
        mbar_init(sm.bar(B_DS_READY), 256);
        mbar_init(sm.bar(B_DQ_FULL), 1);
        mbar_init(sm.bar(B_DQ_FREE), kComputeThreads);
        mbar_init(sm.bar(B_ACC_FULL), 1);
        mbar_init(sm.bar(B_ACC_FREE), kComputeThreads);
        mbar_init(sm.bar(B_DRAIN), 1);
        mbar_init(sm.bar(B_STG_FULL), kComputeThreads);
        mbar_init(sm.bar(B_STG_FULL + 1), kComputeThreads);
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
    // launched as a programmatic dependent of the prepass: the set-up above
    // overlaps its tail; its vectors and counters are read only from here on
    griddep_wait();
#ifdef TND_TRACE
    if (threadIdx.x == 0 && blockIdx.x < 1024) g_cta_span[blockIdx.x][0] = global_ns();
    uint32_t trace_n = 0;
#endif
    uint32_t drain_arm[6] = {0, 0, 0, 0, 0, 0};   // producer: phases armed per load barrier

    if (warp == 0) {
        // ================================================================ producer
        uint32_t ui = 0, ku = 0, gt = 0;
        uint32_t armed_q[2] = {0, 0}, armed_dy[2] = {0, 0}, armed_k = 0, armed_v = 0;
        int *counter = reinterpret_cast<int *>(a.status + kWorkCounter);
        bool ok = true;
        while (ok) {
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
            TRACE(EV_UNIT, (uint32_t)u);
            if (U.ntiles == 0) continue;
            const int z_kv = (int)(U.sd.tk + (int64_t)U.jb * BC);
            // V first: its buffer frees at the previous unit's last dP^T
            if (ku >= 1 && !wait_warp(sm, B_V_EMPTY, ku - 1, a)) break;
            if (lane == 0) {
                uint64_t *vb = sm.bar(B_V_FULL);
                mbar_arrive_expect_tx(vb, G_::kKvTile);
                for (uint32_t cb = 0; cb < G_::NCB; ++cb)
                    tma_load_3d(sm.base + G_::OFF_V + cb * kColBlk, &tmV, vb, 64 * cb, U.g, z_kv);
            }
            ++armed_v;
            for (int t = 0; t < U.ntiles; ++t, ++gt) {
                const int qb = U.qb_lo + t / G, h = U.g * G + t % G;
                const uint32_t s = gt & 1u, k = gt >> 1;
                const int64_t q0 = (int64_t)qb * BR;
                const int z = (int)(U.sd.tq + q0);
                if (k >= 1 && !wait_warp(sm, B_Q_EMPTY + s, k - 1, a)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    uint64_t *fb = sm.bar(B_Q_FULL + s);
                    mbar_arrive_expect_tx(fb, G_::kQTile + G_::kVecBytes);
                    uint8_t *qt = sm.base + G_::OFF_Q + s * G_::kQTile;
                    for (uint32_t cb = 0; cb < G_::NCB; ++cb) tma_load_3d(qt + cb * kColBlk, &tmQ, fb, 64 * cb, h, z);
                    const int64_t vidx = ((int64_t)(U.sd.qblk0 + qb) * a.nq + h) * BR;
                    uint8_t *vec = sm.base + G_::OFF_VEC + s * G_::kVecBytes;
                    bulk_g2s(vec, a.lse2 + vidx, BR * 4, fb);
                    bulk_g2s(vec + BR * 4, a.drow + vidx, BR * 4, fb);
                }
                ++armed_q[s];
                TRACE(EV_L_Q, gt);
                if (k >= 1 && !wait_warp(sm, B_DY_EMPTY + s, k - 1, a)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    uint64_t *fb = sm.bar(B_DY_FULL + s);
                    mbar_arrive_expect_tx(fb, G_::kQTile);
                    uint8_t *dyt = sm.base + G_::OFF_DY + s * G_::kQTile;
                    for (uint32_t cb = 0; cb < G_::NCB; ++cb)
                        tma_load_3d(dyt + cb * kColBlk, &tmDY, fb, 64 * cb, h, z);
                }
                ++armed_dy[s];
                TRACE(EV_L_DY, gt);
                if (t == 0) {
                    // K after the unit's first Q / dY: its buffer frees when the
                    // previous unit's last dQ^T completes
                    if (ku >= 1 && !wait_warp(sm, B_K_EMPTY, ku - 1, a)) {
                        ok = false;
                        break;
                    }
                    // test hook: CTA 0 never loads its first K tile, so the
                    // UMMA issuer's bounded wait for it runs out
                    const bool skip = (a.test_flags & 1) && blockIdx.x == 0 && ku == 0;
                    if (lane == 0 && !skip) {
                        uint64_t *kb = sm.bar(B_K_FULL);
                        mbar_arrive_expect_tx(kb, G_::kKvTile);
                        for (uint32_t cb = 0; cb < G_::NCB; ++cb)
                            tma_load_3d(sm.base + G_::OFF_K + cb * kColBlk, &tmK, kb, 64 * cb, U.g, z_kv);
                    }
                    if (!skip) ++armed_k;
                    TRACE(EV_L_K, gt);
                }
            }
            ++ku;
        }
        drain_arm[0] = armed_q[0];
        drain_arm[1] = armed_q[1];
        drain_arm[2] = armed_dy[0];
        drain_arm[3] = armed_dy[1];
        drain_arm[4] = armed_k;
        drain_arm[5] = armed_v;
        __syncwarp();
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        {
            const uint32_t idS = instr_desc_f16(BF16, 128, BR, false, false);     // S^T, dP^T
            const uint32_t idKV = instr_desc_f16(BF16, 128, HD, false, true);     // dV (A in TMEM), dK
            const uint32_t idQ = instr_desc_f16(BF16, 128, BR, true, true);       // dQ^T
            const uint32_t sbase = smem_u32(sm.base);
            // K-major views (S^T, dP^T and dK's A) and MN-major views (B of
            // dV / dK, both operands of dQ^T)
            const uint64_t dK_k = smem_desc_sw128(sbase + G_::OFF_K, 16, 1024);
            const uint64_t dK_m = smem_desc_sw128(sbase + G_::OFF_K, kColBlk, 1024);
            const uint64_t dV_k = smem_desc_sw128(sbase + G_::OFF_V, 16, 1024);
            const uint64_t dQ_k0 = smem_desc_sw128(sbase + G_::OFF_Q, 16, 1024);
            const uint64_t dQ_m0 = smem_desc_sw128(sbase + G_::OFF_Q, kColBlk, 1024);
            const uint64_t dY_k0 = smem_desc_sw128(sbase + G_::OFF_DY, 16, 1024);
            const uint64_t dY_m0 = smem_desc_sw128(sbase + G_::OFF_DY, kColBlk, 1024);
            const uint64_t dS_k = smem_desc_sw128(sbase + G_::OFF_DS, 16, 1024);
            const uint64_t dS_m = smem_desc_sw128(sbase + G_::OFF_DS, kColBlk, 1024);
            constexpr int KS = HD / 16;     // K steps of S^T / dP^T
            uint32_t ui = 0, ku = 0, gt = 0;
            bool ok = true;
            // S^T(t) = K Q(t)^T into the S buffer: dV(t - 1) has read Pd^T(t - 1)
            // (PV_DONE) and the compute warps have read P^T(t - 1) (their
            // DS_READY(t - 1), awaited before)
            auto issue_s = [&](uint32_t g, bool first) -> bool {
                const uint32_t s = g & 1u;
                if (!wait_uni(sm, B_Q_FULL + s, g >> 1, a)) return false;
                TRACE(EV_W_QFULL, g);
                if (g >= 1 && !wait_uni(sm, B_PV_DONE, g - 1, a)) return false;
                TRACE(EV_W_PVDONE, g);
                if (first && !wait_uni(sm, B_K_FULL, ku, a)) return false;
                TRACE(EV_W_KFULL, g);
                tc_fence_after();
                const uint64_t dq = desc_at(dQ_k0, s * G_::kQTile);
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    const uint32_t off = (kk >> 2) * kColBlk + (kk & 3) * 32;
                    mma_ss_elect(tmem + TM_S, desc_at(dK_k, off), desc_at(dq, off), idS, kk > 0);
                }
                mma_commit_elect(sm.bar(B_S_FULL));
                TRACE(EV_I_S, g);
                return true;
            };
            // dP^T(t) = V dY(t)^T into the dP buffer once the compute warps have
            // read dQ^T(t - 1) out of it
            auto issue_dp = [&](uint32_t g, bool first) -> bool {
                const uint32_t s = g & 1u;
                if (!wait_uni(sm, B_DY_FULL + s, g >> 1, a)) return false;
                TRACE(EV_W_DYFULL, g);
                if (g >= 1 && !wait_uni(sm, B_DQ_FREE, g - 1, a)) return false;
                TRACE(EV_W_DQFREE, g);
                if (first && !wait_uni(sm, B_V_FULL, ku, a)) return false;
                TRACE(EV_W_VFULL, g);
                tc_fence_after();
                const uint64_t dy = desc_at(dY_k0, s * G_::kQTile);
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    const uint32_t off = (kk >> 2) * kColBlk + (kk & 3) * 32;
                    mma_ss_elect(tmem + TM_DP, desc_at(dV_k, off), desc_at(dy, off), idS, kk > 0);
                }
                mma_commit_elect(sm.bar(B_DP_FULL));
                TRACE(EV_I_DP, g);
                return true;
            };
            // Per tile t: dV(t) once P^T(t) is in; dK(t) and dQ^T(t) once dS^T(t)
            // is; then S^T(t + 1) and, once the epilogue has read dQ^T(t) out of
            // the dP buffer, dP^T(t + 1).  A unit's first S^T / dP^T come before
            // its loop.
            while (ok) {
                int u;
                if (!read_unit(sm, ui, a, u)) break;
                ++ui;
                if (u < 0) break;
                const UnitInfo U = unit_info(a, u);
                if (U.ntiles == 0) continue;
                const uint32_t g0 = gt, g_end = gt + (uint32_t)U.ntiles;
                // V arrives before K (K waits for the previous unit's last dQ^T)
                if (!issue_dp(g0, true) || !issue_s(g0, true)) break;
                for (uint32_t g = g0; g < g_end; ++g) {
                    const uint32_t s = g & 1u;
                    const bool first = g == g0;
                    if (first && ku >= 1 && !wait_uni(sm, B_ACC_FREE, ku - 1, a)) {
                        ok = false;
                        break;
                    }
                    TRACE(EV_W_ACCFREE, g);
                    // dV += Pd^T dY(t): A = Pd^T (TMEM, packed), B = dY MN-major (N = HD);
                    // the two K halves follow the two softmax halves.  dY(t) is in:
                    // dP^T(t) was issued after its DY_FULL.
                    const uint64_t dym = desc_at(dY_m0, s * G_::kQTile);
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        if (!wait_uni(sm, B_P_READY + hf, g, a)) {
                            ok = false;
                            break;
                        }
                        TRACE(EV_W_P0 + hf, g);
                        tc_fence_after();
#pragma unroll
                        for (int kq = 0; kq < 4; ++kq) {
                            const int kk = 4 * hf + kq;
                            mma_ts_elect(tmem + 0, tmem + TM_S + pk_col(kk), desc_at(dym, kk * 2048), idKV,
                                         (!first || kk > 0));
                        }
                    }
                    if (!ok) break;
                    mma_commit_elect(sm.bar(B_PV_DONE));
                    mma_commit_elect(sm.bar(B_DY_EMPTY + s));      // dP^T(t) and dV(t) issued: dY(t)'s readers
                    if (g + 1 == g_end) mma_commit_elect(sm.bar(B_V_EMPTY));   // the unit's last dP^T issued
                    TRACE(EV_I_DV, g);
                    if (!wait_uni(sm, B_DS_READY, g, a)) {
                        ok = false;
                        break;
                    }
                    TRACE(EV_W_DS, g);
                    tc_fence_after();
                    // dK += dS^T Q(t): A = dS^T smem K-major, B = Q MN-major
                    const uint64_t dqm = desc_at(dQ_m0, s * G_::kQTile);
#pragma unroll
                    for (int kk = 0; kk < BR / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * kColBlk + (kk & 3) * 32;
                        mma_ss_elect(tmem + HD, desc_at(dS_k, off), desc_at(dqm, kk * 2048), idKV, (!first || kk > 0));
                    }
                    mma_commit_elect(sm.bar(B_Q_EMPTY + s));
                    TRACE(EV_I_DK, g);
                    // dQ^T = K^T dS^T into the dP buffer (the compute warps have read
                    // dP^T(t)): A = K MN-major (M = 128 features), B = dS^T MN-major
#pragma unroll
                    for (int kk = 0; kk < BC / 16; ++kk) {
                        mma_ss_elect(tmem + TM_DP, desc_at(dK_m, kk * 2048), desc_at(dS_m, kk * 2048), idQ, kk > 0);
                    }
                    mma_commit_elect(sm.bar(B_DQ_FULL));
                    TRACE(EV_I_DQ, g);
                    if (g + 1 == g_end) {
                        mma_commit_elect(sm.bar(B_ACC_FULL));
                        mma_commit_elect(sm.bar(B_K_EMPTY));
                    } else if (!issue_s(g + 1, false) || !issue_dp(g + 1, false)) {
                        ok = false;
                        break;
                    }
                }
                if (!ok) break;
                gt = g_end;
                ++ku;
            }
            // every issued UMMA must finish before TMEM is released
            mma_commit_elect(sm.bar(B_DRAIN));
            const long long t0 = clock64();
            while (!mbar_try_wait(sm.bar(B_DRAIN), 0) && clock64() - t0 < a.wait_limit_cycles) {
            }
        }
        __syncwarp();
    } else if (warp < kWriterWarp) {
        // ================================================================ compute warps
        // Two warps per TMEM lane quarter: warps 2-5 take q columns 0-63 of
        // the tile, warps 6-9 columns 64-127 (the same split serves dQ^T,
        // whose TMEM columns are q rows, and dK / dV, whose columns are
        // features).  Per tile t: P^T(t); dS^T(t); the epilogue of tile t.
        const int quarter = warp & 3;
        const int half = (warp - kComputeWarp0) >> 2;
        const int ln = quarter * 32 + lane;                 // TMEM lane: kv row (S^T, dP^T, dK, dV) or feature (dQ^T)
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const float C = a.scale * kLog2e;
        Out *dK = reinterpret_cast<Out *>(a.dk);
        Out *dV = reinterpret_cast<Out *>(a.dv);
        uint32_t ui = 0, ku = 0, gt = 0;
        bool ok = true;
        // dK, dV of a unit (x scale for dK) out of TMEM; thread = kv row,
        // columns [half * HD / 2, (half + 1) * HD / 2)
        auto unit_out = [&](const UnitInfo &U, bool zeros) -> bool {
            const int64_t jj = (int64_t)U.jb * BC + ln;
            const bool row_ok = jj < U.sd.skv;
            const int64_t kv_off = ((U.sd.tk + jj) * a.nkv + U.g) * (int64_t)HD + half * (HD / 2);
            if (zeros) {
                if (row_ok) {
                    for (int c = 0; c < HD / 2; c += 8) {
                        *reinterpret_cast<uint4 *>(dK + kv_off + c) = make_uint4(0, 0, 0, 0);
                        *reinterpret_cast<uint4 *>(dV + kv_off + c) = make_uint4(0, 0, 0, 0);
                    }
                }
                return true;
            }
            if (!wait_warp(sm, B_ACC_FULL, ku, a)) return false;
            tc_fence_after();
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                const uint32_t col0 = (which == 0 ? 0u : (uint32_t)HD) + half * (HD / 2);
                const float mul = which == 0 ? 1.0f : a.scale;
                Out *dst = (which == 0 ? dV : dK) + kv_off;
#pragma unroll
                for (int chunk = 0; chunk < HD / 64; ++chunk) {
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
            return true;
        };
        // Epilogue of tile g: dQ^T out of TMEM (thread = feature ln, q rows
        // 64 half .. + 63), the dP buffer released, the unit's dK / dV out if
        // g ends its unit, then dQ^T staged as fp32 [64 q rows][HD] for the
        // writer warp: rows 0-63 of the tile in its dY stage, rows 64-127 in
        // its Q stage.  DQ_FULL(g) follows dV(g), dP^T(g), dK(g) and dQ^T(g):
        // every reader of both stages and of the dS^T buffer is done.
        auto epilogue = [&](uint32_t g, const UnitInfo &U, bool last) -> bool {
            if (!wait_warp(sm, B_DQ_FULL, g, a)) return false;
            TRACE(EV_C_DQFULL, g);
            tc_fence_after();
            // both 32-column halves loaded together; the dP buffer is released
            // as soon as they are in registers
            const uint32_t s = g & 1u;
            const uint32_t dq_addr = tmem + lane_addr + TM_DP + 64 * half;
            float *stg = reinterpret_cast<float *>(sm.base + (half == 0 ? G_::OFF_DY : G_::OFF_Q) + s * G_::kQTile) + ln;
            uint32_t v0[32], v1[32];
            tmem_ld32_async(dq_addr, v0);
            tmem_ld32_async(dq_addr + 32, v1);
            tmem_wait_ld32(v0);
            tmem_wait_ld32(v1);
            tc_fence_before();
            mbar_arrive(sm.bar(B_DQ_FREE));
            TRACE(EV_C_DQFREE, g);
            if (ln < HD) {
#pragma unroll
                for (int c = 0; c < 32; ++c) stg[c * HD] = __uint_as_float(v0[c]);
#pragma unroll
                for (int c = 0; c < 32; ++c) stg[(32 + c) * HD] = __uint_as_float(v1[c]);
            }
            if (last && !unit_out(U, false)) return false;
            fence_async_smem();
            mbar_arrive(sm.bar(B_STG_FULL + s));
            TRACE(EV_C_EPIDONE, g);
            return true;
        };
        while (ok) {
            int u;
            if (!read_unit(sm, ui, a, u)) break;
            ++ui;
            if (u < 0) break;
            const UnitInfo U = unit_info(a, u);
            if (U.ntiles == 0) {
                unit_out(U, true);
                continue;
            }
            for (int t = 0; t < U.ntiles; ++t, ++gt) {
                const int qb = U.qb_lo + t / G, h = U.g * G + t % G;
                const uint32_t s = gt & 1u;
                const int64_t qc0 = (int64_t)qb * BR + 64 * half;
                const int64_t jj = (int64_t)U.jb * BC + ln;
                const uint64_t keep = keep_columns(a, U.sd, qc0, jj);
                const bool full = __all_sync(0xffffffffu, keep == ~0ull);
                KeepWin kw;
                if (DROP && a.has_drop) keep_fetch(a, U.sd, h, qc0, (int64_t)U.jb * BC + quarter * 32, lane, kw);
                if (!wait_warp(sm, B_Q_FULL + s, gt >> 1, a) || !wait_warp(sm, B_S_FULL, gt, a)) {
                    ok = false;
                    break;
                }
                TRACE(EV_C_SFULL, gt);
                tc_fence_after();
                const float *vec = reinterpret_cast<const float *>(sm.base + G_::OFF_VEC + s * G_::kVecBytes);
                const float4 *lse4 = reinterpret_cast<const float4 *>(vec) + 16 * half;
                const float4 *dvec4 = reinterpret_cast<const float4 *>(vec + BR) + 16 * half;
                const uint64_t zb = (DROP && a.has_drop) ? keep_transpose(kw, lane) : ~0ull;
                // ---- phase 1: P^T from S^T, kept in registers (fp32) for dS; each
                // 32-column chunk of S^T gets Pd^T = P^T o z packed in the dtype in
                // its first 16 columns (the dV operand)
                const uint32_t s_addr = tmem + lane_addr + TM_S + 64 * half;
                float p[64];
                const float cs = PSE ? 1.0f : C;      // with a pse, raw already holds C S^T + pse term
#pragma unroll
                for (int ch = 0; ch < 2; ++ch) {
                    uint32_t raw[32];
                    tmem_ld32(s_addr + 32 * ch, raw);
                    if constexpr (PSE) {
                        float t[32];
                        pse_chunk<BF16>(a, U, h, qc0 + 32 * ch, jj, C, t);
#pragma unroll
                        for (int c = 0; c < 32; ++c) raw[c] = __float_as_uint(fmaf(__uint_as_float(raw[c]), C, t[c]));
                    }
#pragma unroll
                    for (int c4 = 0; c4 < 8; ++c4) {
                        const float4 l = lse4[8 * ch + c4];
                        p[32 * ch + 4 * c4 + 0] = ex2(fmaf(__uint_as_float(raw[4 * c4 + 0]), cs, -l.x));
                        p[32 * ch + 4 * c4 + 1] = ex2(fmaf(__uint_as_float(raw[4 * c4 + 1]), cs, -l.y));
                        p[32 * ch + 4 * c4 + 2] = ex2(fmaf(__uint_as_float(raw[4 * c4 + 2]), cs, -l.z));
                        p[32 * ch + 4 * c4 + 3] = ex2(fmaf(__uint_as_float(raw[4 * c4 + 3]), cs, -l.w));
                    }
                    if (!full) {
                        const uint32_t kh = (uint32_t)(keep >> (32 * ch));
#pragma unroll
                        for (int c = 0; c < 32; ++c) p[32 * ch + c] = ((kh >> c) & 1u) ? p[32 * ch + c] : 0.0f;
                    }
                    uint32_t pk[16];
                    if (DROP && a.has_drop) {
                        const uint32_t zh = (uint32_t)(zb >> (32 * ch));
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            const float z0 = ((zh >> (2 * c)) & 1u) ? a.inv_keep : 0.0f;
                            const float z1 = ((zh >> (2 * c + 1)) & 1u) ? a.inv_keep : 0.0f;
                            pk[c] = pack2<BF16>(p[32 * ch + 2 * c] * z0, p[32 * ch + 2 * c + 1] * z1);
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < 16; ++c) pk[c] = pack2<BF16>(p[32 * ch + 2 * c], p[32 * ch + 2 * c + 1]);
                    }
                    tmem_st16(s_addr + 32 * ch, pk);   // only this chunk's own, already read, columns
                }
                tc_fence_before();
                mbar_arrive(sm.bar(B_P_READY + half));
                TRACE(EV_C_PDONE, gt);
                // ---- phase 2: dS^T = P^T o (z dP^T - D) (P^T from registers: Pd^T is 0
                // where dropout drops a key) into registers, then into the
                // shared-memory dS^T buffer (dK(t - 1) and dQ^T(t - 1) have read it:
                // the epilogue of t - 1 waited for DQ_FULL(t - 1)).
                if (!wait_warp(sm, B_DP_FULL, gt, a)) {
                    ok = false;
                    break;
                }
                TRACE(EV_C_DPFULL, gt);
                tc_fence_after();
                const uint32_t dp_addr = tmem + lane_addr + TM_DP + 64 * half;
                uint32_t dsk[32];
#pragma unroll
                for (int ch = 0; ch < 2; ++ch) {
                    uint32_t raw[32];
                    tmem_ld32(dp_addr + 32 * ch, raw);
                    const uint32_t zh = (uint32_t)(zb >> (32 * ch));
#pragma unroll
                    for (int c4 = 0; c4 < 8; ++c4) {
                        const float4 dv = dvec4[8 * ch + c4];
                        float dp[4] = {__uint_as_float(raw[4 * c4]), __uint_as_float(raw[4 * c4 + 1]),
                                       __uint_as_float(raw[4 * c4 + 2]), __uint_as_float(raw[4 * c4 + 3])};
                        if (DROP && a.has_drop) {
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                dp[e] = ((zh >> (4 * c4 + e)) & 1u) ? dp[e] * a.inv_keep : 0.0f;
                        }
                        const float *pc = p + 32 * ch + 4 * c4;
                        dsk[16 * ch + 2 * c4] = pack2<BF16>(pc[0] * (dp[0] - dv.x), pc[1] * (dp[1] - dv.y));
                        dsk[16 * ch + 2 * c4 + 1] = pack2<BF16>(pc[2] * (dp[2] - dv.z), pc[3] * (dp[3] - dv.w));
                    }
                }
                uint8_t *row = sm.base + G_::OFF_DS + half * kColBlk + ln * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 v = make_uint4(dsk[4 * c], dsk[4 * c + 1], dsk[4 * c + 2], dsk[4 * c + 3]);
                    *reinterpret_cast<uint4 *>(row + ((c ^ (ln & 7)) << 4)) = v;
                }
                fence_async_smem();
                tc_fence_before();
                mbar_arrive(sm.bar(B_DS_READY));
                TRACE(EV_C_DSDONE, gt);
                if (!epilogue(gt, U, t + 1 == U.ntiles)) {
                    ok = false;
                    break;
                }
            }
        }
    } else {
        // ================================================================ dQ writer
        // For each tile, in order: once the compute warps have staged dQ^T,
        // waits until the (q block, head) counter shows that every earlier
        // contributor's update is complete, then stores (first contributor)
        // or adds (later ones) the two staged 64-row halves into the fp32
        // accumulator with TMA, releases the tile's Q and dY stages to the
        // producer as each half has been read, and advances the counter once
        // the writes are complete.
        if (lane == 0) {
            uint32_t ui = 0, gt = 0;
            bool ok = true;
            // counter release owed for the last issued tile.  In chain order
            // it is settled at once (a later release holds up the next
            // contributor: measured slower).  In arrival order only first
            // contributors release, and their writes are waited for once the
            // next tile is issued, as long as the writer has a staged tile
            // and a ready chain to go on with; before any wait the release is
            // settled, so the writer never waits while holding back a
            // counter another CTA may wait on
            int *owed = nullptr;
            int owed_val = 0;
            auto settle = [&]() {
                if (owed) {
                    bulk_wait0();
                    fence_async_global();
                    fence_acq_rel_gpu();
                    st_relaxed_gpu(owed, owed_val);
                    owed = nullptr;
                }
            };
            while (ok) {
                int u;
                if (!mbar_test_wait(sm.bar(B_UNIT_FULL + (ui & 1u)), (ui >> 1) & 1u)) settle();
                if (!read_unit1(sm, ui, a, u)) break;
                ++ui;
                if (u < 0) break;
                const UnitInfo U = unit_info(a, u);
                for (int t = 0; t < U.ntiles; ++t, ++gt) {
                    const int qb = U.qb_lo + t / G, h = U.g * G + t % G;
                    const int qg = U.sd.qblk0 + qb;
                    const QBlockInfo qi = a.qblk[qg];
                    int *flag = a.flags + (int64_t)qg * a.nq + h;
                    const int pos = qi.jhi - U.jb;
                    const uint32_t s = gt & 1u;
                    if (!mbar_test_wait(sm.bar(B_STG_FULL + s), (gt >> 1) & 1u)) {
                        settle();
                        if (!wait_k(sm, B_STG_FULL + s, gt >> 1, a)) {
                            ok = false;
                            break;
                        }
                    }
                    TRACE(EV_W_STG, gt);
                    // ordered: every earlier contributor's update is complete;
                    // arrival order: the first contributor's store is
                    const int need = a.deterministic ? pos : min(pos, 1);
                    if (need > 0) {
                        if (ld_acquire_gpu(flag) < need) {
                            settle();
                            const long long t0 = clock64();
                            while (ld_acquire_gpu(flag) < need) {
                                if (*sm.abort_flag()) {
                                    ok = false;
                                    break;
                                }
                                if (clock64() - t0 > a.wait_limit_cycles) {
                                    // detail: the awaited position and the (q block, head) counter
                                    set_status(a.status, TND_ERR_DEVICE_TIMEOUT,
                                               0x80000000u | ((uint32_t)pos << 24) | (uint32_t)(qg * a.nq + h));
                                    *sm.abort_flag() = 1;
                                    ok = false;
                                    break;
                                }
                                __nanosleep(32);
                            }
                            if (!ok) break;
                        }
                        fence_async_global();   // the counter's acquire before the async-proxy adds
                    }
                    TRACE(EV_W_CHAIN, gt);
                    const int z = (int)(U.sd.tq + (int64_t)qb * BR);
                    // the half staged in the Q stage first, as its own bulk group:
                    // the next Q load (needed sooner than the next dY) waits for it
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const int hs = 1 - i;
                        const uint8_t *stg = sm.base + (hs == 0 ? G_::OFF_DY : G_::OFF_Q) + s * G_::kQTile;
                        const int64_t r0 = (int64_t)qb * BR + 64 * hs;
                        const int rows = (int)max((int64_t)0, min((int64_t)64, (int64_t)U.sd.sq - r0));
                        if (rows == 64) {
                            if (pos == 0) tma_store_3d(&tmDQ, stg, 0, h, z + 64 * hs);
                            else tma_reduce_add_3d(&tmDQ, stg, 0, h, z + 64 * hs);
                        } else {
                            // ragged last block of a sequence: only its own rows
                            for (int r = 0; r < rows; ++r) {
                                float *dst = a.dqacc + ((U.sd.tq + r0 + r) * a.nq + h) * (int64_t)HD;
                                if (pos == 0) bulk_s2g(dst, stg + r * HD * 4, HD * 4);
                                else bulk_reduce_add_f32(dst, stg + r * HD * 4, HD * 4);
                            }
                        }
                        bulk_commit();
                    }
                    TRACE(EV_W_ISSUED, gt);
                    if (owed) {
                        // every group but this tile's two: the previous tile's writes
                        bulk_wait2();
                        fence_async_global();
                        fence_acq_rel_gpu();
                        st_relaxed_gpu(owed, owed_val);
                        owed = nullptr;
                    }
                    bulk_wait_read1();                              // the Q-stage half
                    mbar_arrive(sm.bar(B_Q_EMPTY + s));
                    bulk_wait_read0();                              // the dY-stage half
                    mbar_arrive(sm.bar(B_DY_EMPTY + s));
                    TRACE(EV_W_READ, gt);
                    if (a.deterministic || pos == 0) {
                        owed = flag;
                        owed_val = pos + 1;
                        if (a.deterministic) settle();
                    }
                    TRACE(EV_W_WRITTEN, gt);
                }
            }
            settle();
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
#ifdef TND_TRACE
    if (threadIdx.x == 0 && blockIdx.x < 1024) g_cta_span[blockIdx.x][1] = global_ns();
    if ((threadIdx.x & 31) == 0 && blockIdx.x < kTraceCtas) g_trace_n[blockIdx.x][threadIdx.x >> 5] = trace_n;
#endif
    griddep_launch_dependents();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    // after an abort, TMA loads whose data nobody waited for may still be in
    // flight: they must land before the CTA's shared memory is released
    if (warp == 0 && lane == 0 && *sm.abort_flag()) {
        const int bars[6] = {B_Q_FULL, B_Q_FULL + 1, B_DY_FULL, B_DY_FULL + 1, B_K_FULL, B_V_FULL};
#pragma unroll
        for (int i = 0; i < 6; ++i)
            if (drain_arm[i]) drain_k(sm, bars[i], drain_arm[i] - 1, a);
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

// [rows, heads, hd] tensor of 16-bit elements, boxes of 64 features x 1 head x `box_rows` rows
bool make_map(CUtensorMap *m, const void *ptr, int64_t rows, int64_t heads, int hd, int box_rows, bool bf16)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)hd, (cuuint64_t)heads, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)hd * 2, (cuuint64_t)(heads * hd * 2)};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                    const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// dQ accumulator [rows, heads, hd] fp32, boxes of hd features x 1 head x 64 rows (no swizzle)
bool make_acc_map(CUtensorMap *m, const float *ptr, int64_t rows, int64_t heads, int hd)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)hd, (cuuint64_t)heads, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)hd * 4, (cuuint64_t)(heads * hd * 4)};
    cuuint32_t box[3] = {(cuuint32_t)hd, 1, 64};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <bool BF16, int HD, bool DROP, bool PSE>
cudaError_t launch_hd(const GradArgs &a, cudaStream_t s)
{
    CUtensorMap mq, mk, mv, mdy, mdq;
    if (!make_map(&mq, a.q, a.tq, a.nq, HD, BR, BF16) || !make_map(&mk, a.k, a.tkv, a.nkv, HD, BC, BF16) ||
        !make_map(&mv, a.v, a.tkv, a.nkv, HD, BC, BF16) || !make_map(&mdy, a.dy, a.tq, a.nq, HD, BR, BF16) ||
        !make_acc_map(&mdq, a.dqacc, a.tq, a.nq, HD))
        return cudaErrorInvalidValue;
    const int grid = std::min<int>(a.num_sms, a.n_units);
    constexpr uint32_t smem = Geo<HD>::kSmemBytes;
    cudaError_t e =
        cudaFuncSetAttribute(grad_tc_kernel<BF16, HD, DROP, PSE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_dependent(grad_tc_kernel<BF16, HD, DROP, PSE>, dim3(grid), dim3(kThreads), smem, s, a, mq, mk, mv,
                            mdy, mdq);
}

// dQ = scale * accumulator in the output dtype, one block per (128-row q
// block, head) with heads in x (blocks running together cover neighbouring
// pieces of the same rows); rows of q blocks that no kv block reaches get
// zeros.  Thread t takes float4 column t % (HD / 4) of every (256 / (HD / 4))-th
// row, four rows' loads in flight before their stores, eight blocks per SM.
template <typename Out, int HD>
__global__ void __launch_bounds__(256, 8) dq_finalize_kernel(GradArgs a)
{
    constexpr int kF4 = HD / 4;                 // float4 per row
    constexpr int kRowStep = 256 / kF4;         // rows per pass of the block
    constexpr int kBatch = 4;
    const int h = blockIdx.x, qg = blockIdx.y;
    griddep_wait();   // programmatic dependent of the gradient kernel
    const int2 qr = a.qblk_rows[qg];
    const SeqDesc sd = a.seqs[qr.x];
    const bool covered = a.qblk[qg].jlo >= 0;
    const int rows = min(BR, sd.sq - qr.y);
    const int c4 = threadIdx.x % kF4, r0 = threadIdx.x / kF4;
    const int64_t stride = (int64_t)a.nq * HD;                  // elements between consecutive rows
    const int64_t base = ((sd.tq + qr.y + r0) * a.nq + h) * (int64_t)HD + 4 * c4;
    Out *dQ = reinterpret_cast<Out *>(a.dq);
    for (int rb = 0; rb < BR; rb += kBatch * kRowStep) {
        float4 v[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int r = r0 + rb + k * kRowStep;
            v[k] = (covered && r < rows) ? __ldcs(reinterpret_cast<const float4 *>(a.dqacc + base + (rb + k * kRowStep) * stride))
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int r = r0 + rb + k * kRowStep;
            if (r >= rows) break;
            uint2 pk;
            pk.x = pack2<std::is_same<Out, __nv_bfloat16>::value>(v[k].x * a.scale, v[k].y * a.scale);
            pk.y = pack2<std::is_same<Out, __nv_bfloat16>::value>(v[k].z * a.scale, v[k].w * a.scale);
            *reinterpret_cast<uint2 *>(dQ + base + (rb + k * kRowStep) * stride) = pk;
        }
    }
}

}  // namespace

bool grad_tc_supported(int dtype, int d) { return (dtype == TND_BF16 || dtype == TND_F16) && (d == 64 || d == 128); }

cudaError_t launch_grad_tc(const GradArgs &a, cudaStream_t s)
{
    if (a.n_units == 0) return cudaSuccess;
    const bool bf16 = a.dtype == TND_BF16;
    const bool drop = a.has_drop != 0;
    if (a.pse.ptr) {
        // with a pse: the dropout-capable instances (keep-bits applied when the call has them)
        if (a.d == 128) return bf16 ? launch_hd<true, 128, true, true>(a, s) : launch_hd<false, 128, true, true>(a, s);
        if (a.d == 64) return bf16 ? launch_hd<true, 64, true, true>(a, s) : launch_hd<false, 64, true, true>(a, s);
        return cudaErrorInvalidValue;
    }
    if (a.d == 128) {
        if (bf16) return drop ? launch_hd<true, 128, true, false>(a, s) : launch_hd<true, 128, false, false>(a, s);
        return drop ? launch_hd<false, 128, true, false>(a, s) : launch_hd<false, 128, false, false>(a, s);
    }
    if (a.d == 64) {
        if (bf16) return drop ? launch_hd<true, 64, true, false>(a, s) : launch_hd<true, 64, false, false>(a, s);
        return drop ? launch_hd<false, 64, true, false>(a, s) : launch_hd<false, 64, false, false>(a, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_dq_finalize(const GradArgs &a, cudaStream_t s)
{
    if (a.n_qblk == 0) return cudaSuccess;
    const dim3 grid((unsigned)a.nq, (unsigned)a.n_qblk);
    const bool bf16 = a.dtype == TND_BF16;
    if (a.d == 128)
        return bf16 ? launch_dependent(dq_finalize_kernel<__nv_bfloat16, 128>, grid, dim3(256), 0, s, a)
                    : launch_dependent(dq_finalize_kernel<__half, 128>, grid, dim3(256), 0, s, a);
    return bf16 ? launch_dependent(dq_finalize_kernel<__nv_bfloat16, 64>, grid, dim3(256), 0, s, a)
                : launch_dependent(dq_finalize_kernel<__half, 64>, grid, dim3(256), 0, s, a);
}

}  // namespace tnd

#ifdef TND_TRACE
// Diagnostic build only: copies the event log out (and clears it).
extern "C" int tnd_debug_trace(unsigned long long *events, unsigned int *counts, unsigned long long *spans)
{
    using namespace tnd;
    if (cudaMemcpyFromSymbol(events, g_trace, sizeof(g_trace)) != cudaSuccess) return 1;
    if (cudaMemcpyFromSymbol(counts, g_trace_n, sizeof(g_trace_n)) != cudaSuccess) return 1;
    if (cudaMemcpyFromSymbol(spans, g_cta_span, sizeof(g_cta_span)) != cudaSuccess) return 1;
    static unsigned int zero[kTraceCtas][11] = {};
    return cudaMemcpyToSymbol(g_trace_n, zero, sizeof(zero)) != cudaSuccess;
}
#endif
