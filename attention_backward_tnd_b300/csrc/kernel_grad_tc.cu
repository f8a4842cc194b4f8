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
// Warp roles (512 threads, one CTA per SM, persistent over work units taken
// in plan order from a counter):
//   warp 0      TMA producer: K and V (one buffer each) per unit,
//               Q / dY and the tile's lse2 / D vectors per tile, dropout
//               keep-bits staged in shared memory
//   warp 1      TMEM allocator and single-thread UMMA issuer
//   warps 2-9   softmax-gradient warps: thread = TMEM lane = kv row, two
//               warps per lane quarter, each on 32 of the tile's 64 q columns
//   warps 10-13 epilogue: dQ^T tile TMEM -> shared staging (thread = feature),
//               dK / dV TMEM -> global (thread = kv row) at unit end
//   warp 14     dQ writer: orders and issues the accumulator updates
//   warp 15     counter releases of completed accumulator updates
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
constexpr int NSTAGE = 3;               // Q / dY ring depth
constexpr int kThreads = 512;
constexpr int kSoftmaxWarp0 = 2;        // warps 2-9 (two per TMEM lane quarter)
constexpr int kEpilogueWarp0 = 10;      // warps 10-13
constexpr int kWriterWarp = 14;
constexpr int kReleaseWarp = 15;
constexpr uint32_t kRelRing = 32;       // release queue entries
constexpr uint32_t kTmemCols = 512;

// TMEM columns.  Two 64-column S buffers hold, per tile, S^T (fp32), then
// P^T packed in place, then the tile's dQ^T (fp32) once dV has read P^T.
// Two 64-column dP buffers hold dP^T, then dS^T packed in place.
constexpr uint32_t TM_DV = 0, TM_DK = 128, TM_S0 = 256, TM_DP0 = 384;

// shared memory layout (offsets from a 1024-byte aligned base)
constexpr uint32_t kKvTile = BC * HD * 2;     // 32768: two 64-column blocks of 128 rows x 128 B
constexpr uint32_t kKvColBlk = BC * 128;      // 16384
constexpr uint32_t kQTile = BR * HD * 2;      // 16384: two 64-column blocks of 64 rows x 128 B
constexpr uint32_t kQColBlk = BR * 128;       // 8192
constexpr uint32_t kStgBytes = BR * HD * 2;   // 16384: half a dQ tile, fp32 [32 rows][128 features]
constexpr uint32_t kDsBytes = BC * 128;       // 16384: dS^T, 128 kv rows x 64 q (bf16 / fp16)
constexpr uint32_t kVecBytes = 2 * BR * 4;    // per stage: lse2[64], D[64]
constexpr uint32_t OFF_K = 0;                                 // 1 buffer
constexpr uint32_t OFF_V = OFF_K + kKvTile;                   // 1 buffer
constexpr uint32_t OFF_Q = OFF_V + kKvTile;
constexpr uint32_t OFF_DY = OFF_Q + NSTAGE * kQTile;
constexpr uint32_t OFF_DS = OFF_DY + NSTAGE * kQTile;         // 1 buffer
constexpr uint32_t OFF_STG = OFF_DS + kDsBytes;               // 2 half-tile slots (half k: k % 2)
constexpr uint32_t OFF_VEC = OFF_STG + 2 * kStgBytes;
constexpr uint32_t OFF_BITS = OFF_VEC + NSTAGE * kVecBytes;   // per stage: [64 rows][4 words]
constexpr uint32_t OFF_BAR = OFF_BITS + NSTAGE * BR * 4 * 4;
constexpr uint32_t kNumBars = 38;   // 37 used
constexpr uint32_t OFF_MISC = OFF_BAR + kNumBars * 8;
constexpr uint32_t OFF_REL = OFF_MISC + 64;                   // release queue: {int *flag; int value}
constexpr uint32_t kSmemUsed = OFF_REL + kRelRing * 16;
// The whole 227 KB opt-in: one CTA per SM either way, and every operand
// descriptor's reach (tile base + strides) stays inside the allocation.
constexpr uint32_t kSmemBytes = 232448;
static_assert(kSmemUsed + 1024 + 64 <= kSmemBytes, "shared memory budget (64 B: diagnostic counters)");
static_assert(OFF_STG % 1024 == 0 && OFF_DS % 1024 == 0 && OFF_VEC % 16 == 0, "alignment");

// mbarrier indices.  Every per-tile barrier whose waiter may lag by more than
// one tile is split per buffer ([2], tile t uses t % 2): a parity wait is only
// sound while the barrier is at most one completion past the awaited one.
enum : int {
    B_K_FULL = 0,      //      count 1 + tx
    B_K_EMPTY = 1,     //      count 1 (commit after the unit's last dQ^T)
    B_V_FULL = 2,      //      count 1 + tx
    B_V_EMPTY = 3,     //      count 1 (commit after the unit's last dP)
    B_Q_FULL = 4,      // [3]  count 32 + tx (Q / dY stage t % 3)
    B_Q_EMPTY = 7,     // [3]  count 1 (commit)
    B_S_FULL = 10,     // [2]  count 1 (commit)
    B_P_READY = 12,    // [2]  count 256
    B_PV_DONE = 14,    // [2]  count 1 (commit after dV: P^T consumed, S buffer writable)
    B_DP_FULL = 16,    // [2]  count 1 (commit)
    B_DS_READY = 18,   // [2]  count 256 (the softmax may run a tile ahead of the MMA warp)
    B_DK_DONE = 20,    // [2]  unused (dK(t) completion is implied by DQ_FREE(t))
    B_DQ_FULL = 22,    // [2]  count 1 (commit); also: the dS smem buffer consumed
    B_DQ_FREE = 24,    // [2]  count 128 (dQ^T read out of its S buffer)
    B_ACC_FULL = 26,   //      count 1 (commit)
    B_ACC_FREE = 27,   //      count 128
    B_UNIT_FULL = 28,  // [2]  count 1
    B_UNIT_EMPTY = 30, // [2]  count 14 (MMA + 8 softmax + 4 epilogue warps + writer)
    B_DRAIN = 32,      //      count 1 (commit)
    B_STG_FULL = 33,   // [2]  count 128 (per staging slot)
    B_STG_FREE = 35,   // [2]  count 1
};

// misc words
constexpr uint32_t MISC_TMEM = 0, MISC_RING = 1, MISC_ABORT = 3, MISC_REL_TAIL = 4, MISC_REL_HEAD = 5,
                   MISC_REL_DONE = 6;

struct RelEntry {
    int *flag;
    int value;
    int pad;
};

struct Smem {
    uint8_t *base;
    __device__ uint64_t *bar(int i) const { return reinterpret_cast<uint64_t *>(base + OFF_BAR) + i; }
    __device__ uint32_t *misc() const { return reinterpret_cast<uint32_t *>(base + OFF_MISC); }
    __device__ volatile int *abort_flag() const { return reinterpret_cast<volatile int *>(misc() + MISC_ABORT); }
};

#ifdef TND_WAIT_STATS
// Diagnostic build only: cycles each warp role spends in each wait, summed
// over warps (lane 0) and CTAs.  Slots 0-39: barrier waits; 40: role time;
// 41: dQ counter spins; 42: bulk source-read waits; 43: bulk completion waits;
// 44: proxy fence; 45: counter release batches.
__device__ unsigned long long g_wait_stats[6][56];
__device__ __forceinline__ int wait_role()
{
    const int w = threadIdx.x >> 5;
    return w == 0 ? 0 : w == 1 ? 1 : w < 10 ? 2 : w < 14 ? 3 : w == 14 ? 4 : 5;
}
__device__ __forceinline__ void wait_stat(int slot, long long t0)
{
    if ((threadIdx.x & 31) == 0) atomicAdd(&g_wait_stats[wait_role()][slot], (unsigned long long)(clock64() - t0));
}
#define WAIT_STAT(slot, t0) wait_stat(slot, t0)
// last wait entered by each warp of each CTA: (barrier, completion)
__device__ unsigned int g_wait_last[160][16][2];
__device__ __forceinline__ void wait_note(int bar, uint32_t k)
{
    if ((threadIdx.x & 31) == 0 && blockIdx.x < 160) {
        g_wait_last[blockIdx.x][threadIdx.x >> 5][0] = (unsigned)bar;
        g_wait_last[blockIdx.x][threadIdx.x >> 5][1] = k;
    }
}
#define WAIT_NOTE(bar, k) wait_note(bar, k)
#else
#define WAIT_NOTE(bar, k) ((void)0)
#define WAIT_STAT(slot, t0) ((void)0)
#endif

#ifdef TND_TRACE
// Diagnostic build only: an event timeline of CTA 0, per warp (lane 0):
// {start clock, end clock, (event << 20) | tile}.  Events 0-39: barrier waits;
// 64 + barrier: arrivals; 100 + slot: UMMA issue of S, dP, dV, dK, dQ.
constexpr int kTraceLen = 4096;
__device__ long long g_trace[16][kTraceLen][3];
__device__ unsigned int g_trace_n[16];
// every CTA: global timer at start and end, tiles processed (MMA thread)
__device__ unsigned long long g_cta_time[1024][3];
__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void trace_ev(uint32_t code, long long t0)
{
    // per-warp event counts in the unused tail of the dynamic shared memory:
    // zeroed at kernel start, copied out at its end
    extern __shared__ uint8_t smem_raw[];
    unsigned int *s_trace_n = reinterpret_cast<unsigned int *>(
        ((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023)) + kSmemUsed);
    if ((threadIdx.x & 31) == 0 && blockIdx.x == 0) {
        const int w = threadIdx.x >> 5;
        volatile unsigned int *n = s_trace_n;
        if (code == 0xffffffffu) {
            if (t0 == 0) n[w] = 0;
            else g_trace_n[w] = n[w];
            return;
        }
        const long long t1 = clock64();   // before the counter's shared-memory load
        const unsigned i = n[w];
        n[w] = i + 1;
        if (i < (unsigned)kTraceLen) {
            g_trace[w][i][0] = t0;
            g_trace[w][i][1] = t1;
            g_trace[w][i][2] = code;
        }
    }
}
#define TRACE_EV(ev, k, t0) trace_ev(((uint32_t)(ev) << 20) | ((uint32_t)(k) & 0xfffffu), t0)
#define TRACE_ARR(bar, k) trace_ev(((uint32_t)(64 + (bar)) << 20) | ((uint32_t)(k) & 0xfffffu), clock64())
#else
#define TRACE_EV(ev, k, t0) ((void)0)
#define TRACE_ARR(bar, k) ((void)0)
#endif
#if defined(TND_WAIT_STATS) || defined(TND_TRACE)
#define ISSUE_T0(var) const long long var = clock64()
#define ISSUE_MARK(slot, var, k) \
    do {                         \
        WAIT_STAT(slot, var);    \
        TRACE_EV(100 + (slot) - 46, k, var); \
    } while (0)
#else
#define ISSUE_T0(var) ((void)0)
#define ISSUE_MARK(slot, var, k) ((void)0)
#endif

// Wait for completion `k` (0-based) of barrier `bar`, bounded.
__device__ __forceinline__ bool wait_k(const Smem &sm, int bar, uint32_t k, const GradArgs &a)
{
    uint64_t *b = sm.bar(bar);
    const uint32_t parity = k & 1u;
    const long long t0 = clock64();
    bool ok = true;
    WAIT_NOTE(bar, k);
    while (!mbar_try_wait(b, parity)) {
        if (*sm.abort_flag()) {
            ok = false;
            break;
        }
        if (clock64() - t0 > a.wait_limit_cycles) {
            // detail: completion index, warp, barrier
            set_status(a.status, TND_ERR_DEVICE_TIMEOUT,
                       (k << 12) | ((threadIdx.x >> 5) << 6) | (uint32_t)bar);
            *sm.abort_flag() = 1;
            ok = false;
            break;
        }
    }
    WAIT_STAT(bar, t0);
    TRACE_EV(bar, k, t0);
    return ok;
}

// Single-thread polling variant for the UMMA issuer: mbarrier.test_wait does
// not suspend the thread, so it reacts to the phase flip without a resume delay.
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
__device__ __forceinline__ bool wait_poll(const Smem &sm, int bar, uint32_t k, const GradArgs &a)
{
    uint64_t *b = sm.bar(bar);
    const uint32_t parity = k & 1u;
    const long long t0 = clock64();
    bool ok = true;
    while (!mbar_test_wait(b, parity)) {
        if (*sm.abort_flag()) {
            ok = false;
            break;
        }
        if (clock64() - t0 > a.wait_limit_cycles) {
            set_status(a.status, TND_ERR_DEVICE_TIMEOUT, (k << 12) | ((threadIdx.x >> 5) << 6) | (uint32_t)bar);
            *sm.abort_flag() = 1;
            ok = false;
            break;
        }
    }
    TRACE_EV(bar, k, t0);
    return ok;
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

// Dropout keep-bits.  Bit p of the packed mask (little-endian within each
// byte) is bit p % 64 of the little-endian 64-bit word p / 64.  Row ii of head
// h starts at bit mask_base + (h * sq + ii) * skv; a tile needs the 128 bits
// of kv block jb.  With an 8-byte aligned mask, three aligned words cover any
// bit offset; fetch_keep_rows issues them for rows q0 + lane and q0 + lane + 32
// (independent loads, one memory latency per tile), keep_row_words extracts
// the four 32-bit words.  Words that reach past the mask's end, and an
// unaligned mask, take the byte path.
__device__ __forceinline__ int64_t keep_row_bit(const SeqDesc &sd, int h, int64_t ii, int jb)
{
    return sd.mask_base + ((int64_t)h * sd.sq + ii) * sd.skv + (int64_t)jb * kKvBlock;
}

__device__ __forceinline__ void fetch_keep_rows(const GradArgs &a, const SeqDesc &sd, int h, int64_t q0, int jb,
                                                int lane, uint64_t (&mw)[2][3])
{
    const bool aligned = (reinterpret_cast<uintptr_t>(a.drop_mask) & 7) == 0;
    const uint64_t *m64 = reinterpret_cast<const uint64_t *>(a.drop_mask);
    const int64_t nwords = a.mask_bytes >> 3;   // whole words inside the mask
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int64_t ii = q0 + lane + 32 * rr;
        const int64_t w0 = keep_row_bit(sd, h, ii, jb) >> 6;
#pragma unroll
        for (int e = 0; e < 3; ++e) {
            mw[rr][e] = (aligned && ii < sd.sq && w0 + e < nwords) ? __ldg(m64 + w0 + e) : 0ull;
        }
    }
}

__device__ __forceinline__ uint4 keep_row_words(const uint64_t (&w)[3], const GradArgs &a, const SeqDesc &sd, int h,
                                                int64_t ii, int jb)
{
    if (ii >= sd.sq) return make_uint4(0, 0, 0, 0);
    const int64_t p0 = keep_row_bit(sd, h, ii, jb);
    const bool aligned = (reinterpret_cast<uintptr_t>(a.drop_mask) & 7) == 0;
    uint32_t out[4];
    if (aligned && (p0 >> 6) + 3 <= (a.mask_bytes >> 3)) {
        const int sh = (int)(p0 & 63);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int b = sh + 32 * k, q = b >> 6, off = b & 63;   // q <= 2; the word never crosses w[2]
            // registers, not an indexed array: q is not a compile-time constant
            const uint64_t wq = q == 0 ? w[0] : q == 1 ? w[1] : w[2];
            const uint64_t wn = q == 0 ? w[1] : w[2];
            const uint64_t lo = wq >> off;
            const uint64_t hi = (off > 32 && q < 2) ? (wn << (64 - off)) : 0ull;
            out[k] = (uint32_t)(lo | hi);
        }
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t pos = p0 + 32 * k;
            const int64_t byte0 = pos >> 3;
            uint64_t acc = 0;
#pragma unroll
            for (int bb = 0; bb < 5; ++bb) {
                const int64_t bi = byte0 + bb;
                acc |= (uint64_t)((bi < a.mask_bytes) ? a.drop_mask[bi] : 0) << (8 * bb);
            }
            out[k] = (uint32_t)(acc >> (pos & 7));
        }
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
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

// Shared-memory descriptors are built once per buffer; adding (byte offset
// >> 4) to one moves its start address (the 14-bit field never overflows:
// every address is below 256 KB).
__device__ __forceinline__ uint64_t desc_at(uint64_t base_desc, uint32_t byte_off)
{
    return base_desc + (uint64_t)(byte_off >> 4);
}

// TMEM column of the k-th 16-row K slice of a packed 16-bit operand (Pd^T,
// dS^T): each softmax half packs its 32 q columns into the first 16 columns
// of its own 32-column range, so slices 0-1 sit at columns 0-15 and 2-3 at
// columns 32-47.
__device__ __forceinline__ uint32_t pk_col(int kk) { return (uint32_t)((kk >> 1) * 32 + (kk & 1) * 8); }

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
        mbar_init(sm.bar(B_K_FULL), 1);
        mbar_init(sm.bar(B_K_EMPTY), 1);
        for (int i = 0; i < NSTAGE; ++i) {
            mbar_init(sm.bar(B_Q_FULL + i), 32);
            mbar_init(sm.bar(B_Q_EMPTY + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(sm.bar(B_STG_FULL + i), 128);
            mbar_init(sm.bar(B_STG_FREE + i), 1);
            mbar_init(sm.bar(B_S_FULL + i), 1);
            mbar_init(sm.bar(B_P_READY + i), 256);
            mbar_init(sm.bar(B_PV_DONE + i), 1);
            mbar_init(sm.bar(B_DP_FULL + i), 1);
            mbar_init(sm.bar(B_UNIT_FULL + i), 1);
            mbar_init(sm.bar(B_UNIT_EMPTY + i), 14);
        }
        mbar_init(sm.bar(B_V_FULL), 1);
        mbar_init(sm.bar(B_V_EMPTY), 1);
        mbar_init(sm.bar(B_DS_READY), 256);
        mbar_init(sm.bar(B_DS_READY + 1), 256);
        for (int i = 0; i < 2; ++i) {
            mbar_init(sm.bar(B_DK_DONE + i), 1);
            mbar_init(sm.bar(B_DQ_FULL + i), 1);
            mbar_init(sm.bar(B_DQ_FREE + i), 128);
        }
        mbar_init(sm.bar(B_ACC_FULL), 1);
        mbar_init(sm.bar(B_ACC_FREE), 128);
        mbar_init(sm.bar(B_DRAIN), 1);

        *sm.abort_flag() = 0;
        sm.misc()[MISC_REL_TAIL] = 0;
        sm.misc()[MISC_REL_HEAD] = 0;
        sm.misc()[MISC_REL_DONE] = 0;
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
#ifdef TND_TRACE
    unsigned long long mma_tiles = 0;
#endif
#ifdef TND_WAIT_STATS
    const long long t_role = clock64();
#endif
#ifdef TND_TRACE
    trace_ev(0xffffffffu, 0);
    if (threadIdx.x == 0 && blockIdx.x < 1024) g_cta_time[blockIdx.x][0] = global_ns();
#endif

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
            if (ku >= 1 && !wait_warp(sm, B_K_EMPTY, ku - 1, a)) break;
            if (lane == 0) {
                uint64_t *fb = sm.bar(B_K_FULL);
                mbar_arrive_expect_tx(fb, kKvTile);
                uint8_t *kt = sm.base + OFF_K;
                tma_load_3d(kt, &tmK, fb, 0, U.g, z_kv);
                tma_load_3d(kt + kKvColBlk, &tmK, fb, 64, U.g, z_kv);
            }
            bool ok = true;
            for (int t = 0; t < U.ntiles; ++t, ++gt) {
                const int qb = U.qb_lo + t / G, h = U.g * G + t % G;
                const uint32_t s = gt % NSTAGE, k = gt / NSTAGE;
                const int64_t q0 = (int64_t)qb * BR;
                // dropout keep-bits of the tile: 128 kv bits of each of its 64 q
                // rows, two rows per lane, fetched before the stage wait
                uint64_t mw[2][3];
                if (a.has_drop) fetch_keep_rows(a, U.sd, h, q0, U.jb, lane, mw);
                if (k >= 1 && !wait_warp(sm, B_Q_EMPTY + s, k - 1, a)) {
                    ok = false;
                    break;
                }
                if (a.has_drop) {
                    uint32_t *bits = reinterpret_cast<uint32_t *>(sm.base + OFF_BITS + s * BR * 16);
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr) {
                        const uint4 v = keep_row_words(mw[rr], a, U.sd, h, q0 + lane + 32 * rr, U.jb);
                        *reinterpret_cast<uint4 *>(bits + (lane + 32 * rr) * 4) = v;
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
                    TRACE_ARR(B_Q_FULL, gt);
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
        // outstanding TMA writes must land before the CTA can leave.  K and V
        // loads were issued for units [0, ku) (V possibly not for the last one
        // if the wait before it failed: draining a phase that never started
        // only costs the bounded wait).
        if (*sm.abort_flag() && lane == 0) {
            for (uint32_t s = 0; s < NSTAGE && s < gt; ++s) {
                const uint32_t last = ((gt - 1 - s) / NSTAGE) * NSTAGE + s;  // last tile that used stage s
                drain_k(sm, B_Q_FULL + s, last / NSTAGE, a);
            }
            if (ku >= 1) {
                drain_k(sm, B_K_FULL, ku - 1, a);
                drain_k(sm, B_V_FULL, ku - 1, a);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            const uint32_t idS = instr_desc_f16(BF16, 128, BR, false, false);    // S^T, dP^T
            const uint32_t idKV = instr_desc_f16(BF16, 128, HD, false, true);    // dV, dK (A in TMEM)
            const uint32_t idQ = instr_desc_f16(BF16, 128, BR, true, true);      // dQ^T
            const uint32_t sbase = smem_u32(sm.base);
            // K-major views (S^T, dP^T operands) and MN-major views (dV, dK, dQ^T operands)
            const uint64_t dK_k0 = smem_desc_sw128(sbase + OFF_K, 16, 1024);
            const uint64_t dK_m0 = smem_desc_sw128(sbase + OFF_K, kKvColBlk, 1024);
            const uint64_t dV_k = smem_desc_sw128(sbase + OFF_V, 16, 1024);
            const uint64_t dQ_k0 = smem_desc_sw128(sbase + OFF_Q, 16, 1024);
            const uint64_t dQ_m0 = smem_desc_sw128(sbase + OFF_Q, kQColBlk, 1024);
            const uint64_t dY_k0 = smem_desc_sw128(sbase + OFF_DY, 16, 1024);
            const uint64_t dY_m0 = smem_desc_sw128(sbase + OFF_DY, kQColBlk, 1024);
            const uint64_t dS_m = smem_desc_sw128(sbase + OFF_DS, kQColBlk, 1024);
            uint32_t ui = 0, ku = 0, gt = 0;
            bool ok = true;
            while (ok) {
                int u;
                if (!read_unit1(sm, ui, a, u)) break;
                ++ui;
                if (u < 0) break;
                const UnitInfo U = unit_info(a, u);
                if (U.ntiles == 0) continue;
                if (!wait_poll(sm, B_K_FULL, ku, a)) break;
                tc_fence_after();
                const uint64_t dK_k = dK_k0, dK_m = dK_m0;
                const uint32_t g_end = gt + (uint32_t)U.ntiles;
                // S^T(t) = K Q(t)^T, K-major both, into S buffer t % 2 once the
                // epilogue has read out dQ^T(t - 2) from it
                auto issue_s = [&](uint32_t g_t, bool need_q) -> bool {
                    const uint32_t s = g_t % NSTAGE, b = g_t & 1u;
                    if (need_q && !wait_poll(sm, B_Q_FULL + s, g_t / NSTAGE, a)) return false;
                    if (g_t >= 2 && !wait_poll(sm, B_DQ_FREE + b, (g_t >> 1) - 1, a)) return false;
                    tc_fence_after();
                    ISSUE_T0(ti);
                    const uint64_t dq = desc_at(dQ_k0, s * kQTile);
#pragma unroll
                    for (int kk = 0; kk < HD / 16; ++kk) {
                        const uint32_t off_k = (kk >> 2) * kKvColBlk + (kk & 3) * 32;
                        const uint32_t off_q = (kk >> 2) * kQColBlk + (kk & 3) * 32;
                        mma_ss(tmem + TM_S0 + b * 64, desc_at(dK_k, off_k), desc_at(dq, off_q), idS, kk > 0);
                    }
                    mma_commit(sm.bar(B_S_FULL + b));
                    ISSUE_MARK(46, ti, g_t);
                    return true;
                };
                // dP^T(t) = V dY(t)^T into dP buffer t % 2.  Issued right after S^T(t),
                // whose waits cover it: Q_FULL(t) (dY(t) landed) and DQ_FREE(t - 2),
                // which the epilogue arrives after observing the commit that follows
                // dQ^T(t - 2), and a commit tracks every earlier UMMA of the thread, so
                // dK(t - 2) has read dS^T(t - 2) out of this buffer by then.  Each
                // barrier wait on this thread costs hundreds of cycles of tensor-pipe
                // idle time, hence no wait of its own.
                auto issue_dp = [&](uint32_t g_t) -> bool {
                    const uint32_t s = g_t % NSTAGE, b = g_t & 1u;
                    ISSUE_T0(ti47);
                    const uint64_t dy = desc_at(dY_k0, s * kQTile);
#pragma unroll
                    for (int kk = 0; kk < HD / 16; ++kk) {
                        const uint32_t off_v = (kk >> 2) * kKvColBlk + (kk & 3) * 32;
                        const uint32_t off_y = (kk >> 2) * kQColBlk + (kk & 3) * 32;
                        mma_ss(tmem + TM_DP0 + b * 64, desc_at(dV_k, off_v), desc_at(dy, off_y), idS, kk > 0);
                    }
                    mma_commit(sm.bar(B_DP_FULL + b));
                    ISSUE_MARK(47, ti47, g_t);
                    if (g_t + 1 == g_end) mma_commit(sm.bar(B_V_EMPTY));   // last reader of V
                    return true;
                };
                if (!issue_s(gt, true)) break;
                if (!wait_poll(sm, B_V_FULL, ku, a)) break;
                tc_fence_after();
                if (!issue_dp(gt)) break;
                for (int t = 0; t < U.ntiles; ++t) {
                    const uint32_t g_t = gt + t, s = g_t % NSTAGE, b = g_t & 1u;
                    // the next tile's S^T and dP^T go ahead of this tile's gradients
                    if (t + 1 < U.ntiles && (!issue_s(g_t + 1, true) || !issue_dp(g_t + 1))) {
                        ok = false;
                        break;
                    }
                    if (t == 0 && ku >= 1 && !wait_poll(sm, B_ACC_FREE, ku - 1, a)) {
                        ok = false;
                        break;
                    }
                    // dV += Pd^T dY(t): A = Pd^T (TMEM, packed), B = dY MN-major (N = 128)
                    if (!wait_poll(sm, B_P_READY + b, g_t >> 1, a)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    ISSUE_T0(ti48);
                    const uint64_t dqm = desc_at(dQ_m0, s * kQTile), dym = desc_at(dY_m0, s * kQTile);
#pragma unroll
                    for (int kk = 0; kk < BR / 16; ++kk) {
                        mma_ts(tmem + TM_DV, tmem + TM_S0 + b * 64 + pk_col(kk), desc_at(dym, kk * 2048), idKV,
                               (t > 0 || kk > 0));
                    }
                    mma_commit(sm.bar(B_PV_DONE + b));
                    ISSUE_MARK(48, ti48, g_t);
                    // dK += dS^T Q(t): A = dS^T (TMEM, packed), B = Q MN-major
                    if (!wait_poll(sm, B_DS_READY + b, g_t >> 1, a)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    ISSUE_T0(ti49);
#pragma unroll
                    for (int kk = 0; kk < BR / 16; ++kk) {
                        mma_ts(tmem + TM_DK, tmem + TM_DP0 + b * 64 + pk_col(kk), desc_at(dqm, kk * 2048), idKV,
                               (t > 0 || kk > 0));
                    }
                    mma_commit(sm.bar(B_Q_EMPTY + s));
                    ISSUE_MARK(49, ti49, g_t);
                    // dQ^T(t) = K^T dS^T into S buffer t % 2: dV(t) has read P^T from it
                    // (the softmax arrives DS_READY(t) only after observing PV_DONE(t)):
                    // A = K MN-major (M = 128 features), B = dS^T MN-major (N = 64)
                    tc_fence_after();
                    ISSUE_T0(ti50);
#pragma unroll
                    for (int kk = 0; kk < BC / 16; ++kk) {
                        mma_ss(tmem + TM_S0 + b * 64, desc_at(dK_m, kk * 2048), desc_at(dS_m, kk * 2048),
                               idQ, kk > 0);
                    }
                    mma_commit(sm.bar(B_DQ_FULL + b));
                    ISSUE_MARK(50, ti50, g_t);
                }
                if (!ok) break;
                mma_commit(sm.bar(B_ACC_FULL));
                mma_commit(sm.bar(B_K_EMPTY));
                gt += U.ntiles;
#ifdef TND_TRACE
                mma_tiles += U.ntiles;
#endif
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
        // Two warps per TMEM lane quarter: warps 2-5 take q columns 0-31 of the
        // tile, warps 6-9 columns 32-63.
        const int quarter = warp & 3;
        const int half = (warp - kSoftmaxWarp0) >> 2;
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
                const uint32_t keep = (uint32_t)(keep_columns(a, U.sd, q0, jj) >> (32 * half));
                const bool full = __all_sync(0xffffffffu, keep == 0xffffffffu);
                if (!wait_warp(sm, B_Q_FULL + s, gt / NSTAGE, a) || !wait_warp(sm, B_S_FULL + b, gt >> 1, a)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float4 *lse4 = reinterpret_cast<const float4 *>(sm.base + OFF_VEC + s * kVecBytes) + 8 * half;
                const float4 *dvec4 = lse4 + BR / 4;
                uint32_t zbits = 0xffffffffu;
                if (a.has_drop) {
                    const uint32_t *bits = reinterpret_cast<const uint32_t *>(sm.base + OFF_BITS + s * BR * 16);
                    zbits = 0;
#pragma unroll 8
                    for (int c = 0; c < 32; ++c) zbits |= ((bits[(32 * half + c) * 4 + quarter] >> lane) & 1u) << c;
                }
                // ---- phase 1: P^T from S^T, Pd^T = P^T o z into TMEM (16 packed columns)
                float p[32];
                uint32_t raw[32];
                const uint32_t s_addr = tmem + lane_addr + TM_S0 + b * 64;
                tmem_ld32(s_addr + 32 * half, raw);
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) {
                    const float4 l = lse4[c4];
                    p[4 * c4 + 0] = ex2(fmaf(__uint_as_float(raw[4 * c4 + 0]), C, -l.x));
                    p[4 * c4 + 1] = ex2(fmaf(__uint_as_float(raw[4 * c4 + 1]), C, -l.y));
                    p[4 * c4 + 2] = ex2(fmaf(__uint_as_float(raw[4 * c4 + 2]), C, -l.z));
                    p[4 * c4 + 3] = ex2(fmaf(__uint_as_float(raw[4 * c4 + 3]), C, -l.w));
                }
                if (!full) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) p[c] = ((keep >> c) & 1u) ? p[c] : 0.0f;
                }
                uint32_t pk[16];
                if (a.has_drop) {
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const float z0 = ((zbits >> (2 * c)) & 1u) ? a.inv_keep : 0.0f;
                        const float z1 = ((zbits >> (2 * c + 1)) & 1u) ? a.inv_keep : 0.0f;
                        pk[c] = pack2<BF16>(p[2 * c] * z0, p[2 * c + 1] * z1);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 16; ++c) pk[c] = pack2<BF16>(p[2 * c], p[2 * c + 1]);
                }
                tmem_st16(s_addr + 32 * half, pk);      // packed into this half's own columns
                tc_fence_before();
                mbar_arrive(sm.bar(B_P_READY + b));
                TRACE_ARR(B_P_READY, gt);
                // ---- phase 2: dS^T = P^T o (z dP^T - D) into TMEM and shared memory
                if (!wait_warp(sm, B_DP_FULL + b, gt >> 1, a)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t dp_addr = tmem + lane_addr + TM_DP0 + b * 64;
                tmem_ld32(dp_addr + 32 * half, raw);
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) {
                    const float4 dv = dvec4[c4];
                    float dp[4] = {__uint_as_float(raw[4 * c4]), __uint_as_float(raw[4 * c4 + 1]),
                                   __uint_as_float(raw[4 * c4 + 2]), __uint_as_float(raw[4 * c4 + 3])};
                    if (a.has_drop) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) dp[e] = ((zbits >> (4 * c4 + e)) & 1u) ? dp[e] * a.inv_keep : 0.0f;
                    }
                    pk[2 * c4] = pack2<BF16>(p[4 * c4] * (dp[0] - dv.x), p[4 * c4 + 1] * (dp[1] - dv.y));
                    pk[2 * c4 + 1] = pack2<BF16>(p[4 * c4 + 2] * (dp[2] - dv.z), p[4 * c4 + 3] * (dp[3] - dv.w));
                }
                tmem_st16(dp_addr + 32 * half, pk);
                // the dS^T buffer: the dQ^T GEMM of tile t - 1 must have read it
                if (gt >= 1 && !wait_warp(sm, B_DQ_FULL + (b ^ 1u), (gt - 1) >> 1, a)) {
                    ok = false;
                    break;
                }
                {
                    uint8_t *row = sm.base + OFF_DS + jl * 128;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int chunk = 4 * half + c;
                        uint4 v = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                        *reinterpret_cast<uint4 *>(row + ((chunk ^ (jl & 7)) << 4)) = v;
                    }
                }
                fence_async_smem();
                tc_fence_before();
                // dV(t) has consumed P^T: DS_READY(t) then also frees the S buffer
                // for dQ^T(t), and the MMA warp needs no wait of its own for it
                if (!wait_warp(sm, B_PV_DONE + b, gt >> 1, a)) {
                    ok = false;
                    break;
                }
                mbar_arrive(sm.bar(B_DS_READY + b));
                TRACE_ARR(B_DS_READY, gt);
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
                if (!wait_warp(sm, B_DQ_FULL + (gt & 1u), gt >> 1, a)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t v[BR];
                const uint32_t dq_addr = tmem + lane_addr + TM_S0 + (gt & 1u) * 64;
                tmem_ld32(dq_addr, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
                tmem_ld32(dq_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
                tc_fence_before();
                mbar_arrive(sm.bar(B_DQ_FREE + (gt & 1u)));
                TRACE_ARR(B_DQ_FREE, gt);
                // staging: a ring of two [32 q rows][128 features] fp32 slots;
                // half tile k (q rows 32 (k % 2) .. +31 of tile k / 2) goes to slot
                // k % 2 once the writer's bulk operation has read half k - 2
#pragma unroll
                for (int hs = 0; hs < 2; ++hs) {
                    const uint32_t k = 2 * gt + hs;
                    if (k >= 2 && !wait_warp(sm, B_STG_FREE + hs, (k >> 1) - 1, a)) {
                        ok = false;
                        break;
                    }
                    float *slot = stg + hs * (kStgBytes / 4);
#pragma unroll
                    for (int c = 0; c < BR / 2; ++c) slot[c * HD] = __uint_as_float(v[hs * (BR / 2) + c]);
                    fence_async_smem();
                    mbar_arrive(sm.bar(B_STG_FULL + hs));
                    TRACE_ARR(B_STG_FULL, 2 * gt + hs);
                }
                if (!ok) break;
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
            TRACE_ARR(B_ACC_FREE, ku);
            ++ku;
        }
    } else if (warp == kWriterWarp) {
        // ================================================================ dQ writer
        // Adds each staged dQ^T tile into the fp32 accumulator of its (q block,
        // head): the first contributor stores, later ones add, each after the
        // previous contributor's counter says its update has completed.  A
        // tile goes out as two bulk groups (q rows 0-31, 32-63) so that the
        // epilogue refills one staging half while the other is read.  Once a
        // tile's groups have completed (checked while handling the next tile)
        // its counter update goes to the release warp's queue, so this thread
        // never runs a GPU-scope fence and never holds an unreleased counter
        // while it waits on another one.
        if (lane == 0) {
            uint32_t ui = 0, gt = 0, rel_tail = 0;
            int *pend_flag = nullptr;
            int pend_val = 0;
            const uint8_t *stg = sm.base + OFF_STG;
            RelEntry *ring = reinterpret_cast<RelEntry *>(sm.base + OFF_REL);
            const uint32_t *rel_head = sm.misc() + MISC_REL_HEAD;
            bool ok = true;
            // the previous tile's groups have completed: counter queued.  Done
            // before this tile's operations: other CTAs' chains wait on it
            auto finish_prev = [&]() -> bool {
                if (!pend_flag) return true;
                const long long tw = clock64();
                (void)tw;
                bulk_wait0();
                fence_async_global();
                WAIT_STAT(43, tw);
                const long long t0 = clock64();
                while (rel_tail - ld_acquire_cta_shared(rel_head) >= kRelRing) {
                    if (*sm.abort_flag() || clock64() - t0 > a.wait_limit_cycles) return false;
                }
                RelEntry &e = ring[rel_tail % kRelRing];
                e.flag = pend_flag;
                e.value = pend_val;
                st_release_cta_shared(sm.misc() + MISC_REL_TAIL, ++rel_tail);
                pend_flag = nullptr;
                return true;
            };
            while (ok) {
                int u;
                if (!read_unit1(sm, ui, a, u)) break;
                ++ui;
                if (u < 0) break;
                const UnitInfo U = unit_info(a, u);
                for (int t = 0; t < U.ntiles; ++t, ++gt) {
                    const int qb = U.qb_lo + t / G, h = U.g * G + t % G;
                    const int qg = U.sd.qblk0 + qb;
                    // contributor range and the counter, both loaded while the
                    // epilogue is still staging the tile
                    const QBlockInfo qi = a.qblk[qg];
                    int *flag = a.flags + (int64_t)qg * a.nq + h;
                    const int seen = ld_acquire_gpu(flag);
                    const int64_t q0 = (int64_t)qb * BR;
                    const int rows = (int)min((int64_t)BR, (int64_t)U.sd.sq - q0);
                    if (!wait_k(sm, B_STG_FULL, gt, a) || !finish_prev()) {
                        ok = false;
                        break;
                    }
                    const int pos = qi.jhi - U.jb;
                    if (pos > 0 && seen < pos) {
                        const long long tf = clock64();
                        (void)tf;
                        const long long t0 = clock64();
                        WAIT_NOTE(60, (uint32_t)(qg * a.nq + h) | ((uint32_t)pos << 24));
                        while (ld_acquire_gpu(flag) < pos) {
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
                        WAIT_STAT(41, tf);
                    }
                    if (pos > 0) fence_async_global();    // counter acquire before the bulk reduction
                    const int z = (int)(U.sd.tq + q0);
#pragma unroll 1
                    for (int hs = 0; hs < 2; ++hs) {
                        if (hs == 1 && !wait_k(sm, B_STG_FULL + 1, gt, a)) {
                            ok = false;
                            break;
                        }
                        const uint8_t *slot = stg + hs * kStgBytes;
                        const int r0 = hs * (BR / 2);
                        if (rows == BR) {
                            if (pos == 0) tma_store_3d(&tmDQ, slot, 0, h, z + r0);
                            else tma_reduce_add_3d(&tmDQ, slot, 0, h, z + r0);
                        } else {
                            // ragged last block of a sequence: only its own rows
                            for (int r = r0; r < min(rows, r0 + BR / 2); ++r) {
                                float *dst = a.dqacc + ((int64_t)(z + r) * a.nq + h) * HD;
                                if (pos == 0) bulk_s2g(dst, slot + (r - r0) * HD * 4, HD * 4);
                                else bulk_reduce_add_f32(dst, slot + (r - r0) * HD * 4, HD * 4);
                            }
                        }
                        bulk_commit();
                        // slot 0 is freed once half 1 is in flight, slot 1 at the end of
                        // the tile, so no slot waits for the next tile's counter
                        const long long tr = clock64();
                        (void)tr;
                        if (hs == 1) {
                            bulk_wait_read1();
                            mbar_arrive(sm.bar(B_STG_FREE));
                            TRACE_ARR(B_STG_FREE, 2 * gt);
                            bulk_wait_read0();
                            mbar_arrive(sm.bar(B_STG_FREE + 1));
                            TRACE_ARR(B_STG_FREE, 2 * gt + 1);
                        }
                        WAIT_STAT(42, tr);
                    }
                    if (!ok) break;
                    pend_flag = flag;
                    pend_val = pos + 1;
                }
            }
            if (ok) finish_prev();
            bulk_wait0();
            st_release_cta_shared(sm.misc() + MISC_REL_DONE, 1u);
        }
        __syncwarp();
    } else {
        // ================================================================ counter releases
        // Publishes queued counter values with one GPU-scope fence per batch:
        // the queue entry was pushed (CTA-scope release) after its bulk group
        // completed, so fence + relaxed store is a release of those writes.
        if (lane == 0) {
            uint32_t head = 0;
            const RelEntry *ring = reinterpret_cast<const RelEntry *>(sm.base + OFF_REL);
            long long idle0 = clock64();
            while (true) {
                const uint32_t tail = ld_acquire_cta_shared(sm.misc() + MISC_REL_TAIL);
                if (tail != head) {
                    const long long tr = clock64();
                    (void)tr;
                    fence_acq_rel_gpu();
                    for (; head != tail; ++head) {
                        const RelEntry &e = ring[head % kRelRing];
                        st_relaxed_gpu(e.flag, e.value);
                    }
                    st_release_cta_shared(sm.misc() + MISC_REL_HEAD, head);   // entries read before reuse
                    WAIT_STAT(45, tr);
                    idle0 = clock64();
                    continue;
                }
                if (ld_acquire_cta_shared(sm.misc() + MISC_REL_DONE)) {
                    if (ld_acquire_cta_shared(sm.misc() + MISC_REL_TAIL) == head) break;
                    continue;
                }
                if (*sm.abort_flag()) break;
                if (clock64() - idle0 > 4 * a.wait_limit_cycles) {
                    set_status(a.status, TND_ERR_DEVICE_TIMEOUT, 0x300u);
                    *sm.abort_flag() = 1;
                    break;
                }
                __nanosleep(256);
            }
        }
        __syncwarp();
    }

#ifdef TND_WAIT_STATS
    WAIT_STAT(40, t_role);
#endif
#ifdef TND_TRACE
    trace_ev(0xffffffffu, 1);
    if (threadIdx.x == 32 && blockIdx.x < 1024) {
        g_cta_time[blockIdx.x][1] = global_ns();
        g_cta_time[blockIdx.x][2] = mma_tiles;
    }
#endif
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

// dQ accumulator [rows, heads, 128] fp32, boxes of 128 features x 1 head x `box_rows` rows (no swizzle)
bool make_acc_map(CUtensorMap *m, const float *ptr, int64_t rows, int64_t heads, int box_rows)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)HD, (cuuint64_t)heads, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)HD * 4, (cuuint64_t)(heads * HD * 4)};
    cuuint32_t box[3] = {HD, 1, (cuuint32_t)box_rows};
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
        !make_acc_map(&mdq, a.dqacc, a.tq, a.nq, BR / 2))
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

#ifdef TND_WAIT_STATS
}  // namespace tnd
extern "C" int tnd_debug_wait_last(unsigned int *out)
{
    return cudaMemcpyFromSymbol(out, tnd::g_wait_last, sizeof(tnd::g_wait_last)) != cudaSuccess;
}
extern "C" int tnd_debug_wait_stats(unsigned long long *out, int reset)
{
    if (cudaMemcpyFromSymbol(out, tnd::g_wait_stats, sizeof(tnd::g_wait_stats)) != cudaSuccess) return 1;
    if (reset) {
        static unsigned long long zero[6][56] = {};
        if (cudaMemcpyToSymbol(tnd::g_wait_stats, zero, sizeof(zero)) != cudaSuccess) return 1;
    }
    return 0;
}
namespace tnd {
#endif
#ifdef TND_TRACE
}  // namespace tnd
extern "C" int tnd_debug_trace(long long *events, unsigned int *counts, int reset)
{
    if (cudaMemcpyFromSymbol(events, tnd::g_trace, sizeof(tnd::g_trace)) != cudaSuccess) return 1;
    if (cudaMemcpyFromSymbol(counts, tnd::g_trace_n, sizeof(tnd::g_trace_n)) != cudaSuccess) return 1;
    if (reset) {
        static unsigned int zero[16] = {};
        if (cudaMemcpyToSymbol(tnd::g_trace_n, zero, sizeof(zero)) != cudaSuccess) return 1;
    }
    return 0;
}
extern "C" int tnd_debug_cta_times(unsigned long long *out)
{
    return cudaMemcpyFromSymbol(out, tnd::g_cta_time, sizeof(tnd::g_cta_time)) != cudaSuccess;
}
namespace tnd {
#endif

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
