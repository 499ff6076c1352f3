// based_kernels.cuh: sm_103a kernels of the Based causal forward pass.
//
// Method (the "based_forward.py" kernel-task spec, spec_md and perf_md): with the symmetric
// 2nd-order feature map f(x) (constant, linear, squared and pairwise-product terms, P = 1 + K +
// K(K+1)/2 features; with per-feature coefficients it reproduces phi(q).phi(k) = 1 + q.k +
// (q.k)^2/2 exactly), every head is cut into chunks of 128 rows and, per chunk c,
//     s   = q_c k_c^T                              (tensor core -> TMEM, fp32)
//     A   = 1 + sigma s + sigma^2 s^2 / 2, j <= i   (fp32 polynomial -> bf16 in TMEM)
//     O   = A [v_c | 1] + f~(q_c) D [S | z]        (tensor core; the ones column gives rowsum A,
//                                                    z gives the inter-chunk denominator)
//     o   = O_num / (O_den + 1e-6)
//     S  += v_c^T f(k_c),  z += f(k_c)^T 1         (tensor core, fp32 accumulation in TMEM)
// where f~(q) carries the feature coefficients (1, 1, 1/2 on squares, 1 on cross products) and
// D multiplies feature c of the fp32 state by sigma^degree(c) (1, sigma, sigma^2) as the state is
// rounded to its bf16 operand, so that f~(q) D f(k) = 1 + sigma q.k + sigma^2 (q.k)^2 / 2. The per-head chunk sequence is split across CTAs; the state each CTA starts from is
// the sum of the partial states of the chunks before it (aggregate pass + scan), so the forward
// kernel never waits on another CTA.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <type_traits>

#include "sm103_ptx.cuh"

namespace based {

constexpr int kChunk = 128;            // rows per chunk = MMA M
constexpr int kMaxChain = 4;           // partial states a forward CTA sums into its prefix itself
constexpr int kFwdThreads = 512;       // 4 warpgroups
constexpr int kAggThreads = 512;       // 4 warpgroups
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // a bounded wait gives up after 1 s
constexpr uint64_t kDrainLimitNs = 100000000ull;  // drain of in-flight copies after an abort

// Status word: bit 0 = some wait timed out; bits 8..15 = site of the first timeout.
__device__ unsigned int g_status;

// Optional stage timestamps (clock64) for pipeline analysis, compiled in only with -DBASED_TRACE:
// g_trace[(cta * 64 + chunk) * 32 + event], chunks >= 64 are not recorded.
#ifdef BASED_TRACE
__device__ unsigned long long *g_trace;
#define BASED_TRACE_INIT unsigned long long *const trace_buf_ = g_trace
#define BASED_TRACE_EV(n, ev)                                                                 \
    do {                                                                                      \
        if (trace_buf_ != nullptr && (n) < 64)                                                \
            trace_buf_[(static_cast<size_t>(blockIdx.x) * 64 + (n)) * 32 + (ev)] = clock64(); \
    } while (0)
#else
#define BASED_TRACE_INIT \
    do {                 \
    } while (0)
#define BASED_TRACE_EV(n, ev) \
    do {                      \
    } while (0)
#endif
enum TraceEvent {
    TE_TMA_ISSUE = 0, TE_A_READY, TE_AV_ISSUED, TE_QK_ISSUED, TE_UPD_ISSUED, TE_RO_ISSUED,
    TE_POLY_BEGIN, TE_POLY_END, TE_PHIK_BEGIN, TE_PHIK_END, TE_PHIQ_BEGIN, TE_PHIQ_END,
    TE_EPI_BEGIN, TE_EPI_OFREE, TE_EPI_END, TE_CONV_BEGIN, TE_CONV_READ, TE_CONV_END,
    TE_POLY_LD0, TE_POLY_ST0, TE_POLY_LD1, TE_POLY_ST1,
    TE_LEAD_ISSUE = 23, TE_LEAD_BUILD0, TE_LEAD_BUILD1, TE_LEAD_UPD  // lead-in chunk i at index i
};

enum WaitSite : uint32_t {
    SITE_STAGE_FREE = 1, SITE_TMA_FULL, SITE_S_FULL, SITE_A_FULL, SITE_O_FULL, SITE_O_FREE,
    SITE_AV_DONE, SITE_PHIQ_FULL, SITE_PHIQ_FREE, SITE_PHIK_FULL, SITE_PHIK_FREE, SITE_UPD_DONE,
    SITE_SBF_FULL, SITE_CONV_READ, SITE_AGG_DONE, SITE_DRAIN, SITE_SLOT_READ, SITE_ZRED, SITE_SELFTEST = 255
};

__device__ __forceinline__ void record_timeout(uint32_t site) {
    atomicCAS(&g_status, 0u, 1u | (site << 8));
    atomicOr(&g_status, 1u);
}

// Gives up a wait: aborts the CTA and records the site (rare path, kept out of line).
__device__ __noinline__ void give_up_wait(volatile int *abort_flag, uint32_t site) {
    if (abort_flag != nullptr) *abort_flag = 1;
    record_timeout(site);
}

// Bounded mbarrier wait. Returns false if the CTA aborted or the wait ran out (then it aborts
// the CTA and records the site). Never spins longer than the limit.
__device__ __forceinline__ bool wait_bar_inline(uint32_t bar, uint32_t parity,
                                                volatile int *abort_flag, uint32_t site,
                                                uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (abort_flag != nullptr && *abort_flag) return false;
        if ((it & 15u) == 0u && global_timer_ns() - t0 > limit_ns) {
            give_up_wait(abort_flag, site);
            return false;
        }
    }
}
// The same wait as an out-of-line call: every role shares one copy of the loop, which keeps the
// kernel's code (and its instruction-cache footprint) small.
__device__ __noinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                           uint32_t site, uint64_t limit_ns) {
    return wait_bar_inline(bar, parity, abort_flag, site, limit_ns);
}
// Bounded wait with the completed-phase test inline (a few instructions at each call site) and the
// waiting loop out of line: a wait that finds its phase complete costs no call.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                         uint32_t site, uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_bar_slow(bar, parity, abort_flag, site, limit_ns);
}

// ------------------------------------------------------------------------------------------------
// Compile-time layout for one (K, V) pair.
// ------------------------------------------------------------------------------------------------
__host__ __device__ constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

template <int K_, int V_>
struct Cfg {
    static constexpr int K = K_, V = V_;
    static_assert(K == 8 || K == 16, "K must be 8 or 16");
    static_assert(V == 64 || V == 128, "V must be 64 or 128");
    // Feature blocks of 16 features (bf16: one 32-byte row per token per block).
    static constexpr int NBLK = (K == 16) ? 10 : 3;
    static constexpr int PP = NBLK * 16;  // padded feature count (153 -> 160, 45 -> 48)
    // V = 64: z rides as row 64 of S^T, the ones column of [v | 1] is a spare operand block, and
    // TMEM/SMEM leave room to double-buffer O and the bf16 state operand (pipelined order
    // AV, QK, UPD, RO). V = 128: a small extra MMA accumulates z; single buffers (order AV, RO,
    // QK, UPD).
    static constexpr bool ZROW = (V == 64);
    static constexpr bool FAST = (V == 64);
    static constexpr int NO = V + 16;        // O columns: V numerators, den (rowsum + z_hi), z_lo
    // A stored state (aggregate slot) is feature-major: element (feature c, row r) at
    // c * SROWS + r, rows r < V of S^T and row V = z, so that the threads of a warp (consecutive
    // rows) access consecutive floats.
    static constexpr int SROWS = V + 1;
    static constexpr int SLOT = SROWS * PP;  // floats per stored state

    // TMEM columns (forward kernel)
    static constexpr int TM_S = 0;                                  // S^T (lanes = value dim)
    static constexpr int TM_SC = align_up(PP, 32);                  // s (fp32 scores)
    static constexpr int TM_A = FAST ? TM_SC + 128 : TM_SC;         // A (bf16), over s if V=128
    static constexpr int TM_O0 = FAST ? TM_A + 64 : TM_SC + 128;    // O (lanes = query rows)
    static constexpr int TM_O1 = FAST ? TM_O0 + NO : TM_O0;
    static constexpr int TM_Z = align_up(TM_O1 + NO, 32);           // z tiles (V = 128)
    static_assert(ZROW ? (TM_O1 + NO <= 512) : (TM_Z + 32 <= 512), "TMEM overflow");

    // Shared memory (forward kernel), byte offsets from a 1024-aligned base.
    static constexpr int RAW = kChunk * 32;    // one raw q or k tile: 128 rows x 16 bf16
    static constexpr int VT = kChunk * V * 2;  // one v tile
    static constexpr int PHI = NBLK * 4096;    // one feature tile: NBLK blocks of 128 x 16 bf16
    static constexpr int SBF_ROWS = V + 16;    // rows of the bf16 state operand [S | z_hi z_lo 0]
    static constexpr int SBF_BLK = SBF_ROWS * 32;
    static constexpr int SBF = NBLK * SBF_BLK;
    static constexpr int NSBF = FAST ? 2 : 1;
    // q/k/v stages in flight: as many as fit (loads are issued NST - 1 chunks ahead)
    static constexpr int NST = (K == 16) ? 2 : 3;
    static constexpr int OFF_RAWQ = 0;
    static constexpr int OFF_RAWK = OFF_RAWQ + NST * RAW;
    static constexpr int OFF_V = OFF_RAWK + NST * RAW;
    // ones block: one 16-token k-step of an MN-major SW128 atom (2 KB), re-used by every k-step.
    // A v tile reaches it with a positive leading-byte offset: the stages' v tiles the one right
    // after them, the lead-in stages' v tiles a copy at the end of shared memory.
    static constexpr int ONES = ZROW ? 2048 : 0;
    static constexpr int OFF_ONES = OFF_V + NST * VT;
    static constexpr int OFF_PHIK = OFF_ONES + ONES;
    static constexpr int OFF_PHIQ = OFF_PHIK + PHI;
    static constexpr int OFF_SBF = OFF_PHIQ + PHI;
    static constexpr int OFF_ZONES = align_up(OFF_SBF + NSBF * SBF, 1024);
    // output staging for TMA stores: 128 rows x 32 fp32 (SW128), one quarter/half of a tile
    static constexpr int OST = kChunk * 128;
    // two staging buffers where they fit, so that a piece never waits for the previous one's
    // store to have left shared memory
    static constexpr int NOST = (K == 16 && V == 128) ? 1 : 2;
    // rows of one output TMA box: with a single staging buffer every epilogue warp stores its own
    // 32 rows (no cross-warp barrier); with two, one thread stores all 128 rows of a piece
    static constexpr int EPI_ROWS = NOST == 1 ? 32 : 128;
    static constexpr int OFF_OST = OFF_ZONES + 1024;
    static constexpr int OFF_BAR = OFF_OST + NOST * OST;
    // Lead-in stages (V = 64): k and v tiles of NLS lead-in chunks in flight. They use memory
    // that the range's chunks first need after the lead-in: for K = 16 the state operand buffers
    // (stages 0, 1) and the output staging (stage 2); for K = 8, whose state operands are small,
    // a region of their own (stages 0, 1) and the output staging (stage 2).
    static constexpr int NLS = FAST ? 3 : 0;
    static constexpr int OFF_LEAD = align_up(OFF_BAR + 256, 1024);
    static constexpr int LEAD_OWN = (FAST && K == 8) ? 2 * (VT + RAW) : 0;
    static constexpr int LEAD_BASE = K == 16 ? OFF_SBF : OFF_LEAD;
    __host__ __device__ static constexpr int lead_v(int i) { return i < 2 ? LEAD_BASE + i * VT : OFF_OST; }
    __host__ __device__ static constexpr int lead_k(int i) {
        return i < 2 ? LEAD_BASE + 2 * VT + i * RAW : OFF_OST + VT;
    }
    static_assert(!FAST || K != 16 || 2 * (VT + RAW) <= NSBF * SBF, "lead-in stages over the state operands");
    static_assert(!FAST || VT + RAW <= NOST * OST, "lead-in stage over the output staging");
    static constexpr int OFF_LONES = align_up(OFF_LEAD + LEAD_OWN, 1024);
    static constexpr int SMEM_FWD = OFF_LONES + (FAST ? ONES : 0) + 1024;  // + alignment slack
    // The z MMA reads 8 feature blocks (32 KB) from the phi(k) tile start; they must be inside
    // the allocation even when the tile has fewer blocks (their rows of D are never read).
    static_assert(ZROW || OFF_PHIK + 8 * 4096 <= OFF_BAR, "z MMA window leaves shared memory");
    static_assert(SMEM_FWD <= 232448, "shared memory budget");

    // Shared memory (aggregate kernel): A_NPHIK f(k) buffers and as many k/v stages as fit (at
    // most 8), so that the loads run far enough ahead to hide the memory latency. Three f(k)
    // buffers where they leave room for 4+ stages (the builders then run two chunks ahead of the
    // state update); for K = 16, V = 128 one, since a second would cost the fifth stage and the
    // state update (no z MMAs) is short next to the memory latency; else two.
    // V = 128: per-warp partial sums of z (two buffers, used by alternate pieces, of 8 builder
    // warps x half a feature row, fp32)
    static constexpr int A_ZRED = ZROW ? 0 : 2 * 8 * ((NBLK + 1) / 2) * 16 * 4;
    static constexpr int A_NPHIK = (!ZROW && K == 16) ? 1
                                   : (232448 - 4352 - align_up(3 * PHI, 1024)) / (RAW + VT) >= 4 ? 3 : 2;
    // (alignment slack, barriers, z partial sums, ones block)
    static constexpr int A_NST_FIT =
        (232448 - 1024 - 256 - A_ZRED - ONES - align_up(A_NPHIK * PHI, 1024)) / (RAW + VT);
    static constexpr int A_NST = A_NST_FIT < 8 ? A_NST_FIT : 8;
    static constexpr int A_OFF_PHIK = 0;
    static constexpr int A_OFF_RAWK = align_up(A_NPHIK * PHI, 1024);
    static constexpr int A_OFF_V = A_OFF_RAWK + A_NST * RAW;
    static constexpr int A_OFF_ONES = A_OFF_V + A_NST * VT;
    static constexpr int A_OFF_BAR = A_OFF_ONES + ONES;
    static constexpr int A_OFF_ZRED = A_OFF_BAR + 256;
    static constexpr int SMEM_AGG = A_OFF_ZRED + A_ZRED + 1024;
    static_assert(8 * (2 * A_NST + 2 * A_NPHIK + 6) + 8 <= A_OFF_ZRED - A_OFF_BAR, "barriers (aggregate)");
    static_assert(SMEM_AGG <= 232448, "shared memory budget (aggregate)");
};

// Swizzled byte offsets inside 32-byte-row (SW32) and 128-byte-row (SW128) tiles whose base is
// aligned to the swizzle atom: the 16-byte chunk index is XORed with address bits above the row.
__device__ __forceinline__ uint32_t sw32(int row, int half) {
    return static_cast<uint32_t>(row * 32 + ((half ^ ((row >> 2) & 1)) << 4));
}
__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
    return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}
// Advance a shared-memory descriptor's start address by `bytes` (stays inside the 14-bit field).
__device__ __forceinline__ uint64_t dadd(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }
// v_c operand at k-step j (16 tokens = 2048 bytes of an MN-major SW128 tile). With a ones block
// as the second 64-wide atom (LBO measured from the start address), the LBO shrinks as the start
// advances, so every k-step reads the same 2 KB ones block.
template <bool ONES_ATOM>
__device__ __forceinline__ uint64_t v_step(uint64_t d, int j) {
    const uint64_t step = static_cast<uint64_t>(2048 * j) >> 4;
    return ONES_ATOM ? d + step - (step << 16) : d + step;
}

__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&p);
}
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
    return (static_cast<uint64_t>(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
}
// Two fp32 values (as a packed pair) times two fp32 factors in one packed multiply.
__device__ __forceinline__ void mul_f32x2(float &a, float &b, uint64_t f) {
    uint64_t x = pack_f32x2(a, b), y;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(y) : "l"(x), "l"(f));
    a = __uint_as_float(static_cast<uint32_t>(y));
    b = __uint_as_float(static_cast<uint32_t>(y >> 32));
}
// bf16x2 of the Taylor weights 1 + c1 s + c2 s^2 for two fp32 scores, evaluated as
// fma(s, fma(c2, s, c1), 1) on packed fp32 pairs (square kept in fp32).
__device__ __forceinline__ uint32_t taylor2(uint32_t s_lo, uint32_t s_hi, uint64_t C2, uint64_t C1,
                                           uint64_t ONE) {
    uint32_t out;
    asm("{\n\t.reg .b64 s2, t2, a2;\n\t.reg .b32 alo, ahi;\n\t"
        "mov.b64 s2, {%1, %2};\n\t"
        "fma.rn.f32x2 t2, s2, %3, %4;\n\t"
        "fma.rn.f32x2 a2, s2, t2, %5;\n\t"
        "mov.b64 {alo, ahi}, a2;\n\t"
        "cvt.rn.bf16x2.f32 %0, ahi, alo;\n\t}"
        : "=r"(out)
        : "r"(s_lo), "r"(s_hi), "l"(C2), "l"(C1), "l"(ONE));
    return out;
}

// Builds one token's row of a feature tile from its raw 16-wide bf16 row (SW32 tile) into NBLK
// SW32 blocks of 16 features. Products are exact bf16 products rounded once (mul.rn.bf16x2).
// K = 16: block 0 = x, 1 = x_a^2, 1+d (d = 1..7) = x_a x_{(a+d) mod 16}, 9 = [x_a x_{a+8} (a<8),
//         1, 0 x 7].
// K = 8:  block 0 = [x, x_a^2], 1 = [x_a x_{a+1}, x_a x_{a+2}] (mod 8), 2 = [x_a x_{a+3} (mod 8),
//         x_a x_{a+4} (a<4), 1, 0 x 3].
// Every unordered pair a < b appears exactly once. The squares are multiplied by half2 (a bf16
// pair): (1, 1) gives f(k), (1/2, 1/2) the query side f~(q) with halved squares, so that
// f~(q).f(k) = 1 + q.k + (q.k)^2 / 2 (a power of two is exact, so both sides share this one code
// path). The scale is not applied to q: the state conversion multiplies feature c of the fp32
// state by scale^degree(c) before the state is rounded to bf16, so that the scale enters once,
// in fp32, and q is never rounded after scaling. Only blocks f_lo <= f < f_hi are built (two
// threads can share a token row).
// Out of line: the q and k builders share one copy of the code, which keeps the kernel's
// instruction-cache footprint small.
constexpr uint32_t kBf16One2 = 0x3F803F80u;   // bf16 pair (1.0, 1.0)
constexpr uint32_t kBf16Half2 = 0x3F003F00u;  // bf16 pair (0.5, 0.5)
template <int K>
__device__ __noinline__ void build_features(uint32_t raw, uint32_t phi, int t, uint32_t half2, int f_lo,
                                            int f_hi) {
    const uint32_t rb = raw + static_cast<uint32_t>(t) * 32u;
    const uint32_t sw = static_cast<uint32_t>(((t >> 2) & 1) << 4);
    const uint4 lo = ld_shared_v4(rb + sw);
    auto store_blk = [&](int f, uint32_t p0, uint32_t p1, uint32_t p2, uint32_t p3, uint32_t p4,
                         uint32_t p5, uint32_t p6, uint32_t p7) {
        const uint32_t base = phi + static_cast<uint32_t>(f) * 4096u + static_cast<uint32_t>(t) * 32u;
        st_shared_v4(base + sw, p0, p1, p2, p3);
        st_shared_v4(base + (16u ^ sw), p4, p5, p6, p7);
    };
    constexpr uint32_t ONE_ZERO = 0x00003F80u;  // bf16 pair (1.0, 0.0)
    auto sq = [&](uint32_t x) { return bmul2(bmul2(x, half2), x); };
    auto in = [&](int f) { return f_lo <= f && f < f_hi; };
    if constexpr (K == 16) {
        const uint4 hi = ld_shared_v4(rb + (16u ^ sw));
        const uint32_t X[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
        if (in(0)) store_blk(0, X[0], X[1], X[2], X[3], X[4], X[5], X[6], X[7]);
        if (in(1))
            store_blk(1, sq(X[0]), sq(X[1]), sq(X[2]), sq(X[3]), sq(X[4]), sq(X[5]), sq(X[6]), sq(X[7]));
#pragma unroll
        for (int d = 1; d <= 7; ++d) {
            if (!in(1 + d)) continue;
            uint32_t P[8];
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                uint32_t R;
                if (d % 2 == 0) {
                    R = X[(m + d / 2) & 7];
                } else {
                    R = __byte_perm(X[(m + (d - 1) / 2) & 7], X[(m + (d + 1) / 2) & 7], 0x5432);
                }
                P[m] = bmul2(X[m], R);
            }
            store_blk(1 + d, P[0], P[1], P[2], P[3], P[4], P[5], P[6], P[7]);
        }
        if (in(9))
            store_blk(9, bmul2(X[0], X[4]), bmul2(X[1], X[5]), bmul2(X[2], X[6]), bmul2(X[3], X[7]),
                      ONE_ZERO, 0u, 0u, 0u);
    } else {
        const uint32_t X[4] = {lo.x, lo.y, lo.z, lo.w};
        if (in(0)) store_blk(0, X[0], X[1], X[2], X[3], sq(X[0]), sq(X[1]), sq(X[2]), sq(X[3]));
        uint32_t R1[4], R3[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            R1[m] = __byte_perm(X[m], X[(m + 1) & 3], 0x5432);
            R3[m] = __byte_perm(X[(m + 1) & 3], X[(m + 2) & 3], 0x5432);
        }
        if (in(1))
            store_blk(1, bmul2(X[0], R1[0]), bmul2(X[1], R1[1]), bmul2(X[2], R1[2]), bmul2(X[3], R1[3]),
                      bmul2(X[0], X[1]), bmul2(X[1], X[2]), bmul2(X[2], X[3]), bmul2(X[3], X[0]));
        if (in(2))
            store_blk(2, bmul2(X[0], R3[0]), bmul2(X[1], R3[1]), bmul2(X[2], R3[2]), bmul2(X[3], R3[3]),
                      bmul2(X[0], X[2]), bmul2(X[1], X[3]), ONE_ZERO, 0u);
    }
}

// f(k) of token t for feature blocks [F0, F1) (half of the row, fixed at compile time), stored as
// build_features stores it with half2 = (1, 1) (the same products, bit for bit), with every
// feature also added to z[16 (f - F0) + j] (fp32; feature j of block f), so that the aggregate
// pass gets z = sum f(k) without an MMA.
template <int K, int F0, int F1>
__device__ __forceinline__ void build_k_features_acc(uint32_t raw, uint32_t phi, int t, float (&z)[(F1 - F0) * 16]) {
    const uint32_t rb = raw + static_cast<uint32_t>(t) * 32u;
    const uint32_t sw = static_cast<uint32_t>(((t >> 2) & 1) << 4);
    auto put = [&](int f, const uint32_t (&w)[8]) {
        const uint32_t base = phi + static_cast<uint32_t>(f) * 4096u + static_cast<uint32_t>(t) * 32u;
        st_shared_v4(base + sw, w[0], w[1], w[2], w[3]);
        st_shared_v4(base + (16u ^ sw), w[4], w[5], w[6], w[7]);
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            z[16 * (f - F0) + 2 * m] += __uint_as_float(w[m] << 16);
            z[16 * (f - F0) + 2 * m + 1] += __uint_as_float(w[m] & 0xFFFF0000u);
        }
    };
    constexpr uint32_t ONE_ZERO = 0x00003F80u;  // bf16 pair (1.0, 0.0)
    const uint4 lo = ld_shared_v4(rb + sw);
    if constexpr (K == 16) {
        const uint4 hi = ld_shared_v4(rb + (16u ^ sw));
        const uint32_t X[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
        for (int f = F0; f < F1; ++f) {
            uint32_t w[8];
            if (f == 0) {
#pragma unroll
                for (int m = 0; m < 8; ++m) w[m] = X[m];
            } else if (f == 1) {
#pragma unroll
                for (int m = 0; m < 8; ++m) w[m] = bmul2(X[m], X[m]);
            } else if (f <= 8) {
                const int d = f - 1;
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const uint32_t R = (d % 2 == 0)
                                           ? X[(m + d / 2) & 7]
                                           : __byte_perm(X[(m + (d - 1) / 2) & 7], X[(m + (d + 1) / 2) & 7], 0x5432);
                    w[m] = bmul2(X[m], R);
                }
            } else {
                w[0] = bmul2(X[0], X[4]);
                w[1] = bmul2(X[1], X[5]);
                w[2] = bmul2(X[2], X[6]);
                w[3] = bmul2(X[3], X[7]);
                w[4] = ONE_ZERO;
                w[5] = w[6] = w[7] = 0u;
            }
            put(f, w);
        }
    } else {
        const uint32_t X[4] = {lo.x, lo.y, lo.z, lo.w};
#pragma unroll
        for (int f = F0; f < F1; ++f) {
            uint32_t w[8];
            if (f == 0) {
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    w[m] = X[m];
                    w[4 + m] = bmul2(X[m], X[m]);
                }
            } else if (f == 1) {
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    w[m] = bmul2(X[m], __byte_perm(X[m], X[(m + 1) & 3], 0x5432));
                    w[4 + m] = bmul2(X[m], X[(m + 1) & 3]);
                }
            } else {
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    w[m] = bmul2(X[m], __byte_perm(X[(m + 1) & 3], X[(m + 2) & 3], 0x5432));
                w[4] = bmul2(X[0], X[2]);
                w[5] = bmul2(X[1], X[3]);
                w[6] = ONE_ZERO;
                w[7] = 0u;
            }
            put(f, w);
        }
    }
}

// Sums n values over the 32 lanes of a warp (v[0..n) per lane, fp32) by recursive halving: at
// each step a lane keeps one half of its values, adds its partner's copy of that half and sends
// the other half, so the warp moves about n values in total instead of 5 n. Where the count
// turns odd the remaining lane bits are summed whole (those lanes then hold equal sums).
// After the call lane l holds z_final_count(n, 16) sums of consecutive values from index base.
__host__ __device__ constexpr int z_final_count(int n, int o) {
    return o == 0 ? n : (n % 2 == 0 ? z_final_count(n / 2, o / 2) : z_final_count(n, o / 2));
}
// lane bits whose lanes hold duplicate sums (only the lane with those bits clear stores them)
__host__ __device__ constexpr int z_dup_mask(int n, int o) {
    return o == 0 ? 0 : (n % 2 == 0 ? z_dup_mask(n / 2, o / 2) : (o | z_dup_mask(n, o / 2)));
}
template <int NV, int n, int o>
__device__ __forceinline__ void z_reduce_scatter(float (&v)[NV], int lane, int &base) {
    if constexpr (o > 0) {
        if constexpr (n % 2 == 0) {
            const bool up = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < n / 2; ++i) {
                const float send = up ? v[i] : v[i + n / 2];
                const float keep = up ? v[i + n / 2] : v[i];
                v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, o);
            }
            if (up) base += n / 2;
            z_reduce_scatter<NV, n / 2, o / 2>(v, lane, base);
        } else {
#pragma unroll
            for (int i = 0; i < n; ++i) v[i] += __shfl_xor_sync(0xFFFFFFFFu, v[i], o);
            z_reduce_scatter<NV, n, o / 2>(v, lane, base);
        }
    }
}

// ------------------------------------------------------------------------------------------------
// Work partition. The heads are dealt into L lanes (lane r: heads h = r, r + L, ...), and each
// lane's B*(H/L)*n_c chunks, ordered head-major, are cut into G contiguous ranges, the same cut
// in every lane. CTA j L + r takes range j of lane r. The L CTAs of a group then work on the same
// positions of L adjacent heads at the same time, and the q/k rows of those heads, which share
// 128-byte lines, are read from DRAM once instead of once per head.
// ------------------------------------------------------------------------------------------------
// Lanes: as many as adjacent heads' q/k rows fill a 128-byte line (4 for K = 16, 8 for K = 8),
// halved until they divide H and the CTA count (sms CTAs over N chunks) splits evenly over them.
__host__ __device__ inline int choose_lanes(int K, int H, long long N, int sms) {
    int L = 128 / (2 * K);
    while (L > 1 && (H % L != 0 || (N > sms && sms % L != 0) || sms < L)) L /= 2;
    return L;
}
struct Part {
    long long g0, g1;
};
__host__ __device__ __forceinline__ Part cta_range(long long N, int G, int i) {
    return Part{N * i / G, N * (i + 1) / G};
}
// The range ends inside a head, so its last stretch of chunks has a partial state to publish.
__host__ __device__ __forceinline__ bool has_aggregate(long long N, int G, int i, int n_c) {
    const Part p = cta_range(N, G, i);
    return p.g1 > p.g0 && (p.g1 % n_c) != 0;
}
// The range starts inside a head and stays inside it, so its aggregate continues the previous
// range's prefix.
__host__ __device__ __forceinline__ bool continues_prefix(long long N, int G, int i, int n_c) {
    if (i == 0) return false;
    const Part p = cta_range(N, G, i);
    return p.g1 > p.g0 && (p.g0 % n_c) != 0 && (p.g0 / n_c) == ((p.g1 - 1) / n_c);
}
// Partial states that make up the prefix of range i (which starts inside a head): slots
// i - m .. i - 1, where the ranges i - m + 1 .. i - 1 continue the prefix of the one before them.
// m stops at max_chain (1 when a scan has already summed each run into its last slot).
__host__ __device__ __forceinline__ int prefix_chain_len(long long N, int G, int i, int n_c, int max_chain) {
    int m = 1;
    for (int j = i - 1; m < max_chain && continues_prefix(N, G, j, n_c); --j) ++m;
    return m;
}

// ------------------------------------------------------------------------------------------------
// Work plan of the aggregate pass (host side; also used by the partition check)
// ------------------------------------------------------------------------------------------------
constexpr int kMaxRanges = 256;             // upper bound on G (one range per SM)
constexpr int kMaxPieces = 2 * kMaxRanges;  // stretches + aggregate-CTA boundaries inside them

// The stretches (the last stretch of every range that ends inside a head), concatenated in range
// order and cut into n_cta segments of equal length, one per aggregate CTA, so that no CTA waits
// on a long stretch while others idle. A segment's part in one stretch is a piece; each piece's
// partial state has its own slot (slot index = piece index, pieces in concatenated order).
struct AggPieces {
    int n_cta;                           // aggregate CTAs
    int n;                               // pieces (= slots)
    uint16_t cta_first[kMaxRanges + 1];  // CTA j sums pieces [cta_first[j], cta_first[j + 1])
    int32_t g0[kMaxPieces];              // first chunk (global chunk index) of each piece
    int32_t len[kMaxPieces];             // chunks of each piece
};
// Prefix of forward CTA r: the sum of slots slot[r] .. slot[r] + cnt[r] - 1 (cnt = 0: the range
// starts at a head start and needs none).
struct Prefixes {
    uint16_t slot[kMaxRanges];
    uint8_t cnt[kMaxRanges];
};
// Runs of slots that a scan turns into inclusive prefixes: one per chain of stretches in a head
// with two or more pieces.
struct ScanRuns {
    int n;                         // number of runs
    uint16_t start[kMaxRanges];    // first slot of the run
    uint16_t len[kMaxRanges];      // slots in the run (>= 2)
};
struct AggPlan {
    AggPieces pieces;
    Prefixes pre;
    ScanRuns runs;
    bool scan;  // some prefix has more than kMaxChain slots: the scan kernel runs, every cnt is 1
};

// Completes a plan whose pieces are set: the prefix of every range that starts inside a head (the
// pieces of the chain of stretches before it in that head) and, when some prefix has more than
// kMaxChain pieces, the scan runs (one per chain of two or more pieces; each prefix is then the
// last slot of its chain's part of the run).
inline void finish_agg_plan(long long N, int G, int n_c, int ns, const int *st_range, const int *first_piece,
                            const int *last_piece, AggPlan &P) {
    int stretch_of[kMaxRanges], last_of[kMaxRanges];
    for (int i = 0; i < G; ++i) stretch_of[i] = -1;
    for (int s = 0; s < ns; ++s) stretch_of[st_range[s]] = s;
    P.scan = false;
    for (int r = 0; r < G; ++r) {
        P.pre.cnt[r] = 0;
        P.pre.slot[r] = 0;
        last_of[r] = -1;
        if (cta_range(N, G, r).g0 % n_c == 0) continue;
        const int m = prefix_chain_len(N, G, r, n_c, G);
        const int f = first_piece[stretch_of[r - m]], l = last_piece[stretch_of[r - 1]];
        P.pre.slot[r] = static_cast<uint16_t>(f);
        P.pre.cnt[r] = static_cast<uint8_t>(l - f + 1 < 255 ? l - f + 1 : 255);
        last_of[r] = l;
        if (l - f + 1 > kMaxChain) P.scan = true;
    }
    P.runs.n = 0;
    if (!P.scan) return;
    for (int s = 0; s < ns; ++s) {
        if (continues_prefix(N, G, st_range[s], n_c)) continue;
        int t = s + 1;
        while (t < ns && st_range[t] == st_range[t - 1] + 1 && continues_prefix(N, G, st_range[t], n_c)) ++t;
        const int f = first_piece[s], l = last_piece[t - 1];
        if (l - f + 1 >= 2) {
            P.runs.start[P.runs.n] = static_cast<uint16_t>(f);
            P.runs.len[P.runs.n] = static_cast<uint16_t>(l - f + 1);
            ++P.runs.n;
        }
    }
    for (int r = 0; r < G; ++r)
        if (P.pre.cnt[r] > 0) {
            P.pre.slot[r] = static_cast<uint16_t>(last_of[r]);
            P.pre.cnt[r] = 1;
        }
}

// Builds the plan for G ranges over N chunks (n_c per head). Two candidates: one aggregate CTA per
// stretch, or the stretches cut evenly over up to max_cta CTAs (only if it needs at most max_slots
// slots). The balanced cut is taken when its estimated critical path, in chunks of aggregate work,
// is clearly shorter: the longest CTA load, plus about two chunks for the extra pieces' slot
// writes, plus about six when the plan needs the scan kernel (measured on GB300: an aggregate
// chunk takes about 0.5 us, the scan and its launch about 3 us).
inline void make_agg_plan(long long N, int G, int n_c, int max_cta, int max_slots, AggPlan &P) {
    int ns = 0;
    int st_range[kMaxRanges];
    long long st_g0[kMaxRanges], st_len[kMaxRanges], L = 0, longest = 0;
    for (int i = 0; i < G; ++i) {
        if (!has_aggregate(N, G, i, n_c)) continue;
        const Part p = cta_range(N, G, i);
        const long long hs = ((p.g1 - 1) / n_c) * n_c;
        const long long ga = p.g0 > hs ? p.g0 : hs;
        st_range[ns] = i;
        st_g0[ns] = ga;
        st_len[ns] = p.g1 - ga;
        L += st_len[ns];
        longest = st_len[ns] > longest ? st_len[ns] : longest;
        ++ns;
    }
    int first_piece[kMaxRanges], last_piece[kMaxRanges];
    // one aggregate CTA per stretch
    AggPieces &A = P.pieces;
    A.n_cta = ns;
    for (int s = 0; s < ns; ++s) {
        A.cta_first[s] = static_cast<uint16_t>(s);
        A.g0[s] = static_cast<int32_t>(st_g0[s]);
        A.len[s] = static_cast<int32_t>(st_len[s]);
        first_piece[s] = last_piece[s] = s;
    }
    A.cta_first[ns] = static_cast<uint16_t>(ns);
    A.n = ns;
    finish_agg_plan(N, G, n_c, ns, st_range, first_piece, last_piece, P);
    const int cap = max_cta < kMaxRanges ? max_cta : kMaxRanges;
    const int n_cta = static_cast<int>(L < cap ? L : cap);
    if (ns == 0 || n_cta <= ns) return;
    constexpr long long kPiecePenalty = 2, kScanPenalty = 6;
    const long long cost_one = longest + (P.scan ? kScanPenalty : 0);
    const long long bal_load = (L + n_cta - 1) / n_cta;
    if (10 * (bal_load + kPiecePenalty) >= 85 * cost_one / 10) return;  // no clear gain even without a scan
    // the balanced cut: CTA j sums concatenated positions [L j / n_cta, L (j + 1) / n_cta)
    static thread_local AggPlan B;
    int bfirst[kMaxRanges], blast[kMaxRanges];
    int n = 0, s = 0;
    long long s_off = 0;  // concatenated offset of stretch s
    B.pieces.n_cta = n_cta;
    for (int j = 0; j < n_cta; ++j) {
        const long long x1 = L * (j + 1) / n_cta;
        B.pieces.cta_first[j] = static_cast<uint16_t>(n);
        for (long long x = L * j / n_cta; x < x1;) {
            while (x >= s_off + st_len[s]) s_off += st_len[s++];
            const long long end = x1 < s_off + st_len[s] ? x1 : s_off + st_len[s];
            if (n >= kMaxPieces || n >= max_slots) return;  // keep one CTA per stretch
            B.pieces.g0[n] = static_cast<int32_t>(st_g0[s] + (x - s_off));
            B.pieces.len[n] = static_cast<int32_t>(end - x);
            if (x == s_off) bfirst[s] = n;
            blast[s] = n;
            ++n;
            x = end;
        }
    }
    B.pieces.cta_first[n_cta] = static_cast<uint16_t>(n);
    B.pieces.n = n;
    finish_agg_plan(N, G, n_c, ns, st_range, bfirst, blast, B);
    const long long cost_bal = bal_load + kPiecePenalty + (B.scan ? kScanPenalty : 0);
    if (100 * cost_bal < 85 * cost_one) P = B;
}

// ------------------------------------------------------------------------------------------------
// Forward CTAs' ranges (host plan, read by the forward kernel). Range j of a lane is its chunks
// [g0[j], g0[j + 1]). A range that starts inside a head continues the state of that head's chunks
// before it, which it gets in one of two ways, the same for every range of a call:
//  - from slots: the aggregate pass wrote partial states, and the CTA sums slots slot[j] ..
//    slot[j] + cnt[j] - 1 (cnt = 0 at a head start); the chunks are cut evenly (cta_range);
//  - by a lead-in (V = 64, lead_in set): the CTA first runs the state update alone over the
//    g0[j] % n_c chunks of its head before g0[j], so that the call is the forward kernel alone;
//    the cut then gives each range as many chunks as its lead-in leaves room for (lead_cut).
// ------------------------------------------------------------------------------------------------
struct Ranges {
    int32_t g0[kMaxRanges + 1];
    uint16_t slot[kMaxRanges];
    uint8_t cnt[kMaxRanges];
    // launch order: CTA group i (blockIdx / L) takes range order[i]. The block scheduler hands
    // out CTAs in index order, so the ranges that cost most go first: calls issued back to back
    // start a call's CTAs on the SMs the previous call frees first, and those finish their
    // set-up before that call has ended.
    uint16_t order[kMaxRanges];
    int32_t lead_in;
};

// Cost model of a CTA, in thousandths of the time of one chunk of the forward pipeline (fitted to
// stage traces of single calls on GB300, V = 64, K = 16; one chunk is about 1.77 us):
// kStartCost for its start and end (set-up, the first loads, the pipeline's fill and drain),
// kLeadStart more when it has a lead-in, kLeadCost per lead-in chunk (the f(k) tile and the state
// update alone), 1000 per chunk of its range. The traces give 252 per lead-in chunk; calls issued
// back to back run lead-ins slower (more memory traffic at every call's start), and the cut with
// 325 measured fastest there (B4 T4096 H16 41.5 us per call against 44.2 with 252, 42.1 with
// 350, 46.0 with 220).
constexpr long long kStartCost = 4950, kLeadStart = 815, kLeadCost = 325;
__host__ __device__ inline long long range_cost(long long lead, long long len) {
    return kStartCost + (lead > 0 ? kLeadStart + lead * kLeadCost : 0) + 1000 * len;
}

// Lead-in cut of a lane's N chunks (n_c per head) into at most G ranges: the smallest makespan M
// (cost model above) for which the greedy cut, in which each range takes every chunk that M
// leaves room for after its lead-in, covers all N chunks. Writes the cut to R.g0 (ranges past
// the last are empty, g0 = N), sets R.lead_in, clears R.cnt, and returns M. A greedy range that
// ends further into a head leaves the next range less room, by less than it gained (kLeadCost <
// 1000) except when it leaves a head start (kLeadStart), so coverage grows with M nearly
// everywhere: the bisection finds the smallest M up to such steps, and the cut it returns always
// covers the chunks with every range within M.
inline long long lead_cut(long long N, int G, int n_c, Ranges &R) {
    auto greedy = [&](long long M, bool write) -> bool {
        long long g = 0;
        int j = 0;
        for (; j < G && g < N; ++j) {
            const long long s = g % n_c;
            const long long room = (M - range_cost(s, 0)) / 1000;
            if (room < 1) return false;
            if (write) R.g0[j] = static_cast<int32_t>(g);
            g = g + room < N ? g + room : N;
        }
        if (g < N) return false;
        if (write)
            for (; j <= G; ++j) R.g0[j] = static_cast<int32_t>(N);
        return true;
    };
    long long lo = 0, hi = range_cost(0, N);  // hi: the first range takes everything
    while (hi - lo > 1) {
        const long long mid = lo + (hi - lo) / 2;
        if (greedy(mid, false)) hi = mid;
        else lo = mid;
    }
    greedy(hi, true);
    R.lead_in = 1;
    for (int j = 0; j < G; ++j) {
        R.slot[j] = 0;
        R.cnt[j] = 0;
        R.order[j] = static_cast<uint16_t>(j);
    }
    // the non-empty ranges by cost, highest first (insertion sort: G <= 256); ties keep their order
    auto cost = [&](int j) { return range_cost(R.g0[j] % n_c, R.g0[j + 1] - R.g0[j]); };
    int used = 0;
    while (used < G && R.g0[used + 1] > R.g0[used]) ++used;
    for (int a = 1; a < used; ++a) {
        const uint16_t x = R.order[a];
        const long long cx = cost(x);
        int b = a;
        for (; b > 0 && cost(R.order[b - 1]) < cx; --b) R.order[b] = R.order[b - 1];
        R.order[b] = x;
    }
    return hi;
}

// Walks the chunks of a range without divisions: (b, h, c) advance like an odometer.
// g is a chunk index of one head lane (see choose_lanes): lane r's heads are h = hv L + r,
// hv < Hl = H / L.
struct Cursor {
    int n, last, c, hv, h, b, n_c, Hl, L, r;
    __host__ __device__ __forceinline__ void init(long long g, int nchunks, int n_c_, int Hl_, int L_, int r_) {
        n_c = n_c_;
        Hl = Hl_;
        L = L_;
        r = r_;
        n = 0;
        last = nchunks - 1;
        const long long head = g / n_c;
        c = static_cast<int>(g - head * n_c);
        hv = static_cast<int>(head % Hl);
        b = static_cast<int>(head / Hl);
        h = hv * L + r;
    }
    __host__ __device__ __forceinline__ void next() {
        ++n;
        if (++c == n_c) {
            c = 0;
            if (++hv == Hl) {
                hv = 0;
                ++b;
            }
            h = hv * L + r;
        }
    }
    __device__ __forceinline__ int t0() const { return c * kChunk; }
    // a non-zero state precedes this chunk (inter-chunk read-out needed)
    __device__ __forceinline__ bool has_ro() const { return c > 0; }
    // a later chunk of this range continues the head (state update needed)
    __device__ __forceinline__ bool has_upd() const { return !(n == last || c == n_c - 1); }
    // the update accumulates onto a carried state
    __device__ __forceinline__ bool upd_acc() const { return c > 0; }
};

// ------------------------------------------------------------------------------------------------
// Forward kernel
// warp 0: TMA producer | warp 1: intra-chunk MMA issuer | warp 2: owns TMEM | warp 3: state MMA
// issuer | warps 4-7: Taylor weights A | warps 8-11: feature tiles + output epilogue |
// warps 12-15: state conversion S^T (fp32 TMEM) -> bf16 operand. V = 64: warps 2 and 15 compute
// Taylor weights too (warp 15 has no rows of S^T to convert).
// ------------------------------------------------------------------------------------------------
enum FwdBar {
    FB_TMA_FULL0 = 0, FB_STAGE_FREE0 = 3, FB_S_FULL = 6, FB_A_FULL, FB_O_FULL0, FB_O_FULL1,
    FB_O_FREE0, FB_O_FREE1, FB_AV_DONE, FB_PHIQ_FULL, FB_PHIQ_FREE, FB_PHIK_FULL, FB_PHIK_FREE,
    FB_UPD_DONE, FB_CONV_READ, FB_SBF_FULL, FB_DRAIN, FB_DRAIN_B, FB_AV_DONE1, FB_SBF_FULL1,
    FB_LFULL0, FB_LFREE0 = FB_LFULL0 + 3, FB_COUNT = FB_LFREE0 + 3  // lead-in stages (NLS <= 3)
};

// OBF: the output tile is written as bf16 (round to nearest even from the fp32 quotient) instead
// of fp32. LEADIN: the ranges that start inside a head run lead-ins (else they load their prefix
// from slots); each instance carries only its own way, which keeps the hot code of the other
// roles small.
template <int K, int V, bool OBF, bool LEADIN>
__global__ void __launch_bounds__(kFwdThreads, 1)
based_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                 const float *__restrict__ prefix, int T, int H, int n_c, long long N, int G, int L,
                 int lane_slots, float scale, const __grid_constant__ Ranges rg, int wait_prev) {
    using CF = Cfg<K, V>;
    constexpr bool FAST = CF::FAST;
    static_assert(!LEADIN || FAST, "lead-ins are built for V = 64");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + CF::OFF_BAR + 8 * FB_COUNT);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + CF::OFF_BAR + 8 * FB_COUNT + 4);
    auto BAR = [&](int i) -> uint32_t { return sb + CF::OFF_BAR + 8u * static_cast<uint32_t>(i); };
    // Conversion k fills state operand buffer k % NSBF and completes a phase of that buffer's
    // SBF_FULL barrier. With two buffers (V = 64) the state update of the next chunk is issued
    // before this chunk's read-out, so conversion k + 1 may complete before the read-out waits for
    // conversion k; one barrier per buffer keeps that waiter within one phase of its barrier.
    auto sbf_full_bar = [&](int k) -> int { return (CF::NSBF == 2 && (k & 1)) ? FB_SBF_FULL1 : FB_SBF_FULL; };
    auto sbf_full_par = [&](int k) -> uint32_t { return static_cast<uint32_t>(CF::NSBF == 2 ? (k >> 1) & 1 : k & 1); };

    // range j of head lane r (N, G: chunks and ranges of one lane; lane_slots: slots per lane)
    const int j_range = rg.order[static_cast<int>(blockIdx.x) / L], r_lane = static_cast<int>(blockIdx.x) % L;
    const int Hl = H / L;
    const long long g0 = rg.g0[j_range], g1 = rg.g0[j_range + 1];
    const int nchunks = static_cast<int>(g1 - g0);
    if (nchunks <= 0) return;
    // Lead-in (V = 64): the chunks of the first head before g0, whose state update alone runs
    // first. Lead-in chunk i is loaded into lead-in stage i % NLS (k and v only), chunk n of the
    // range into stage n % NST.
    const int n_lead = LEADIN ? static_cast<int>(g0 % n_c) : 0;
    constexpr int NLS = CF::NLS > 0 ? CF::NLS : 1;
    constexpr int kLeadAhead = 3;  // lead-in chunks prefetched into L2 ahead of the newest load
    constexpr bool kLeadOverSbf = LEADIN && K == 16;  // lead-in stages over the state operands
    auto stage_of = [&](int n) -> int { return n % CF::NST; };
    auto stage_par = [&](int n) -> uint32_t { return static_cast<uint32_t>((n / CF::NST) & 1); };
    BASED_TRACE_INIT;
    if (threadIdx.x == 0) BASED_TRACE_EV(63, 20);  // CTA start
#ifdef BASED_TRACE
    if (threadIdx.x == 0 && trace_buf_ != nullptr)
        trace_buf_[(static_cast<size_t>(blockIdx.x) * 64 + 63) * 32 + 22] = global_timer_ns();
#endif

    // k, v tiles of lead-in chunk i (cursor position cu) into lead-in stage i % NLS, completing on
    // LFULL
    auto issue_lead = [&](int i, const Cursor &cu) {
        const int ls = i % NLS;
        const uint32_t bar = BAR(FB_LFULL0 + ls);
        BASED_TRACE_EV(i, TE_LEAD_ISSUE);
        mbar_arrive_expect_tx(bar, CF::RAW + CF::VT);
        tma_load_4d(sb + CF::lead_k(ls), &tm_k, bar, 0, cu.h, cu.t0(), cu.b);
        tma_load_4d(sb + CF::lead_v(ls), &tm_v, bar, 0, cu.h, cu.t0(), cu.b);
    };
    // q, k, v tiles of chunk n (cursor position cu) into stage n % NST, completing on TMA_FULL
    auto issue_loads = [&](int n, const Cursor &cu) {
        const int s = n % CF::NST;
        const uint32_t bar = BAR(FB_TMA_FULL0 + s);
        BASED_TRACE_EV(n, TE_TMA_ISSUE);
        mbar_arrive_expect_tx(bar, 2 * CF::RAW + CF::VT);
        tma_load_4d(sb + CF::OFF_RAWQ + s * CF::RAW, &tm_q, bar, 0, cu.h, cu.t0(), cu.b);
        tma_load_4d(sb + CF::OFF_RAWK + s * CF::RAW, &tm_k, bar, 0, cu.h, cu.t0(), cu.b);
        tma_load_4d(sb + CF::OFF_V + s * CF::VT, &tm_v, bar, 0, cu.h, cu.t0(), cu.b);
        if constexpr (V == 128)
            tma_load_4d(sb + CF::OFF_V + s * CF::VT + 16384, &tm_v, bar, 64, cu.h, cu.t0(), cu.b);
    };
    const int n_early = nchunks < CF::NST ? nchunks : CF::NST;  // loads issued during set-up
    const int n_lead_early = n_lead < NLS ? n_lead : NLS;

    // ---- set-up: barriers, constant tiles, TMEM -------------------------------------------------
    if (threadIdx.x == 0) {
        // arrivals per phase: 1 = producer / commit, else one elected lane per warp of a group;
        // STAGE_FREE: one commit from each MMA issuer. V = 64: six warps compute the Taylor
        // weights and three convert the state (see the role split below).
        constexpr uint32_t NW = FAST ? 6 : 4, NC = FAST ? 3 : 4;
        const uint32_t counts[FB_COUNT] = {1, 1, 1, 2, 2, 2, 1, NW, 1, 1, 4, 4, 1, 4, 1, 4, 1, 1, NC, NC, 1, 1, 1, NC,
                                           1, 1, 1, 1, 1, 1};
        for (int i = 0; i < FB_COUNT; ++i) mbar_init(BAR(i), counts[i]);
        *abort_flag = 0;
        fence_mbar_init();
        // the first loads go out now (this thread is the TMA producer), so that their memory
        // latency overlaps the rest of the set-up
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        prefetch_tensormap(&tm_o);
        // The first kernel of a call is launched as a programmatic dependent of the previous
        // kernel in the stream (whose outputs may be q, k or v, and which may still read o):
        // nothing of this grid touches global memory before this thread's first loads, and those
        // wait for that kernel. After an aggregate pass the previous call has already completed.
        if (wait_prev) griddep_wait();
        if (LEADIN && n_lead > 0) {
            // the lead-in's first loads, then the next kLeadAhead lead-in chunks into L2 (each later
            // load prefetches the chunk kLeadAhead after it), so that the lead-in's loads wait on
            // L2 rather than DRAM
            Cursor cl;
            cl.init(g0 - n_lead, n_lead, n_c, Hl, L, r_lane);
            for (int i = 0; i < n_lead_early; ++i, cl.next()) issue_lead(i, cl);
            for (int i = n_lead_early; i < n_lead && i < NLS + kLeadAhead; ++i, cl.next()) {
                tma_prefetch_4d(&tm_k, 0, cl.h, cl.t0(), cl.b);
                tma_prefetch_4d(&tm_v, 0, cl.h, cl.t0(), cl.b);
            }
        }
        Cursor cu;
        cu.init(g0, nchunks, n_c, Hl, L, r_lane);
        for (int n = 0; n < n_early; ++n, cu.next()) issue_loads(n, cu);
    }
    // bf16 state operands: zero once (rows V+2.. stay zero; rows 0..V+1 are rewritten per use).
    // Lead-in stages over them: the conversion warps zero rows V+2.. after the lead-in instead.
    if (!(kLeadOverSbf && n_lead > 0))
        for (int i = threadIdx.x; i < CF::NSBF * CF::SBF / 16; i += kFwdThreads)
            st_shared_v4(sb + CF::OFF_SBF + 16u * i, 0u, 0u, 0u, 0u);
    if constexpr (CF::ZROW) {
        // ones block: an MN-major SW128 block whose element 0 is 1.0 in every token row. It is
        // the extra operand block behind v_c: A rows 64..127 of the state update (so that row 64
        // of S^T accumulates z) and B columns 64..79 of A [v | 1] (column 64 = rowsum A).
        for (int i = threadIdx.x; i < 2 * CF::ONES / 16; i += kFwdThreads)
            st_shared_v4(sb + (i < CF::ONES / 16 ? CF::OFF_ONES : CF::OFF_LONES - CF::ONES) + 16u * i, 0u, 0u, 0u,
                         0u);
        __syncthreads();
        if (threadIdx.x < 32)
            st_shared_u16(sb + (threadIdx.x < 16 ? CF::OFF_ONES : CF::OFF_LONES) + sw128(threadIdx.x & 15, 0), 0x3F80);
    }
    // ones column as a K-major SW32 operand: N row 0 = 16 ones, rows 1..15 = 0.
    if (threadIdx.x < 32)
        st_shared_v4(sb + CF::OFF_ZONES + 16u * threadIdx.x, threadIdx.x < 2 ? 0x3F803F80u : 0u,
                     threadIdx.x < 2 ? 0x3F803F80u : 0u, threadIdx.x < 2 ? 0x3F803F80u : 0u,
                     threadIdx.x < 2 ? 0x3F803F80u : 0u);
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_holder), 512);
        tmem_relinquish();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    if (threadIdx.x == 0) BASED_TRACE_EV(63, 21);  // set-up done
    // the next call's first kernel may start launching now; it waits for this grid before it
    // touches memory
    griddep_launch_dependents();

    if (warp == 0) {
        // ================================ TMA producer =========================================
        if (lane == 0) {
            int lead_issued = n_lead_early, issued = n_early;
            bool ok = true;
            if (LEADIN && n_lead > n_lead_early) {
                Cursor cl, cp;  // cp: kLeadAhead chunks ahead (L2 prefetch)
                cl.init(g0 - n_lead, n_lead, n_c, Hl, L, r_lane);
                cp.init(g0 - n_lead, n_lead, n_c, Hl, L, r_lane);
                for (int i = 0; i < n_lead_early; ++i) cl.next();
                for (int i = 0; i < NLS + kLeadAhead; ++i) cp.next();
                for (int i = n_lead_early; i < n_lead; ++i, cl.next()) {
                    const int ls = i % NLS;
                    if (!(ok = wait_bar(BAR(FB_LFREE0 + ls), ((i / NLS) - 1) & 1, abort_flag, SITE_STAGE_FREE)))
                        break;
                    issue_lead(i, cl);
                    ++lead_issued;
                    if (i + kLeadAhead < n_lead) {
                        tma_prefetch_4d(&tm_k, 0, cp.h, cp.t0(), cp.b);
                        tma_prefetch_4d(&tm_v, 0, cp.h, cp.t0(), cp.b);
                        cp.next();
                    }
                }
            }
            Cursor cu;
            cu.init(g0, nchunks, n_c, Hl, L, r_lane);
            for (int n = 0; n < n_early; ++n) cu.next();
            for (int n = n_early; ok && n < nchunks; ++n, cu.next()) {
                const int s = n % CF::NST;
                if (!wait_bar(BAR(FB_STAGE_FREE0 + s), ((n / CF::NST) - 1) & 1, abort_flag,
                              SITE_STAGE_FREE))
                    break;
                issue_loads(n, cu);
                ++issued;
            }
            if (*abort_flag) {  // let copies already in flight land before the CTA exits
                for (int m = issued - CF::NST; m < issued; ++m)
                    if (m >= 0)
                        wait_bar(BAR(FB_TMA_FULL0 + m % CF::NST), (m / CF::NST) & 1, nullptr,
                                 SITE_DRAIN, kDrainLimitNs);
                for (int m = lead_issued - NLS; m < lead_issued; ++m)
                    if (m >= 0)
                        wait_bar(BAR(FB_LFULL0 + m % NLS), (m / NLS) & 1, nullptr, SITE_DRAIN, kDrainLimitNs);
            }
        }
    } else if (warp == 1 || warp == 3) {
        // ============================== MMA issuers ============================================
        // Two threads issue MMAs, so that neither stream waits on the other's inputs: warp 1 the
        // intra-chunk products (s = q k^T, O = A [v | 1]), warp 3 the state products (S^T +=
        // [v | 1]^T f(k), O += f~(q) [S | z]). Each thread's MMAs run in its issue order; the
        // read-out accumulates into the O tile of a chunk only after AV_DONE shows that
        // A [v | 1] (which initialises it) has completed.
        if (lane == 0) {
            const uint32_t t_s = tmem + CF::TM_S, t_sc = tmem + CF::TM_SC, t_a = tmem + CF::TM_A,
                           t_z = tmem + CF::TM_Z;
            const uint32_t t_o0 = tmem + CF::TM_O0, t_o1 = tmem + CF::TM_O1;
            // Operand descriptors, computed once: per k-step and per stage only the start address
            // advances. Raw q/k tiles are K-major SW32; v_c is an MN-major SW128 operand whose
            // second 64-wide block is the ones block (V = 64, LBO depends on the stage) or the
            // upper half of v_c (V = 128).
            auto va_desc = [&](int s) {  // k-step 0 of stage s
                const uint32_t lbo = CF::ZROW ? CF::OFF_ONES - CF::OFF_V - s * CF::VT : 16384u;
                return smem_desc(sb + CF::OFF_V + s * CF::VT, lbo, 1024, LAYOUT_SW128);
            };
            const uint64_t d_va0 = va_desc(0), d_va1 = va_desc(1), d_va2 = va_desc(CF::NST > 2 ? 2 : 1);
            const uint64_t d_zones = smem_desc(sb + CF::OFF_ZONES, 16, 256, LAYOUT_SW32);
            Cursor cu;
            cu.init(g0, nchunks, n_c, Hl, L, r_lane);
            if (warp == 1) {
                // ---- intra-chunk stream: QK(0); per chunk QK(n + 1) and AV(n) ----
                constexpr uint32_t ID_QK = idesc_bf16_f32(128, 128, 0, 0);
                constexpr uint32_t ID_AV = idesc_bf16_f32(128, FAST ? CF::NO : V, 0, 1);
                constexpr uint32_t ID_RS = idesc_bf16_f32(128, 16, 0, 0);
                const uint64_t d_q = smem_desc(sb + CF::OFF_RAWQ, 16, 256, LAYOUT_SW32);
                const uint64_t d_k = smem_desc(sb + CF::OFF_RAWK, 16, 256, LAYOUT_SW32);
                // s = q k^T of chunk m into the scores tile, completing on S_FULL
                auto issue_qk = [&](int m) -> bool {
                    const int sm = stage_of(m);
                    if (!wait_bar(BAR(FB_TMA_FULL0 + sm), stage_par(m), abort_flag, SITE_TMA_FULL))
                        return false;
                    tc_fence_after();
                    mma_ss(t_sc, dadd(d_q, sm * CF::RAW), dadd(d_k, sm * CF::RAW), ID_QK, 0);
                    mma_commit(BAR(FB_S_FULL));
                    return true;
                };
                bool ok = issue_qk(0);
                for (int n = 0; ok && n < nchunks; ++n, cu.next()) {
                    const int s = stage_of(n);
                    const int ob = FAST ? (n & 1) : 0;
                    const uint64_t d_va = s == 0 ? d_va0 : (s == 1 ? d_va1 : d_va2);
                    const uint32_t t_out = ob ? t_o1 : t_o0;
                    if (!(ok = wait_bar(BAR(FB_A_FULL), n & 1, abort_flag, SITE_A_FULL))) break;
                    BASED_TRACE_EV(n, TE_A_READY);
                    // V = 64: the scores tile is free once A(n) is complete, so QK(n + 1) goes
                    // first when its tiles have landed, and the Taylor weights of chunk n + 1 are
                    // computed while AV(n) runs (they wait for AV_DONE before they overwrite A).
                    bool qk_next = false;
                    if constexpr (FAST) {
                        const int m = n + 1;
                        if (m < nchunks && mbar_test_wait(BAR(FB_TMA_FULL0 + stage_of(m)), stage_par(m))) {
                            if (!(ok = issue_qk(m))) break;
                            qk_next = true;
                            BASED_TRACE_EV(n, TE_QK_ISSUED);
                        }
                    }
                    if (FAST ? (n >= 2) : (n >= 1)) {
                        const uint32_t par = FAST ? (((n >> 1) - 1) & 1) : ((n - 1) & 1);
                        if (!(ok = wait_bar(BAR(FB_O_FREE0 + ob), par, abort_flag, SITE_O_FREE))) break;
                    }
                    tc_fence_after();
                    // O = A [v_c | 1]: numerators and rowsum A (V = 64: one MMA per 16 keys over
                    // the v block and the ones block; V = 128: a separate 16-column MMA for the
                    // rowsum)
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        mma_ts(t_out, t_a + 8 * j, v_step<CF::ZROW>(d_va, j), ID_AV, j > 0);
                    if constexpr (!FAST) {
#pragma unroll
                        for (int j = 0; j < 8; ++j) mma_ts(t_out + V, t_a + 8 * j, d_zones, ID_RS, j > 0);
                    }
                    // one AV_DONE barrier per O buffer (V = 64), so that this stream, which may run a
                    // chunk ahead, never completes two phases of a barrier the other still waits on
                    mma_commit(BAR(ob ? FB_AV_DONE1 : FB_AV_DONE));
                    if (!cu.has_ro()) mma_commit(BAR(FB_O_FULL0 + ob));  // no read-out follows
                    mma_commit(BAR(FB_STAGE_FREE0 + s));                  // QK(n) and AV(n) read it
                    BASED_TRACE_EV(n, TE_AV_ISSUED);
                    if (n + 1 < nchunks && !qk_next) {
                        if constexpr (!FAST) {
                            // the next s overwrites A (same TMEM columns): wait until A was read
                            if (!(ok = wait_bar(BAR(FB_AV_DONE), n & 1, abort_flag, SITE_AV_DONE))) break;
                        }
                        if (!(ok = issue_qk(n + 1))) break;
                        BASED_TRACE_EV(n, TE_QK_ISSUED);
                    }
                }
                // every MMA issued must finish before TMEM is released
                mma_commit(BAR(FB_DRAIN));
                wait_bar(BAR(FB_DRAIN), 0, nullptr, SITE_DRAIN, kDrainLimitNs);
            } else {
                // ---- state stream: per chunk UPD(n) and RO(n) ----
                constexpr uint32_t ID_RO = idesc_bf16_f32(128, CF::NO, 0, 0);
                constexpr uint32_t ID_UPD = idesc_bf16_f32(128, CF::PP, 1, 1);
                constexpr uint32_t ID_Z = idesc_bf16_f32(128, 16, 1, 0);
                const uint64_t d_sbf0 = smem_desc(sb + CF::OFF_SBF, 16, 256, LAYOUT_SW32);
                const uint64_t d_sbf1 = smem_desc(sb + CF::OFF_SBF + (CF::NSBF - 1) * CF::SBF, 16, 256, LAYOUT_SW32);
                const uint64_t d_phik = smem_desc(sb + CF::OFF_PHIK, 4096, 256, LAYOUT_SW32);
                const uint64_t d_phiq = smem_desc(sb + CF::OFF_PHIQ, 16, 256, LAYOUT_SW32);
                // ro_idx: read-outs (= conversions consumed); upd_idx, qn: fills of the f(k) and
                // the f~(q) tile consumed
                int ro_idx = 0, upd_idx = 0, qn = 0;
                bool ok = true;
                // release_stage >= 0: that stage is released as soon as f~(q_c) is built (the
                // builders have read its raw tiles; the commit tracks the state update issued
                // before, which read v_c)
                auto issue_ro = [&](int n, uint32_t t_out, int release_stage) -> bool {
                    // O += f~(q_c) [S | z_hi z_lo], after O = A [v_c | 1] has completed
                    if (!wait_bar(BAR(FB_PHIQ_FULL), qn & 1, abort_flag, SITE_PHIQ_FULL)) return false;
                    if (release_stage >= 0) mma_commit(BAR(FB_STAGE_FREE0 + release_stage));
                    // conversion ro_idx (one SBF_FULL barrier per state operand buffer)
                    if (!wait_bar(BAR(sbf_full_bar(ro_idx)), sbf_full_par(ro_idx), abort_flag, SITE_SBF_FULL))
                        return false;
                    const int ob = FAST ? (n & 1) : 0;
                    const uint32_t avp = FAST ? ((n >> 1) & 1) : (n & 1);
                    if (!wait_bar(BAR(ob ? FB_AV_DONE1 : FB_AV_DONE), avp, abort_flag, SITE_AV_DONE))
                        return false;
                    tc_fence_after();
                    const uint64_t db = (ro_idx & 1) ? d_sbf1 : d_sbf0;
#pragma unroll
                    for (int f = 0; f < CF::NBLK; ++f)
                        mma_ss(t_out, dadd(d_phiq, 4096 * f), dadd(db, CF::SBF_BLK * f), ID_RO, 1);
                    mma_commit(BAR(FB_PHIQ_FREE));
                    ++ro_idx;
                    ++qn;
                    return true;
                };
                auto issue_upd = [&](int n, uint64_t d_va) -> bool {
                    // S^T += [v_c | 1]^T f(k_c)  (z as row 64, or via the z MMAs)
                    if (!wait_bar(BAR(FB_PHIK_FULL), upd_idx & 1, abort_flag, SITE_PHIK_FULL)) return false;
                    if (cu.upd_acc()) {
                        // the previous conversion must have read S^T before it changes
                        const int r = FAST ? ro_idx : ro_idx - 1;
                        if (!wait_bar(BAR(FB_CONV_READ), r & 1, abort_flag, SITE_CONV_READ)) return false;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t acc = (j > 0 || cu.upd_acc()) ? 1u : 0u;
                        mma_ss(t_s, v_step<CF::ZROW>(d_va, j), dadd(d_phik, 512 * j), ID_UPD, acc);
                        if constexpr (!CF::ZROW) {
                            mma_ss(t_z, dadd(d_phik, 512 * j), d_zones, ID_Z, acc);
                            if constexpr (CF::PP > 128)  // features 32..159 (only 128.. read)
                                mma_ss(t_z + 16, dadd(d_phik, 2 * 4096 + 512 * j), d_zones, ID_Z, acc);
                        }
                    }
                    mma_commit(BAR(FB_UPD_DONE));
                    mma_commit(BAR(FB_PHIK_FREE));
                    BASED_TRACE_EV(n, TE_UPD_ISSUED);
                    ++upd_idx;
                    return true;
                };
                if constexpr (LEADIN) {
                    // Lead-in: S^T += [v_c | 1]^T f(k_c) over the head's chunks before the range.
                    // Their f(k) tiles alternate between the f(k) and the f~(q) tile, so that the
                    // next one is built while this one is summed. One UPD_DONE phase marks the
                    // whole lead-in for the conversion.
                    const uint64_t d_phiq_k = smem_desc(sb + CF::OFF_PHIQ, 4096, 256, LAYOUT_SW32);
                    for (int i = 0; ok && i < n_lead; ++i) {
                        const int ls = i % NLS;
                        const bool alt = i & 1;
                        if (!(ok = wait_bar(BAR(alt ? FB_PHIQ_FULL : FB_PHIK_FULL), (alt ? qn : upd_idx) & 1,
                                            abort_flag, alt ? SITE_PHIQ_FULL : SITE_PHIK_FULL)))
                            break;
                        tc_fence_after();
                        const uint64_t d_va = smem_desc(sb + CF::lead_v(ls), CF::OFF_LONES - CF::lead_v(ls), 1024,
                                                        LAYOUT_SW128);
                        const uint64_t d_f = alt ? d_phiq_k : d_phik;
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            mma_ss(t_s, v_step<CF::ZROW>(d_va, j), dadd(d_f, 512 * j), ID_UPD,
                                   (i > 0 || j > 0) ? 1u : 0u);
                        mma_commit(BAR(alt ? FB_PHIQ_FREE : FB_PHIK_FREE));
                        mma_commit(BAR(FB_LFREE0 + ls));  // UPD read v_c (f(k) is built)
                        BASED_TRACE_EV(i, TE_LEAD_UPD);
                        if (alt) ++qn;
                        else ++upd_idx;
                    }
                    if (ok && n_lead > 0) mma_commit(BAR(FB_UPD_DONE));
                }
                for (int n = 0; ok && n < nchunks; ++n, cu.next()) {
                    const int s = stage_of(n);
                    const int ob = FAST ? (n & 1) : 0;
                    const uint64_t d_va = s == 0 ? d_va0 : (s == 1 ? d_va1 : d_va2);
                    const uint32_t t_out = ob ? t_o1 : t_o0;
                    // V = 64 updates first (double-buffered state operand); V = 128 reads out
                    // first, so that the single state operand is consumed before it is rewritten
                    if (FAST && cu.has_upd() && !(ok = issue_upd(n, d_va))) break;
                    if (cu.has_ro()) {
                        if (!(ok = issue_ro(n, t_out, FAST ? s : -1))) break;
                        mma_commit(BAR(FB_O_FULL0 + ob));
                        BASED_TRACE_EV(n, TE_RO_ISSUED);
                    }
                    if (!FAST && cu.has_upd() && !(ok = issue_upd(n, d_va))) break;
                    // UPD(n) read v_c; f(k), f~(q) are built (V = 64 with a read-out: released above)
                    if (!(FAST && cu.has_ro())) mma_commit(BAR(FB_STAGE_FREE0 + s));
                }
                mma_commit(BAR(FB_DRAIN_B));
                wait_bar(BAR(FB_DRAIN_B), 0, nullptr, SITE_DRAIN, kDrainLimitNs);
            }
        }
    } else if (warp == 2 && !FAST) {
        // warp 2: no role besides owning the TMEM allocation
    } else if (warp < 8 || (FAST && warp == 15)) {
        // ======================= Taylor weights: A = poly(s), causal mask =======================
        // Query rows 32 q4 .. 32 q4 + 31 (TMEM lane quarter q4 = warp % 4) need key blocks
        // 0..q4 of 32 keys. V = 64: warps 2 and 15, otherwise idle (warp 15 has no state rows to
        // convert), share the two longest row quarters, so that no warp computes more than two
        // blocks: warp 6 blocks 0-1 and warp 2 block 2 of quarter 2, warp 7 blocks 0-1 and
        // warp 15 blocks 2-3 of quarter 3.
        const int q4 = warp & 3;
        const bool helper = FAST && (warp == 2 || warp == 15);
        const int kb_lo = helper ? 2 : 0;
        const int kb_hi = (FAST && !helper && q4 >= 2) ? 1 : q4;
        const uint32_t lo = static_cast<uint32_t>(q4 * 32) << 16;
        const float c1 = scale, c2 = 0.5f * scale * scale;
        const uint64_t C1 = pack_f32x2(c1, c1), C2 = pack_f32x2(c2, c2), ONE = pack_f32x2(1.f, 1.f);
        if constexpr (FAST) {
            // A blocks above the diagonal block stay zero (never rewritten)
            uint32_t z16[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) z16[j] = 0u;
            if (!helper)
                for (int kb = q4 + 1; kb < 4; ++kb) tmem_st_x16(tmem + lo + CF::TM_A + 16 * kb, z16);
            tmem_wait_st();
        }
        // mask of the diagonal block, per bf16 pair (keys 2i, 2i+1 against row = lane)
        auto diag_mask = [&](int i) -> uint32_t {
            return (2 * i <= lane ? 0x0000FFFFu : 0u) | (2 * i + 1 <= lane ? 0xFFFF0000u : 0u);
        };
        for (int n = 0; n < nchunks; ++n) {
            if (!wait_bar(BAR(FB_S_FULL), n & 1, abort_flag, SITE_S_FULL)) break;
            tc_fence_after();
            if (warp == 7 && lane == 0) BASED_TRACE_EV(n, TE_POLY_BEGIN);
            uint32_t ra[32], rb[32];
            tmem_ld_x32(tmem + lo + CF::TM_SC + 32 * kb_lo, ra);
            // weights of key block kb from its 32 scores, as 16 bf16 pairs
            auto pack_weights = [&](int kb, const uint32_t (&r)[32], uint32_t (&packed)[16]) {
                const bool diag = kb == q4;
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    packed[i] = taylor2(r[2 * i], r[2 * i + 1], C2, C1, ONE) &
                                (diag ? diag_mask(i) : 0xFFFFFFFFu);
            };
            if constexpr (FAST) {
                // At most two key blocks per warp, both loaded and weighted before A, which AV of
                // the previous chunk may still be reading, is overwritten (QK of this chunk can be
                // issued before that AV).
                const bool two = kb_lo < kb_hi;
                if (two) tmem_ld_x32(tmem + lo + CF::TM_SC + 32 * (kb_lo + 1), rb);
                tmem_wait_ld_dep(ra);
                if (warp == 7 && lane == 0) BASED_TRACE_EV(n, TE_POLY_LD0);
                uint32_t pa[16], pb[16];
                pack_weights(kb_lo, ra, pa);
                if (two) {
                    tmem_wait_ld_dep(rb);
                    pack_weights(kb_lo + 1, rb, pb);
                }
                if (n > 0 && !wait_bar(BAR(((n - 1) & 1) ? FB_AV_DONE1 : FB_AV_DONE), ((n - 1) >> 1) & 1,
                                       abort_flag, SITE_AV_DONE))
                    break;
                tc_fence_after();
                tmem_st_x16(tmem + lo + CF::TM_A + 16 * kb_lo, pa);
                if (two) tmem_st_x16(tmem + lo + CF::TM_A + 16 * (kb_lo + 1), pb);
            } else {
                // Key blocks 0..q4, one per step with the load of the next one in flight. Rolled
                // by two blocks (one copy of the body keeps the code small). A columns
                // [16 kb, 16 kb + 16) overlay s columns already read.
                auto weights = [&](int kb, const uint32_t (&r)[32]) {
                    uint32_t packed[16];
                    pack_weights(kb, r, packed);
                    tmem_st_x16(tmem + lo + CF::TM_A + 16 * kb, packed);
                };
#pragma unroll 1
                for (int kb = kb_lo; kb <= kb_hi; kb += 2) {
                    const bool two = kb + 1 <= kb_hi;
                    if (two) tmem_ld_x32(tmem + lo + CF::TM_SC + 32 * (kb + 1), rb);
                    tmem_wait_ld_dep(ra);
                    if (warp == 7 && lane == 0) BASED_TRACE_EV(n, kb == 0 ? TE_POLY_LD0 : TE_POLY_LD1);
                    weights(kb, ra);
                    if (two) {
                        if (kb + 2 <= kb_hi) tmem_ld_x32(tmem + lo + CF::TM_SC + 32 * (kb + 2), ra);
                        tmem_wait_ld_dep(rb);
                        weights(kb + 1, rb);
                    }
                }
                // A overlays s, so the blocks above the diagonal block are cleared each time
                uint32_t z16[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) z16[j] = 0u;
#pragma unroll 1
                for (int kb = q4 + 1; kb < 4; ++kb) tmem_st_x16(tmem + lo + CF::TM_A + 16 * kb, z16);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(FB_A_FULL));
            if (warp == 7 && lane == 0) BASED_TRACE_EV(n, TE_POLY_END);
        }
    } else if (warp < 12) {
        // =============== feature tiles f(k_c), f~(q_c) and the output epilogue ==================
        const int t = (warp - 8) * 32 + lane;  // token of the chunk = TMEM lane = output row
        const int q4 = warp & 3;
        const uint32_t lo = static_cast<uint32_t>(q4 * 32) << 16;
        int qn = 0, upd_idx = 0;  // fills of the f~(q) and the f(k) tile
        bool ok = true;

        // Output tile: o = O_num / (O_den + 1e-6), written through staging buffers as pieces of
        // 128-byte rows (32 fp32 or 64 bf16 columns, SW128) by TMA stores, so that the output
        // traffic never occupies the load/store path the TMEM accesses of the other roles use.
        // Either each warp stages and stores its own 32 rows (EPI_ROWS = 32: the four warps never
        // wait for each other), or the four warps meet at a named barrier and one thread stores
        // the 128-row piece (fewer stores).
        // Rows past T are clipped by the tensor map; a box that starts past T is not issued.
        int piece = 0;  // output pieces staged so far (selects the staging buffer)
        auto epilogue = [&](int m, int eb, int eh, int et0) -> bool {
            const int ob = FAST ? (m & 1) : 0;
            const uint32_t par = FAST ? ((m >> 1) & 1) : (m & 1);
            if (!wait_bar(BAR(FB_O_FULL0 + ob), par, abort_flag, SITE_O_FULL)) return false;
            tc_fence_after();
            if (warp == 11 && lane == 0) BASED_TRACE_EV(m, TE_EPI_BEGIN);
            const uint32_t to = tmem + lo + (ob ? CF::TM_O1 : CF::TM_O0);
            uint32_t d[2], r0[32], r1[32];
            tmem_ld_x2(to + V, d);
            tmem_ld_x32(to, r0);
            tmem_ld_x32(to + 32, r1);
            tmem_wait_ld();
            const float inv = __frcp_rn(__uint_as_float(d[0]) + __uint_as_float(d[1]) + 1e-6f);
            auto release_o = [&]() {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(FB_O_FREE0 + ob));  // O read completely
                if (warp == 11 && lane == 0) BASED_TRACE_EV(m, TE_EPI_OFREE);
            };
            if constexpr (V == 64) release_o();
            constexpr int PCOLS = OBF ? 64 : 32;  // output columns per 128-byte staged row
#pragma unroll
            for (int p = 0; p < V / PCOLS; ++p) {
                if constexpr (V == 128) {
                    if (p == 64 / PCOLS) {
                        tmem_ld_x32(to + 64, r0);
                        tmem_ld_x32(to + 96, r1);
                        tmem_wait_ld();
                        release_o();
                    }
                }
                constexpr bool WARP_BOX = CF::EPI_ROWS == 32;
                const uint32_t ost = sb + CF::OFF_OST + (piece % CF::NOST) * CF::OST + q4 * 4096;
                ++piece;
                // the store that last used this buffer has read it
                if (WARP_BOX ? lane == 0 : t == 0) {
                    if constexpr (CF::NOST == 2) bulk_wait_group_read<1>();
                    else bulk_wait_group_read<0>();
                }
                if (WARP_BOX) __syncwarp();
                else named_bar_sync(1, 128);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint32_t a = ost + static_cast<uint32_t>(lane) * 128u + ((c ^ (lane & 7)) << 4);
                    if constexpr (OBF) {
                        // 16 bytes = 8 bf16 columns: columns 0..31 from r0, 32..63 from r1
                        const uint32_t *x = (c < 4 ? r0 : r1) + 8 * (c & 3);
                        auto o2 = [&](int j) {
                            return pack_bf16x2(__uint_as_float(x[j]) * inv, __uint_as_float(x[j + 1]) * inv);
                        };
                        st_shared_v4(a, o2(0), o2(2), o2(4), o2(6));
                    } else {
                        const uint32_t *r = (p & 1) ? r1 : r0;
                        st_shared_v4(a, __float_as_uint(__uint_as_float(r[4 * c]) * inv),
                                     __float_as_uint(__uint_as_float(r[4 * c + 1]) * inv),
                                     __float_as_uint(__uint_as_float(r[4 * c + 2]) * inv),
                                     __float_as_uint(__uint_as_float(r[4 * c + 3]) * inv));
                    }
                }
                fence_proxy_async_smem();
                if (WARP_BOX) {
                    __syncwarp();
                    if (lane == 0 && et0 + 32 * q4 < T) {
                        tma_store_4d(&tm_o, ost, PCOLS * p, eh, et0 + 32 * q4, eb);
                        bulk_commit_group();
                    }
                } else {
                    named_bar_sync(1, 128);
                    if (t == 0) {
                        tma_store_4d(&tm_o, ost - q4 * 4096, PCOLS * p, eh, et0, eb);
                        bulk_commit_group();
                    }
                }
            }
            if (warp == 11 && lane == 0) BASED_TRACE_EV(m, TE_EPI_END);
            return true;
        };
        auto build_q = [&](int n, int s) -> bool {
            if (qn > 0 && !wait_bar(BAR(FB_PHIQ_FREE), (qn - 1) & 1, abort_flag, SITE_PHIQ_FREE))
                return false;
            if (warp == 8 && lane == 0) BASED_TRACE_EV(n, TE_PHIQ_BEGIN);
            build_features<K>(sb + CF::OFF_RAWQ + s * CF::RAW, sb + CF::OFF_PHIQ, t, kBf16Half2, 0, CF::NBLK);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(FB_PHIQ_FULL));
            if (warp == 8 && lane == 0) BASED_TRACE_EV(n, TE_PHIQ_END);
            ++qn;
            return true;
        };
        auto build_k = [&](int n, int s) -> bool {
            if (upd_idx > 0 &&
                !wait_bar(BAR(FB_PHIK_FREE), (upd_idx - 1) & 1, abort_flag, SITE_PHIK_FREE))
                return false;
            if (warp == 8 && lane == 0) BASED_TRACE_EV(n, TE_PHIK_BEGIN);
            build_features<K>(sb + CF::OFF_RAWK + s * CF::RAW, sb + CF::OFF_PHIK, t, kBf16One2, 0, CF::NBLK);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(FB_PHIK_FULL));
            if (warp == 8 && lane == 0) BASED_TRACE_EV(n, TE_PHIK_END);
            ++upd_idx;
            return true;
        };
        if constexpr (LEADIN) {
            // lead-in: f(k) of the head's chunks before the range, alternately into the f(k) and
            // the f~(q) tile
            for (int i = 0; ok && i < n_lead; ++i) {
                const int ls = i % NLS;
                if (!(ok = wait_bar(BAR(FB_LFULL0 + ls), (i / NLS) & 1, abort_flag, SITE_TMA_FULL))) break;
                const bool alt = i & 1;
                const int fill = alt ? qn : upd_idx;
                if (fill > 0 && !(ok = wait_bar(BAR(alt ? FB_PHIQ_FREE : FB_PHIK_FREE), (fill - 1) & 1, abort_flag,
                                                alt ? SITE_PHIQ_FREE : SITE_PHIK_FREE)))
                    break;
                if (warp == 8 && lane == 0) BASED_TRACE_EV(i, TE_LEAD_BUILD0);
                build_features<K>(sb + CF::lead_k(ls), sb + (alt ? CF::OFF_PHIQ : CF::OFF_PHIK), t, kBf16One2, 0,
                                  CF::NBLK);
                if (warp == 8 && lane == 0) BASED_TRACE_EV(i, TE_LEAD_BUILD1);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(alt ? FB_PHIQ_FULL : FB_PHIK_FULL));
                if (alt) ++qn;
                else ++upd_idx;
            }
        }
        Cursor cu;
        cu.init(g0, nchunks, n_c, Hl, L, r_lane);
        int pb = 0, ph = 0, pt0 = 0;  // coordinates of the previous chunk (for its epilogue)
        for (int n = 0; ok && n < nchunks; ++n, cu.next()) {
            const int s = stage_of(n);
            if (!FAST && n > 0 && !(ok = epilogue(n - 1, pb, ph, pt0))) break;
            if (cu.has_ro() || cu.has_upd()) {
                if (!(ok = wait_bar(BAR(FB_TMA_FULL0 + s), stage_par(n), abort_flag, SITE_TMA_FULL)))
                    break;
                if (FAST) {  // the state update comes first in the MMA order
                    if (cu.has_upd() && !(ok = build_k(n, s))) break;
                    if (cu.has_ro() && !(ok = build_q(n, s))) break;
                } else {
                    if (cu.has_ro() && !(ok = build_q(n, s))) break;
                    if (cu.has_upd() && !(ok = build_k(n, s))) break;
                }
            }
            if (FAST && n > 0 && !(ok = epilogue(n - 1, pb, ph, pt0))) break;
            pb = cu.b;
            ph = cu.h;
            pt0 = cu.t0();
        }
        if (ok) epilogue(nchunks - 1, pb, ph, pt0);
        // the staging buffers must outlive the last store
        if (CF::EPI_ROWS == 32 ? lane == 0 : t == 0) bulk_wait_group_all();
    } else {
        // ============== state conversion: S^T (fp32, TMEM) -> bf16 operand [S | z_hi z_lo] =====
        // warps 12-15 (V = 64: warps 12-14, the warps whose TMEM lanes hold rows 0..64 of S^T)
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane;  // TMEM lane = row of S^T = value index
        const uint32_t lo = static_cast<uint32_t>(q4 * 32) << 16;
        constexpr int LAST_ROW = CF::ZROW ? V : V - 1;
        const bool warp_has_rows = q4 * 32 <= LAST_ROW;
        constexpr int BATCH = V == 64 ? (CF::NBLK + 1) / 2 : 4;  // blocks per TMEM round trip

        // One block of a state row as bf16: rows r < V are S^T rows; with the z row (V = 64) row V
        // is z rounded to bf16 and row V + 1 its rounding remainder (z as a hi/lo pair, about 16
        // significant bits). One code path for both kinds of row keeps the code small.
        // The scale enters here, once, in fp32: feature c of the state is multiplied by
        // scale^degree(c) as the state is rounded to its bf16 operand, i.e. by scale for the K
        // linear features (c < K), by 1 for the constant feature (kConst: K = 16 block 9 column 8,
        // K = 8 block 2 column 12) and by scale^2 for every square and cross product; with the
        // query features f~(q) this gives 1 + scale q.k + scale^2 (q.k)^2 / 2.
        const uint64_t S11 = pack_f32x2(scale, scale), S22 = pack_f32x2(scale * scale, scale * scale);
        const uint64_t SC2 = pack_f32x2(1.0f, scale * scale);  // the pair that holds the constant feature
        constexpr int kConst = K == 16 ? 9 * 16 + 8 : 2 * 16 + 12;
        auto put_block = [&](uint32_t sbf, int f, const uint32_t *xs) {
            const uint32_t blk = sbf + CF::SBF_BLK * f;
            if (r <= LAST_ROW) {
                float x[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) x[j] = __uint_as_float(xs[j]);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int p0 = 16 * f + 2 * j;
                    mul_f32x2(x[2 * j], x[2 * j + 1], p0 < K ? S11 : (p0 == kConst ? SC2 : S22));
                }
                uint32_t hi[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) hi[j] = pack_bf16x2(x[2 * j], x[2 * j + 1]);
                st_shared_v4(blk + sw32(r, 0), hi[0], hi[1], hi[2], hi[3]);
                st_shared_v4(blk + sw32(r, 1), hi[4], hi[5], hi[6], hi[7]);
                if (CF::ZROW && r == V) {
                    uint32_t lw[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        lw[j] = pack_bf16x2(x[2 * j] - __uint_as_float(hi[j] << 16),
                                            x[2 * j + 1] - __uint_as_float(hi[j] & 0xFFFF0000u));
                    st_shared_v4(blk + sw32(V + 1, 0), lw[0], lw[1], lw[2], lw[3]);
                    st_shared_v4(blk + sw32(V + 1, 1), lw[4], lw[5], lw[6], lw[7]);
                }
            }
        };
        auto put_z = [&](uint32_t sbf, int p, float z) {
            z *= p < K ? scale : (p == kConst ? 1.0f : scale * scale);
            const int f = p >> 4, j = p & 15;
            const __nv_bfloat16 h = __float2bfloat16_rn(z);
            const __nv_bfloat16 l = __float2bfloat16_rn(z - __bfloat162float(h));
            const uint32_t a = sbf + CF::SBF_BLK * f + 2u * (j & 7);
            st_shared_u16(a + sw32(V, j >> 3), *reinterpret_cast<const uint16_t *>(&h));
            st_shared_u16(a + sw32(V + 1, j >> 3), *reinterpret_cast<const uint16_t *>(&l));
        };
        auto convert = [&](int cidx, int n) -> bool {
            // SBF_FULL counts one arrival per conversion warp; a warp must not arrive for this
            // conversion while the previous phase of the same barrier is still open (a warp
            // without rows finishes early, and the next state update only waits for CONV_READ).
            if (cidx >= CF::NSBF && !wait_bar(BAR(sbf_full_bar(cidx - CF::NSBF)), sbf_full_par(cidx - CF::NSBF),
                                              abort_flag, SITE_SBF_FULL))
                return false;
            if (warp == 12 && lane == 0) BASED_TRACE_EV(n, TE_CONV_BEGIN);
            const uint32_t sbf = sb + CF::OFF_SBF + (cidx % CF::NSBF) * CF::SBF;
            float za = 0.f, zb = 0.f;
            if constexpr (!CF::ZROW) {
                uint32_t a, b;
                tmem_ld_x1(tmem + lo + CF::TM_Z, a);
                tmem_ld_x1(tmem + lo + CF::TM_Z + 16, b);
                tmem_wait_ld();
                za = __uint_as_float(a);
                zb = __uint_as_float(b);
            }
            if (warp_has_rows) {
                // One feature block per step, the load of the next one in flight while the current
                // one is converted; S^T is released once its last block is in registers. Rolled by
                // two blocks (one copy of the body keeps the code small).
                uint32_t xa[16], xb[16];
                tmem_ld_x16(tmem + lo + CF::TM_S, xa);
#pragma unroll 1
                for (int f = 0; f < CF::NBLK; f += 2) {
                    const bool two = f + 1 < CF::NBLK;
                    if (two) tmem_ld_x16(tmem + lo + CF::TM_S + 16 * (f + 1), xb);
                    tmem_wait_ld_dep(xa);
                    reg_fence(xb);
                    if (f + 2 >= CF::NBLK) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(BAR(FB_CONV_READ));  // S^T may change now
                        if (warp == 12 && lane == 0) BASED_TRACE_EV(n, TE_CONV_READ);
                    }
                    put_block(sbf, f, xa);
                    if (two) {
                        if (f + 2 < CF::NBLK) tmem_ld_x16(tmem + lo + CF::TM_S + 16 * (f + 2), xa);
                        put_block(sbf, f + 1, xb);
                    }
                }
            } else {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(FB_CONV_READ));
            }
            if constexpr (!CF::ZROW) {
                if (r < CF::PP && r < 128) put_z(sbf, r, za);
                if (r + 32 >= 128 && r + 32 < CF::PP) put_z(sbf, r + 32, zb);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(sbf_full_bar(cidx)));
            if (warp == 12 && lane == 0) BASED_TRACE_EV(n, TE_CONV_END);
            return true;
        };

        int cidx = 0;
        // A range that starts inside a head continues from the prefix state of the chunks before
        // it: load it into TMEM, then convert it like any other state.
        if (!LEADIN && rg.cnt[j_range] > 0) {
            // The prefix is the sum of the partial states of the pieces of the head before this
            // range: slots slot .. slot + m - 1 (m <= kMaxChain; m = 1 when a scan has
            // already summed them).
            const int m = rg.cnt[j_range];
            // launched as a dependent of the aggregate / scan kernel: only this read of their
            // output waits for them (every other role starts right away)
            griddep_wait();
#ifdef BASED_TRACE
            if (r == 0 && trace_buf_ != nullptr)
                trace_buf_[(static_cast<size_t>(blockIdx.x) * 64 + 63) * 32 + 24] = global_timer_ns();
#endif
            const float *slot =
                prefix + (static_cast<size_t>(rg.slot[j_range]) + static_cast<size_t>(r_lane) * lane_slots) * CF::SLOT;
            // One code path per chain length, so that every load it issues is needed and all of a
            // step's loads are in flight together; the terms are summed in range order.
            auto load_prefix = [&](auto chain_len) {
                constexpr int M = decltype(chain_len)::value;
                auto chain = [&](const float *e) -> float {
                    float x = __ldg(e);
#pragma unroll
                    for (int i = 1; i < M; ++i) x += __ldg(e + static_cast<size_t>(i) * CF::SLOT);
                    return x;
                };
                if (warp_has_rows) {
                    // two feature blocks of loads in flight per step; element (c, r) at
                    // c * SROWS + r, so a warp reads consecutive floats
                    const bool mine = r <= LAST_ROW;
                    const float *col = slot + (mine ? r : 0);
#pragma unroll 1
                    for (int f = 0; f < CF::NBLK; f += 2) {
                        uint32_t x[2][16];
#pragma unroll
                        for (int h = 0; h < 2; ++h)
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                const int c = 16 * (f + h) + j;
                                x[h][j] = (mine && c < CF::PP)
                                              ? __float_as_uint(chain(col + static_cast<size_t>(c) * CF::SROWS))
                                              : 0u;
                            }
                        tmem_st_x16(tmem + lo + CF::TM_S + 16 * f, x[0]);
                        if (f + 1 < CF::NBLK) tmem_st_x16(tmem + lo + CF::TM_S + 16 * (f + 1), x[1]);
                    }
                }
                if constexpr (!CF::ZROW) {
                    const float *zcol = slot + V;
                    const float za = r < CF::PP ? chain(zcol + static_cast<size_t>(r) * CF::SROWS) : 0.0f;
                    const float zb = r + 32 < CF::PP ? chain(zcol + static_cast<size_t>(r + 32) * CF::SROWS) : 0.0f;
                    tmem_st_x1(tmem + lo + CF::TM_Z, __float_as_uint(za));
                    tmem_st_x1(tmem + lo + CF::TM_Z + 16, __float_as_uint(zb));
                }
            };
            static_assert(kMaxChain == 4, "one prefix load path per chain length");
            if (m == 1) load_prefix(std::integral_constant<int, 1>{});
            else if (m == 2) load_prefix(std::integral_constant<int, 2>{});
            else if (m == 3) load_prefix(std::integral_constant<int, 3>{});
            else load_prefix(std::integral_constant<int, 4>{});
            tmem_wait_st();
            convert(cidx++, 63);
        }
        int u = 0;
        bool ok = true;
        if (LEADIN && n_lead > 0) {
            // the state summed by the lead-in: one UPD_DONE phase for all of its chunks
            ok = wait_bar(BAR(FB_UPD_DONE), 0, abort_flag, SITE_UPD_DONE);
            if (ok) {
                tc_fence_after();
                if constexpr (kLeadOverSbf) {
                    // lead-in stages were over the state operands: rows V + 2 .. of both are
                    // zeroed again (the lead-in's reads of them are complete)
                    constexpr int kPad = (CF::SBF_ROWS - V - 2) * 2;  // 16-byte pieces per block
                    for (int i = static_cast<int>(threadIdx.x) - 12 * 32; i < CF::NSBF * CF::NBLK * kPad; i += 3 * 32)
                        st_shared_v4(sb + CF::OFF_SBF + CF::SBF_BLK * (i / kPad) + (V + 2) * 32 + 16 * (i % kPad), 0u,
                                     0u, 0u, 0u);
                    // (each warp's proxy fence in the conversion covers these stores before its
                    // SBF_FULL arrival)
                }
                ok = convert(cidx++, 63);
            }
            u = 1;
        }
        Cursor cu;
        cu.init(g0, nchunks, n_c, Hl, L, r_lane);
        for (int n = 0; ok && n < nchunks; ++n, cu.next()) {
            if (!cu.has_upd()) continue;
            if (!wait_bar(BAR(FB_UPD_DONE), u & 1, abort_flag, SITE_UPD_DONE)) break;
            tc_fence_after();
            if (!convert(cidx++, n)) break;
            ++u;
        }
    }

    // ---- teardown ------------------------------------------------------------------------------
    // (every thread must be done with TMEM before it is released: the single-lane roles reach
    // this barrier after the other lanes of their warps, so it counts threads, not warps)
    tc_fence_before();
    cta_sync();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
#ifdef BASED_TRACE
    if (threadIdx.x == 0 && trace_buf_ != nullptr)
        trace_buf_[(static_cast<size_t>(blockIdx.x) * 64 + 63) * 32 + 23] = global_timer_ns();
#endif
}

// ------------------------------------------------------------------------------------------------
// Aggregate kernel: the partial states [S^T | z] of the pieces of the stretches (the last stretch
// of every range that ends inside a head), each written as fp32 into its slot. CTA j sums the
// chunks of pieces cta_first[j] .. cta_first[j + 1] - 1 in order, into two TMEM accumulators used
// in turn, so that one piece's slot is written while the next piece is summed.
// warp 0: TMA producer | warp 1: MMA issuer | warp 2: owns TMEM | warp 3: idle | warps 4-11: f(k)
// tiles (half of each token row per warp; V = 128: also z of each piece, summed in registers) |
// warps 12-15: slot writers (512 threads; with 384, one piece per CTA, warps 8-11 write the slot
// after building)
// ------------------------------------------------------------------------------------------------
// Barriers of the aggregate kernel with S k/v stages and NP f(k) buffers: TMA_FULL[S],
// STAGE_FREE[S], PHIK_FULL[NP], PHIK_FREE[NP], per accumulator AGG_DONE[2] (its piece is summed)
// and SLOT_READ[2] (its slot is written), DRAIN, ZRED (V = 128: the builder warps' partial sums of
// a piece's z are in shared memory).
template <int S, int NP>
struct AggBar {
    static constexpr int TMA_FULL0 = 0, STAGE_FREE0 = S, PHIK_FULL0 = 2 * S, PHIK_FREE0 = 2 * S + NP,
                         AGG_DONE0 = 2 * S + 2 * NP, SLOT_READ0 = AGG_DONE0 + 2, DRAIN = SLOT_READ0 + 2,
                         ZRED = DRAIN + 1, COUNT = ZRED + 1;
    static_assert(8 * COUNT + 8 <= 256, "barrier area");
};
constexpr uint32_t kAggAccStride = 256;  // TMEM columns between the two accumulators

// Walks the chunks of pieces p .. p_end - 1 in order (the piece table is read once per piece).
struct PieceWalk {
    Cursor cu;
    const AggPieces *ap;
    int p, p_end, j, len, n_c, Hl, L, r;
    __device__ __forceinline__ void start_piece() {
        len = ap->len[p];
        cu.init(ap->g0[p], len, n_c, Hl, L, r);
    }
    __device__ __forceinline__ void init(const AggPieces &a, int p0, int p1, int n_c_, int Hl_, int L_, int r_) {
        ap = &a;
        p = p0;
        p_end = p1;
        j = 0;
        len = 0;
        n_c = n_c_;
        Hl = Hl_;
        L = L_;
        r = r_;
        if (p < p_end) start_piece();
    }
    __device__ __forceinline__ bool first() const { return j == 0; }
    __device__ __forceinline__ bool last() const { return j == len - 1; }
    __device__ __forceinline__ void next() {
        if (++j == len) {
            j = 0;
            if (++p < p_end) start_piece();
        } else {
            cu.next();
        }
    }
};

template <int K, int V>
__global__ void __launch_bounds__(kAggThreads, 1)
based_agg_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 float *__restrict__ slots, int H, int n_c, int L, const __grid_constant__ AggPieces ap) {
    using CF = Cfg<K, V>;
    constexpr int S = CF::A_NST;
    constexpr int NP = CF::A_NPHIK;
    using AB = AggBar<S, NP>;
    constexpr int AB_TMA_FULL0 = AB::TMA_FULL0, AB_STAGE_FREE0 = AB::STAGE_FREE0,
                  AB_PHIK_FULL0 = AB::PHIK_FULL0, AB_PHIK_FREE0 = AB::PHIK_FREE0,
                  AB_AGG_DONE0 = AB::AGG_DONE0, AB_SLOT_READ0 = AB::SLOT_READ0, AB_DRAIN = AB::DRAIN,
                  AB_COUNT = AB::COUNT;
    // CTA a L + r sums CTA a's pieces of head lane r into that lane's slots
    const int a_cta = static_cast<int>(blockIdx.x) / L, r_lane = static_cast<int>(blockIdx.x) % L;
    const int Hl = H / L;
    if (a_cta >= ap.n_cta) return;
    slots += static_cast<size_t>(r_lane) * ap.n * CF::SLOT;
    const int p0 = ap.cta_first[a_cta], p1 = ap.cta_first[a_cta + 1];
    int nchunks = 0;
    for (int p = p0; p < p1; ++p) nchunks += ap.len[p];
    if (nchunks <= 0) return;

    extern __shared__ uint8_t smem_raw[];
    BASED_TRACE_INIT;
#ifdef BASED_TRACE
    if (threadIdx.x == 0 && trace_buf_ != nullptr)
        trace_buf_[(static_cast<size_t>(blockIdx.x) * 64 + 40) * 32 + 8] = global_timer_ns();
#endif
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + CF::A_OFF_BAR + 8 * AB_COUNT);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + CF::A_OFF_BAR + 8 * AB_COUNT + 4);
    auto BAR = [&](int i) -> uint32_t { return sb + CF::A_OFF_BAR + 8u * static_cast<uint32_t>(i); };

    // k, v tiles of the CTA's chunk u (cursor position cu) into stage u % S, completing on TMA_FULL.
    // Their L2 lines are marked for eviction first: this pass reads them once, and without the mark
    // they push out the slots written earlier in the pass, which the forward kernel reads next
    // (measured: 0.4 - 1.1 % faster calls on B=4..8 T=16384 H=32).
    auto issue_loads = [&](int u, const Cursor &cu) {
        const int s = u % S;
        const uint32_t bar = BAR(AB_TMA_FULL0 + s);
        const uint64_t pol = l2_policy_evict_first();
        BASED_TRACE_EV(u + 40, 0);
        mbar_arrive_expect_tx(bar, CF::RAW + CF::VT);
        tma_load_4d_hint(sb + CF::A_OFF_RAWK + s * CF::RAW, &tm_k, bar, 0, cu.h, cu.t0(), cu.b, pol);
        tma_load_4d_hint(sb + CF::A_OFF_V + s * CF::VT, &tm_v, bar, 0, cu.h, cu.t0(), cu.b, pol);
        if constexpr (V == 128)
            tma_load_4d_hint(sb + CF::A_OFF_V + s * CF::VT + 16384, &tm_v, bar, 64, cu.h, cu.t0(), cu.b, pol);
    };
    const int n_early = nchunks < S ? nchunks : S;  // loads issued during set-up
    if (threadIdx.x == 0) {
        for (int i = 0; i < AB_COUNT; ++i) {
            const bool phik_full = i >= AB_PHIK_FULL0 && i < AB_PHIK_FULL0 + NP;
            const bool slot_read = i >= AB_SLOT_READ0 && i < AB_SLOT_READ0 + 2;
            mbar_init(BAR(i), (phik_full || i == AB::ZRED) ? 8u : (slot_read ? 4u : 1u));
        }
        *abort_flag = 0;
        fence_mbar_init();
        // the first loads go out now (this thread is the TMA producer)
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        // launched as a programmatic dependent of the previous kernel in the stream (whose
        // outputs may be k or v, and which may still read the slots): nothing of this grid touches
        // global memory before this thread's first loads, and those wait for that kernel
        griddep_wait();
        PieceWalk w;
        w.init(ap, p0, p1, n_c, Hl, L, r_lane);
        for (int u = 0; u < n_early; ++u, w.next()) issue_loads(u, w.cu);
    }
    if constexpr (CF::ZROW) {
        for (int i = threadIdx.x; i < CF::ONES / 16; i += blockDim.x)
            st_shared_v4(sb + CF::A_OFF_ONES + 16u * i, 0u, 0u, 0u, 0u);
        __syncthreads();
        if (threadIdx.x < 16)
            st_shared_u16(sb + CF::A_OFF_ONES + sw128(threadIdx.x, 0), 0x3F80);
    }
    // one accumulator (256 columns) when the CTA sums one piece, else two
    const uint32_t tmem_cols = p1 - p0 > 1 ? 2 * kAggAccStride : kAggAccStride;
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_holder), tmem_cols);
        tmem_relinquish();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    // the scan / forward kernel may start launching now (the previous kernel has completed): it
    // waits for this grid before it reads the slots
    griddep_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            int issued = n_early;
            PieceWalk w;
            w.init(ap, p0, p1, n_c, Hl, L, r_lane);
            for (int u = 0; u < n_early; ++u) w.next();
            for (int u = n_early; u < nchunks; ++u, w.next()) {
                const int s = u % S;
                if (!wait_bar(BAR(AB_STAGE_FREE0 + s), ((u / S) - 1) & 1, abort_flag, SITE_STAGE_FREE))
                    break;
                issue_loads(u, w.cu);
                ++issued;
            }
            if (*abort_flag) {
                for (int m = issued - S; m < issued; ++m)
                    if (m >= 0)
                        wait_bar(BAR(AB_TMA_FULL0 + (m % S)), (m / S) & 1, nullptr, SITE_DRAIN,
                                 kDrainLimitNs);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t ID_UPD = idesc_bf16_f32(128, CF::PP, 1, 1);
            PieceWalk w;
            w.init(ap, p0, p1, n_c, Hl, L, r_lane);
            int kk = 0;  // pieces of this CTA started
            for (int u = 0; u < nchunks; ++u, w.next()) {
                const int s = u % S, pb = u % NP, b = kk & 1;
                // accumulator b is free once the slot of the piece two before was written
                if (w.first() && kk >= 2 &&
                    !wait_bar(BAR(AB_SLOT_READ0 + b), ((kk - 2) >> 1) & 1, abort_flag, SITE_SLOT_READ))
                    break;
                if (!wait_bar(BAR(AB_TMA_FULL0 + s), (u / S) & 1, abort_flag, SITE_TMA_FULL)) break;
                if (!wait_bar(BAR(AB_PHIK_FULL0 + pb), (u / NP) & 1, abort_flag, SITE_PHIK_FULL)) break;
                BASED_TRACE_EV(u + 40, 1);
                tc_fence_after();
                const uint32_t t_s = tmem + b * kAggAccStride;
                const uint32_t lbo_a = CF::ZROW ? (CF::A_OFF_ONES - (CF::A_OFF_V + s * CF::VT)) : 16384u;
                const uint64_t d_va = smem_desc(sb + CF::A_OFF_V + s * CF::VT, lbo_a, 1024, LAYOUT_SW128);
                const uint64_t d_phik = smem_desc(sb + CF::A_OFF_PHIK + pb * CF::PHI, 4096, 256, LAYOUT_SW32);
                const bool carry = !w.first();
                // (V = 128: z is summed by the builders, not by an MMA)
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t acc = (j > 0 || carry) ? 1u : 0u;
                    mma_ss(t_s, v_step<CF::ZROW>(d_va, j), dadd(d_phik, 512 * j), ID_UPD, acc);
                }
                mma_commit(BAR(AB_PHIK_FREE0 + pb));
                mma_commit(BAR(AB_STAGE_FREE0 + s));
                if (w.last()) {
                    mma_commit(BAR(AB_AGG_DONE0 + b));  // piece kk summed
                    ++kk;
                }
                BASED_TRACE_EV(u + 40, 2);
            }
            // every MMA issued must finish before TMEM is released
            mma_commit(BAR(AB_DRAIN));
            wait_bar(BAR(AB_DRAIN), 0, nullptr, SITE_DRAIN, kDrainLimitNs);
        }
    } else if (warp < 4) {
        // warps 2 and 3: no role (warp 2 owns the TMEM allocation)
    } else if (warp < 12) {
        // feature builders (warps 4-11): token t of the chunk, warps 4-7 the first half of its
        // feature blocks and warps 8-11 the second half, cycling through the f(k) buffers
        const int t = (warp & 3) * 32 + lane;
        constexpr int H0 = (CF::NBLK + 1) / 2;  // feature blocks of the first half of a row
        if constexpr (CF::ZROW) {
            const int f_lo = warp < 8 ? 0 : H0, f_hi = warp < 8 ? H0 : CF::NBLK;
            for (int u = 0; u < nchunks; ++u) {
                const int s = u % S, pb = u % NP;
                if (!wait_bar(BAR(AB_TMA_FULL0 + s), (u / S) & 1, abort_flag, SITE_TMA_FULL)) break;
                if (u >= NP && !wait_bar(BAR(AB_PHIK_FREE0 + pb), ((u / NP) - 1) & 1, abort_flag,
                                         SITE_PHIK_FREE))
                    break;
                if (warp == 4 && lane == 0) BASED_TRACE_EV(u + 40, 3);
                build_features<K>(sb + CF::A_OFF_RAWK + s * CF::RAW, sb + CF::A_OFF_PHIK + pb * CF::PHI, t,
                                  kBf16One2, f_lo, f_hi);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(AB_PHIK_FULL0 + pb));
                if (warp == 4 && lane == 0) BASED_TRACE_EV(u + 40, 4);
            }
        } else {
            // V = 128: the builders also sum z = sum f(k) of each piece: per thread over its
            // tokens, then over the warp's lanes, then over the four warps of its half of the row
            // (through shared memory), into the slot's z column
            auto build_sum = [&](auto half) {
                constexpr int F0 = decltype(half)::value ? H0 : 0;
                constexpr int F1 = decltype(half)::value ? CF::NBLK : H0;
                constexpr int NZ = (F1 - F0) * 16;
                float *red = reinterpret_cast<float *>(smem + CF::A_OFF_ZRED);
                float z[NZ];
#pragma unroll
                for (int i = 0; i < NZ; ++i) z[i] = 0.0f;
                PieceWalk w;
                w.init(ap, p0, p1, n_c, Hl, L, r_lane);
                int kk = 0;
                for (int u = 0; u < nchunks; ++u, w.next()) {
                    const int s = u % S, pb = u % NP;
                    if (!wait_bar(BAR(AB_TMA_FULL0 + s), (u / S) & 1, abort_flag, SITE_TMA_FULL)) break;
                    if (u >= NP && !wait_bar(BAR(AB_PHIK_FREE0 + pb), ((u / NP) - 1) & 1, abort_flag,
                                             SITE_PHIK_FREE))
                        break;
                    if (warp == 4 && lane == 0) BASED_TRACE_EV(u + 40, 3);
                    build_k_features_acc<K, F0, F1>(sb + CF::A_OFF_RAWK + s * CF::RAW,
                                                    sb + CF::A_OFF_PHIK + pb * CF::PHI, t, z);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(BAR(AB_PHIK_FULL0 + pb));
                    if (warp == 4 && lane == 0) BASED_TRACE_EV(u + 40, 4);
                    if (!w.last()) continue;
                    // piece kk is built: its z
                    int zbase = 0;
                    z_reduce_scatter<NZ, NZ, 16>(z, lane, zbase);
                    // partials of warp (half, q4) in buffer kk % 2: [buffer][half][q4][H0 * 16]
                    float *mine = red + ((kk & 1) * 8 + decltype(half)::value * 4 + (warp & 3)) * (H0 * 16);
                    constexpr int NF = z_final_count(NZ, 16);
                    if ((lane & z_dup_mask(NZ, 16)) == 0) {
#pragma unroll
                        for (int i = 0; i < NF; ++i) mine[zbase + i] = z[i];
                    }
#pragma unroll
                    for (int i = 0; i < NZ; ++i) z[i] = 0.0f;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(BAR(AB::ZRED));
                    if (!wait_bar(BAR(AB::ZRED), kk & 1, abort_flag, SITE_ZRED)) break;
                    // feature c of the row: the four warps' partials of its half
                    const int tb = (warp - 4) * 32 + lane;  // 0..255
                    if (tb < CF::PP) {
                        const int hf = tb < H0 * 16 ? 0 : 1, ci = tb - hf * H0 * 16;
                        const float *part = red + ((kk & 1) * 8 + hf * 4) * (H0 * 16) + ci;
                        const float zc = (part[0] + part[H0 * 16]) + (part[2 * H0 * 16] + part[3 * H0 * 16]);
                        slots[static_cast<size_t>(p0 + kk) * CF::SLOT + static_cast<size_t>(tb) * CF::SROWS + V] = zc;
                    }
                    ++kk;
                }
            };
            if (warp < 8) build_sum(std::integral_constant<int, 0>{});
            else build_sum(std::integral_constant<int, 1>{});
        }
    }
    // Slot writers: S^T rows (V = 64: and z, row 64) of each summed piece -> its fp32 slot (V = 128:
    // the builders write z), element (c, r) at
    // c * SROWS + r. With several pieces per CTA they are warps 12-15 (512 threads), so that the
    // f(k) builders never wait for a slot; with one piece per CTA (384 threads) warps 8-11 write it
    // after building.
    const bool dedicated_writers = blockDim.x > 384;
    if (dedicated_writers ? warp >= 12 : (warp >= 8 && warp < 12)) {
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane;
        const uint32_t lo = static_cast<uint32_t>(q4 * 32) << 16;
        constexpr int LAST_ROW = CF::ZROW ? V : V - 1;
        for (int kk = 0; kk < p1 - p0; ++kk) {
            const int b = kk & 1;
            if (!wait_bar(BAR(AB_AGG_DONE0 + b), (kk >> 1) & 1, abort_flag, SITE_AGG_DONE)) break;
            tc_fence_after();
            if (q4 == 0 && lane == 0) BASED_TRACE_EV(40, 5);
            float *slot = slots + static_cast<size_t>(p0 + kk) * CF::SLOT;
            const uint32_t acc = tmem + lo + b * kAggAccStride;
            if (q4 * 32 <= LAST_ROW) {
                // two feature blocks per TMEM round trip
#pragma unroll 1
                for (int f = 0; f < CF::NBLK; f += 2) {
                    uint32_t x[2][16];
                    tmem_ld_x16(acc + 16 * f, x[0]);
                    if (f + 1 < CF::NBLK) tmem_ld_x16(acc + 16 * (f + 1), x[1]);
                    tmem_wait_ld_dep(x[0]);
                    tmem_wait_ld_dep(x[1]);
                    if (r <= LAST_ROW) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            if (f + h >= CF::NBLK) break;
                            float *dst = slot + static_cast<size_t>(16 * (f + h)) * CF::SROWS + r;
#pragma unroll
                            for (int j = 0; j < 16; ++j) dst[j * CF::SROWS] = __uint_as_float(x[h][j]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(AB_SLOT_READ0 + b));  // the accumulator may be reused
        }
    }

#ifdef BASED_TRACE
    if (threadIdx.x == 0 && trace_buf_ != nullptr)
        trace_buf_[(static_cast<size_t>(blockIdx.x) * 64 + 40) * 32 + 9] = global_timer_ns();
#endif
    tc_fence_before();
    cta_sync();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, tmem_cols);
    }
}


// ------------------------------------------------------------------------------------------------
// Scan: within each run of ranges that continue one head's prefix, turn the per-range partial
// states into inclusive prefixes (slot i = sum of the partial states of ranges <= i in the run).
// The runs are listed by the host: block (x, l runs.n + r) handles a slice of the elements of run r
// of head lane l.
// ------------------------------------------------------------------------------------------------
__global__ void based_scan_kernel(float *__restrict__ slots, int slot_elems, int lane_slots,
                                  const __grid_constant__ ScanRuns runs) {
    griddep_launch_dependents();
    griddep_wait();  // the aggregate kernel's slots are complete and visible
    if (runs.n == 0) return;
    // blockIdx.y = lane * runs.n + run (every head lane has the same runs)
    const int r = static_cast<int>(blockIdx.y) % runs.n, lane = static_cast<int>(blockIdx.y) / runs.n;
    const int i0 = runs.start[r] + lane * lane_slots, len = runs.len[r];
    const int vec = slot_elems / 4;  // slots are whole float4s
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < vec; e += gridDim.x * blockDim.x) {
        float4 *p = reinterpret_cast<float4 *>(slots + static_cast<size_t>(i0) * slot_elems) + e;
        float4 acc = p[0];
        // up to four slots per step, their loads issued together (one round trip instead of one per
        // slot); the sums stay in range order
        for (int j0 = 1; j0 < len; j0 += 4) {
            float4 x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (j0 + u < len) x[u] = p[static_cast<size_t>(j0 + u) * vec];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (j0 + u < len) {
                    acc.x += x[u].x;
                    acc.y += x[u].y;
                    acc.z += x[u].z;
                    acc.w += x[u].w;
                    p[static_cast<size_t>(j0 + u) * vec] = acc;
                }
            }
        }
    }
}

// One-thread kernel whose barrier nobody signals: exercises the bounded-wait path.
__global__ void based_selftest_wait_kernel(unsigned long long limit_ns, int *result) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    abort_flag = 0;
    fence_mbar_init();
    const bool ok = wait_bar(b, 0, reinterpret_cast<volatile int *>(&abort_flag), SITE_SELFTEST,
                             limit_ns);
    *result = ok ? 1 : 0;
}

}  // namespace based
