// based_kernels.cuh: sm_103a kernels of the Based causal forward pass.
//
// Method (the "based_forward.py" kernel-task spec, spec_md and perf_md): with the symmetric
// 2nd-order feature map f(x) (constant, linear, squared and pairwise-product terms, P = 1 + K +
// K(K+1)/2 features, which reproduces phi(q).phi(k) = 1 + q.k + (q.k)^2/2 exactly once each
// feature carries its coefficient), every head is cut into chunks of 128 rows and, per chunk c,
//     s   = q_c k_c^T                      (tensor core, TMEM)
//     A   = (1 + sigma s + sigma^2 s^2 / 2) masked to j <= i   (fp32 polynomial -> bf16 TMEM)
//     O   = A v_c + f(q_c) [S | z]         (tensor core; z gives the inter-chunk denominator)
//     o   = O_num / (rowsum(A) + O_den + 1e-6)
//     S  += v_c^T f(k_c),  z += f(k_c)^T 1  (tensor core, fp32 accumulation in TMEM)
// The per-head chunk sequence is split across CTAs; the state each CTA starts from is the sum of
// the partial states of the chunks before it (aggregate pass + scan), so the forward kernel never
// waits on another CTA.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "sm103_ptx.cuh"

namespace based {

constexpr int kChunk = 128;            // rows per chunk = MMA M
constexpr int kFwdThreads = 512;       // 4 warpgroups
constexpr int kAggThreads = 384;       // 3 warpgroups
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // a bounded wait gives up after 1 s
constexpr uint64_t kDrainLimitNs = 100000000ull;  // drain of in-flight copies after an abort

// Status word: bit 0 = some wait timed out; bits 8..15 = site of the first timeout.
__device__ unsigned int g_status;

enum WaitSite : uint32_t {
    SITE_STAGE_FREE = 1, SITE_TMA_FULL, SITE_S_FULL, SITE_A_FULL, SITE_O_FULL, SITE_O_FREE,
    SITE_AV_DONE, SITE_PHIQ_FULL, SITE_PHIQ_FREE, SITE_PHIK_FULL, SITE_PHIK_FREE, SITE_UPD_DONE,
    SITE_SBF_FULL, SITE_AGG_DONE, SITE_DRAIN, SITE_SELFTEST = 255
};

__device__ __forceinline__ void record_timeout(uint32_t site) {
    atomicCAS(&g_status, 0u, 1u | (site << 8));
    atomicOr(&g_status, 1u);
}

// Bounded mbarrier wait. Returns false if the CTA aborted or the wait ran out (then it aborts
// the CTA and records the site). Never spins longer than the limit.
__device__ __noinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                      uint32_t site, uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (abort_flag != nullptr && *abort_flag) return false;
        if ((it & 15u) == 0u && global_timer_ns() - t0 > limit_ns) {
            if (abort_flag != nullptr) *abort_flag = 1;
            record_timeout(site);
            return false;
        }
    }
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
    // z rides as row V of S^T when that row exists inside the 128-row MMA (V = 64); otherwise a
    // separate small MMA accumulates it.
    static constexpr bool ZROW = (V == 64);
    static constexpr int NO = V + 16;        // O columns: V numerators, den hi, den lo, padding
    static constexpr int SROWS = V + 1;      // rows of a stored state: V rows of S^T + z
    static constexpr int SLOT = SROWS * PP;  // floats per stored state

    // TMEM columns (forward kernel)
    static constexpr int TM_S = 0;                               // S^T (lanes = value dim)
    static constexpr int TM_SA = align_up(PP, 32);               // s (fp32) then A (bf16)
    static constexpr int TM_O = TM_SA + 128;                     // O (lanes = query rows)
    static constexpr int TM_Z = align_up(TM_O + NO, 32);         // z tiles (V = 128)
    static_assert(TM_Z + 32 <= 512, "TMEM overflow");
    // TMEM columns (aggregate kernel)
    static constexpr int TA_Z = align_up(PP, 32);
    static_assert(TA_Z + 32 <= 256, "TMEM overflow (aggregate)");

    // Shared memory (forward kernel), byte offsets from a 1024-aligned base.
    static constexpr int RAW = kChunk * 32;    // one raw q or k tile: 128 rows x 16 bf16
    static constexpr int VT = kChunk * V * 2;  // one v tile
    static constexpr int PHI = NBLK * 4096;    // one feature tile: NBLK blocks of 128 x 16 bf16
    static constexpr int SBF_ROWS = V + 16;    // rows of the bf16 state operand [S | z_hi z_lo 0]
    static constexpr int SBF_BLK = SBF_ROWS * 32;
    static constexpr int SBF = NBLK * SBF_BLK;
    static constexpr int OFF_RAWQ = 0;
    static constexpr int OFF_RAWK = OFF_RAWQ + 2 * RAW;
    static constexpr int OFF_V = OFF_RAWK + 2 * RAW;
    static constexpr int OFF_ONES = OFF_V + 2 * VT;
    static constexpr int OFF_PHIK = OFF_ONES + (ZROW ? VT : 0);
    static constexpr int OFF_PHIQ = OFF_PHIK + PHI;
    static constexpr int OFF_SBF = OFF_PHIQ + PHI;
    static constexpr int OFF_ZONES = align_up(OFF_SBF + SBF, 1024);
    static constexpr int OFF_BAR = OFF_ZONES + 1024;
    static constexpr int SMEM_FWD = OFF_BAR + 256 + 1024;  // + alignment slack
    // The z MMA reads 8 feature blocks (32 KB) from the phi(k) tile start; they must be inside
    // the allocation even when the tile has fewer blocks (their rows of D are never read).
    static_assert(ZROW || OFF_PHIK + 8 * 4096 <= OFF_BAR, "z MMA window leaves shared memory");
    static_assert(SMEM_FWD <= 232448, "shared memory budget");

    // Shared memory (aggregate kernel)
    static constexpr int A_OFF_PHIK = 0;
    static constexpr int A_OFF_RAWK = align_up(PHI, 1024);
    static constexpr int A_OFF_V = A_OFF_RAWK + 2 * RAW;
    static constexpr int A_OFF_ONES = A_OFF_V + 2 * VT;
    static constexpr int A_OFF_ZONES = A_OFF_ONES + (ZROW ? VT : 0);
    static constexpr int A_OFF_BAR = A_OFF_ZONES + 1024;
    static constexpr int SMEM_AGG = A_OFF_BAR + 256 + 1024;
    static_assert(ZROW || A_OFF_PHIK + 8 * 4096 <= A_OFF_BAR, "z MMA window (aggregate)");
};

// Swizzled byte offsets inside 32-byte-row (SW32) and 128-byte-row (SW128) tiles whose base is
// aligned to the swizzle atom: the 16-byte chunk index is XORed with address bits above the row.
__device__ __forceinline__ uint32_t sw32(int row, int half) {
    return static_cast<uint32_t>(row * 32 + ((half ^ ((row >> 2) & 1)) << 4));
}
__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
    return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
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

// Coefficient of feature p = 16 f + j of the symmetric feature map (see build_features): the
// scaled polynomial sigma (q.k) + sigma^2 (q.k)^2 / 2 splits into linear terms (sigma), squares
// (sigma^2 / 2) and distinct cross products (sigma^2); the constant feature has 1, padding 0.
template <int K>
__device__ __forceinline__ float feature_coef(int f, int j, float c_lin, float c_sq, float c_x) {
    if (K == 16) {
        if (f == 0) return c_lin;
        if (f == 1) return c_sq;
        if (f <= 8) return c_x;
        return j < 8 ? c_x : (j == 8 ? 1.0f : 0.0f);
    } else {
        if (f == 0) return j < 8 ? c_lin : c_sq;
        if (f == 1) return c_x;
        return j < 12 ? c_x : (j == 12 ? 1.0f : 0.0f);
    }
}

// Builds the feature tile row of one token from its raw 16-wide bf16 row (SW32 tile) into NBLK
// SW32 blocks of 16 features. Products are exact bf16 products rounded once (mul.rn.bf16x2).
// K = 16: block 0 = x, 1 = x_a^2, 1+d (d = 1..7) = x_a x_{(a+d) mod 16}, 9 = [x_a x_{a+8} (a<8),
//         1, 0 x 7].
// K = 8:  block 0 = [x, x_a^2], 1 = [x_a x_{a+1}, x_a x_{a+2}] (mod 8), 2 = [x_a x_{a+3} (mod 8),
//         x_a x_{a+4} (a<4), 1, 0 x 3].
// Every unordered pair a < b appears exactly once.
template <int K>
__device__ __forceinline__ void build_features(uint32_t raw, uint32_t phi, int t) {
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
    if constexpr (K == 16) {
        const uint4 hi = ld_shared_v4(rb + (16u ^ sw));
        const uint32_t X[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
        store_blk(0, X[0], X[1], X[2], X[3], X[4], X[5], X[6], X[7]);
        store_blk(1, bmul2(X[0], X[0]), bmul2(X[1], X[1]), bmul2(X[2], X[2]), bmul2(X[3], X[3]),
                  bmul2(X[4], X[4]), bmul2(X[5], X[5]), bmul2(X[6], X[6]), bmul2(X[7], X[7]));
#pragma unroll
        for (int d = 1; d <= 7; ++d) {
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
        store_blk(9, bmul2(X[0], X[4]), bmul2(X[1], X[5]), bmul2(X[2], X[6]), bmul2(X[3], X[7]),
                  ONE_ZERO, 0u, 0u, 0u);
    } else {
        const uint32_t X[4] = {lo.x, lo.y, lo.z, lo.w};
        store_blk(0, X[0], X[1], X[2], X[3], bmul2(X[0], X[0]), bmul2(X[1], X[1]),
                  bmul2(X[2], X[2]), bmul2(X[3], X[3]));
        uint32_t R1[4], R3[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            R1[m] = __byte_perm(X[m], X[(m + 1) & 3], 0x5432);
            R3[m] = __byte_perm(X[(m + 1) & 3], X[(m + 2) & 3], 0x5432);
        }
        store_blk(1, bmul2(X[0], R1[0]), bmul2(X[1], R1[1]), bmul2(X[2], R1[2]), bmul2(X[3], R1[3]),
                  bmul2(X[0], X[1]), bmul2(X[1], X[2]), bmul2(X[2], X[3]), bmul2(X[3], X[0]));
        store_blk(2, bmul2(X[0], R3[0]), bmul2(X[1], R3[1]), bmul2(X[2], R3[2]), bmul2(X[3], R3[3]),
                  bmul2(X[0], X[2]), bmul2(X[1], X[3]), ONE_ZERO, 0u);
    }
}

// ------------------------------------------------------------------------------------------------
// Work partition: the B*H*n_c chunks, ordered head-major, are cut into G contiguous ranges.
// ------------------------------------------------------------------------------------------------
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

struct ChunkInfo {
    int b, h, c, t0;
    bool has_ro, has_upd, upd_acc;
};
__device__ __forceinline__ ChunkInfo chunk_info(long long g, long long g1, int n_c, int H) {
    ChunkInfo ci;
    const long long head = g / n_c;
    ci.c = static_cast<int>(g % n_c);
    ci.b = static_cast<int>(head / H);
    ci.h = static_cast<int>(head % H);
    ci.t0 = ci.c * kChunk;
    ci.has_ro = ci.c > 0;                                     // a non-zero state precedes
    ci.has_upd = !((g == g1 - 1) || (ci.c == n_c - 1));       // a later chunk of this range uses it
    ci.upd_acc = ci.c > 0;                                    // accumulate onto the carried state
    return ci;
}

// ------------------------------------------------------------------------------------------------
// Forward kernel
// ------------------------------------------------------------------------------------------------
enum FwdBar {
    FB_TMA_FULL0 = 0, FB_TMA_FULL1, FB_STAGE_FREE0, FB_STAGE_FREE1, FB_S_FULL, FB_A_FULL,
    FB_O_FULL, FB_O_FREE, FB_AV_DONE, FB_PHIQ_FULL, FB_PHIQ_FREE, FB_PHIK_FULL, FB_PHIK_FREE,
    FB_UPD_DONE, FB_SBF_FULL, FB_DRAIN, FB_COUNT
};

template <int K, int V>
__global__ void __launch_bounds__(kFwdThreads, 1)
based_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, float *__restrict__ out,
                 const float *__restrict__ prefix, int T, int H, int n_c, long long N, int G,
                 float scale) {
    using CF = Cfg<K, V>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + CF::OFF_BAR + 8 * FB_COUNT);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + CF::OFF_BAR + 8 * FB_COUNT + 4);
    auto BAR = [&](int i) -> uint32_t { return sb + CF::OFF_BAR + 8u * static_cast<uint32_t>(i); };

    const Part part = cta_range(N, G, blockIdx.x);
    const long long g0 = part.g0, g1 = part.g1;
    const int nchunks = static_cast<int>(g1 - g0);
    if (nchunks <= 0) return;

    // ---- set-up: barriers, constant tiles, TMEM -------------------------------------------------
    if (threadIdx.x == 0) {
        const uint32_t counts[FB_COUNT] = {1, 1, 1, 1, 1, 4, 1, 4, 1, 4, 1, 4, 1, 1, 4, 1};
        for (int i = 0; i < FB_COUNT; ++i) mbar_init(BAR(i), counts[i]);
        *abort_flag = 0;
        fence_mbar_init();
    }
    // bf16 state operand: zero once (rows V+2.. stay zero; rows 0..V+1 are rewritten per use).
    for (int i = threadIdx.x; i < CF::SBF / 16; i += kFwdThreads)
        st_shared_v4(sb + CF::OFF_SBF + 16u * i, 0u, 0u, 0u, 0u);
    if constexpr (CF::ZROW) {
        // ones tile: the extra A rows (64..127) of the state update, as an MN-major SW128 block;
        // row (token) r holds 1.0 at element 0, so that row 64 of S^T accumulates z.
        for (int i = threadIdx.x; i < CF::VT / 16; i += kFwdThreads)
            st_shared_v4(sb + CF::OFF_ONES + 16u * i, 0u, 0u, 0u, 0u);
        __syncthreads();
        if (threadIdx.x < kChunk)
            st_shared_u16(sb + CF::OFF_ONES + sw128(threadIdx.x, 0), 0x3F80);
    } else {
        // ones column for the z MMA: K-major SW32 operand, N row 0 = 16 ones, rows 1..15 = 0.
        if (threadIdx.x < 32)
            st_shared_v4(sb + CF::OFF_ZONES + 16u * threadIdx.x,
                         threadIdx.x < 2 ? 0x3F803F80u : 0u, threadIdx.x < 2 ? 0x3F803F80u : 0u,
                         threadIdx.x < 2 ? 0x3F803F80u : 0u, threadIdx.x < 2 ? 0x3F803F80u : 0u);
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_holder), 512);
        tmem_relinquish();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    const float c_lin = scale, c_sq = 0.5f * scale * scale, c_x = scale * scale;

    if (warp == 0) {
        // ================================ TMA producer =========================================
        if (lane == 0) {
            prefetch_tensormap(&tm_q);
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
            int issued = 0;
            for (int n = 0; n < nchunks; ++n) {
                const int s = n & 1;
                if (n >= 2 && !wait_bar(BAR(FB_STAGE_FREE0 + s), ((n >> 1) - 1) & 1, abort_flag,
                                        SITE_STAGE_FREE))
                    break;
                const ChunkInfo ci = chunk_info(g0 + n, g1, n_c, H);
                const uint32_t bar = BAR(FB_TMA_FULL0 + s);
                mbar_arrive_expect_tx(bar, 2 * CF::RAW + CF::VT);
                tma_load_4d(sb + CF::OFF_RAWQ + s * CF::RAW, &tm_q, bar, 0, ci.h, ci.t0, ci.b);
                tma_load_4d(sb + CF::OFF_RAWK + s * CF::RAW, &tm_k, bar, 0, ci.h, ci.t0, ci.b);
                tma_load_4d(sb + CF::OFF_V + s * CF::VT, &tm_v, bar, 0, ci.h, ci.t0, ci.b);
                if constexpr (V == 128)
                    tma_load_4d(sb + CF::OFF_V + s * CF::VT + 16384, &tm_v, bar, 64, ci.h, ci.t0,
                                ci.b);
                ++issued;
            }
            if (*abort_flag) {  // let copies already in flight land before the CTA exits
                for (int m = issued - 2; m < issued; ++m)
                    if (m >= 0)
                        wait_bar(BAR(FB_TMA_FULL0 + (m & 1)), (m >> 1) & 1, nullptr, SITE_DRAIN,
                                 kDrainLimitNs);
            }
        }
    } else if (warp == 1) {
        // ================================ MMA issuer ===========================================
        if (lane == 0) {
            const uint32_t t_s = tmem + CF::TM_S, t_sa = tmem + CF::TM_SA, t_o = tmem + CF::TM_O,
                           t_z = tmem + CF::TM_Z;
            constexpr uint32_t ID_QK = idesc_bf16_f32(128, 128, 0, 0);
            constexpr uint32_t ID_AV = idesc_bf16_f32(128, V, 0, 1);
            constexpr uint32_t ID_RO = idesc_bf16_f32(128, CF::NO, 0, 0);
            constexpr uint32_t ID_UPD = idesc_bf16_f32(128, CF::PP, 1, 1);
            constexpr uint32_t ID_Z = idesc_bf16_f32(128, 16, 1, 0);
            auto issue_qk = [&](int s) {
                const uint64_t a = smem_desc(sb + CF::OFF_RAWQ + s * CF::RAW, 16, 256, LAYOUT_SW32);
                const uint64_t b = smem_desc(sb + CF::OFF_RAWK + s * CF::RAW, 16, 256, LAYOUT_SW32);
                mma_ss(t_sa, a, b, ID_QK, 0);
            };
            int ro_idx = 0, upd_idx = 0;
            bool ok = wait_bar(BAR(FB_TMA_FULL0), 0, abort_flag, SITE_TMA_FULL);
            if (ok) {
                tc_fence_after();
                issue_qk(0);
                mma_commit(BAR(FB_S_FULL));
            }
            for (int n = 0; ok && n < nchunks; ++n) {
                const int s = n & 1;
                const ChunkInfo ci = chunk_info(g0 + n, g1, n_c, H);
                if (!(ok = wait_bar(BAR(FB_A_FULL), n & 1, abort_flag, SITE_A_FULL))) break;
                if (n > 0 && !(ok = wait_bar(BAR(FB_O_FREE), (n - 1) & 1, abort_flag, SITE_O_FREE)))
                    break;
                tc_fence_after();
                // O = A v_c (A: bf16 in TMEM; v_c: MN-major SW128, 16 tokens per step)
                const uint32_t vb = sb + CF::OFF_V + s * CF::VT;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    mma_ts(t_o, t_sa + 8 * j, smem_desc(vb + 2048 * j, 16384, 1024, LAYOUT_SW128),
                           ID_AV, j > 0);
                mma_commit(BAR(FB_AV_DONE));
                if (ci.has_ro) {
                    // O += f(q_c) [S | z_hi z_lo]
                    if (!(ok = wait_bar(BAR(FB_PHIQ_FULL), ro_idx & 1, abort_flag, SITE_PHIQ_FULL)))
                        break;
                    if (!(ok = wait_bar(BAR(FB_SBF_FULL), ro_idx & 1, abort_flag, SITE_SBF_FULL)))
                        break;
                    tc_fence_after();
#pragma unroll
                    for (int f = 0; f < CF::NBLK; ++f)
                        mma_ss(t_o, smem_desc(sb + CF::OFF_PHIQ + 4096 * f, 16, 256, LAYOUT_SW32),
                               smem_desc(sb + CF::OFF_SBF + CF::SBF_BLK * f, 16, 256, LAYOUT_SW32),
                               ID_RO, 1);
                    mma_commit(BAR(FB_PHIQ_FREE));
                    ++ro_idx;
                }
                mma_commit(BAR(FB_O_FULL));
                // s of the next chunk overwrites A: wait until the A v_c product has read it.
                if (!(ok = wait_bar(BAR(FB_AV_DONE), n & 1, abort_flag, SITE_AV_DONE))) break;
                if (n + 1 < nchunks) {
                    const int s1 = (n + 1) & 1;
                    if (!(ok = wait_bar(BAR(FB_TMA_FULL0 + s1), ((n + 1) >> 1) & 1, abort_flag,
                                        SITE_TMA_FULL)))
                        break;
                    tc_fence_after();
                    issue_qk(s1);
                    mma_commit(BAR(FB_S_FULL));
                }
                if (ci.has_upd) {
                    // S^T += [v_c | 1]^T f(k_c)  (and z via the ones row or the z MMA)
                    if (!(ok = wait_bar(BAR(FB_PHIK_FULL), upd_idx & 1, abort_flag, SITE_PHIK_FULL)))
                        break;
                    tc_fence_after();
                    const uint32_t lbo_a = CF::ZROW ? (CF::OFF_ONES - (CF::OFF_V + s * CF::VT)) : 16384u;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t acc = (j > 0 || ci.upd_acc) ? 1u : 0u;
                        mma_ss(t_s, smem_desc(vb + 2048 * j, lbo_a, 1024, LAYOUT_SW128),
                               smem_desc(sb + CF::OFF_PHIK + 512 * j, 4096, 256, LAYOUT_SW32),
                               ID_UPD, acc);
                        if constexpr (!CF::ZROW) {
                            const uint64_t zb = smem_desc(sb + CF::OFF_ZONES, 16, 256, LAYOUT_SW32);
                            mma_ss(t_z, smem_desc(sb + CF::OFF_PHIK + 512 * j, 4096, 256, LAYOUT_SW32),
                                   zb, ID_Z, acc);
                            if constexpr (CF::PP > 128)  // features 32..159 (only 128.. read)
                                mma_ss(t_z + 16,
                                       smem_desc(sb + CF::OFF_PHIK + 2 * 4096 + 512 * j, 4096, 256,
                                                 LAYOUT_SW32),
                                       zb, ID_Z, acc);
                        }
                    }
                    mma_commit(BAR(FB_UPD_DONE));
                    mma_commit(BAR(FB_PHIK_FREE));
                    ++upd_idx;
                }
                mma_commit(BAR(FB_STAGE_FREE0 + s));
            }
            // every MMA issued must finish before TMEM is released
            mma_commit(BAR(FB_DRAIN));
            wait_bar(BAR(FB_DRAIN), 0, nullptr, SITE_DRAIN, kDrainLimitNs);
        }
    } else if (warp < 4) {
        // warps 2 and 3: no role (warp 2 owns the TMEM allocation)
    } else if (warp < 8) {
        // ======================= rows: polynomial of chunk n, epilogue of chunk n-1 ============
        const int q4 = warp & 3;
        const int row = q4 * 32 + lane;
        const uint32_t lo = static_cast<uint32_t>(q4 * 32) << 16;
        const float c1 = scale, c2 = 0.5f * scale * scale;
        tmem_st_x2(tmem + lo + CF::TM_O + V, 0u, 0u);  // den columns start at zero
        tmem_wait_st();

        auto epilogue = [&](int m, float rowsum) -> bool {
            const ChunkInfo ci = chunk_info(g0 + m, g1, n_c, H);
            if (!wait_bar(BAR(FB_O_FULL), m & 1, abort_flag, SITE_O_FULL)) return false;
            tc_fence_after();
            uint32_t d[2];
            tmem_ld_x2(tmem + lo + CF::TM_O + V, d);
            uint32_t r[32];
            tmem_ld_x32(tmem + lo + CF::TM_O, r);
            tmem_wait_ld();
            const float den = rowsum + __uint_as_float(d[0]) + __uint_as_float(d[1]) + 1e-6f;
            const float inv = __frcp_rn(den);
            const int t = ci.t0 + row;
            float *dst = out + ((static_cast<size_t>(ci.b) * T + t) * H + ci.h) * V;
            const bool valid = t < T;
#pragma unroll
            for (int p = 0; p < V / 32; ++p) {
                if (p > 0) {
                    tmem_ld_x32(tmem + lo + CF::TM_O + 32 * p, r);
                    tmem_wait_ld();
                }
                if (p == V / 32 - 1) {
                    // O fully read: zero the den columns for the next chunk and release O.
                    tmem_st_x2(tmem + lo + CF::TM_O + V, 0u, 0u);
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(BAR(FB_O_FREE));
                }
                if (valid) {
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        st_global_cs_v4(dst + 32 * p + e, __uint_as_float(r[e]) * inv,
                                        __uint_as_float(r[e + 1]) * inv,
                                        __uint_as_float(r[e + 2]) * inv,
                                        __uint_as_float(r[e + 3]) * inv);
                }
            }
            return true;
        };

        float rs_prev = 0.0f;
        bool ok = true;
        for (int n = 0; n < nchunks; ++n) {
            if (!(ok = wait_bar(BAR(FB_S_FULL), n & 1, abort_flag, SITE_S_FULL))) break;
            tc_fence_after();
            float rs = 0.0f;
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) {
                uint32_t packed[16];
                if (kb <= q4) {
                    uint32_t r[32];
                    tmem_ld_x32(tmem + lo + CF::TM_SA + 32 * kb, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const float s0 = __uint_as_float(r[j]), s1 = __uint_as_float(r[j + 1]);
                        float a0 = fmaf(s0, fmaf(c2, s0, c1), 1.0f);
                        float a1 = fmaf(s1, fmaf(c2, s1, c1), 1.0f);
                        if (kb == q4) {  // causal mask on the diagonal block: key j <= row
                            if (j > lane) a0 = 0.0f;
                            if (j + 1 > lane) a1 = 0.0f;
                        }
                        const __nv_bfloat162 p = __floats2bfloat162_rn(a0, a1);
                        rs += __low2float(p) + __high2float(p);
                        packed[j >> 1] = *reinterpret_cast<const uint32_t *>(&p);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) packed[j] = 0u;
                }
                // A columns [16 kb, 16 kb + 16) overlay s columns that were already read.
                tmem_st_x16(tmem + lo + CF::TM_SA + 16 * kb, packed);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(FB_A_FULL));
            if (n > 0 && !(ok = epilogue(n - 1, rs_prev))) break;
            rs_prev = rs;
        }
        if (ok) epilogue(nchunks - 1, rs_prev);
    } else if (warp < 12) {
        // ================================ feature builders =====================================
        const int t = (warp - 8) * 32 + lane;
        int ro_idx = 0, upd_idx = 0;
        for (int n = 0; n < nchunks; ++n) {
            const int s = n & 1;
            const ChunkInfo ci = chunk_info(g0 + n, g1, n_c, H);
            if (!ci.has_ro && !ci.has_upd) continue;
            if (!wait_bar(BAR(FB_TMA_FULL0 + s), (n >> 1) & 1, abort_flag, SITE_TMA_FULL)) break;
            if (ci.has_ro) {
                if (ro_idx > 0 &&
                    !wait_bar(BAR(FB_PHIQ_FREE), (ro_idx - 1) & 1, abort_flag, SITE_PHIQ_FREE))
                    break;
                build_features<K>(sb + CF::OFF_RAWQ + s * CF::RAW, sb + CF::OFF_PHIQ, t);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(FB_PHIQ_FULL));
                ++ro_idx;
            }
            if (ci.has_upd) {
                if (upd_idx > 0 &&
                    !wait_bar(BAR(FB_PHIK_FREE), (upd_idx - 1) & 1, abort_flag, SITE_PHIK_FREE))
                    break;
                build_features<K>(sb + CF::OFF_RAWK + s * CF::RAW, sb + CF::OFF_PHIK, t);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(FB_PHIK_FULL));
                ++upd_idx;
            }
        }
    } else {
        // ============== state conversion: S^T (fp32, TMEM) -> bf16 operand [S | z_hi z_lo] =====
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane;  // TMEM lane = row of S^T = value index
        const uint32_t lo = static_cast<uint32_t>(q4 * 32) << 16;
        constexpr int LAST_ROW = CF::ZROW ? V : V - 1;
        const bool warp_has_rows = q4 * 32 <= LAST_ROW;

        auto convert = [&]() {
            if (warp_has_rows) {
#pragma unroll 1
                for (int f = 0; f < CF::NBLK; ++f) {
                    uint32_t x[16];
                    tmem_ld_x16(tmem + lo + CF::TM_S + 16 * f, x);
                    tmem_wait_ld();
                    float v[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        v[j] = __uint_as_float(x[j]) * feature_coef<K>(f, j, c_lin, c_sq, c_x);
                    const uint32_t blk = sb + CF::OFF_SBF + CF::SBF_BLK * f;
                    if (r < V) {
                        st_shared_v4(blk + sw32(r, 0), pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                     pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
                        st_shared_v4(blk + sw32(r, 1), pack_bf16x2(v[8], v[9]),
                                     pack_bf16x2(v[10], v[11]), pack_bf16x2(v[12], v[13]),
                                     pack_bf16x2(v[14], v[15]));
                    } else if (CF::ZROW && r == V) {
                        // z as a hi/lo pair of bf16 rows: about 16 significant bits
                        uint32_t hi[8], lw[8];
#pragma unroll
                        for (int j = 0; j < 16; j += 2) {
                            const __nv_bfloat162 h2 = __floats2bfloat162_rn(v[j], v[j + 1]);
                            hi[j >> 1] = *reinterpret_cast<const uint32_t *>(&h2);
                            lw[j >> 1] = pack_bf16x2(v[j] - __low2float(h2), v[j + 1] - __high2float(h2));
                        }
                        st_shared_v4(blk + sw32(V, 0), hi[0], hi[1], hi[2], hi[3]);
                        st_shared_v4(blk + sw32(V, 1), hi[4], hi[5], hi[6], hi[7]);
                        st_shared_v4(blk + sw32(V + 1, 0), lw[0], lw[1], lw[2], lw[3]);
                        st_shared_v4(blk + sw32(V + 1, 1), lw[4], lw[5], lw[6], lw[7]);
                    }
                }
            }
            if constexpr (!CF::ZROW) {
                // z tiles: lane r of tile a holds feature r, lane r of tile b holds feature r + 32
                uint32_t za, zb;
                tmem_ld_x1(tmem + lo + CF::TM_Z, za);
                tmem_ld_x1(tmem + lo + CF::TM_Z + 16, zb);
                tmem_wait_ld();
                auto put = [&](int p, float z) {
                    const int f = p >> 4, j = p & 15;
                    const float zc = z * feature_coef<K>(f, j, c_lin, c_sq, c_x);
                    const __nv_bfloat16 h = __float2bfloat16_rn(zc);
                    const __nv_bfloat16 l = __float2bfloat16_rn(zc - __bfloat162float(h));
                    const uint32_t a = sb + CF::OFF_SBF + CF::SBF_BLK * f + 2u * (j & 7);
                    st_shared_u16(a + sw32(V, j >> 3), *reinterpret_cast<const uint16_t *>(&h));
                    st_shared_u16(a + sw32(V + 1, j >> 3), *reinterpret_cast<const uint16_t *>(&l));
                };
                if (r < CF::PP && r < 128) put(r, __uint_as_float(za));
                if (r + 32 >= 128 && r + 32 < CF::PP) put(r + 32, __uint_as_float(zb));
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(FB_SBF_FULL));
        };

        // A range that starts inside a head continues from the prefix state of the chunks before
        // it: load it into TMEM, then convert it like any other state.
        if (g0 % n_c != 0) {
            const float *slot = prefix + static_cast<size_t>(blockIdx.x - 1) * CF::SLOT;
            if (warp_has_rows) {
                const bool mine = r <= LAST_ROW;
#pragma unroll 1
                for (int f = 0; f < CF::NBLK; ++f) {
                    uint32_t x[16];
#pragma unroll
                    for (int j = 0; j < 16; j += 4) {
                        float4 v4 = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (mine)
                            v4 = *reinterpret_cast<const float4 *>(slot + static_cast<size_t>(r) * CF::PP +
                                                                   16 * f + j);
                        x[j] = __float_as_uint(v4.x);
                        x[j + 1] = __float_as_uint(v4.y);
                        x[j + 2] = __float_as_uint(v4.z);
                        x[j + 3] = __float_as_uint(v4.w);
                    }
                    tmem_st_x16(tmem + lo + CF::TM_S + 16 * f, x);
                }
            }
            if constexpr (!CF::ZROW) {
                const float *zrow = slot + static_cast<size_t>(V) * CF::PP;
                const float za = r < CF::PP ? zrow[r] : 0.0f;
                const float zb = r + 32 < CF::PP ? zrow[r + 32] : 0.0f;
                tmem_st_x1(tmem + lo + CF::TM_Z, __float_as_uint(za));
                tmem_st_x1(tmem + lo + CF::TM_Z + 16, __float_as_uint(zb));
            }
            tmem_wait_st();
            convert();
        }
        int u = 0;
        for (int n = 0; n < nchunks; ++n) {
            const ChunkInfo ci = chunk_info(g0 + n, g1, n_c, H);
            if (!ci.has_upd) continue;
            if (!wait_bar(BAR(FB_UPD_DONE), u & 1, abort_flag, SITE_UPD_DONE)) break;
            tc_fence_after();
            convert();
            ++u;
        }
    }

    // ---- teardown ------------------------------------------------------------------------------
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------------------------------------
// Aggregate kernel: the partial state [S^T | z] of the last stretch of a range that ends inside a
// head, written as fp32 rows into slot blockIdx.x.
// ------------------------------------------------------------------------------------------------
enum AggBar {
    AB_TMA_FULL0 = 0, AB_TMA_FULL1, AB_STAGE_FREE0, AB_STAGE_FREE1, AB_PHIK_FULL, AB_PHIK_FREE,
    AB_AGG_DONE, AB_DRAIN, AB_COUNT
};

template <int K, int V>
__global__ void __launch_bounds__(kAggThreads, 1)
based_agg_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 float *__restrict__ slots, int H, int n_c, long long N, int G) {
    using CF = Cfg<K, V>;
    if (!has_aggregate(N, G, blockIdx.x, n_c)) return;
    const Part part = cta_range(N, G, blockIdx.x);
    const long long ga = part.g0 > ((part.g1 - 1) / n_c) * n_c ? part.g0 : ((part.g1 - 1) / n_c) * n_c;
    const long long g1 = part.g1;
    const int nchunks = static_cast<int>(g1 - ga);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + CF::A_OFF_BAR + 8 * AB_COUNT);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + CF::A_OFF_BAR + 8 * AB_COUNT + 4);
    auto BAR = [&](int i) -> uint32_t { return sb + CF::A_OFF_BAR + 8u * static_cast<uint32_t>(i); };

    if (threadIdx.x == 0) {
        const uint32_t counts[AB_COUNT] = {1, 1, 1, 1, 4, 1, 1, 1};
        for (int i = 0; i < AB_COUNT; ++i) mbar_init(BAR(i), counts[i]);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if constexpr (CF::ZROW) {
        for (int i = threadIdx.x; i < CF::VT / 16; i += kAggThreads)
            st_shared_v4(sb + CF::A_OFF_ONES + 16u * i, 0u, 0u, 0u, 0u);
        __syncthreads();
        if (threadIdx.x < kChunk)
            st_shared_u16(sb + CF::A_OFF_ONES + sw128(threadIdx.x, 0), 0x3F80);
    } else {
        if (threadIdx.x < 32)
            st_shared_v4(sb + CF::A_OFF_ZONES + 16u * threadIdx.x,
                         threadIdx.x < 2 ? 0x3F803F80u : 0u, threadIdx.x < 2 ? 0x3F803F80u : 0u,
                         threadIdx.x < 2 ? 0x3F803F80u : 0u, threadIdx.x < 2 ? 0x3F803F80u : 0u);
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_holder), 256);
        tmem_relinquish();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
            int issued = 0;
            for (int n = 0; n < nchunks; ++n) {
                const int s = n & 1;
                if (n >= 2 && !wait_bar(BAR(AB_STAGE_FREE0 + s), ((n >> 1) - 1) & 1, abort_flag,
                                        SITE_STAGE_FREE))
                    break;
                const ChunkInfo ci = chunk_info(ga + n, g1, n_c, H);
                const uint32_t bar = BAR(AB_TMA_FULL0 + s);
                mbar_arrive_expect_tx(bar, CF::RAW + CF::VT);
                tma_load_4d(sb + CF::A_OFF_RAWK + s * CF::RAW, &tm_k, bar, 0, ci.h, ci.t0, ci.b);
                tma_load_4d(sb + CF::A_OFF_V + s * CF::VT, &tm_v, bar, 0, ci.h, ci.t0, ci.b);
                if constexpr (V == 128)
                    tma_load_4d(sb + CF::A_OFF_V + s * CF::VT + 16384, &tm_v, bar, 64, ci.h, ci.t0,
                                ci.b);
                ++issued;
            }
            if (*abort_flag) {
                for (int m = issued - 2; m < issued; ++m)
                    if (m >= 0)
                        wait_bar(BAR(AB_TMA_FULL0 + (m & 1)), (m >> 1) & 1, nullptr, SITE_DRAIN,
                                 kDrainLimitNs);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t ID_UPD = idesc_bf16_f32(128, CF::PP, 1, 1);
            constexpr uint32_t ID_Z = idesc_bf16_f32(128, 16, 1, 0);
            const uint32_t t_s = tmem, t_z = tmem + CF::TA_Z;
            for (int n = 0; n < nchunks; ++n) {
                const int s = n & 1;
                if (!wait_bar(BAR(AB_TMA_FULL0 + s), (n >> 1) & 1, abort_flag, SITE_TMA_FULL)) break;
                if (!wait_bar(BAR(AB_PHIK_FULL), n & 1, abort_flag, SITE_PHIK_FULL)) break;
                tc_fence_after();
                const uint32_t vb = sb + CF::A_OFF_V + s * CF::VT;
                const uint32_t lbo_a = CF::ZROW ? (CF::A_OFF_ONES - (CF::A_OFF_V + s * CF::VT)) : 16384u;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t acc = (j > 0 || n > 0) ? 1u : 0u;
                    mma_ss(t_s, smem_desc(vb + 2048 * j, lbo_a, 1024, LAYOUT_SW128),
                           smem_desc(sb + CF::A_OFF_PHIK + 512 * j, 4096, 256, LAYOUT_SW32), ID_UPD,
                           acc);
                    if constexpr (!CF::ZROW) {
                        const uint64_t zb = smem_desc(sb + CF::A_OFF_ZONES, 16, 256, LAYOUT_SW32);
                        mma_ss(t_z, smem_desc(sb + CF::A_OFF_PHIK + 512 * j, 4096, 256, LAYOUT_SW32),
                               zb, ID_Z, acc);
                        if constexpr (CF::PP > 128)
                            mma_ss(t_z + 16,
                                   smem_desc(sb + CF::A_OFF_PHIK + 2 * 4096 + 512 * j, 4096, 256,
                                             LAYOUT_SW32),
                                   zb, ID_Z, acc);
                    }
                }
                mma_commit(BAR(AB_PHIK_FREE));
                mma_commit(BAR(AB_STAGE_FREE0 + s));
            }
            mma_commit(BAR(AB_AGG_DONE));
            wait_bar(BAR(AB_AGG_DONE), 0, nullptr, SITE_DRAIN, kDrainLimitNs);
        }
    } else if (warp < 4) {
        // warps 2 and 3: no role (warp 2 owns the TMEM allocation)
    } else if (warp < 8) {
        // feature builders: token t of the chunk
        const int t = (warp - 4) * 32 + lane;
        for (int n = 0; n < nchunks; ++n) {
            const int s = n & 1;
            if (!wait_bar(BAR(AB_TMA_FULL0 + s), (n >> 1) & 1, abort_flag, SITE_TMA_FULL)) break;
            if (n > 0 && !wait_bar(BAR(AB_PHIK_FREE), (n - 1) & 1, abort_flag, SITE_PHIK_FREE)) break;
            build_features<K>(sb + CF::A_OFF_RAWK + s * CF::RAW, sb + CF::A_OFF_PHIK, t);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(AB_PHIK_FULL));
        }
    } else {
        // writer: S^T rows (and z) -> fp32 slot
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane;
        const uint32_t lo = static_cast<uint32_t>(q4 * 32) << 16;
        constexpr int LAST_ROW = CF::ZROW ? V : V - 1;
        float *slot = slots + static_cast<size_t>(blockIdx.x) * CF::SLOT;
        if (wait_bar(BAR(AB_AGG_DONE), 0, abort_flag, SITE_AGG_DONE)) {
            tc_fence_after();
            if (q4 * 32 <= LAST_ROW) {
#pragma unroll 1
                for (int f = 0; f < CF::NBLK; ++f) {
                    uint32_t x[16];
                    tmem_ld_x16(tmem + lo + 16 * f, x);
                    tmem_wait_ld();
                    if (r <= LAST_ROW) {
                        float *dst = slot + static_cast<size_t>(r) * CF::PP + 16 * f;
#pragma unroll
                        for (int j = 0; j < 16; j += 4)
                            *reinterpret_cast<float4 *>(dst + j) =
                                make_float4(__uint_as_float(x[j]), __uint_as_float(x[j + 1]),
                                            __uint_as_float(x[j + 2]), __uint_as_float(x[j + 3]));
                    }
                }
            }
            if constexpr (!CF::ZROW) {
                uint32_t za, zb;
                tmem_ld_x1(tmem + lo + CF::TA_Z, za);
                tmem_ld_x1(tmem + lo + CF::TA_Z + 16, zb);
                tmem_wait_ld();
                float *zrow = slot + static_cast<size_t>(V) * CF::PP;
                if (r < CF::PP && r < 128) zrow[r] = __uint_as_float(za);
                if (r + 32 >= 128 && r + 32 < CF::PP) zrow[r + 32] = __uint_as_float(zb);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// ------------------------------------------------------------------------------------------------
// Scan: within each run of ranges that continue one head's prefix, turn the per-range partial
// states into inclusive prefixes (slot i = sum of the partial states of ranges <= i in the run).
// ------------------------------------------------------------------------------------------------
__global__ void based_scan_kernel(float *__restrict__ slots, int slot_elems, int n_c, long long N,
                                  int G) {
    const int i = blockIdx.y;
    if (!has_aggregate(N, G, i, n_c) || continues_prefix(N, G, i, n_c)) return;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= slot_elems) return;
    float acc = slots[static_cast<size_t>(i) * slot_elems + e];
    for (int j = i + 1; j < G && continues_prefix(N, G, j, n_c) && has_aggregate(N, G, j, n_c); ++j) {
        float *p = slots + static_cast<size_t>(j) * slot_elems + e;
        acc += *p;
        *p = acc;
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
