// based_fwd.cu: C ABI of the Based causal forward pass (declared in include/based.h).
//
// Host side: argument checks, the work partition, tensor maps, the library-owned workspace and
// the launch sequence  [aggregate -> scan] -> forward  on the caller's stream. All arithmetic of
// the method runs in the kernels of based_kernels.cuh.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/based.h"
#include "based_kernels.cuh"
#include "based_plan.h"

namespace {

using namespace based;

thread_local char tl_cuda_error[256] = "";

int cuda_fail(cudaError_t e, const char *what) {
    snprintf(tl_cuda_error, sizeof(tl_cuda_error), "%s: %s", what, cudaGetErrorString(e));
    return BASED_ERR_CUDA;
}
#define BASED_CUDA(call)                                   \
    do {                                                   \
        cudaError_t e_ = (call);                           \
        if (e_ != cudaSuccess) return cuda_fail(e_, #call); \
    } while (0)

// cuTensorMapEncodeTiled, fetched from the driver at run time (no link-time libcuda dependency).
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// (dim0, H, T, B) tensor of 2-byte (bf16) or 4-byte (fp32) elements with a
// (box0, 1, box_rows, 1) box. promo: how far L2 widens a miss of the box's rows.
int make_map(CUtensorMap *map, const void *base, int d0, int B, int T, int H, int box0,
             CUtensorMapSwizzle swz, CUtensorMapL2promotion promo, bool fp32 = false,
             int box_rows = kChunk) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) {
        snprintf(tl_cuda_error, sizeof(tl_cuda_error), "cuTensorMapEncodeTiled unavailable");
        return BASED_ERR_CUDA;
    }
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d0), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(B)};
    const cuuint64_t es = fp32 ? 4 : 2;
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(d0) * es,
                                   static_cast<cuuint64_t>(H) * d0 * es,
                                   static_cast<cuuint64_t>(T) * H * d0 * es};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(box0), 1, static_cast<cuuint32_t>(box_rows), 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                     const_cast<void *>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                     promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(tl_cuda_error, sizeof(tl_cuda_error), "cuTensorMapEncodeTiled failed (%d)",
                 static_cast<int>(r));
        return BASED_ERR_CUDA;
    }
    return BASED_OK;
}

struct Plan {
    int n_c;        // chunks per head
    int L;          // head lanes (choose_lanes); every lane has the same partition and plan
    long long N;    // chunks of one lane
    int G;          // ranges of one lane (forward CTAs: G L)
    bool lead_in;   // ranges that start inside a head run a lead-in (else: slots, see Ranges)
    bool need_agg;  // the aggregate pass runs (slots, and some range ends inside a head)
    int slot_floats;
    size_t ws_bytes;
    AggPlan agg;    // pieces of the aggregate pass, the forward CTAs' prefixes, the scan runs
    Ranges rg;      // the forward CTAs' ranges and how each gets its prefix
};

constexpr int kMaxDevices = 64;
struct DeviceState {
    std::mutex m;
    bool init = false;
    int sms = 0;
    int cc_major = 0, cc_minor = 0;
    bool attrs_done[2][2][2] = {};  // [K == 16][V == 128][bf16 output]
    void *ws = nullptr;
    size_t ws_bytes = 0;
    // Workspaces that a larger one replaced. They are never freed: a CUDA graph may have captured
    // a call that uses one, and replaying it must not write to freed memory.
    std::vector<void *> retired_ws;
    void *hbuf = nullptr;  // based_fwd_host staging (q | k | v | o)
    size_t hbuf_bytes = 0;
    // based_fwd_host pipeline: copy-in, compute and copy-out streams, per-piece events, and the
    // compute stream's workspace
    static constexpr int kHostPieces = 8;
    cudaStream_t hs_in = nullptr, hs_comp = nullptr, hs_out = nullptr;
    cudaEvent_t hfork = nullptr, hdone = nullptr;
    cudaEvent_t hin[kHostPieces] = {}, hcomp[kHostPieces] = {};
    void *hws = nullptr;
    size_t hws_bytes = 0;
};
DeviceState g_dev[kMaxDevices];

int current_device(int *dev) {
    BASED_CUDA(cudaGetDevice(dev));
    if (*dev < 0 || *dev >= kMaxDevices) return BASED_ERR_NO_DEVICE;
    DeviceState &d = g_dev[*dev];
    std::lock_guard<std::mutex> lk(d.m);
    if (!d.init) {
        cudaDeviceProp prop;
        BASED_CUDA(cudaGetDeviceProperties(&prop, *dev));
        d.sms = prop.multiProcessorCount;
        d.cc_major = prop.major;
        d.cc_minor = prop.minor;
        d.init = true;
    }
    if (!(d.cc_major == 10 && d.cc_minor == 3)) return BASED_ERR_NO_DEVICE;
    return BASED_OK;
}

int slot_floats(int K, int V) { return (V + 1) * ((K == 16) ? 160 : 48); }

// max_ws: workspace bytes the plan may use at most (the balanced aggregate pass needs a slot per
// piece, up to about twice the ranges; with less it falls back to one slot per range)
Plan build_plan(int B, int T, int H, int K, int V, int sms, size_t max_ws) {
    Plan p;
    const LaneSplit ls = lane_split(B, T, H, K, sms);
    p.n_c = ls.n_c;
    p.L = ls.L;
    p.N = ls.N;
    p.G = ls.G;
    p.need_agg = false;
    for (int i = 0; i < p.G; ++i)
        if (has_aggregate(p.N, p.G, i, p.n_c)) p.need_agg = true;
    p.slot_floats = slot_floats(K, V);
    const size_t slot_bytes = static_cast<size_t>(p.slot_floats) * sizeof(float);
    const size_t max_slots = max_ws / slot_bytes / p.L;  // per lane
    make_agg_plan(p.N, p.G, p.n_c, p.G, max_slots < kMaxPieces ? static_cast<int>(max_slots) : kMaxPieces, p.agg);
    p.lead_in = false;
    if (p.need_agg) {
        // lead-ins instead of slots, where the cost model finds them faster
        const int used = choose_lead_in(p.N, p.G, p.n_c, V, p.agg, p.rg);
        if (used > 0) {
            p.lead_in = true;
            p.need_agg = false;
            p.G = used;  // the ranges past the last are empty: no CTAs for them
        }
    }
    if (!p.lead_in) {
        for (int j = 0; j <= p.G; ++j) p.rg.g0[j] = static_cast<int32_t>(cta_range(p.N, p.G, j).g0);  // j = G: N
        p.rg.lead_in = 0;
        for (int j = 0; j < p.G; ++j) {
            p.rg.order[j] = static_cast<uint16_t>(j);
            p.rg.slot[j] = p.agg.pre.slot[j];
            p.rg.cnt[j] = p.agg.pre.cnt[j];
        }
    }
    p.ws_bytes = p.need_agg ? static_cast<size_t>(p.L) * p.agg.pieces.n * slot_bytes : 0;
    return p;
}

// The plan of a shape, from a per-thread cache of the last few shapes: a call repeats the shape
// of the calls before it far more often than not, and building a plan (the aggregate plan, the
// bisection of the lead-in cut) costs host time comparable to a small call's kernel time. The
// reference stays valid until this thread's next make_plan call.
const Plan &make_plan(int B, int T, int H, int K, int V, int sms, size_t max_ws = ~static_cast<size_t>(0)) {
    struct Entry {
        int key[6];
        size_t max_ws;
        bool used;
        Plan plan;
    };
    constexpr int kEntries = 4;
    static thread_local Entry cache[kEntries];
    static thread_local int next = 0;
    const int key[6] = {B, T, H, K, V, sms};
    for (Entry &e : cache)
        if (e.used && e.max_ws == max_ws && std::memcmp(e.key, key, sizeof(key)) == 0) return e.plan;
    Entry &e = cache[next];
    next = (next + 1) % kEntries;
    e.plan = build_plan(B, T, H, K, V, sms, max_ws);
    std::memcpy(e.key, key, sizeof(key));
    e.max_ws = max_ws;
    e.used = true;
    return e.plan;
}

// The kernels index the slots with the plan's tables and check none of them on the device: the
// ranges must cut the lane's chunks in order, each lead-in must stay inside its head, every
// prefix must read only slots the aggregate pass writes, every piece must lie in its lane's
// chunks, and every scan run must stay within the slots. A plan that breaks this is a library
// bug; the call then fails before anything is launched (the partition check in the tests
// exercises the same invariants over many shapes).
bool plan_in_bounds(const Plan &p) {
    if (p.G < 1 || p.G > kMaxRanges || p.rg.g0[0] != 0 || p.rg.g0[p.G] != p.N) return false;
    if (p.rg.lead_in != (p.lead_in ? 1 : 0)) return false;
    {
        bool seen[kMaxRanges] = {};  // the launch order is a permutation of the ranges
        for (int i = 0; i < p.G; ++i) {
            if (p.rg.order[i] >= p.G || seen[p.rg.order[i]]) return false;
            seen[p.rg.order[i]] = true;
        }
    }
    for (int j = 0; j < p.G; ++j) {
        if (p.rg.g0[j + 1] <= p.rg.g0[j]) return false;
        if (p.lead_in && p.rg.cnt[j] != 0) return false;
        if (!p.need_agg && p.rg.cnt[j] != 0) return false;
    }
    if (!p.need_agg) return true;
    for (int j = 0; j < p.G; ++j)
        if (p.rg.cnt[j] != p.agg.pre.cnt[j] || p.rg.slot[j] != p.agg.pre.slot[j]) return false;
    const AggPieces &A = p.agg.pieces;
    if (A.n < 1 || A.n > kMaxPieces || A.n_cta < 1 || A.n_cta > p.G) return false;
    if (A.cta_first[0] != 0 || A.cta_first[A.n_cta] != A.n) return false;
    for (int j = 0; j < A.n_cta; ++j)
        if (A.cta_first[j + 1] < A.cta_first[j]) return false;
    for (int q = 0; q < A.n; ++q)
        if (A.len[q] < 1 || A.g0[q] < 0 || static_cast<long long>(A.g0[q]) + A.len[q] > p.N) return false;
    for (int r = 0; r < p.G; ++r) {
        const int cnt = p.agg.pre.cnt[r];
        if (cnt == 0) continue;
        if (cnt > (p.agg.scan ? 1 : kMaxChain) || p.agg.pre.slot[r] + cnt > A.n) return false;
    }
    if (p.agg.scan)
        for (int i = 0; i < p.agg.runs.n; ++i)
            if (p.agg.runs.len[i] < 2 || p.agg.runs.start[i] + p.agg.runs.len[i] > A.n) return false;
    return true;
}

// out_elem: bytes per output element (4 for fp32, 2 for bf16)
int check_args(const void *q, const void *k, const void *v, int B, int T, int H, int K, int V,
               const void *o, size_t out_elem = 4) {
    if (!q || !k || !v || !o) return BASED_ERR_NULL_POINTER;
    if (K != 8 && K != 16) return BASED_ERR_UNSUPPORTED_K;
    if (V != 64 && V != 128) return BASED_ERR_UNSUPPORTED_V;
    if (B < 1 || T < 1 || H < 1) return BASED_ERR_BAD_SHAPE;
    if (static_cast<long long>(B) * T * H >= (1ll << 31)) return BASED_ERR_BAD_SHAPE;
    auto al = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!al(q) || !al(k) || !al(v) || !al(o)) return BASED_ERR_MISALIGNED;
    const size_t rows = static_cast<size_t>(B) * T * H;
    auto overlap = [](const void *a, size_t na, const void *b, size_t nb) {
        const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
        return x < y + nb && y < x + na;
    };
    const size_t ob = rows * V * out_elem;
    if (overlap(o, ob, q, rows * K * 2) || overlap(o, ob, k, rows * K * 2) ||
        overlap(o, ob, v, rows * V * 2))
        return BASED_ERR_ALIASING;
    return BASED_OK;
}

// Launches kernel<<<grid, block, smem, st>>>(args...), as a programmatic dependent of the
// previous kernel in the stream when `dependent` is set.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t st, bool dependent, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = dependent ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

template <int K, int V, bool OBF>
int launch(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int T, int H,
           float scale, void *o, float *ws, const Plan &p, DeviceState &d, cudaStream_t st,
           cudaEvent_t ev_begin, cudaEvent_t ev_end) {
    using CF = Cfg<K, V>;
    // the forward kernel's instances: prefixes from slots, and lead-ins (V = 64; for V = 128 the
    // same instance)
    void (*const fwd_slots)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, const float *, int, int, int,
                            long long, int, int, int, float, Ranges, int) = based_fwd_kernel<K, V, OBF, false>;
    decltype(fwd_slots) fwd_lead = based_fwd_kernel<K, V, OBF, CF::FAST>;
    {
        std::lock_guard<std::mutex> lk(d.m);
        bool &done = d.attrs_done[K == 16][V == 128][OBF];
        if (!done) {
            BASED_CUDA(cudaFuncSetAttribute(fwd_slots, cudaFuncAttributeMaxDynamicSharedMemorySize, CF::SMEM_FWD));
            BASED_CUDA(cudaFuncSetAttribute(fwd_lead, cudaFuncAttributeMaxDynamicSharedMemorySize, CF::SMEM_FWD));
            BASED_CUDA(cudaFuncSetAttribute(based_agg_kernel<K, V>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize, CF::SMEM_AGG));
            done = true;
        }
    }
    CUtensorMap mq, mk, mv, mo;
    int rc;
    const CUtensorMapSwizzle sw_qk = CU_TENSOR_MAP_SWIZZLE_32B;
    // A q or k row of one head is 16 or 32 bytes of a 128-byte line shared with adjacent heads.
    // A miss fetches 64 bytes, or the whole line when four head lanes of 32-byte rows (K = 16)
    // read all of it at about the same time. Without lanes the rest of a longer fetch would be
    // read by other CTAs long after it left L2 (on inputs much larger than L2); with eight lanes
    // of 16-byte rows (K = 8) 64 bytes measure about 1 % faster. No promotion measures like 128.
    const CUtensorMapL2promotion promo_qk =
        (K == 16 && p.L == 4) ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_64B;
    if ((rc = make_map(&mq, q, K, B, T, H, 16, sw_qk, promo_qk)) != BASED_OK) return rc;
    if ((rc = make_map(&mk, k, K, B, T, H, 16, sw_qk, promo_qk)) != BASED_OK) return rc;
    if ((rc = make_map(&mv, v, V, B, T, H, 64, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B)) !=
        BASED_OK)
        return rc;
    // output boxes of 128-byte rows: 32 fp32 or 64 bf16 columns
    if ((rc = make_map(&mo, o, V, B, T, H, OBF ? 64 : 32, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_128B, !OBF, CF::EPI_ROWS)) != BASED_OK)
        return rc;
    if (p.need_agg) {
        // 512 threads (dedicated slot writers) when a CTA sums several pieces, else 384
        const int threads = p.agg.pieces.n > p.agg.pieces.n_cta ? kAggThreads : 384;
        // a programmatic dependent of the previous kernel in the stream (it waits for that kernel
        // before its first access to memory), unless the caller brackets the call with events
        BASED_CUDA(launch_dependent(based_agg_kernel<K, V>, dim3(p.agg.pieces.n_cta * p.L), dim3(threads),
                                    CF::SMEM_AGG, st, !ev_begin, mk, mv, ws, H, p.n_c, p.L, p.agg.pieces));
        if (p.agg.scan) {  // otherwise each forward CTA sums the (at most kMaxChain) slots it needs
            dim3 grid((p.slot_floats / 4 + 255) / 256, p.agg.runs.n * p.L);
            BASED_CUDA(launch_dependent(based_scan_kernel, grid, dim3(256), 0, st, true, ws,
                                        p.slot_floats, p.agg.pieces.n, p.agg.runs));
        }
    }
    if (ev_begin) BASED_CUDA(cudaEventRecord(ev_begin, st));
    // The forward kernel is launched as a programmatic dependent of the kernel before it: after
    // the aggregate pass it starts while that pass finishes (only its read of the prefix slots
    // waits for it); as the first kernel of the call it waits for the previous kernel of the stream
    // before its first access to memory. When the caller brackets the call with events, every
    // kernel is an ordinary launch.
    const bool dependent = !ev_begin;
    BASED_CUDA(launch_dependent(p.lead_in ? fwd_lead : fwd_slots, dim3(p.G * p.L), dim3(kFwdThreads), CF::SMEM_FWD, st,
                                dependent, mq, mk, mv, mo, static_cast<const float *>(ws), T, H, p.n_c,
                                p.N, p.G, p.L, p.agg.pieces.n, scale, p.rg, p.need_agg ? 0 : 1));
    if (ev_end) BASED_CUDA(cudaEventRecord(ev_end, st));
    return BASED_OK;
}

// obf: o holds bf16 (else fp32)
// max_ws: the most workspace the plan may use (the fixed scratch of based_fwd_noalloc)
int run(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int T, int H, int K, int V,
        float scale, void *o, bool obf, void *ws, size_t ws_bytes, bool own_ws, based_stream_t stream,
        void *ev_begin = nullptr, void *ev_end = nullptr, size_t max_ws = ~static_cast<size_t>(0)) {
    int rc = check_args(q, k, v, B, T, H, K, V, o, obf ? 2 : 4);
    if (rc != BASED_OK) return rc;
    int dev;
    if ((rc = current_device(&dev)) != BASED_OK) return rc;
    DeviceState &d = g_dev[dev];
    const Plan &p = make_plan(B, T, H, K, V, d.sms, max_ws);
    if (!plan_in_bounds(p)) {
        snprintf(tl_cuda_error, sizeof(tl_cuda_error), "internal error: work plan out of bounds");
        return BASED_ERR_BAD_ARGUMENT;
    }
    if (!(scale > 0.0f) || std::isnan(scale)) scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(K)));
    if (own_ws) {
        std::lock_guard<std::mutex> lk(d.m);
        if (p.ws_bytes > d.ws_bytes) {
            void *w = nullptr;
            BASED_CUDA(cudaMalloc(&w, p.ws_bytes));
            if (d.ws) d.retired_ws.push_back(d.ws);  // kept: a captured graph may still use it
            d.ws = w;
            d.ws_bytes = p.ws_bytes;
        }
        ws = d.ws;
        ws_bytes = d.ws_bytes;
    } else if (p.ws_bytes > 0) {
        if (!ws || ws_bytes < p.ws_bytes || (reinterpret_cast<uintptr_t>(ws) & 15u))
            return BASED_ERR_WORKSPACE;
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    float *w = static_cast<float *>(ws);
    cudaEvent_t eb = static_cast<cudaEvent_t>(ev_begin), ee = static_cast<cudaEvent_t>(ev_end);
    if (obf) {
        if (K == 16 && V == 64) return launch<16, 64, true>(q, k, v, B, T, H, scale, o, w, p, d, st, eb, ee);
        if (K == 16 && V == 128) return launch<16, 128, true>(q, k, v, B, T, H, scale, o, w, p, d, st, eb, ee);
        if (K == 8 && V == 64) return launch<8, 64, true>(q, k, v, B, T, H, scale, o, w, p, d, st, eb, ee);
        return launch<8, 128, true>(q, k, v, B, T, H, scale, o, w, p, d, st, eb, ee);
    }
    if (K == 16 && V == 64) return launch<16, 64, false>(q, k, v, B, T, H, scale, o, w, p, d, st, eb, ee);
    if (K == 16 && V == 128) return launch<16, 128, false>(q, k, v, B, T, H, scale, o, w, p, d, st, eb, ee);
    if (K == 8 && V == 64) return launch<8, 64, false>(q, k, v, B, T, H, scale, o, w, p, d, st, eb, ee);
    return launch<8, 128, false>(q, k, v, B, T, H, scale, o, w, p, d, st, eb, ee);
}

// Scratch of based_fwd_noalloc: a fixed array in the library's device image, so that the entry
// point never allocates. Its host-side name is only a handle; the device address is looked up per
// device with cudaGetSymbolAddress.
__device__ __align__(256) unsigned char g_noalloc_scratch[BASED_NOALLOC_SCRATCH_BYTES];

struct NoAllocState {
    std::mutex m;
    void *ptr = nullptr;  // device address of g_noalloc_scratch on this device
};
NoAllocState g_noalloc[kMaxDevices];

// Device address of the scratch array on device `dev` (current), looked up on first use.
int noalloc_scratch(int dev, void **ptr) {
    NoAllocState &s = g_noalloc[dev];
    std::lock_guard<std::mutex> lk(s.m);
    if (s.ptr == nullptr) {
        void *p = nullptr;
        BASED_CUDA(cudaGetSymbolAddress(&p, g_noalloc_scratch));
        s.ptr = p;
    }
    *ptr = s.ptr;
    return BASED_OK;
}

}  // namespace

extern "C" {

int based_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int T, int H, int K,
              int V, float scale, float *o, based_stream_t stream) {
    return run(q, k, v, B, T, H, K, V, scale, o, false, nullptr, 0, true, stream);
}

int based_fwd_timed(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int T, int H,
                    int K, int V, float scale, float *o, based_stream_t stream, void *ev_begin,
                    void *ev_end) {
    return run(q, k, v, B, T, H, K, V, scale, o, false, nullptr, 0, true, stream, ev_begin, ev_end);
}

int based_fwd_noalloc(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int T, int H,
                      int K, int V, float scale, float *o, based_stream_t stream) {
    int rc = check_args(q, k, v, B, T, H, K, V, o);
    if (rc != BASED_OK) return rc;
    int dev;
    if ((rc = current_device(&dev)) != BASED_OK) return rc;
    // the plan that fits the fixed scratch (one slot per range when balanced pieces do not fit)
    const size_t ws_need = make_plan(B, T, H, K, V, g_dev[dev].sms, BASED_NOALLOC_SCRATCH_BYTES).ws_bytes;
    if (ws_need > BASED_NOALLOC_SCRATCH_BYTES) return BASED_ERR_SCRATCH_LIMIT;
    void *scratch = nullptr;
    if (ws_need > 0 && (rc = noalloc_scratch(dev, &scratch)) != BASED_OK) return rc;
    return run(q, k, v, B, T, H, K, V, scale, o, false, scratch, ws_need, false, stream, nullptr,
               nullptr, BASED_NOALLOC_SCRATCH_BYTES);
}

int based_fwd_kernel_count(int B, int T, int H, int K, int V) {
    if ((K != 8 && K != 16) || (V != 64 && V != 128) || B < 1 || T < 1 || H < 1) return 0;
    int dev;
    if (current_device(&dev) != BASED_OK) return 0;
    const Plan &p = make_plan(B, T, H, K, V, g_dev[dev].sms);
    return p.need_agg ? (p.agg.scan ? 3 : 2) : 1;
}

size_t based_fwd_workspace_size(int B, int T, int H, int K, int V) {
    if ((K != 8 && K != 16) || (V != 64 && V != 128) || B < 1 || T < 1 || H < 1) return 0;
    int dev;
    if (current_device(&dev) != BASED_OK) return 0;
    return make_plan(B, T, H, K, V, g_dev[dev].sms).ws_bytes;
}

int based_fwd_ws(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int T, int H,
                 int K, int V, float scale, float *o, void *workspace, size_t ws_bytes,
                 based_stream_t stream) {
    return run(q, k, v, B, T, H, K, V, scale, o, false, workspace, ws_bytes, false, stream);
}

int based_fwd_bf16_out(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int T, int H,
                       int K, int V, float scale, uint16_t *o, void *workspace, size_t ws_bytes,
                       based_stream_t stream, void *ev_begin, void *ev_end) {
    return run(q, k, v, B, T, H, K, V, scale, o, true, workspace, ws_bytes, workspace == nullptr,
               stream, ev_begin, ev_end);
}

int based_fwd_host(const uint16_t *q_host, const uint16_t *k_host, const uint16_t *v_host, int B,
                   int T, int H, int K, int V, float scale, float *o_host, based_stream_t stream) {
    if (!q_host || !k_host || !v_host || !o_host) return BASED_ERR_NULL_POINTER;
    if (K != 8 && K != 16) return BASED_ERR_UNSUPPORTED_K;
    if (V != 64 && V != 128) return BASED_ERR_UNSUPPORTED_V;
    if (B < 1 || T < 1 || H < 1 || static_cast<long long>(B) * T * H >= (1ll << 31))
        return BASED_ERR_BAD_SHAPE;
    int dev, rc;
    if ((rc = current_device(&dev)) != BASED_OK) return rc;
    DeviceState &d = g_dev[dev];
    // The problem is cut into up to 8 pieces of independent heads: ranges of batch entries (each
    // a contiguous block) or, for a single batch entry, ranges of heads (pitched blocks of rows). A three-stage pipeline runs them: one
    // stream copies every piece in, one computes each piece once its copy has landed, one copies
    // each result out once it is computed, so that both copy directions and the kernels overlap.
    constexpr int P = DeviceState::kHostPieces;
    // whole batch entries where there are several (contiguous copies); head ranges otherwise
    const int nb = B < P ? B : P;
    const int nh = B > 1 ? 1 : (H < P ? H : P);
    const size_t rows = static_cast<size_t>(B) * T * H;
    auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    const size_t bq = up(rows * K * 2), bv = up(rows * V * 2), bo = up(rows * V * 4);
    const size_t need = 2 * bq + bv + bo;
    // the most workspace any piece needs (pieces run one after another on the compute stream; a
    // piece has B / nb or B / nb + 1 batch entries and H / nh or H / nh + 1 heads)
    size_t ws_piece = 0;
    for (int pb : {B / nb, (B + nb - 1) / nb})
        for (int hp : {H / nh, (H + nh - 1) / nh})
            if (pb > 0 && hp > 0) {
                const size_t w = up(make_plan(pb, T, hp, K, V, d.sms).ws_bytes);
                ws_piece = w > ws_piece ? w : ws_piece;
            }
    uint8_t *base, *wsb;
    {
        std::lock_guard<std::mutex> lk(d.m);
        if (need > d.hbuf_bytes) {
            if (d.hbuf) {
                cudaError_t e = cudaFree(d.hbuf);
                d.hbuf = nullptr;
                d.hbuf_bytes = 0;
                if (e != cudaSuccess) return cuda_fail(e, "cudaFree(staging)");
            }
            BASED_CUDA(cudaMalloc(&d.hbuf, need));
            d.hbuf_bytes = need;
        }
        if (ws_piece > d.hws_bytes) {
            if (d.hws) {
                cudaError_t e = cudaFree(d.hws);
                d.hws = nullptr;
                d.hws_bytes = 0;
                if (e != cudaSuccess) return cuda_fail(e, "cudaFree(host-path workspace)");
            }
            BASED_CUDA(cudaMalloc(&d.hws, ws_piece));
            d.hws_bytes = ws_piece;
        }
        if (!d.hfork) {
            BASED_CUDA(cudaStreamCreateWithFlags(&d.hs_in, cudaStreamNonBlocking));
            BASED_CUDA(cudaStreamCreateWithFlags(&d.hs_comp, cudaStreamNonBlocking));
            BASED_CUDA(cudaStreamCreateWithFlags(&d.hs_out, cudaStreamNonBlocking));
            BASED_CUDA(cudaEventCreateWithFlags(&d.hdone, cudaEventDisableTiming));
            for (int i = 0; i < P; ++i) {
                BASED_CUDA(cudaEventCreateWithFlags(&d.hin[i], cudaEventDisableTiming));
                BASED_CUDA(cudaEventCreateWithFlags(&d.hcomp[i], cudaEventDisableTiming));
            }
            BASED_CUDA(cudaEventCreateWithFlags(&d.hfork, cudaEventDisableTiming));
        }
        base = static_cast<uint8_t *>(d.hbuf);
        wsb = static_cast<uint8_t *>(d.hws);
    }
    uint16_t *dq = reinterpret_cast<uint16_t *>(base);
    uint16_t *dk = reinterpret_cast<uint16_t *>(base + bq);
    uint16_t *dv = reinterpret_cast<uint16_t *>(base + 2 * bq);
    float *dout = reinterpret_cast<float *>(base + 2 * bq + bv);
    cudaStream_t caller = reinterpret_cast<cudaStream_t>(stream);
    // fork: the pipeline starts after the work already queued on the caller's stream
    BASED_CUDA(cudaEventRecord(d.hfork, caller));
    BASED_CUDA(cudaStreamWaitEvent(d.hs_in, d.hfork, 0));
    BASED_CUDA(cudaStreamWaitEvent(d.hs_comp, d.hfork, 0));
    BASED_CUDA(cudaStreamWaitEvent(d.hs_out, d.hfork, 0));
    size_t off = 0;  // rows of the compact pieces before this one
    for (int i = 0; i < nb * nh; ++i) {
        const int ib = i / nh, ih = i % nh;
        const int b0 = static_cast<int>(static_cast<long long>(B) * ib / nb);
        const int b1 = static_cast<int>(static_cast<long long>(B) * (ib + 1) / nb);
        const int h0 = static_cast<int>(static_cast<long long>(H) * ih / nh);
        const int h1 = static_cast<int>(static_cast<long long>(H) * (ih + 1) / nh);
        const int pb = b1 - b0, hp = h1 - h0;
        const size_t prow = static_cast<size_t>(pb) * T;  // (b, t) rows of the piece
        const size_t src = (static_cast<size_t>(b0) * T * H + h0);  // first element row on the host
        uint16_t *pq = dq + off * K, *pk = dk + off * K, *pv = dv + off * V;
        float *po = dout + off * V;
        off += prow * hp;
        // A piece of whole batch entries is one contiguous block: copy it as such (the 2D path
        // moves short rows, such as 192-byte q rows, far below the link's bandwidth).
        const bool whole = hp == H;
        auto copy_in = [&](uint16_t *dst, const uint16_t *hsrc, int dim) -> cudaError_t {
            const size_t w = static_cast<size_t>(hp) * dim * 2;
            return whole ? cudaMemcpyAsync(dst, hsrc + src * dim, prow * w, cudaMemcpyHostToDevice, d.hs_in)
                         : cudaMemcpy2DAsync(dst, w, hsrc + src * dim, static_cast<size_t>(H) * dim * 2, w, prow,
                                             cudaMemcpyHostToDevice, d.hs_in);
        };
        BASED_CUDA(copy_in(pq, q_host, K));
        BASED_CUDA(copy_in(pk, k_host, K));
        BASED_CUDA(copy_in(pv, v_host, V));
        BASED_CUDA(cudaEventRecord(d.hin[i], d.hs_in));
        BASED_CUDA(cudaStreamWaitEvent(d.hs_comp, d.hin[i], 0));
        rc = run(pq, pk, pv, pb, T, hp, K, V, scale, po, false, wsb, ws_piece, false,
                 reinterpret_cast<based_stream_t>(d.hs_comp));
        if (rc != BASED_OK) return rc;
        BASED_CUDA(cudaEventRecord(d.hcomp[i], d.hs_comp));
        BASED_CUDA(cudaStreamWaitEvent(d.hs_out, d.hcomp[i], 0));
        if (whole)
            BASED_CUDA(cudaMemcpyAsync(o_host + src * V, po, prow * hp * V * 4, cudaMemcpyDeviceToHost, d.hs_out));
        else
            BASED_CUDA(cudaMemcpy2DAsync(o_host + src * V, static_cast<size_t>(H) * V * 4, po,
                                         static_cast<size_t>(hp) * V * 4, static_cast<size_t>(hp) * V * 4, prow,
                                         cudaMemcpyDeviceToHost, d.hs_out));
    }
    // join: the caller's stream continues after the last copy out, then the call waits for it
    BASED_CUDA(cudaEventRecord(d.hdone, d.hs_out));
    BASED_CUDA(cudaStreamWaitEvent(caller, d.hdone, 0));
    BASED_CUDA(cudaStreamSynchronize(caller));
    // The call has synchronised: report (and clear) a bounded wait that gave up since the status
    // word was last cleared, so that a timed-out kernel never passes for a result.
    unsigned int st = 0;
    if ((rc = based_device_status(dev, &st, 1)) != BASED_OK) return rc;
    return st != 0 ? BASED_ERR_DEVICE_TIMEOUT : BASED_OK;
}

int based_device_status(int device, unsigned int *status, int clear) {
    if (!status) return BASED_ERR_NULL_POINTER;
    int prev;
    BASED_CUDA(cudaGetDevice(&prev));
    if (device != prev) BASED_CUDA(cudaSetDevice(device));
    cudaError_t e = cudaMemcpyFromSymbol(status, based::g_status, sizeof(unsigned int));
    if (e == cudaSuccess && clear) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(based::g_status, &zero, sizeof(unsigned int));
    }
    if (device != prev) cudaSetDevice(prev);
    if (e != cudaSuccess) return cuda_fail(e, "status word");
    return BASED_OK;
}

int based_selftest_wait_timeout(unsigned long long limit_ns) {
    if (limit_ns < 1000ull) limit_ns = 1000ull;
    if (limit_ns > 2000000000ull) limit_ns = 2000000000ull;
    int dev;
    BASED_CUDA(cudaGetDevice(&dev));
    unsigned int before;
    int rc = based_device_status(dev, &before, 1);
    if (rc != BASED_OK) return rc;
    int *res = nullptr;
    BASED_CUDA(cudaMalloc(&res, sizeof(int)));
    based::based_selftest_wait_kernel<<<1, 1>>>(limit_ns, res);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    int h = -1;
    if (e == cudaSuccess) e = cudaMemcpy(&h, res, sizeof(int), cudaMemcpyDeviceToHost);
    cudaFree(res);
    if (e != cudaSuccess) return cuda_fail(e, "selftest kernel");
    unsigned int st;
    rc = based_device_status(dev, &st, 0);  // left set: other entry points must report it
    if (rc != BASED_OK) return rc;
    // the wait must have given up (result 0) and recorded site 255
    if (h != 0 || (st & 1u) == 0u || ((st >> 8) & 0xFFu) != 255u) return BASED_ERR_BAD_ARGUMENT;
    return BASED_OK;
}

const char *based_fwd_strerror(int code) {
    switch (code) {
        case BASED_OK: return "ok";
        case BASED_ERR_NULL_POINTER: return "null pointer";
        case BASED_ERR_UNSUPPORTED_K: return "unsupported K (must be 8 or 16)";
        case BASED_ERR_UNSUPPORTED_V: return "unsupported V (must be 64 or 128)";
        case BASED_ERR_BAD_SHAPE: return "bad shape (B, T, H >= 1 and B*T*H < 2^31)";
        case BASED_ERR_MISALIGNED: return "device pointer not 16-byte aligned";
        case BASED_ERR_ALIASING: return "output overlaps an input";
        case BASED_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case BASED_ERR_CUDA: return "CUDA error";
        case BASED_ERR_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait";
        case BASED_ERR_NO_DEVICE: return "current device is not an sm_103 GPU";
        case BASED_ERR_BAD_ARGUMENT: return "invalid argument";
        case BASED_ERR_SCRATCH_LIMIT:
            return "shape needs more scratch than the fixed BASED_NOALLOC_SCRATCH_BYTES array";
        default: return "unknown error code";
    }
}

const char *based_strerror(int code) { return based_fwd_strerror(code); }

const char *based_last_cuda_error(void) { return tl_cuda_error; }

int based_abi_version(void) { return 10100; }

#ifdef BASED_TRACE
// Trace builds only: device buffer of (CTAs x 64 x 32) uint64 stage timestamps, or NULL to stop.
__attribute__((visibility("default"))) int based_trace_set(void *buf) {
    cudaError_t e = cudaMemcpyToSymbol(based::g_trace, &buf, sizeof(void *));
    return e == cudaSuccess ? 0 : cuda_fail(e, "trace buffer");
}
#endif

}  // extern "C"
