/*
 * based.h: C ABI of the GB300 (sm_103a) Based causal forward pass.
 *
 * Based is causal linear attention whose kernel is the 2nd-order Taylor polynomial of exp:
 * with s[i,j] = scale * (q_i . k_j),
 *     A[i,j] = 1 + s[i,j] + s[i,j]^2 / 2        for j <= i (0 otherwise)
 *     o_i    = (sum_j A[i,j] v_j) / (sum_j A[i,j] + 1e-6)
 * Source: the "based_forward.py" kernel-task spec (tools/factory/specs/based_forward.py),
 * spec_md (definition and the feature-map identity phi(q).phi(k) = 1 + q.k + (q.k)^2/2 with
 * phi(x) = [1, x, x(x)x/sqrt(2)]) and contract_md (argument shapes, scale semantics, causality).
 *
 * Conventions shared by every entry point:
 *   - Layouts are row-major and contiguous: q, k are (B, T, H, K); v and o are (B, T, H, V).
 *     q, k, v hold bfloat16 values given as their 16-bit patterns; o receives float32.
 *   - Supported sizes: K in {8, 16}; V in {64, 128}; B, H >= 1; 1 <= T; B*T*H < 2^31.
 *     T need not be a multiple of anything.
 *   - scale multiplies q only, before the dot product. A scale that is <= 0 or NaN selects the
 *     default K^-0.5 (the C stand-in for the spec's scale=None).
 *   - Inputs are read-only. o must not overlap q, k or v.
 *   - Device pointers must be 16-byte aligned (the kernels move tiles with TMA).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy default stream)
 *     unless stated otherwise, and never synchronise the device implicitly, except that the
 *     first call on a device (or a call that needs a larger workspace than any before it)
 *     allocates the library-owned workspace with cudaMalloc.
 *   - Return value: 0 on success or a negative BASED_ERR_* code. Argument errors are detected
 *     on the host before anything is launched. based_fwd_strerror() names every code.
 *
 * Ownership: the caller owns q, k, v, o. The library owns one workspace per device, which holds
 * per-segment partial states (fp32) for the chunk-parallel state scan; it lives until process
 * exit. Shapes whose work plan gives the CTAs lead-ins instead (V = 64, where the plan finds that
 * faster: each CTA that starts inside a head sums that head's earlier chunks itself) use no
 * workspace (based_fwd_workspace_size() returns 0). The library allocates no device memory per call, with one exception: based_fwd (and
 * based_fwd_timed, and based_fwd_bf16_out with a NULL workspace) grow the library-owned
 * workspace with cudaMalloc when a shape needs more than any call before it. A workspace that a
 * larger one replaces is never freed, so that a CUDA graph which captured an earlier call still
 * replays into valid memory. Callers that must not allocate at all use based_fwd_ws (caller-owned
 * workspace) or based_fwd_noalloc (fixed scratch). Concurrent calls that use the library-owned
 * workspace on the same device must be ordered by the caller (same stream, or events);
 * based_fwd_ws() takes a caller-owned workspace instead and has no such restriction.
 */
#ifndef BASED_GB300_H
#define BASED_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define BASED_API __attribute__((visibility("default")))
#else
#define BASED_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream handle, ABI-compatible with cudaStream_t / CUstream. */
typedef struct CUstream_st *based_stream_t;

enum {
    BASED_OK = 0,
    BASED_ERR_NULL_POINTER = -1,   /* q, k, v or o is NULL */
    BASED_ERR_UNSUPPORTED_K = -2,  /* K not in {8, 16} */
    BASED_ERR_UNSUPPORTED_V = -3,  /* V not in {64, 128} */
    BASED_ERR_BAD_SHAPE = -4,      /* B, T or H < 1, or B*T*H too large */
    BASED_ERR_MISALIGNED = -5,     /* a device pointer is not 16-byte aligned */
    BASED_ERR_ALIASING = -6,       /* o overlaps q, k or v */
    BASED_ERR_WORKSPACE = -7,      /* workspace NULL or smaller than based_fwd_workspace_size() */
    BASED_ERR_CUDA = -8,           /* a CUDA runtime/driver call failed (see based_last_cuda_error) */
    BASED_ERR_DEVICE_TIMEOUT = -9, /* a kernel gave up a bounded wait (based_device_status) */
    BASED_ERR_NO_DEVICE = -10,     /* no sm_103 device is current */
    BASED_ERR_BAD_ARGUMENT = -11,  /* any other invalid argument */
    BASED_ERR_SCRATCH_LIMIT = -12  /* shape needs more than BASED_NOALLOC_SCRATCH_BYTES of scratch */
};

/*
 * based_fwd: the causal Based forward pass on device buffers.
 *   q, k   device, bf16 bit patterns, (B,T,H,K) contiguous        (read only)
 *   v      device, bf16 bit patterns, (B,T,H,V) contiguous        (read only)
 *   scale  query scale; <= 0 or NaN selects K^-0.5
 *   o      device, float32, (B,T,H,V) contiguous                   (written)
 *   stream CUDA stream the kernels are launched on
 * Computes o_i = phi(q_i)^T S_i / (phi(q_i)^T z_i + 1e-6) with S_i = sum_{j<=i} phi(k_j) v_j^T
 * and z_i = sum_{j<=i} phi(k_j) (spec_md, "Why this is not an O(T^2) op"), using the
 * library-owned workspace.
 */
BASED_API int based_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int T, int H, int K,
              int V, float scale, float *o, based_stream_t stream);

/* Bytes of workspace based_fwd_ws() needs for this shape on the current device (0 if none). */
BASED_API size_t based_fwd_workspace_size(int B, int T, int H, int K, int V);

/* based_fwd with a caller-owned device workspace of ws_bytes bytes (16-byte aligned). The
 * workspace is scratch: its contents on entry are ignored and on return are unspecified. Calls
 * that share one workspace must not overlap on the GPU. */
BASED_API int based_fwd_ws(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int T, int H,
                 int K, int V, float scale, float *o, void *workspace, size_t ws_bytes,
                 based_stream_t stream);

/*
 * based_fwd_bf16_out: based_fwd with a bfloat16 output, which halves the largest data stream of
 * the call (the kernel-task spec's output contract allows "bf16 or fp32"; fp32 is the default).
 *   q, k, v, B, T, H, K, V, scale, stream: as for based_fwd.
 *   o          device, bf16 bit patterns, (B,T,H,V) contiguous, 16-byte aligned (written). Each
 *              element is the fp32 result based_fwd computes, rounded to nearest even.
 *   workspace  NULL: the library-owned workspace (as based_fwd); otherwise a caller-owned device
 *              workspace of ws_bytes bytes (as based_fwd_ws).
 *   ev_begin, ev_end  NULL, or caller-created CUDA events recorded around the forward kernel
 *              (as based_fwd_timed).
 * Errors: as based_fwd and based_fwd_ws; o must not overlap q, k or v.
 */
BASED_API int based_fwd_bf16_out(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int T,
                                 int H, int K, int V, float scale, uint16_t *o, void *workspace,
                                 size_t ws_bytes, based_stream_t stream, void *ev_begin, void *ev_end);

/*
 * based_fwd_noalloc: based_fwd for callers that may not allocate device memory while they run,
 * e.g. a serving loop whose device memory is planned up front by its own allocator, or code
 * that cannot afford the device-wide synchronisation cudaMalloc/cudaFree can cause. The paper
 * and the kernel-task spec have no counterpart to this entry point: it only changes where the
 * scratch lives.
 *   Arguments, layouts, scale and the result are those of based_fwd. Scratch (the per-segment
 *   partial states) lives in one fixed array of BASED_NOALLOC_SCRATCH_BYTES bytes that is part of
 *   the library's device image: every GPU that loads the library holds it until process exit.
 *   The call itself runs no cudaMalloc, cudaFree or other allocating routine.
 *   - The work plan is limited to what fits the array: where based_fwd would cut the aggregate
 *     pass into more pieces (one partial-state slot each) than fit, this entry point keeps one
 *     slot per range (82,560 bytes per SM for K = 16, V = 128, so 16 MiB covers up to 203 SMs).
 *     Shapes whose scratch would still exceed the array are rejected with
 *     BASED_ERR_SCRATCH_LIMIT before anything is launched.
 *   - The first call on a device looks up the array's device address (and loads the library's
 *     device code there if that has not happened yet); make that first call before any stream
 *     capture.
 *   - Every call on a device shares the one array, which keeps the last call's contents. No
 *     scratch element has to start at zero: each call writes every element it reads before
 *     reading it. Calls that overlap on the GPU (other streams, other threads) race on the array
 *     and give wrong results: order them (same stream, or events).
 */
#define BASED_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
BASED_API int based_fwd_noalloc(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int T,
                                int H, int K, int V, float scale, float *o, based_stream_t stream);

/*
 * based_fwd_host: the same computation on HOST buffers, end to end. The problem is cut into up to
 * eight pieces of independent heads (ranges of batch entries, or of heads when B = 1) that run through
 * a three-stage pipeline on library-owned streams: copy in (pitched cudaMemcpy2DAsync), compute,
 * copy out, so that both copy directions and the kernels overlap. The pipeline starts after the
 * work already queued on `stream`, which then continues after it; the call synchronises `stream`
 * before returning. Page-locked host memory makes the copies asynchronous DMA; pageable memory
 * also works, more slowly. The device buffers, streams, events and workspace are cached per
 * device and grown on demand (cudaMalloc), so this call is not reentrant for one device.
 * After its final synchronisation the call reads and clears the device status word
 * (based_device_status): if any kernel of this library gave up a bounded wait since the word was
 * last cleared, it returns BASED_ERR_DEVICE_TIMEOUT, and o_host must not be used.
 */
BASED_API int based_fwd_host(const uint16_t *q_host, const uint16_t *k_host, const uint16_t *v_host, int B,
                   int T, int H, int K, int V, float scale, float *o_host, based_stream_t stream);

/* based_fwd that also records two caller-created CUDA events (cudaEvent_t, may be NULL) on
 * `stream`: ev_begin right before the forward kernel and ev_end right after it, so that the
 * caller can time that kernel alone (the aggregate and scan kernels, when launched, come before
 * ev_begin). Same arguments, semantics and workspace as based_fwd otherwise. */
BASED_API int based_fwd_timed(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int T,
                              int H, int K, int V, float scale, float *o, based_stream_t stream,
                              void *ev_begin, void *ev_end);

/* Number of kernels one based_fwd call launches for this shape on the current device: 1 (the
 * forward kernel alone: no CTA needs the state of chunks before its range, or the CTAs run
 * lead-ins), 2 (aggregate, forward: every prefix is the sum of at most four partial
 * states, which the forward kernel adds itself) or 3 (aggregate, scan, forward: some prefix has
 * more); 0 for an unsupported shape. */
BASED_API int based_fwd_kernel_count(int B, int T, int H, int K, int V);

/* Reads (and, if clear != 0, resets) the device status word of `device`: 0 means no kernel of
 * this library gave up a bounded wait since the last reset; otherwise bit 0 is set and bits
 * 8..15 name the first wait site that timed out. Synchronous. Returns 0 or BASED_ERR_CUDA. */
BASED_API int based_device_status(int device, unsigned int *status, int clear);

/* Launches a one-thread kernel that waits on a barrier nothing ever signals, with the given
 * limit in nanoseconds (clamped to [1e3, 2e9]), and returns after it gave up. The status word is
 * cleared before the launch and left reporting a timeout at site 255 afterwards, so that a caller
 * can check how other entry points report it; clear it with based_device_status(dev, &s, 1).
 * Exercises the bounded-wait path without hanging the GPU. Synchronous. Returns 0 if the wait
 * timed out as expected, else an error code. */
BASED_API int based_selftest_wait_timeout(unsigned long long limit_ns);

/* Human-readable name of a return code (a static string; never NULL). */
BASED_API const char *based_fwd_strerror(int code);

/* The same as based_fwd_strerror (the name earlier versions of this library exported). */
BASED_API const char *based_strerror(int code);

/* The last CUDA error string seen by the library on this thread ("" if none). */
BASED_API const char *based_last_cuda_error(void);

/* Version of this ABI (major * 10000 + minor * 100 + patch). */
BASED_API int based_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BASED_GB300_H */
