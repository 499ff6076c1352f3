/*
 * Based causal forward pass: plain CPU oracle in fp64.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may call, link or load this file;
 * it exists so that tests, the smoke check and the CPU-baseline leg of the benchmark can check
 * the CUDA kernels against an independent, slow and obviously correct computation. It shares
 * no code, header, table or constant with the CUDA library.
 *
 * Source: the "based_forward.py" kernel-task spec (tools/factory/specs/based_forward.py).
 * Everything below restates, in loops, what that spec defines:
 *
 *   spec_md, first block: with s[i,j] = scale * (q_i . k_j),
 *       A[i,j] = 1 + s[i,j] + s[i,j]^2 / 2   for j <= i, 0 otherwise
 *       o_i    = (sum_j A[i,j] v_j) / (sum_j A[i,j] + 1e-6)
 *   spec_md, "Why this is not an O(T^2) op": phi(x) = [1, x, x(x)x / sqrt(2)], length
 *       P = 1 + K + K*K, and phi(q).phi(k) = 1 + q.k + (q.k)^2 / 2, so
 *       o_i = phi(q_i)^T S_i / (phi(q_i)^T z_i + 1e-6), S_i = sum_{j<=i} phi(k_j) v_j^T,
 *       z_i = sum_{j<=i} phi(k_j).
 *   contract_md: scale multiplies q only, before the dot product; the 1e-6 guard is added
 *       after the full row sum; attention is causal and includes the diagonal.
 *   reference_src: the chunked evaluation order (direct polynomial inside a chunk, feature-map
 *       state across chunks, state updated after the chunk's outputs are formed).
 *
 * Two independent evaluations are provided:
 *   based_oracle_direct_rows  the O(T^2) double sum of the definition, for chosen (head,row)
 *                             pairs (brute force; used on tiny inputs and on sampled rows);
 *   based_oracle_chunked      the feature-map form over chunks of any length C >= 1, for
 *                             chosen heads (the timed CPU baseline).
 * Inputs are fp64 arrays (callers convert the exact bf16 values). Layouts follow the spec's
 * contract: q,k (B,T,H,K) and v (B,T,H,V), row-major and contiguous. Outputs are fp64.
 *
 * Readings where the spec is silent (spec_md and contract_md fix none of these):
 *   - the scale is used as given (the caller passes the fp32 value the kernel receives);
 *   - T need not be a multiple of 64 or of the chunk length: the last chunk is short;
 *   - the output is returned in fp64 and compared against the kernel's fp32 output.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* Length of phi(x) for a K-dimensional x: 1 + K + K*K ("Why this is not an O(T^2) op"). */
int based_oracle_feature_len(int K) { return 1 + K + K * K; }

/* phi(x) = [1, x, vec(x (x) x) / sqrt(2)], the outer product flattened row-major (index a*K+b),
 * exactly as the spec's feature map builds it. */
void based_oracle_phi(const double *x, int K, double *out) {
    const double inv_sqrt2 = 1.0 / sqrt(2.0);
    out[0] = 1.0;
    for (int a = 0; a < K; ++a) out[1 + a] = x[a];
    for (int a = 0; a < K; ++a)
        for (int b = 0; b < K; ++b) out[1 + K + a * K + b] = x[a] * x[b] * inv_sqrt2;
}

/* ---------------------------------------------------------------------------------------------
 * Small thread pool helper: run fn(i, ctx) for i in [0, n) on nthreads threads.
 * ------------------------------------------------------------------------------------------- */
typedef void (*work_fn)(int64_t i, void *ctx);
typedef struct {
    work_fn fn;
    void *ctx;
    int64_t n;
    int64_t next;
    pthread_mutex_t lock;
} pool_t;

static void *pool_worker(void *arg) {
    pool_t *p = (pool_t *)arg;
    for (;;) {
        pthread_mutex_lock(&p->lock);
        int64_t i = p->next++;
        pthread_mutex_unlock(&p->lock);
        if (i >= p->n) break;
        p->fn(i, p->ctx);
    }
    return NULL;
}

static int resolve_threads(int nthreads) {
    if (nthreads > 0) return nthreads;
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static void run_pool(work_fn fn, void *ctx, int64_t n, int nthreads) {
    pool_t p;
    p.fn = fn;
    p.ctx = ctx;
    p.n = n;
    p.next = 0;
    pthread_mutex_init(&p.lock, NULL);
    int nt = resolve_threads(nthreads);
    if (nt > n) nt = (int)(n > 0 ? n : 1);
    if (nt <= 1) {
        pool_worker(&p);
    } else {
        pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
        for (int t = 0; t < nt; ++t) pthread_create(&th[t], NULL, pool_worker, &p);
        for (int t = 0; t < nt; ++t) pthread_join(th[t], NULL);
        free(th);
    }
    pthread_mutex_destroy(&p.lock);
}

/* Element (b,t,h,c) of a (B,T,H,D) contiguous tensor, with head index bh = b*H + h. */
static inline const double *row_ptr(const double *x, int bh, int t, int T, int H, int D) {
    int b = bh / H, h = bh % H;
    return x + (((int64_t)b * T + t) * H + h) * (int64_t)D;
}

/* ---------------------------------------------------------------------------------------------
 * Direct form (spec_md, first block), evaluated at chosen (head, row) pairs.
 * ------------------------------------------------------------------------------------------- */
typedef struct {
    const double *q, *k, *v;
    int T, H, K, V;
    double scale;
    const int64_t *pairs; /* n pairs of (bh, i) */
    double *o_rows;       /* (n, V) */
    double *den_rows;     /* (n) or NULL */
} direct_ctx;

static void direct_one(int64_t r, void *vctx) {
    direct_ctx *c = (direct_ctx *)vctx;
    const int bh = (int)c->pairs[2 * r];
    const int i = (int)c->pairs[2 * r + 1];
    double *num = c->o_rows + r * (int64_t)c->V;
    for (int e = 0; e < c->V; ++e) num[e] = 0.0;
    double den = 0.0;
    const double *qi = row_ptr(c->q, bh, i, c->T, c->H, c->K);
    for (int j = 0; j <= i; ++j) { /* causal, diagonal included */
        const double *kj = row_ptr(c->k, bh, j, c->T, c->H, c->K);
        const double *vj = row_ptr(c->v, bh, j, c->T, c->H, c->V);
        double dot = 0.0;
        for (int a = 0; a < c->K; ++a) dot += (c->scale * qi[a]) * kj[a]; /* scale on q only */
        const double s = dot;
        const double A = 1.0 + s + s * s / 2.0;
        for (int e = 0; e < c->V; ++e) num[e] += A * vj[e];
        den += A;
    }
    for (int e = 0; e < c->V; ++e) num[e] = num[e] / (den + 1e-6);
    if (c->den_rows) c->den_rows[r] = den;
}

/* Returns 0 on success, -1 on bad arguments. */
int based_oracle_direct_rows(const double *q, const double *k, const double *v, int B, int T, int H,
                             int K, int V, double scale, const int64_t *pairs, int64_t n_pairs,
                             double *o_rows, double *den_rows, int nthreads) {
    if (!q || !k || !v || !pairs || !o_rows || B < 1 || T < 1 || H < 1 || K < 1 || V < 1) return -1;
    for (int64_t r = 0; r < n_pairs; ++r) {
        if (pairs[2 * r] < 0 || pairs[2 * r] >= (int64_t)B * H) return -1;
        if (pairs[2 * r + 1] < 0 || pairs[2 * r + 1] >= T) return -1;
    }
    direct_ctx c = {q, k, v, T, H, K, V, scale, pairs, o_rows, den_rows};
    run_pool(direct_one, &c, n_pairs, nthreads);
    return 0;
}

/* ---------------------------------------------------------------------------------------------
 * Chunked feature-map form (reference_src loop + the identity of "Why this is not an O(T^2) op").
 * For each chosen head, S (P x V) and z (P) start at zero; for each chunk of C rows:
 *   num_r = phi(q_r) S + sum_{j in chunk, j <= r} A[r,j] v_j
 *   den_r = phi(q_r) . z + sum_{j in chunk, j <= r} A[r,j]
 *   o_r   = num_r / (den_r + 1e-6)
 * and only then S += sum_j phi(k_j) v_j^T, z += sum_j phi(k_j) over the chunk's rows.
 * ------------------------------------------------------------------------------------------- */
typedef struct {
    const double *q, *k, *v;
    int T, H, K, V, C;
    double scale;
    const int64_t *heads; /* n chosen bh indices */
    double *o;            /* (n, T, V) */
    double *den;          /* (n, T) or NULL */
} chunk_ctx;

static void chunked_one(int64_t hidx, void *vctx) {
    chunk_ctx *c = (chunk_ctx *)vctx;
    const int bh = (int)c->heads[hidx];
    const int K = c->K, V = c->V, T = c->T, C = c->C;
    const int P = based_oracle_feature_len(K);
    double *S = (double *)calloc((size_t)P * V, sizeof(double));
    double *z = (double *)calloc((size_t)P, sizeof(double));
    double *pq = (double *)malloc(sizeof(double) * (size_t)P);
    double *pk = (double *)malloc(sizeof(double) * (size_t)P);
    double *qs = (double *)malloc(sizeof(double) * (size_t)K);
    double *num = (double *)malloc(sizeof(double) * (size_t)V);
    double *o = c->o + hidx * (int64_t)T * V;

    for (int i0 = 0; i0 < T; i0 += C) {
        const int n = (T - i0 < C) ? (T - i0) : C;
        /* outputs of this chunk, from the state of all earlier chunks plus the direct term */
        for (int r = 0; r < n; ++r) {
            const double *qr = row_ptr(c->q, bh, i0 + r, T, c->H, K);
            for (int a = 0; a < K; ++a) qs[a] = c->scale * qr[a]; /* q <- scale * q */
            based_oracle_phi(qs, K, pq);
            double den = 0.0;
            for (int e = 0; e < V; ++e) num[e] = 0.0;
            for (int p = 0; p < P; ++p) { /* inter-chunk: phi(q) S and phi(q) . z */
                for (int e = 0; e < V; ++e) num[e] += pq[p] * S[(int64_t)p * V + e];
                den += pq[p] * z[p];
            }
            for (int j = 0; j <= r; ++j) { /* intra-chunk: causal polynomial weights */
                const double *kj = row_ptr(c->k, bh, i0 + j, T, c->H, K);
                const double *vj = row_ptr(c->v, bh, i0 + j, T, c->H, V);
                double s = 0.0;
                for (int a = 0; a < K; ++a) s += qs[a] * kj[a];
                const double A = 1.0 + s + 0.5 * s * s;
                for (int e = 0; e < V; ++e) num[e] += A * vj[e];
                den += A;
            }
            double *orow = o + (int64_t)(i0 + r) * V;
            for (int e = 0; e < V; ++e) orow[e] = num[e] / (den + 1e-6);
            if (c->den) c->den[hidx * (int64_t)T + i0 + r] = den;
        }
        /* fold the chunk into the state */
        for (int j = 0; j < n; ++j) {
            const double *kj = row_ptr(c->k, bh, i0 + j, T, c->H, K);
            const double *vj = row_ptr(c->v, bh, i0 + j, T, c->H, V);
            based_oracle_phi(kj, K, pk);
            for (int p = 0; p < P; ++p) {
                for (int e = 0; e < V; ++e) S[(int64_t)p * V + e] += pk[p] * vj[e];
                z[p] += pk[p];
            }
        }
    }
    free(S);
    free(z);
    free(pq);
    free(pk);
    free(qs);
    free(num);
}

/* heads == NULL means every head 0..B*H-1 in order. Returns 0 on success, -1 on bad arguments. */
int based_oracle_chunked(const double *q, const double *k, const double *v, int B, int T, int H,
                         int K, int V, double scale, int chunk, const int64_t *heads,
                         int64_t n_heads, double *o, double *den, int nthreads) {
    if (!q || !k || !v || !o || B < 1 || T < 1 || H < 1 || K < 1 || V < 1 || chunk < 1) return -1;
    int64_t *all = NULL;
    if (!heads) {
        n_heads = (int64_t)B * H;
        all = (int64_t *)malloc(sizeof(int64_t) * (size_t)n_heads);
        for (int64_t i = 0; i < n_heads; ++i) all[i] = i;
        heads = all;
    }
    for (int64_t i = 0; i < n_heads; ++i)
        if (heads[i] < 0 || heads[i] >= (int64_t)B * H) {
            free(all);
            return -1;
        }
    chunk_ctx c = {q, k, v, T, H, K, V, chunk, scale, heads, o, den};
    run_pool(chunked_one, &c, n_heads, nthreads);
    free(all);
    return 0;
}

/* Number of worker threads a call with nthreads <= 0 would use. */
int based_oracle_default_threads(void) { return resolve_threads(0); }
