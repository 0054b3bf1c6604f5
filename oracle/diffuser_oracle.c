/*
 * diffuser_oracle.c -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.
 *
 * A plain, slow, fp64 CPU statement of what the Diffuser hot path computes:
 * the fixed sparse edge set (local window, global tokens, random edges, or the
 * BigBird block pattern), the row softmax over each row's allowed set, and K
 * personalized-PageRank (PPR) diffusion hops over those weights; and the
 * gradient of that forward with respect to Q, K and V (the backward pass).
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this library.  It shares no code, header, table or helper with the
 * CUDA library; the two meet only in the seeded input buffers.
 *
 * Sources (page title, section / equation):
 *   [D]  "Diffuser: modelling long sequences with multi-hop attention
 *        diffusion" (reading notes on arXiv 2210.11794v2):
 *        sec 2.1 eq S.1-S.5 (masked softmax weights), sec 2.2 (three edge
 *        kinds), sec 2.4 eq S.7 (PPR recursion), sec 2.5 (finite-K form),
 *        sec 2.6 (training through the unrolled recursion; causal use: A
 *        lower-triangular).
 *   [S]  "1.2.1 Static sparsity: Longformer, BigBird and sliding windows":
 *        sec 1 eq 1-4 (scores, mask, softmax, output), sec 1.1 eq 5-6
 *        (window; causal window of r+1 history positions), sec 1.2 eq 12
 *        (symmetric global tokens), sec 2 eq 13 and
 *        the 12-block example (BigBird block pattern), sec 2.1 (duplicate
 *        edges must not enter the denominator twice).
 *   [B]  "038 BigBird: keeping long-sequence information paths with sparse
 *        connections", sec 2 (S_i = W_i u R_i u G; global rows read all).
 *
 * Readings where the pages leave a step open (all restated in the design
 * notes):
 *   - Random target of row i, draw t (0 <= t < R):
 *       j = splitmix64(seed XOR (i*R + t)) mod n   (unsigned 64-bit).
 *     splitmix64 is the published SplitMix64 output function (Steele, Lea and
 *     Flood 2014) applied to one state value.  Draws are directed i -> j, not
 *     resampled: a duplicate is simply dropped by the set union.
 *   - Window: |i - j| <= r truncated at both ends, never refilled ([S] eq 5).
 *   - Globals: symmetric ([S] eq 12): a global row reads every position and
 *     every row reads every global; global rows take no random draws.
 *   - Block pattern: N = ceil(n / b) blocks; window blocks are the centred
 *     odd-sized run around J, truncated at the ends; random block t of block
 *     row J is splitmix64(seed XOR (J*s + t)) mod N; global blocks are
 *     0..gb-1, which read every block and are read by every block; a token
 *     pair is an edge iff its block pair is allowed; the last block may be
 *     ragged ([S] sec 2, eq 13).
 *   - Scale 1/sqrt(d) with d the head width ([S] eq 1, [D] eq S.1).
 *   - Causal graph: the token graph with the mask j <= i applied to all
 *     three edge kinds ([D] sec 2.6; [S] sec 1.1 for the causal window):
 *     window [i-r, i], globals g <= i, a global row reads 0..i, and a random
 *     draw that lands after i is dropped, not redrawn.
 *   - Uniform-spaced extras ("w uni." of [D] sec 4.5, Tab S.7: the random
 *     edges' positions are taken at uniform spacing instead of at random;
 *     the spacing rule is not given): the R positions of row i are the
 *     uniform grid of spacing n/R on the ring of positions, offset by half a
 *     spacing from i:  j_t = (i + floor((2t + 1) n / (2R))) mod n,  t < R.
 *
 * Everything is computed in double precision, in the plainest loop order.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG (-1)
#define ORACLE_NO_MEM (-2)
#define ORACLE_CAPACITY (-3)

/* SplitMix64 output function on one 64-bit state value (published
 * definition; golden-ratio increment, then two xor-shift-multiply rounds). */
uint64_t oracle_splitmix64(uint64_t x) {
    uint64_t z = x + 0x9E3779B97F4A7C15ULL;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Emit the marked columns of one row in ascending order.  `col` may be NULL
 * (counting pass).  Returns the number of marked columns. */
static int64_t emit_row(const unsigned char* mark, int64_t n, int32_t* col,
                        int64_t at, int64_t capacity, int* overflow) {
    int64_t count = 0;
    for (int64_t j = 0; j < n; ++j) {
        if (!mark[j]) continue;
        if (col) {
            if (at + count >= capacity) { *overflow = 1; return count; }
            col[at + count] = (int32_t)j;
        }
        ++count;
    }
    return count;
}

/*
 * Token-level graph ([D] sec 2.2; [S] eq 5, eq 12; [B] sec 2); `dilation`
 * spaces the window's positions ([S] eq 11), 1 for the plain window.
 *   N(i) = {0..n-1}                                   if i in G
 *   N(i) = {j : |i-j| <= r} u G u {random draws}      otherwise
 * The set is held as a 0/1 mark per column, so duplicates collapse and the
 * ascending scan sorts it.  Pass row_ptr/col = NULL to count only.
 * `globals` NULL means G = {0..n_globals-1}; otherwise it must be strictly
 * increasing inside [0, n).
 */
static int token_graph(int64_t n, int32_t r, int32_t dilation, int32_t n_globals,
                       const int32_t* globals, int32_t rand_per_row,
                       uint64_t seed, int causal, int uniform, int64_t* row_ptr, int32_t* col,
                       int64_t col_capacity, int64_t* nnz_out) {
    if (n < 1 || n > INT32_MAX || r < 0 || dilation < 1 || n_globals < 0 || n_globals > n ||
        rand_per_row < 0 || !nnz_out)
        return ORACLE_BAD_ARG;
    unsigned char* is_global = (unsigned char*)calloc((size_t)n, 1);
    unsigned char* mark = (unsigned char*)malloc((size_t)n);
    if (!is_global || !mark) { free(is_global); free(mark); return ORACLE_NO_MEM; }
    for (int32_t t = 0; t < n_globals; ++t) {
        int64_t gpos = globals ? globals[t] : t;
        if (gpos < 0 || gpos >= n || (globals && t > 0 && globals[t] <= globals[t - 1])) {
            free(is_global); free(mark); return ORACLE_BAD_ARG;
        }
        is_global[gpos] = 1;
    }
    int overflow = 0;
    int64_t nnz = 0;
    if (row_ptr) row_ptr[0] = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (is_global[i]) {
            memset(mark, 1, (size_t)n);                 /* a global row reads all */
        } else {
            memset(mark, 0, (size_t)n);
            for (int64_t j = 0; j < n; ++j)              /* window, eq 5 (eq 11 when dilated) */
                if (llabs(i - j) <= (int64_t)r * dilation && llabs(i - j) % dilation == 0)
                    mark[j] = 1;
            for (int64_t j = 0; j < n; ++j)              /* every row reads G, eq 12 */
                if (is_global[j]) mark[j] = 1;
            for (int32_t t = 0; t < rand_per_row; ++t) { /* random draws */
                uint64_t j;
                if (uniform) {                           /* "w uni.": uniform grid from i */
                    int64_t off = ((int64_t)(2 * t + 1) * n) / (2 * (int64_t)rand_per_row);
                    j = (uint64_t)((i + off) % n);
                } else {
                    uint64_t key = (uint64_t)i * (uint64_t)rand_per_row + (uint64_t)t;
                    j = oracle_splitmix64(seed ^ key) % (uint64_t)n;
                }
                mark[j] = 1;
            }
        }
        if (causal)                                      /* causal mask, [D] sec 2.6 */
            for (int64_t j = i + 1; j < n; ++j) mark[j] = 0;
        nnz += emit_row(mark, n, col, nnz, col_capacity, &overflow);
        if (overflow) { free(is_global); free(mark); return ORACLE_CAPACITY; }
        if (row_ptr) row_ptr[i + 1] = nnz;
    }
    *nnz_out = nnz;
    free(is_global);
    free(mark);
    return ORACLE_OK;
}

int oracle_token_graph(int64_t n, int32_t r, int32_t n_globals,
                       const int32_t* globals, int32_t rand_per_row,
                       uint64_t seed, int64_t* row_ptr, int32_t* col,
                       int64_t col_capacity, int64_t* nnz_out) {
    return token_graph(n, r, 1, n_globals, globals, rand_per_row, seed, 0, 0, row_ptr,
                       col, col_capacity, nnz_out);
}

/*
 * Causal token graph ([D] sec 2.6: A lower-triangular, so every window,
 * random and global edge must satisfy j <= i; [S] sec 1.1: the causal window
 * is the r+1 nearest history positions).  The edge set is the token graph
 * above with the mask j <= i applied to every row:
 *   N(i) = {0..i}                                           if i in G
 *   N(i) = ({j : i-r <= j <= i} u G u {random draws}) n [0, i]  otherwise
 * The random draws are the same draws as the bidirectional graph's; those
 * that land in the future are dropped, not redrawn.
 */
int oracle_token_graph_causal(int64_t n, int32_t r, int32_t n_globals,
                              const int32_t* globals, int32_t rand_per_row,
                              uint64_t seed, int64_t* row_ptr, int32_t* col,
                              int64_t col_capacity, int64_t* nnz_out) {
    return token_graph(n, r, 1, n_globals, globals, rand_per_row, seed, 1, 0, row_ptr,
                       col, col_capacity, nnz_out);
}

/*
 * Dilated token graph ([S] sec 1.2 eq 11): the window of row i becomes
 *   {i + k * dilation : -r <= k <= r} cut to the sequence,
 * which is the sliding window for dilation 1; globals and random draws as in
 * the token graph (one that falls on a window position enters once).
 * `causal` applies the mask j <= i as for oracle_token_graph_causal.
 */
int oracle_token_graph_dilated(int64_t n, int32_t r, int32_t dilation, int32_t n_globals,
                               const int32_t* globals, int32_t rand_per_row, uint64_t seed,
                               int32_t causal, int64_t* row_ptr, int32_t* col,
                               int64_t col_capacity, int64_t* nnz_out) {
    return token_graph(n, r, dilation, n_globals, globals, rand_per_row, seed, causal != 0, 0,
                       row_ptr, col, col_capacity, nnz_out);
}

/*
 * Token graph with uniform-spaced extras ([D] sec 4.5, Tab S.7, "w uni."):
 * the token graph (or, with causal != 0, the causal token graph) whose R
 * random draws of row i are replaced by the positions
 *   j_t = (i + floor((2t + 1) n / (2R))) mod n,  t < R
 * (R >= 1 when used; R = 0 gives the plain window-and-globals graph).
 */
int oracle_token_graph_uniform(int64_t n, int32_t r, int32_t n_globals, const int32_t* globals,
                               int32_t rand_per_row, int32_t causal, int64_t* row_ptr,
                               int32_t* col, int64_t col_capacity, int64_t* nnz_out) {
    return token_graph(n, r, 1, n_globals, globals, rand_per_row, 0, causal != 0, 1, row_ptr,
                       col, col_capacity, nnz_out);
}

/*
 * BigBird ITC block graph ([S] sec 2 eq 13 and the 12-block example; [B]
 * sec 2).  Blocks of `block` tokens, N = ceil(n / block).  Block row J reads
 * every block if J < global_blocks; otherwise the window blocks around J,
 * the global blocks and `rand_blocks` random blocks.  Token i reads token j
 * iff block(j) is allowed for block(i).
 */
int oracle_block_graph(int64_t n, int32_t block, int32_t window_blocks,
                       int32_t rand_blocks, int32_t global_blocks,
                       uint64_t seed, int64_t* row_ptr, int32_t* col,
                       int64_t col_capacity, int64_t* nnz_out) {
    if (n < 1 || n > INT32_MAX || block < 1 || window_blocks < 1 ||
        (window_blocks % 2) == 0 || rand_blocks < 0 || global_blocks < 0 ||
        !nnz_out)
        return ORACLE_BAD_ARG;
    int64_t nb = (n + block - 1) / block;
    if (global_blocks > nb) return ORACLE_BAD_ARG;
    int64_t half = (window_blocks - 1) / 2;
    unsigned char* allowed = (unsigned char*)malloc((size_t)nb);
    unsigned char* mark = (unsigned char*)malloc((size_t)n);
    if (!allowed || !mark) { free(allowed); free(mark); return ORACLE_NO_MEM; }
    int overflow = 0;
    int64_t nnz = 0;
    if (row_ptr) row_ptr[0] = 0;
    for (int64_t i = 0; i < n; ++i) {
        int64_t J = i / block;
        memset(allowed, 0, (size_t)nb);
        if (J < global_blocks) {
            memset(allowed, 1, (size_t)nb);              /* global block row */
        } else {
            for (int64_t c = J - half; c <= J + half; ++c)
                if (c >= 0 && c < nb) allowed[c] = 1;     /* window blocks */
            for (int64_t c = 0; c < global_blocks; ++c)
                allowed[c] = 1;                           /* global blocks */
            for (int32_t t = 0; t < rand_blocks; ++t) {   /* random blocks */
                uint64_t key = (uint64_t)J * (uint64_t)rand_blocks + (uint64_t)t;
                allowed[oracle_splitmix64(seed ^ key) % (uint64_t)nb] = 1;
            }
        }
        for (int64_t j = 0; j < n; ++j) mark[j] = allowed[j / block];
        nnz += emit_row(mark, n, col, nnz, col_capacity, &overflow);
        if (overflow) { free(allowed); free(mark); return ORACLE_CAPACITY; }
        if (row_ptr) row_ptr[i + 1] = nnz;
    }
    *nnz_out = nnz;
    free(allowed);
    free(mark);
    return ORACLE_OK;
}

/*
 * Masked row softmax over each row's allowed set ([D] eq S.1-S.5; [S] eq 1-3):
 *   s_ij = (q_i . k_j) / sqrt(d),  A_ij = exp(s_ij - m_i) / sum_t exp(s_it - m_i)
 * with m_i the row maximum (subtracting it changes nothing mathematically).
 * Q, K: [n][d] row-major.  A: one weight per CSR edge, in CSR order.
 */
void oracle_attention_weights(const double* Q, const double* K, int64_t n,
                              int32_t d, const int64_t* row_ptr,
                              const int32_t* col, double* A) {
    const double scale = 1.0 / sqrt((double)d);
    for (int64_t i = 0; i < n; ++i) {
        int64_t e0 = row_ptr[i], e1 = row_ptr[i + 1];
        if (e1 <= e0) continue;
        double m = -INFINITY;
        for (int64_t e = e0; e < e1; ++e) {
            const double* q = Q + i * d;
            const double* k = K + (int64_t)col[e] * d;
            double s = 0.0;
            for (int32_t c = 0; c < d; ++c) s += q[c] * k[c];
            A[e] = s * scale;                       /* raw score for now */
            if (A[e] > m) m = A[e];
        }
        double denom = 0.0;
        for (int64_t e = e0; e < e1; ++e) {
            A[e] = exp(A[e] - m);
            denom += A[e];
        }
        for (int64_t e = e0; e < e1; ++e) A[e] /= denom;
    }
}

/*
 * PPR diffusion ([D] sec 2.4 eq S.7):
 *   Z_0 = V,  Z_{k+1} = (1 - alpha) * A Z_k + alpha * V,  0 <= k < hops.
 * A in CSR (row_ptr, col, weights), V and Z: [n][dv] row-major.  Z receives
 * Z_hops.
 */
int oracle_diffuse(const double* A, const int64_t* row_ptr, const int32_t* col,
                   const double* V, int64_t n, int32_t dv, int32_t hops,
                   double alpha, double* Z) {
    if (hops < 0 || n < 1 || dv < 1) return ORACLE_BAD_ARG;
    double* next = (double*)malloc(sizeof(double) * (size_t)n * (size_t)dv);
    double* acc = (double*)malloc(sizeof(double) * (size_t)dv);
    if (!next || !acc) { free(next); free(acc); return ORACLE_NO_MEM; }
    memcpy(Z, V, sizeof(double) * (size_t)n * (size_t)dv);
    for (int32_t k = 0; k < hops; ++k) {
        for (int64_t i = 0; i < n; ++i) {
            /* acc = (A Z_k)_i = sum over the row's edges e of A_e * Z_k[col_e] */
            for (int32_t c = 0; c < dv; ++c) acc[c] = 0.0;
            for (int64_t e = row_ptr[i]; e < row_ptr[i + 1]; ++e) {
                const double* z = Z + (int64_t)col[e] * dv;
                for (int32_t c = 0; c < dv; ++c) acc[c] += A[e] * z[c];
            }
            for (int32_t c = 0; c < dv; ++c)
                next[i * dv + c] = (1.0 - alpha) * acc[c] + alpha * V[i * dv + c];
        }
        memcpy(Z, next, sizeof(double) * (size_t)n * (size_t)dv);
    }
    free(next);
    free(acc);
    return ORACLE_OK;
}

/* ---- whole forward over independent (batch, head) units -------------------
 * The units share the graph and nothing else, so threads take whole units;
 * the arithmetic inside a unit is exactly the two functions above. */
typedef struct {
    const double *Q, *K, *V;
    double* out;
    int64_t units, n, nnz;
    int32_t d, hops, nthreads, tid;
    double alpha;
    const int64_t* row_ptr;
    const int32_t* col;
    int status;
} oracle_job;

static void* forward_worker(void* arg) {
    oracle_job* job = (oracle_job*)arg;
    double* A = (double*)malloc(sizeof(double) * (size_t)(job->nnz > 0 ? job->nnz : 1));
    if (!A) { job->status = ORACLE_NO_MEM; return NULL; }
    const int64_t stride = job->n * job->d;
    for (int64_t u = job->tid; u < job->units; u += job->nthreads) {
        oracle_attention_weights(job->Q + u * stride, job->K + u * stride, job->n,
                                 job->d, job->row_ptr, job->col, A);
        int st = oracle_diffuse(A, job->row_ptr, job->col, job->V + u * stride,
                                job->n, job->d, job->hops, job->alpha,
                                job->out + u * stride);
        if (st != ORACLE_OK) { job->status = st; break; }
    }
    free(A);
    return NULL;
}

/*
 * Q, K, V, out: [units][n][d] contiguous (units = batch * heads).
 * nthreads >= 1 workers split the units; 1 runs everything on the caller.
 */
int oracle_forward(const double* Q, const double* K, const double* V,
                   int64_t units, int64_t n, int32_t d, const int64_t* row_ptr,
                   const int32_t* col, int32_t hops, double alpha, double* out,
                   int32_t nthreads) {
    if (units < 0 || n < 1 || d < 1 || hops < 0 || nthreads < 1) return ORACLE_BAD_ARG;
    if (nthreads > units) nthreads = (int32_t)(units > 0 ? units : 1);
    oracle_job* jobs = (oracle_job*)calloc((size_t)nthreads, sizeof(oracle_job));
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return ORACLE_NO_MEM; }
    for (int32_t t = 0; t < nthreads; ++t) {
        jobs[t] = (oracle_job){Q, K, V, out, units, n, row_ptr[n], d, hops,
                               nthreads, t, alpha, row_ptr, col, ORACLE_OK};
    }
    int status = ORACLE_OK;
    if (nthreads == 1) {
        forward_worker(&jobs[0]);
    } else {
        int32_t started = 0;
        for (; started < nthreads; ++started)
            if (pthread_create(&th[started], NULL, forward_worker, &jobs[started]) != 0) break;
        if (started < nthreads) status = ORACLE_NO_MEM;  /* join those that did start */
        for (int32_t t = 0; t < started; ++t) pthread_join(th[t], NULL);
        if (status != ORACLE_OK) {
            /* units of workers that never started were not computed */
            free(jobs); free(th); return status;
        }
    }
    for (int32_t t = 0; t < nthreads; ++t)
        if (jobs[t].status != ORACLE_OK) status = jobs[t].status;
    free(jobs);
    free(th);
    return status;
}

/*
 * Backward pass through the unrolled recursion ([D] sec 2.6: training runs the
 * same unrolled K-hop recursion, and the gradient flows back through every
 * round of aggregation into the attention weights and from there into the
 * scores).  For one unit, given dOut = dL/dZ_hops, the chain rule taken step
 * by step in reverse order:
 *   Z_{k+1} = (1 - alpha) A Z_k + alpha V:
 *       dV   += alpha G_{k+1}
 *       dA_e += (1 - alpha) G_{k+1}[i] . Z_k[j]         for each edge e = (i, j)
 *       G_k   = (1 - alpha) A^T G_{k+1}
 *   Z_0 = V:  dV += G_0
 *   softmax over row i:  dS_e = A_e (dA_e - sum_{t in row i} A_t dA_t)
 *   s_ij = q_i . k_j / sqrt(d):  dQ_i += dS_e k_j / sqrt(d),  dK_j += dS_e q_i / sqrt(d)
 * with G_hops = dOut.  The forward states Z_0 .. Z_{hops-1} are kept (the
 * plain store-everything form of automatic differentiation).
 * Q, K, V, dOut, dQ, dK, dV: [units][n][d] contiguous; dQ, dK, dV are written.
 */
int oracle_backward(const double* Q, const double* K, const double* V,
                    const double* dOut, int64_t units, int64_t n, int32_t d,
                    const int64_t* row_ptr, const int32_t* col, int32_t hops,
                    double alpha, double* dQ, double* dK, double* dV) {
    if (units < 0 || n < 1 || d < 1 || hops < 0) return ORACLE_BAD_ARG;
    const int64_t nnz = row_ptr[n];
    const size_t nd = (size_t)n * (size_t)d;
    const double scale = 1.0 / sqrt((double)d);
    double* A = (double*)malloc(sizeof(double) * (size_t)(nnz > 0 ? nnz : 1));
    double* dA = (double*)malloc(sizeof(double) * (size_t)(nnz > 0 ? nnz : 1));
    double* Z = (double*)malloc(sizeof(double) * nd * (size_t)(hops > 0 ? hops : 1));
    double* G = (double*)malloc(sizeof(double) * nd);
    double* Gn = (double*)malloc(sizeof(double) * nd);
    if (!A || !dA || !Z || !G || !Gn) {
        free(A); free(dA); free(Z); free(G); free(Gn);
        return ORACLE_NO_MEM;
    }
    int status = ORACLE_OK;
    for (int64_t u = 0; u < units && status == ORACLE_OK; ++u) {
        const double* q = Q + (size_t)u * nd;
        const double* k = K + (size_t)u * nd;
        const double* v = V + (size_t)u * nd;
        double* dq = dQ + (size_t)u * nd;
        double* dk = dK + (size_t)u * nd;
        double* dv = dV + (size_t)u * nd;
        oracle_attention_weights(q, k, n, d, row_ptr, col, A);
        /* forward states Z_0 .. Z_{hops-1} */
        for (int32_t h = 0; h < hops && status == ORACLE_OK; ++h)
            status = oracle_diffuse(A, row_ptr, col, v, n, d, h, alpha, Z + (size_t)h * nd);
        if (status != ORACLE_OK) break;
        memcpy(G, dOut + (size_t)u * nd, sizeof(double) * nd);
        memset(dv, 0, sizeof(double) * nd);
        memset(dA, 0, sizeof(double) * (size_t)(nnz > 0 ? nnz : 1));
        for (int32_t h = hops - 1; h >= 0; --h) {
            const double* z = Z + (size_t)h * nd;          /* Z_h; G holds G_{h+1} */
            for (size_t x = 0; x < nd; ++x) dv[x] += alpha * G[x];
            memset(Gn, 0, sizeof(double) * nd);
            for (int64_t i = 0; i < n; ++i) {
                for (int64_t e = row_ptr[i]; e < row_ptr[i + 1]; ++e) {
                    const int64_t j = col[e];
                    double dot = 0.0;
                    for (int32_t c = 0; c < d; ++c) dot += G[i * d + c] * z[j * d + c];
                    dA[e] += (1.0 - alpha) * dot;
                    for (int32_t c = 0; c < d; ++c)
                        Gn[j * d + c] += (1.0 - alpha) * A[e] * G[i * d + c];
                }
            }
            memcpy(G, Gn, sizeof(double) * nd);
        }
        for (size_t x = 0; x < nd; ++x) dv[x] += G[x];    /* Z_0 = V */
        memset(dq, 0, sizeof(double) * nd);
        memset(dk, 0, sizeof(double) * nd);
        for (int64_t i = 0; i < n; ++i) {
            double dot = 0.0;                               /* sum_t A_t dA_t over row i */
            for (int64_t e = row_ptr[i]; e < row_ptr[i + 1]; ++e) dot += A[e] * dA[e];
            for (int64_t e = row_ptr[i]; e < row_ptr[i + 1]; ++e) {
                const int64_t j = col[e];
                const double ds = A[e] * (dA[e] - dot) * scale;
                for (int32_t c = 0; c < d; ++c) {
                    dq[i * d + c] += ds * k[j * d + c];
                    dk[j * d + c] += ds * q[i * d + c];
                }
            }
        }
    }
    free(A); free(dA); free(Z); free(G); free(Gn);
    return status;
}
