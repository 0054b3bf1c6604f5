/*
 * diffuser.h -- C ABI of libdiffuser.so, the GB300 (sm_103a) implementation of
 * the Diffuser hot path:
 *
 *   1. a fixed sparse edge set N(i): local window u global tokens u random
 *      edges (token level), or the BigBird ITC block pattern;
 *   2. attention weights A_ij = softmax over N(i) of q_i.k_j / sqrt(d);
 *   3. K personalized-PageRank hops  Z_0 = V,
 *      Z_{k+1} = (1 - alpha) A Z_k + alpha V,  written out as Z_K.
 *
 * Sources (page title, section / equation):
 *   [D] "Diffuser: modelling long sequences with multi-hop attention diffusion"
 *       (reading notes on arXiv 2210.11794v2): sec 2.1 eq S.1-S.5, sec 2.2,
 *       sec 2.4 eq S.7, sec 2.6 (cost model: score once, aggregate K times).
 *   [S] "1.2.1 Static sparsity: Longformer, BigBird and sliding windows":
 *       eq 1-4, sec 1.1 eq 5-6, sec 1.2 eq 12, sec 2 eq 13, sec 2.1.
 *   [B] "038 BigBird: keeping long-sequence information paths with sparse
 *       connections", sec 2.
 *
 * Conventions for every entry point:
 *   - Returns a diffuser_status (0 = DIFFUSER_OK).  No C++ exception crosses
 *     the ABI.  diffuser_last_error() gives a one-line message for the last
 *     failure on the calling thread.
 *   - "device" pointers are CUDA global-memory addresses on the device that
 *     was current when the graph was built; "host" pointers are ordinary CPU
 *     memory.  Every pointer is owned by the caller unless stated otherwise.
 *   - Tensors Q, K, V, out are contiguous [B][H][n][d] (batch, head, token,
 *     feature), 16-byte aligned, in the I/O dtype.  d must be 64.
 *   - Work is enqueued on `stream` (NULL = legacy default stream) and is
 *     asynchronous with respect to the host unless stated otherwise.
 *   - Argument checks happen on the host before anything is enqueued; a
 *     failing call launches nothing.
 */
#ifndef DIFFUSER_H
#define DIFFUSER_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DIFFUSER_API __attribute__((visibility("default")))
#else
#define DIFFUSER_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so that the header needs no CUDA
 * include. */
typedef struct CUstream_st* diffuser_stream;

typedef struct diffuser_graph diffuser_graph;

typedef enum {
    DIFFUSER_OK = 0,
    DIFFUSER_ERR_INVALID_ARG = 1,  /* a null pointer, a size out of range, misalignment */
    DIFFUSER_ERR_UNSUPPORTED = 2,  /* a dtype, head width or option the library does not support */
    DIFFUSER_ERR_OVERFLOW = 3,     /* an edge count or buffer size overflows its index type */
    DIFFUSER_ERR_ALLOC = 4,        /* a device or host allocation failed */
    DIFFUSER_ERR_CUDA = 5,         /* a CUDA runtime call or launch failed */
    DIFFUSER_ERR_DEVICE = 6,       /* a kernel reported an error through its status word */
    DIFFUSER_ERR_WORKSPACE = 7     /* workspace pointer null/misaligned or too small */
} diffuser_status;

typedef enum {
    DIFFUSER_DTYPE_FP32 = 0,       /* float32 I/O; all arithmetic in fp32 FMA */
    DIFFUSER_DTYPE_BF16 = 1        /* bfloat16 I/O; fp32 accumulation and fp32 A, Z_k */
} diffuser_dtype;

/* Text for a status code (static storage, never NULL). */
DIFFUSER_API const char* diffuser_status_string(int status);

/* Message of the last failure on the calling thread ("" if none). */
DIFFUSER_API const char* diffuser_last_error(void);

/* Library version as major*10000 + minor*100 + patch. */
DIFFUSER_API int diffuser_version(void);

/* ---------------------------------------------------------------- graphs
 *
 * A graph is an immutable, deduplicated CSR edge set (rows and columns
 * ascending) plus the device-side layouts the kernels use.  It is built on
 * the device that is current at the call, holds its own device and host
 * memory, and may be shared by any number of streams and calls on that
 * device.  The build is synchronous (it returns when the graph is ready).
 */

/*
 * Token-level Diffuser/Longformer graph ([D] sec 2.2; [S] eq 5, eq 12;
 * [B] sec 2).  For i in G: N(i) = {0..n-1}.  Otherwise
 *   N(i) = {j : |i-j| <= r} u G u {splitmix64(seed ^ (i*R + t)) mod n : t < R}
 * with R = rand_per_row, splitmix64 the published SplitMix64 output
 * function, the modulo unsigned 64-bit, and duplicates entering once.
 *
 *   n            sequence length, 1 <= n <= 2^31-1
 *   r            window radius >= 0 (truncated at the ends, never refilled)
 *   n_globals    |G|, 0 <= n_globals <= n
 *   global_idx   host, n_globals strictly increasing positions in [0,n);
 *                NULL means G = {0..n_globals-1}
 *   rand_per_row R, 0 <= R <= 1024 (draws per non-global row)
 *   seed         64-bit seed of the random draws
 *   out          receives the new graph (caller frees with diffuser_graph_free)
 * Errors: INVALID_ARG (ranges, unsorted globals, null out), OVERFLOW (nnz
 * beyond 2^40), ALLOC, CUDA.
 */
DIFFUSER_API int diffuser_build_graph(int64_t n, int32_t r, int32_t n_globals, const int32_t* global_idx,
                         int32_t rand_per_row, uint64_t seed, diffuser_graph** out);

/*
 * Causal token graph ([D] sec 2.6: for autoregressive use A must be
 * lower-triangular, so every window, global and random edge obeys j <= i;
 * [S] sec 1.1: the causal window is the r+1 history positions).  The edge
 * set of diffuser_build_graph with the same arguments, cut to j <= i:
 *   N(i) = {0..i}                                               if i in G
 *   N(i) = ({j : i-r <= j <= i} u G u {random draws}) n [0, i]  otherwise
 * with the same draws as diffuser_build_graph; a draw that lands after i is
 * dropped, not redrawn.  Every row holds its own position, so no softmax row
 * is empty.  Arguments, ownership and errors: as diffuser_build_graph.  The
 * forward picks its path as for diffuser_build_graph; on the band path a
 * tile reads only the key chunks up to its last row.
 */
DIFFUSER_API int diffuser_build_causal_graph(int64_t n, int32_t r, int32_t n_globals,
                                const int32_t* global_idx, int32_t rand_per_row,
                                uint64_t seed, diffuser_graph** out);

/*
 * Dilated token graph ([S] sec 1.2 eq 11): as diffuser_build_graph (or, with
 * causal != 0, diffuser_build_causal_graph) with the window of row i replaced
 * by the positions {i + k * dilation : -r <= k <= r} inside the sequence
 * (dilation 1 is the sliding window and builds exactly that graph).  Globals
 * and random draws as there; a global or draw that falls on a window position
 * enters once.  dilation >= 1.  A graph with dilation > 1 takes the CSR path.
 * Errors: as diffuser_build_graph.
 */
DIFFUSER_API int diffuser_build_dilated_graph(int64_t n, int32_t r, int32_t dilation,
                                 int32_t n_globals, const int32_t* global_idx,
                                 int32_t rand_per_row, uint64_t seed, int32_t causal,
                                 diffuser_graph** out);

/*
 * Token graph with uniform-spaced extras ([D] sec 4.5, Tab S.7, the "w uni."
 * ablation: the positions of the random edges are taken at uniform spacing
 * instead of at random; the pages do not give the spacing rule).  As
 * diffuser_build_graph (causal != 0: diffuser_build_causal_graph) with the R
 * draws of row i replaced by the uniform grid of spacing n / R on the ring of
 * positions, half a spacing on from i:
 *   j_t = (i + floor((2t + 1) n / (2R))) mod n,  t < R = positions_per_row,
 * entering once where they fall on the window or a global.  No seed: the
 * graph is deterministic.  positions_per_row 0..1024.  The forward picks its
 * path as for diffuser_build_graph.  Errors: as diffuser_build_graph.
 */
DIFFUSER_API int diffuser_build_uniform_graph(int64_t n, int32_t r, int32_t n_globals,
                                              const int32_t* global_idx, int32_t positions_per_row,
                                              int32_t causal, diffuser_graph** out);

/*
 * BigBird ITC block graph ([S] sec 2 eq 13 and its 12-block example; [B]
 * sec 2).  N = ceil(n/block) blocks (the last one may be ragged).  Block row
 * J < global_blocks reads every block.  Any other block row J reads the
 * window_blocks blocks centred on J (truncated at the ends), blocks
 * 0..global_blocks-1, and the blocks splitmix64(seed ^ (J*rand_blocks + t))
 * mod N for t < rand_blocks.  Token i reads token j iff block(j) is allowed
 * for block(i).
 *
 *   block >= 1; window_blocks odd, 1..63; rand_blocks 0..64;
 *   0 <= global_blocks <= N.
 * Errors: as diffuser_build_graph.
 */
DIFFUSER_API int diffuser_build_block_graph(int64_t n, int32_t block, int32_t window_blocks,
                               int32_t rand_blocks, int32_t global_blocks, uint64_t seed,
                               diffuser_graph** out);

/* n and nnz (= number of edges) of a graph; either output may be NULL. */
DIFFUSER_API int diffuser_graph_info(const diffuser_graph* g, int64_t* n, int64_t* nnz);

/*
 * Copy the CSR to caller-owned HOST buffers: row_ptr[n+1] (int64, row_ptr[0]
 * = 0, row_ptr[n] = nnz) and col_idx[nnz] (int32, ascending within a row).
 */
DIFFUSER_API int diffuser_graph_copy_csr(const diffuser_graph* g, int64_t* row_ptr, int32_t* col_idx);

/* Release a graph (NULL is a no-op).  No call using it may still be running. */
DIFFUSER_API void diffuser_graph_free(diffuser_graph* g);

/* ---------------------------------------------------------------- forward */

/*
 * Bytes of device workspace diffuser_forward needs for this graph and shape,
 * whichever kernel path is selected.  On the CSR path the workspace holds
 * the stored weights A (fp32, "score once, aggregate K times", [D] sec 2.4 /
 * 2.6) and the fp32 hop state Z_k.  On the band path it holds the row
 * statistics (maxima, inverse sums), the weights of the edges outside the
 * window (globals, random extras, the global rows), the hop state Z_k (as
 * fp32 rows and as bf16 hi/lo operand rows) and the per-hop partial sums;
 * the window's weights are recomputed from Q and K in every hop and never
 * stored.
 *   B, H >= 1; d == 64; dtype a diffuser_dtype.
 */
DIFFUSER_API int diffuser_workspace_size(const diffuser_graph* g, int64_t B, int64_t H, int32_t d,
                            int32_t dtype, size_t* bytes);

/*
 * The hot path ([D] eq S.1-S.5 then eq S.7; [S] eq 1-4):
 *   A_ij = exp(s_ij - m_i) / sum_{t in N(i)} exp(s_it - m_i),  s_ij = q_i.k_j / sqrt(d)
 *   Z_0 = V,  Z_{k+1} = (1 - alpha) A Z_k + alpha V  (k < hops),  out = Z_hops
 * for every (batch, head) unit independently, all units sharing graph g.
 *
 *   Q, K, V     device, [B][H][n][d] in `dtype`, n = the graph's n
 *   out         device, [B][H][n][d] in `dtype`; must not overlap Q or K; may
 *               equal V only when hops == 0
 *   hops        K >= 0 (0 copies V to out)
 *   alpha       restart weight, 0 <= alpha <= 1 (alpha = 0 is allowed: the
 *               finite recursion is well defined)
 *   workspace   device, >= diffuser_workspace_size bytes, 256-byte aligned;
 *               contents on entry are ignored and on return undefined; one
 *               workspace must not be used by two calls in flight at once
 *   stream      stream on which everything is enqueued
 * Precision: A and Z_k are fp32; bf16 outputs are rounded to nearest-even
 * once, from fp32.  On the band and block paths the first forward with a
 * given B*H on a graph builds a table of each CTA's tiles on the host and
 * uploads it (a few KB of device memory held with the graph, at most four
 * tables per path); a forward issued while the caller's stream is capturing
 * deals the tiles in a fixed snake order instead (the same results, bit for
 * bit).  A forward repeated with the same arguments on an uncaptured stream
 * is recorded once into a CUDA graph held with g and replayed afterwards.
 * Errors: INVALID_ARG, UNSUPPORTED (d != 64, dtype),
 * WORKSPACE, CUDA, and DEVICE when a kernel of an earlier call on g has
 * reported a failure through the graph's status word (see
 * diffuser_graph_status): the check reads a host mirror of the word, so it
 * costs no synchronization and sees failures of calls that have completed;
 * nothing is launched until the word is reset.
 */
DIFFUSER_API int diffuser_forward(const void* Q, const void* K, const void* V, int32_t dtype, int64_t B,
                     int64_t H, int32_t d, const diffuser_graph* g, int32_t hops, float alpha,
                     void* out, void* workspace, size_t workspace_bytes, diffuser_stream stream);

/*
 * Bytes of device workspace diffuser_forward_host needs: the forward's
 * workspace plus device staging for Q, K, V and out.
 */
DIFFUSER_API int diffuser_host_workspace_size(const diffuser_graph* g, int64_t B, int64_t H, int32_t d,
                                 int32_t dtype, size_t* bytes);

/*
 * diffuser_forward on HOST buffers: enqueues the host-to-device copies of Q,
 * K and V, the forward, and the transfer of out back to the host, ordered
 * after earlier work on `stream` and complete when `stream` is.
 * Q, K, V, out are host [B][H][n][d] buffers (page-locked memory makes the
 * copies asynchronous; pageable memory works but the copies then block).
 * On the band path V uploads on an internal side stream while the score
 * kernels run, and a page-locked `out` that is mapped into the device's
 * address space is written directly by the last hop (no separate copy); the
 * host buffers must therefore stay valid and untouched until `stream` has
 * been synchronized.  The caller must synchronize `stream` before reading
 * `out`.  Errors: as diffuser_forward.
 */
DIFFUSER_API int diffuser_forward_host(const void* Q, const void* K, const void* V, int32_t dtype, int64_t B,
                          int64_t H, int32_t d, const diffuser_graph* g, int32_t hops,
                          float alpha, void* out, void* workspace, size_t workspace_bytes,
                          diffuser_stream stream);

/*
 * Backward pass ([D] sec 2.6: training runs the same unrolled K-hop
 * recursion and the gradient flows back through every round of aggregation
 * into the weights and the scores).  Given dOut = dL/dout of the forward with
 * the same Q, K, V, graph, hops and alpha, writes the exact gradients
 *   dV = sum over the hops of alpha G_{k+1}, plus G_0, where G_K = dOut and
 *        G_k = (1 - alpha) A^T G_{k+1};
 *   dA_ij = (1 - alpha) sum_k G_{k+1}[i] . Z_k[j];
 *   dS_ij = A_ij (dA_ij - sum_t A_it dA_it);
 *   dQ_i = sum_j dS_ij k_j / sqrt(d),  dK_j = sum_i dS_ij q_i / sqrt(d).
 * The forward's weights and states Z_1 .. Z_{K-1} are recomputed inside the
 * call.  The first backward on a graph also builds its transposed edge list
 * (on the host, then a synchronous upload: 12 bytes per edge and 8 per
 * position of device memory, plus 24 per position on token graphs with a plain
 * window or 12 per block pair on block graphs, held with the graph), so make
 * that first call outside any stream capture.  All arithmetic is fp32; dQ, dK, dV are written in the I/O dtype.
 * On a token graph with a plain window (dilation 1) the window's edges run as
 * 64 x 64 tiles in shared memory and the other edges (globals outside the
 * window, random extras, the global rows' other keys) on CSR kernels; on a
 * block graph of 64-token blocks every edge runs as tiles, key block by key
 * block; on other graphs, or with DIFFUSER_PATH_CSR selected, CSR kernels take
 * every edge.
 * Sums run in a fixed order: repeated calls give identical bits.  Launches
 * count as SCORE (the recomputed weights, the softmax and score gradients) and
 * HOP (the recomputed and reversed hops).
 *
 *   Q, K, V, dOut   device [B][H][n][d] in dtype, 16-byte aligned
 *   dQ, dK, dV      device [B][H][n][d] in dtype, written; they may not overlap
 *                   the inputs or each other
 *   workspace       diffuser_backward_workspace_size bytes, 256-byte aligned:
 *                   2 units nnz + (3 + max(K, 1)) units n 64 fp32 values, and
 *                   on a token graph with a plain window units (nnz - the
 *                   window's pairs) more: the weights of the edges outside the
 *                   window, copied into key order once per call for the
 *                   transposed hops
 * Asynchronous on `stream`.  Errors: as diffuser_forward.
 */
DIFFUSER_API int diffuser_backward_workspace_size(const diffuser_graph* g, int64_t B, int64_t H,
                                     int32_t d, int32_t dtype, int32_t hops, size_t* bytes);
DIFFUSER_API int diffuser_backward(const void* Q, const void* K, const void* V, const void* dOut,
                      int32_t dtype, int64_t B, int64_t H, int32_t d, const diffuser_graph* g,
                      int32_t hops, float alpha, void* dQ, void* dK, void* dV, void* workspace,
                      size_t workspace_bytes, diffuser_stream stream);

/* ---------------------------------------------------------------- one graph per head */

/*
 * diffuser_forward with a graph of its own for every head ([D] sec 2.2 and
 * [S] sec 2: the random connections may differ per layer and per head; a
 * per-layer graph is one graph object per layer).  Head h of every batch item
 * runs on graphs[h]; the heads' graphs must share n and the device.  Q, K, V,
 * out, hops, alpha, stream and the aliasing rules are those of
 * diffuser_forward.
 *   graphs      host array of H graph pointers (may repeat a graph)
 *   workspace   device, >= diffuser_per_head_workspace_size bytes, 256-byte
 *               aligned: for B > 1, staging for one head's Q, K, V and out
 *               (4 B n d elements; a head's slices are strided in BHSD, so each
 *               head is gathered into it with one strided copy per tensor and
 *               its output scattered back), then the largest per-head
 *               diffuser_forward workspace for B units.  For B = 1 the heads
 *               are contiguous and run in place (no staging).
 * The heads run one after the other on `stream`.  Errors: as
 * diffuser_forward (INVALID_ARG also for a NULL or mismatched graph).
 */
DIFFUSER_API int diffuser_per_head_workspace_size(const diffuser_graph* const* graphs, int64_t B,
                                                  int64_t H, int32_t d, int32_t dtype, size_t* bytes);
DIFFUSER_API int diffuser_forward_per_head(const void* Q, const void* K, const void* V, int32_t dtype,
                                           int64_t B, int64_t H, int32_t d,
                                           const diffuser_graph* const* graphs, int32_t hops,
                                           float alpha, void* out, void* workspace,
                                           size_t workspace_bytes, diffuser_stream stream);

/* ---------------------------------------------------------------- the surrounding layer */

/*
 * The projections around the diffusion module ([D] sec 2.1: per head
 * Q = X W_Q, K = X W_K, V = X W_V; [D] sec 2.4, Fig S.3: the heads' outputs
 * are concatenated and projected by W_O; residual and feed-forward lie
 * outside the module), as dense GEMMs on the tcgen05 tensor cores: bf16
 * operands, fp32 accumulation, bf16 results rounded to nearest-even once.
 * Weights use the [out_features][in_features] layout:
 *   X     device bf16 [B][n][D]   (tokens of batch item b, model width D)
 *   Wqkv  device bf16 [3 H d][D]  row s H d + h d + f is feature f of head h
 *                                 of Q (s = 0), K (s = 1) or V (s = 2)
 *   Wo    device bf16 [D][H d]    column h d + f reads feature f of head h
 *   Q, K, V, Z   device bf16 [B][H][n][d] (the forward's layout)
 *   Y     device bf16 [B][n][D]
 * d == 64; D a multiple of 8, at most 65536; H >= 1.  All pointers 16-byte
 * aligned; outputs may not overlap inputs or each other.  Asynchronous on
 * `stream`.  The first projection call on a device makes a 16-byte device
 * status block and a page-locked host mirror of it (kept for the process);
 * a projection kernel whose bounded wait gives up records a code there
 * (diffuser_projection_status) and later projection calls return
 * DIFFUSER_ERR_DEVICE until it is reset.
 * Errors: INVALID_ARG, UNSUPPORTED, ALLOC, CUDA, DEVICE.
 */
DIFFUSER_API int diffuser_qkv_projection(const void* X, const void* Wqkv, int64_t B, int64_t n, int32_t D,
                                         int32_t H, int32_t d, void* Q, void* K, void* V,
                                         diffuser_stream stream);
/* Y[b][i] = concat_h Z[b][h][i] . Wo^T (the heads' concatenation and W_O). */
DIFFUSER_API int diffuser_output_projection(const void* Z, const void* Wo, int64_t B, int64_t n, int32_t D,
                                            int32_t H, int32_t d, void* Y, diffuser_stream stream);
/* Read (synchronously) the stand-alone projections' status word of the
 * current device; reset != 0 clears it. */
DIFFUSER_API int diffuser_projection_status(int* status, int reset);

/*
 * The whole module on one graph: Q, K, V = the projections of X, Z =
 * diffuser_forward(Q, K, V) (bf16), Y = the output projection of Z.  n is the
 * graph's n.  workspace: device, >= diffuser_layer_workspace_size bytes,
 * 256-byte aligned (Q, K, V, Z, then the forward's workspace).  Kernel
 * failures are recorded in the graph's status word.  Errors: as
 * diffuser_forward and the projections.
 */
DIFFUSER_API int diffuser_layer_workspace_size(const diffuser_graph* g, int64_t B, int32_t D, int32_t H,
                                               int32_t d, size_t* bytes);
DIFFUSER_API int diffuser_layer_forward(const void* X, const void* Wqkv, const void* Wo, int64_t B,
                                        int32_t D, int32_t H, int32_t d, const diffuser_graph* g,
                                        int32_t hops, float alpha, void* Y, void* workspace,
                                        size_t workspace_bytes, diffuser_stream stream);

/* ---------------------------------------------------------------- no-allocation forward */

/*
 * diffuser_forward without any device allocation, for callers that cannot
 * call cudaMalloc while the forward runs: serving loops whose device memory
 * is fixed at start-up, or host frameworks that own every allocation and
 * forbid allocating calls on their hot path (cudaMalloc may synchronize the
 * device and fail under memory pressure at an unpredictable moment).  (The
 * pages have no counterpart: this is a library convenience, not part of the
 * method.)
 *
 * Same arguments and results as diffuser_forward, without the workspace: the
 * weights A and the hop state live in one fixed array in device global
 * memory defined by the library (diffuser_no_alloc_scratch_bytes() bytes,
 * 32 MiB), which every GPU that loads the library holds until the process
 * exits.  It runs the general CSR kernels, with diffuser_forward's CSR-path
 * argument checks, workspace layout and hop sequence.  The graph must be
 * built beforehand (diffuser_build_graph allocates).
 *   - Problems whose weights and hop state need more than the array holds
 *     (units * nnz * 4 + 2 * units * n * 64 * 4 bytes, each part rounded up
 *     to 256) are rejected with DIFFUSER_ERR_WORKSPACE before anything runs.
 *   - Every call overwrites the part of the array it uses; nothing in it has
 *     to start at zero (the weights and each hop's state are written before
 *     they are read).
 *   - The first call on a device looks up the array's device address on that
 *     device (make it before any stream capture); later calls only launch
 *     kernels.  No cudaMalloc, cudaFree or allocating library routine is
 *     called.
 *   - All calls share the array: two calls that overlap on the GPU (on
 *     different streams, or different host threads) race and corrupt each
 *     other's results.  Calls on one stream are serialized and safe.
 * Errors: as diffuser_forward, plus WORKSPACE when the problem is too large.
 */
DIFFUSER_API int diffuser_forward_no_alloc(const void* Q, const void* K, const void* V,
                                           int32_t dtype, int64_t B, int64_t H, int32_t d,
                                           const diffuser_graph* g, int32_t hops, float alpha,
                                           void* out, diffuser_stream stream);

/* Size in bytes of the fixed device array diffuser_forward_no_alloc uses. */
DIFFUSER_API size_t diffuser_no_alloc_scratch_bytes(void);

/* ---------------------------------------------------------------- test exports */

/*
 * Attention weights only ([D] eq S.1-S.5): writes A for every unit in CSR
 * edge order to A_out (device, fp32 [B*H][nnz]).  Same arguments and
 * workspace as diffuser_forward.
 */
DIFFUSER_API int diffuser_attention_weights(const void* Q, const void* K, int32_t dtype, int64_t B, int64_t H,
                               int32_t d, const diffuser_graph* g, float* A_out, void* workspace,
                               size_t workspace_bytes, diffuser_stream stream);

/*
 * Diffusion only ([D] eq S.7) on caller-given weights: A (device, fp32
 * [B*H][nnz] in CSR edge order of g, rows need not sum to 1), V and out as
 * in diffuser_forward.  Runs the same hop kernels as the forward's general
 * path.  workspace >= diffuser_workspace_size bytes.
 */
DIFFUSER_API int diffuser_diffuse_csr(const diffuser_graph* g, const float* A, const void* V, int32_t dtype,
                         int64_t B, int64_t H, int32_t d, int32_t hops, float alpha, void* out,
                         void* workspace, size_t workspace_bytes, diffuser_stream stream);

/* ---------------------------------------------------------------- path and status */

typedef enum {
    DIFFUSER_PATH_AUTO = 0,       /* band tensor-core path where eligible, else CSR */
    DIFFUSER_PATH_CSR = 1         /* always the general CSR SIMT path (forward and backward) */
} diffuser_path;

/*
 * Select the kernel path for later calls in this process (thread-safe; the
 * default is DIFFUSER_PATH_AUTO).  The band path serves token graphs with
 * bf16 I/O, window radius >= 8 and at most 32 globals; it stores the weights
 * in a decomposed window/global/extra layout and runs the window part of
 * every hop on tcgen05 tensor cores (bf16 hi + lo split, fp32 accumulation).
 * The workspace size depends on the path: query diffuser_workspace_size
 * after changing it.  Errors: INVALID_ARG for an unknown path.
 */
DIFFUSER_API int diffuser_set_path(int path);
DIFFUSER_API int diffuser_get_path(void);

/* Kernel families a forward can run on. */
typedef enum {
    DIFFUSER_KERNELS_CSR = 1,     /* general CSR SIMT kernels (fp32 arithmetic) */
    DIFFUSER_KERNELS_BAND = 2,    /* token graphs: tcgen05 window tiles + random-edge gathers */
    DIFFUSER_KERNELS_BLOCK = 3    /* block graphs of 64-token blocks: tcgen05 block-sparse tiles */
} diffuser_kernels;

/*
 * The kernel family diffuser_forward would run for graph g and this dtype
 * under the current path selection (a diffuser_kernels value in *kernels).
 * The band family serves token graphs with bf16 I/O, window radius >= 8,
 * dilation 1 and at most 32 globals; the block family serves block graphs of
 * 64-token blocks with bf16 I/O; everything else runs the CSR family.
 */
DIFFUSER_API int diffuser_kernels_for(const diffuser_graph* g, int32_t dtype, int* kernels);

/*
 * Read (synchronously) the device status word that the graph's kernels set
 * when a bounded internal wait gives up (0 = no error); reset != 0 clears it
 * and its host mirror.  A nonzero word means results computed since the last
 * reset are invalid, and every forward or backward on g returns
 * DIFFUSER_ERR_DEVICE without launching anything until it is reset.
 */
DIFFUSER_API int diffuser_graph_status(const diffuser_graph* g, int* status, int reset);

/*
 * Test export: write `status` into the graph's status word and its host
 * mirror with plain copies (no kernel), as a kernel does when one of its
 * bounded waits gives up.  Lets a test check the error path of the entry
 * points and of the caller's own checks without making any kernel fail.
 */
DIFFUSER_API int diffuser_graph_set_status(const diffuser_graph* g, int status);

/* ---------------------------------------------------------------- measurement */

/* Kinds of kernel launch, for the counters below. */
typedef enum {
    DIFFUSER_KERNEL_BUILD = 0,    /* graph construction */
    DIFFUSER_KERNEL_SCORE = 1,    /* scores + masked softmax -> A */
    DIFFUSER_KERNEL_HOP = 2,      /* one diffusion hop (the window part, on the band path) */
    DIFFUSER_KERNEL_AUX = 3,      /* copies, conversions, split-reduction merges */
    DIFFUSER_KERNEL_GATHER = 4,   /* band path: a hop's random-edge / global gathers */
    DIFFUSER_KERNEL_KINDS = 5
} diffuser_kernel_kind;

/* Number of kernels this library has launched in this process, per kind
 * (array of DIFFUSER_KERNEL_KINDS entries; may be NULL) and in total (return
 * value). */
DIFFUSER_API int64_t diffuser_launch_count(int64_t* per_kind);

/*
 * Device-time profiling of the library's own kernels.  Between begin and
 * end, every launch is bracketed by CUDA events recorded on the stream it is
 * launched on.  end synchronizes those events and writes, per kind, the
 * summed device milliseconds and the number of launches (arrays of
 * DIFFUSER_KERNEL_KINDS entries).  Thread-safe; one profile at a time.
 */
DIFFUSER_API int diffuser_profile_begin(void);
DIFFUSER_API int diffuser_profile_end(double* ms_per_kind, int64_t* launches_per_kind);

#ifdef __cplusplus
}
#endif

#endif /* DIFFUSER_H */
