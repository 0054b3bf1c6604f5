// Backward pass: the gradients dQ, dK, dV of <dOut, Z_K> ("Diffuser:
// modelling long sequences with multi-hop attention diffusion", sec 2.6:
// training runs the same unrolled K-hop recursion, and the gradient flows back
// through every round of aggregation into the weights and from there into the
// scores).  fp32 arithmetic throughout; any graph, either I/O dtype.  With
// G_K = dOut, after recomputing A and Z_1 .. Z_{K-1}, for k = K-1 .. 0:
//
//    dA_e += (1 - alpha) G_{k+1}[i] . Z_k[j]          for every edge e = (i, j);
//    G_k[j] = (1 - alpha) sum_e A_e G_{k+1}[i]         (the transposed graph),
//    dV_acc[j] += alpha G_{k+1}[j]                     (dV = dV_acc + G_0 at k = 0);
//
// then the softmax and the scores: dS_e = A_e (dA_e - sum_t A_t dA_t) / sqrt(64)
// (in place over dA), dQ_i = sum_e dS_e k_j and dK_j = sum_e dS_e q_i.
//
// Two kinds of kernels share the edges.  On a token graph with a plain window
// (dilation 1) row i holds the keys lo(i) .. hi(i) of its window as one run of
// its CSR row (at wp0[i]), and key j the rows whose windows hold it as one run
// of its transposed list (at tw0[j]).  The band kernels take those runs as
// dense tiles: a CTA stages 64 rows of the operand and the weights of a 64 x 64
// block of the window in shared memory, and each thread accumulates a register
// tile (products A Z and A^T G: 8 rows x 2 features per lane; dA: 4 rows x 4
// keys per thread).  The CSR kernels (a warp per row or key, lanes own two
// features, one coalesced operand row per edge) take the other edges -- the
// globals outside the window, the random extras, the global rows' other keys
// -- and add the band kernels' partial sums before their epilogue; on other
// graphs (and with the CSR path forced) they take every edge.  Every sum runs
// in a fixed order (window keys ascending, then the other edges in CSR or
// transposed order), so the result is deterministic.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>
#include <vector>

#include "internal.h"

namespace dfs {
namespace {

constexpr int kBwdWarps = 8;           // warps per CTA; one warp per row or key
constexpr float kScale = 0.125f;       // 1/sqrt(64), exact

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two adjacent features (2l, 2l + 1) of a row, widened to fp32.
__device__ __forceinline__ float2 load2(const float* p) { return *reinterpret_cast<const float2*>(p); }
__device__ __forceinline__ float2 load2(const __nv_bfloat16* p) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
    return make_float2(bf16lo(w), bf16hi(w));
}
// Four adjacent features of a row, widened to fp32.
__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    return make_float4(bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y));
}
__device__ __forceinline__ void store2(float* p, float2 v) { *reinterpret_cast<float2*>(p) = v; }
__device__ __forceinline__ void store2(__nv_bfloat16* p, float2 v) {
    *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(v.x, v.y);
}

struct BwdArgs {
    const int64_t* row_ptr;   // CSR [n + 1]
    const int32_t* col;       // CSR [nnz]
    const int64_t* t_ptr;     // transposed graph: incoming edges of key j at t_ptr[j] .. t_ptr[j+1]-1
    const int32_t* t_row;     // their rows i, ascending
    const int64_t* t_edge;    // their CSR edge ids e
    const int64_t* wp0;       // [n] CSR position of row i's window run; null: no band kernels
    const int64_t* tw0;       // [n] transposed-list position of key j's window run
    const int32_t* bptr;      // block graph (64-token blocks): key blocks of block row J at bcol[bptr[J] ..];
    const int32_t* bcol;      //   null: no block runs
    const int32_t* btptr;     // the row blocks holding key block KB at btrow[btptr[KB] ..], and the
    const int32_t* btrow;     //   key block's place in each such row block's list
    const int32_t* btpos;
    const int32_t* row_order; // [n] the heavy rows by falling edge count, then the others ascending
    const int32_t* key_order; // [n] the same for the keys and their incoming edges
    int64_t heavy_rows, heavy_keys;   // how many come first in each order
    int64_t n, nnz, units;
    int32_t r, causal;        // the window: keys i - r .. i + r (.. i when causal), clipped
    const int64_t* trest;     // [n + 1] where key j's incoming edges outside its window run start in
    int64_t nrest;            //   the key-ordered weights ([units][nrest]); null: none are kept
};

// The keys lo .. hi of row i's window, and the rows lo .. hi whose windows hold key j.
__device__ __forceinline__ void win_row(const BwdArgs& a, int64_t i, int64_t& lo, int64_t& hi) {
    lo = i - a.r > 0 ? i - a.r : 0;
    hi = a.causal ? i : (i + a.r < a.n - 1 ? i + a.r : a.n - 1);
}
__device__ __forceinline__ void win_key(const BwdArgs& a, int64_t j, int64_t& lo, int64_t& hi) {
    lo = a.causal ? j : (j - a.r > 0 ? j - a.r : 0);
    hi = j + a.r < a.n - 1 ? j + a.r : a.n - 1;
}
// The window run [s0, s1) of row i's CSR edges (key j's transposed list) that the
// band kernels take; empty without them, everything on a block graph.
__device__ __forceinline__ void row_run(const BwdArgs& a, int64_t i, int64_t e0, int64_t e1, int64_t& s0,
                                        int64_t& s1) {
    if (a.bptr) { s0 = e0; s1 = e1; return; }
    if (!a.wp0) { s0 = s1 = e0; return; }
    int64_t lo, hi;
    win_row(a, i, lo, hi);
    s0 = a.wp0[i];
    s1 = s0 + (hi - lo + 1);
}
__device__ __forceinline__ void key_run(const BwdArgs& a, int64_t j, int64_t t0, int64_t t1, int64_t& s0,
                                        int64_t& s1) {
    if (a.bptr) { s0 = t0; s1 = t1; return; }
    if (!a.tw0) { s0 = s1 = t0; return; }
    int64_t lo, hi;
    win_key(a, j, lo, hi);
    s0 = a.tw0[j];
    s1 = s0 + (hi - lo + 1);
}
// The (unit, row) of CSR warp gw: the heavy rows (or keys) of every unit first,
// heaviest first, every unit's copy in turn, so that their long lists start with
// the launch; then the other rows unit by unit in order.
__device__ __forceinline__ void warp_item(const BwdArgs& a, int64_t gw, const int32_t* order, int64_t heavy,
                                          int64_t& u, int64_t& i) {
    if (gw < a.units * heavy) {
        const int64_t rk = gw / a.units;
        u = gw - rk * a.units;
        i = order[rk];
    } else {
        const int64_t g2 = gw - a.units * heavy, rest = a.n - heavy;
        u = g2 / rest;
        i = order[heavy + (g2 - u * rest)];
    }
}

// position v of the edges e0 .. e1-1 outside the run [s0, s1)
__device__ __forceinline__ int64_t rest_pos(int64_t e0, int64_t v, int64_t s0, int64_t s1) {
    const int64_t e = e0 + v;
    return e >= s0 ? e + (s1 - s0) : e;
}

// ---------------------------------------------------------------- band kernels
constexpr int kTile = 64;              // rows (keys) of a band tile
constexpr int kChunk = 64;             // keys (rows) of a staged chunk
constexpr int kBandThreads = 256;
constexpr int kWStride = kChunk + 4;   // a staged weight row (float4-aligned)
constexpr int kMaxRange = 1088;        // rows of a key tile whose runs are staged in shared memory
constexpr int kXPer = kChunk * (kHeadDim / 4) / kBandThreads;   // float4s of X a thread stages (dA)
static_assert(kXPer * kBandThreads == kChunk * (kHeadDim / 4), "staging shares");

// The tiles of a band launch: unit-major on token graphs (neighbouring tiles of a
// unit run together); tile-major on block graphs, so that the heavy global block
// rows (keys) of every unit start with the launch.
__device__ __forceinline__ void tile_of(const BwdArgs& a, bool tile_major, int64_t& u, int64_t& t) {
    const int64_t tiles = (a.n + kTile - 1) / kTile;
    if (tile_major) { t = blockIdx.x / a.units; u = blockIdx.x - t * a.units; }
    else { u = blockIdx.x / tiles; t = blockIdx.x - u * tiles; }
}

// Asynchronous global -> shared copies (this thread's; cp_wait<N> leaves the N
// newest groups in flight, a __syncthreads then shares the data): 16 or 4 bytes, or
// zeros when `valid` is false (nothing is read then).
__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void cp16(void* sdst, const void* gsrc, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(sdst)), "l"(gsrc),
                 "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp4(void* sdst, const void* gsrc, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_addr(sdst)), "l"(gsrc),
                 "r"(valid ? 4 : 0) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int kN>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(kN) : "memory"); }

// A chunk's 64 operand rows (first .. first + 63, zeros past last) into xs, in X's
// own type, as asynchronous 16-byte copies.
template <typename TX>
__device__ __forceinline__ void stage_rows_async(TX (*xs)[kHeadDim], const TX* Xu, int64_t first, int64_t last,
                                                 int tid) {
    constexpr int kPerRow = kHeadDim * (int)sizeof(TX) / 16;           // 16-byte pieces of a row
    constexpr int kPer = kChunk * kPerRow / kBandThreads;
    constexpr int kElems = 16 / (int)sizeof(TX);
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        const int idx = tid + kBandThreads * q, rr = idx / kPerRow, c = idx - rr * kPerRow;
        const int64_t j = first + rr;
        cp16(&xs[rr][kElems * c], j <= last ? Xu + j * kHeadDim + kElems * c : Xu, j <= last);
    }
}

// P[i] = sum over the keys j of row i's window of W[e(i, j)] X[j], e(i, j) =
// wp0[i] + j - lo(i); on a block graph (kBlk) over the key blocks of row i's block,
// e(i, j) = row_ptr[i] + 64 (place of j's block in the list) + j % 64.  A CTA: 64
// rows of one unit; warp w rows 8w .. 8w+7, lane l features 2l, 2l+1; the keys in
// chunks of 64 (the window's, or the key blocks), ascending, staged by
// asynchronous copies one chunk ahead (two buffers).
template <typename TX, bool kBlk>
__global__ void __launch_bounds__(kBandThreads)
bwd_band_rows_kernel(BwdArgs a, const float* __restrict__ W, const TX* __restrict__ X, float* __restrict__ P) {
    extern __shared__ __align__(16) uint8_t band_smem[];
    auto xs = reinterpret_cast<TX (*)[kChunk][kHeadDim]>(band_smem);                   // [2]
    auto ws = reinterpret_cast<float (*)[kTile][kWStride]>(band_smem + 2 * kChunk * kHeadDim * sizeof(TX));
    int64_t* s_lo = reinterpret_cast<int64_t*>(ws + 2);        // the tile rows' windows and runs
    int64_t* s_hi = s_lo + kTile;
    int64_t* s_wp = s_hi + kTile;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int64_t u, t;
    tile_of(a, kBlk, u, t);
    const int64_t i0 = t * kTile;
    const int64_t ilast = i0 + kTile - 1 < a.n - 1 ? i0 + kTile - 1 : a.n - 1;
    int64_t klo = 0, khi = 0, c_begin = 0, c_end;
    if (kBlk) {
        c_begin = a.bptr[t];
        c_end = a.bptr[t + 1];
    } else {
        int64_t tmp;
        win_row(a, i0, klo, tmp);
        win_row(a, ilast, tmp, khi);
        c_end = (khi - klo) / kChunk + 1;
    }
    if (tid < kTile) {
        const int64_t i = i0 + tid;
        int64_t lo = 1, hi = 0, wp = 0;            // rows past n: an empty window
        if (i <= ilast) {
            if (kBlk) { lo = 0; hi = a.n - 1; wp = a.row_ptr[i]; }
            else { win_row(a, i, lo, hi); wp = a.wp0[i]; }
        }
        s_lo[tid] = lo; s_hi[tid] = hi; s_wp[tid] = wp;
    }
    __syncthreads();                              // the row table, before the first staging
    const float* Wu = W + (size_t)u * a.nnz;
    const TX* Xu = X + (size_t)u * a.n * kHeadDim;
    constexpr int kWPer = kTile * kChunk / kBandThreads;
    auto stage = [&](int64_t c, int b) {
        const int64_t k0 = kBlk ? (int64_t)a.bcol[c] * kChunk : klo + kChunk * c;
        const int64_t kend = kBlk ? (k0 + kChunk - 1 < a.n - 1 ? k0 + kChunk - 1 : a.n - 1) : khi;
        stage_rows_async(xs[b], Xu, k0, kend, tid);
        const int kk = tid & (kChunk - 1);
        const int64_t j = k0 + kk;
#pragma unroll
        for (int q = 0; q < kWPer; ++q) {
            const int rr = (tid >> 6) + (kBandThreads / kChunk) * q;
            const int64_t lo = s_lo[rr];
            const bool in = j >= lo && j <= s_hi[rr] && j <= kend;
            const int64_t at = kBlk ? s_wp[rr] + kChunk * (c - c_begin) + kk : s_wp[rr] + (j - lo);
            cp4(&ws[b][rr][kk], in ? Wu + at : Wu, in);
        }
        cp_commit();
    };
    float2 acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = make_float2(0.f, 0.f);
    if (c_begin < c_end) stage(c_begin, 0);
    for (int64_t c = c_begin; c < c_end; ++c) {
        const int b = (int)((c - c_begin) & 1);
        if (c + 1 < c_end) { stage(c + 1, b ^ 1); cp_wait<1>(); }
        else cp_wait<0>();
        __syncthreads();                          // chunk c has landed for every thread
#pragma unroll 2
        for (int kk = 0; kk < kChunk; kk += 4) {
            float2 z[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) z[q] = load2(&xs[b][kk + q][2 * lane]);
#pragma unroll
            for (int rr = 0; rr < 8; ++rr) {
                const float4 w4 = *reinterpret_cast<const float4*>(&ws[b][8 * warp + rr][kk]);
                acc[rr] = __ffma2_rn(make_float2(w4.x, w4.x), z[0], acc[rr]);
                acc[rr] = __ffma2_rn(make_float2(w4.y, w4.y), z[1], acc[rr]);
                acc[rr] = __ffma2_rn(make_float2(w4.z, w4.z), z[2], acc[rr]);
                acc[rr] = __ffma2_rn(make_float2(w4.w, w4.w), z[3], acc[rr]);
            }
        }
        __syncthreads();                          // buffer b is read before chunk c + 2 refills it
    }
#pragma unroll
    for (int rr = 0; rr < 8; ++rr) {
        const int64_t i = i0 + 8 * warp + rr;
        if (i < a.n) store2(P + ((size_t)u * a.n + i) * kHeadDim + 2 * lane, acc[rr]);
    }
}

// P[j] = sum over the rows i whose windows (key-block lists, kBlk) hold key j of
// W[e(i, j)] X[i].  A CTA: 64 keys of one unit; warp w keys 8w .. 8w+7, lane l
// features 2l, 2l+1; the rows in chunks of 64 (the window rows', or the row blocks
// holding the key block), ascending, staged one chunk ahead like the rows kernel.
// The runs wp0 of the tile's rows are staged once when there are at most
// kMaxRange of them.
template <typename TX, bool kBlk>
__global__ void __launch_bounds__(kBandThreads)
bwd_band_keys_kernel(BwdArgs a, const float* __restrict__ W, const TX* __restrict__ X, float* __restrict__ P) {
    extern __shared__ __align__(16) uint8_t band_smem[];
    auto xs = reinterpret_cast<TX (*)[kChunk][kHeadDim]>(band_smem);                   // [2]
    auto ws = reinterpret_cast<float (*)[kChunk][kWStride]>(band_smem + 2 * kChunk * kHeadDim * sizeof(TX));
    int64_t* s_wp = reinterpret_cast<int64_t*>(ws + 2);        // [kMaxRange] [row of the chunk][key of the tile]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int64_t u, t;
    tile_of(a, kBlk, u, t);
    const int64_t j0 = t * kTile;
    const int64_t jlast = j0 + kTile - 1 < a.n - 1 ? j0 + kTile - 1 : a.n - 1;
    int64_t rlo = 0, rhi = 0, c_begin = 0, c_end;
    bool staged = false;
    if (kBlk) {
        c_begin = a.btptr[t];
        c_end = a.btptr[t + 1];
    } else {
        int64_t tmp;
        win_key(a, j0, rlo, tmp);
        win_key(a, jlast, tmp, rhi);
        c_end = (rhi - rlo) / kChunk + 1;
        staged = rhi - rlo + 1 <= kMaxRange;
        if (staged)
            for (int64_t i = rlo + tid; i <= rhi; i += kBandThreads) s_wp[i - rlo] = a.wp0[i];
    }
    __syncthreads();                              // the run table, before the first staging
    const float* Wu = W + (size_t)u * a.nnz;
    const TX* Xu = X + (size_t)u * a.n * kHeadDim;
    constexpr int kWPer = kChunk * kTile / kBandThreads;
    auto stage = [&](int64_t c, int b) {
        const int64_t r0 = kBlk ? (int64_t)a.btrow[c] * kChunk : rlo + kChunk * c;
        const int64_t rend = kBlk ? (r0 + kChunk - 1 < a.n - 1 ? r0 + kChunk - 1 : a.n - 1) : rhi;
        const int64_t place = kBlk ? (int64_t)a.btpos[c] * kChunk : 0;
        stage_rows_async(xs[b], Xu, r0, rend, tid);
        const int kk = tid & (kTile - 1);
        const int64_t j = j0 + kk;
#pragma unroll
        for (int q = 0; q < kWPer; ++q) {
            const int rr = (tid >> 6) + (kBandThreads / kTile) * q;
            const int64_t i = r0 + rr;
            bool in;
            int64_t at;
            if (kBlk) {
                in = i <= rend && j <= jlast;
                at = in ? a.row_ptr[i] + place + kk : 0;
            } else {
                int64_t lo, hi;
                win_row(a, i, lo, hi);
                in = i <= rend && j < a.n && j >= lo && j <= hi;
                at = in ? (staged ? s_wp[i - rlo] : a.wp0[i]) + (j - lo) : 0;
            }
            cp4(&ws[b][rr][kk], Wu + at, in);
        }
        cp_commit();
    };
    float2 acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = make_float2(0.f, 0.f);
    if (c_begin < c_end) stage(c_begin, 0);
    for (int64_t c = c_begin; c < c_end; ++c) {
        const int b = (int)((c - c_begin) & 1);
        if (c + 1 < c_end) { stage(c + 1, b ^ 1); cp_wait<1>(); }
        else cp_wait<0>();
        __syncthreads();
#pragma unroll 4
        for (int rr = 0; rr < kChunk; ++rr) {
            const float2 x = load2(&xs[b][rr][2 * lane]);
            const float4 wa = *reinterpret_cast<const float4*>(&ws[b][rr][8 * warp]);
            const float4 wb = *reinterpret_cast<const float4*>(&ws[b][rr][8 * warp + 4]);
            acc[0] = __ffma2_rn(make_float2(wa.x, wa.x), x, acc[0]);
            acc[1] = __ffma2_rn(make_float2(wa.y, wa.y), x, acc[1]);
            acc[2] = __ffma2_rn(make_float2(wa.z, wa.z), x, acc[2]);
            acc[3] = __ffma2_rn(make_float2(wa.w, wa.w), x, acc[3]);
            acc[4] = __ffma2_rn(make_float2(wb.x, wb.x), x, acc[4]);
            acc[5] = __ffma2_rn(make_float2(wb.y, wb.y), x, acc[5]);
            acc[6] = __ffma2_rn(make_float2(wb.z, wb.z), x, acc[6]);
            acc[7] = __ffma2_rn(make_float2(wb.w, wb.w), x, acc[7]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const int64_t j = j0 + 8 * warp + q;
        if (j < a.n) store2(P + ((size_t)u * a.n + j) * kHeadDim + 2 * lane, acc[q]);
    }
}

// A chunk's 64 operand rows, feature-major (xt[f][r]; rows fastest across the
// threads, so the transposing stores are conflict-free), zero past last.
template <typename TX>
__device__ __forceinline__ void stage_rows_t(float (*xt)[kWStride], const TX* Xu, int64_t first, int64_t last,
                                             int tid) {
    float4 v[kXPer];
#pragma unroll
    for (int q = 0; q < kXPer; ++q) {
        const int idx = tid + kBandThreads * q, rr = idx & (kChunk - 1), f4 = idx / kChunk;
        const int64_t j = first + rr;
        v[q] = j <= last ? load4(Xu + j * kHeadDim + 4 * f4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int q = 0; q < kXPer; ++q) {
        const int idx = tid + kBandThreads * q, rr = idx & (kChunk - 1), f4 = idx / kChunk;
        xt[4 * f4][rr] = v[q].x; xt[4 * f4 + 1][rr] = v[q].y; xt[4 * f4 + 2][rr] = v[q].z; xt[4 * f4 + 3][rr] = v[q].w;
    }
}

// dA[e(i, j)] += keep * G[i] . Z[j] over the windows (key-block lists, kBlk) of 64
// rows of one unit: the rows' G staged once (feature-major), the keys' Z in chunks
// of 64 (row-major, 65- or 66-element rows: conflict-free column reads), staged by
// asynchronous copies one chunk ahead; thread (ty, tx) computes rows 4ty .. +3 x
// keys tx + 16c (c < 4) of each chunk, the dA values it updates loaded before its
// dot products.
template <typename TZ>
struct ZRow { static constexpr int kStride = sizeof(TZ) == 4 ? kChunk + 1 : kChunk + 2; };
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename TG, typename TZ, bool kBlk>
__global__ void __launch_bounds__(kBandThreads)
bwd_band_sddmm_kernel(BwdArgs a, const TG* __restrict__ G, const TZ* __restrict__ Z, float* __restrict__ dA,
                      float keep) {
    constexpr int kZS = ZRow<TZ>::kStride;
    extern __shared__ __align__(16) uint8_t band_smem[];
    auto gs = reinterpret_cast<float (*)[kWStride]>(band_smem);                          // [feature][row]
    auto zs = reinterpret_cast<TZ (*)[kChunk][kZS]>(band_smem + kHeadDim * kWStride * sizeof(float));   // [2][key][feature]
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    int64_t u, t;
    tile_of(a, kBlk, u, t);
    const int64_t i0 = t * kTile;
    const int64_t ilast = i0 + kTile - 1 < a.n - 1 ? i0 + kTile - 1 : a.n - 1;
    int64_t klo = 0, khi = 0, c_begin = 0, c_end;
    if (kBlk) {
        c_begin = a.bptr[t];
        c_end = a.bptr[t + 1];
    } else {
        int64_t tmp;
        win_row(a, i0, klo, tmp);
        win_row(a, ilast, tmp, khi);
        c_end = (khi - klo) / kChunk + 1;
    }
    const TG* Gu = G + (size_t)u * a.n * kHeadDim;
    const TZ* Zu = Z + (size_t)u * a.n * kHeadDim;
    float* dAu = dA + (size_t)u * a.nnz;
    auto chunk_keys = [&](int64_t c, int64_t& k0, int64_t& kend) {
        k0 = kBlk ? (int64_t)a.bcol[c] * kChunk : klo + kChunk * c;
        kend = kBlk ? (k0 + kChunk - 1 < a.n - 1 ? k0 + kChunk - 1 : a.n - 1) : khi;
    };
    auto stage = [&](int64_t c, int b) {
        int64_t k0, kend;
        chunk_keys(c, k0, kend);
        constexpr int kPairs = sizeof(TZ) == 4 ? 1 : 2;                 // elements per 4-byte copy
        constexpr int kPer = kChunk * kHeadDim / kPairs / kBandThreads;
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int idx = tid + kBandThreads * q, kk = idx / (kHeadDim / kPairs);
            const int f = kPairs * (idx - kk * (kHeadDim / kPairs));
            const int64_t j = k0 + kk;
            cp4(&zs[b][kk][f], j <= kend ? Zu + j * kHeadDim + f : Zu, j <= kend);
        }
        cp_commit();
    };
    stage_rows_t(gs, Gu, i0, ilast, tid);
    // this thread's rows: window bounds and runs (a block graph's rows take every key
    // of their chunks)
    int64_t rlo[4], rhi[4], rp0[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int64_t i = i0 + 4 * ty + q;
        rlo[q] = 1; rhi[q] = 0; rp0[q] = 0;
        if (i <= ilast) {
            if (kBlk) { rlo[q] = 0; rhi[q] = a.n - 1; rp0[q] = a.row_ptr[i]; }
            else { win_row(a, i, rlo[q], rhi[q]); rp0[q] = a.wp0[i]; }
        }
    }
    if (c_begin < c_end) stage(c_begin, 0);
    for (int64_t c = c_begin; c < c_end; ++c) {
        const int b = (int)((c - c_begin) & 1);
        int64_t k0, kend;
        chunk_keys(c, k0, kend);
        // the dA values this thread updates in chunk c (positions distinct)
        int64_t at[4][4];
        bool in[4][4];
        float old[4][4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const int kk = tx + 16 * cc;
                const int64_t j = k0 + kk;
                in[q][cc] = j >= rlo[q] && j <= rhi[q] && j <= kend;
                at[q][cc] = kBlk ? rp0[q] + kChunk * (c - c_begin) + kk : rp0[q] + (j - rlo[q]);
                old[q][cc] = in[q][cc] ? dAu[at[q][cc]] : 0.f;
            }
        if (c + 1 < c_end) { stage(c + 1, b ^ 1); cp_wait<1>(); }
        else cp_wait<0>();
        __syncthreads();                          // chunk c (and, first, the rows' G) is in
        float acc[4][4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) acc[q][cc] = 0.f;
#pragma unroll 8
        for (int f = 0; f < kHeadDim; ++f) {
            const float4 g4 = *reinterpret_cast<const float4*>(&gs[f][4 * ty]);
            const float gv[4] = {g4.x, g4.y, g4.z, g4.w};
            float zv[4];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) zv[cc] = to_f32(zs[b][tx + 16 * cc][f]);
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) acc[q][cc] = fmaf(gv[q], zv[cc], acc[q][cc]);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
                if (in[q][cc]) dAu[at[q][cc]] = fmaf(keep, acc[q][cc], old[q][cc]);
        __syncthreads();                          // buffer b is read before chunk c + 2 refills it
    }
}

// The band kernels' launches: block-graph runs or window runs.  The product kernels
// take their two staging buffers (and tables) as dynamic shared memory.
template <typename TX>
constexpr size_t rows_smem() {
    return 2 * kChunk * kHeadDim * sizeof(TX) + 2 * kTile * kWStride * sizeof(float) + 3 * kTile * sizeof(int64_t);
}
template <typename TX>
constexpr size_t keys_smem() {
    return 2 * kChunk * kHeadDim * sizeof(TX) + 2 * kChunk * kWStride * sizeof(float) + kMaxRange * sizeof(int64_t);
}
template <typename K>
void allow_smem(K kernel, size_t bytes) {
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}
template <typename TX>
void band_rows(const BwdArgs& a, dim3 grid, cudaStream_t s, const float* W, const TX* X, float* P) {
    static std::once_flag once;
    std::call_once(once, [] {
        allow_smem(bwd_band_rows_kernel<TX, true>, rows_smem<TX>());
        allow_smem(bwd_band_rows_kernel<TX, false>, rows_smem<TX>());
    });
    if (a.bptr) bwd_band_rows_kernel<TX, true><<<grid, kBandThreads, rows_smem<TX>(), s>>>(a, W, X, P);
    else bwd_band_rows_kernel<TX, false><<<grid, kBandThreads, rows_smem<TX>(), s>>>(a, W, X, P);
}
template <typename TX>
void band_keys(const BwdArgs& a, dim3 grid, cudaStream_t s, const float* W, const TX* X, float* P) {
    static std::once_flag once;
    std::call_once(once, [] {
        allow_smem(bwd_band_keys_kernel<TX, true>, keys_smem<TX>());
        allow_smem(bwd_band_keys_kernel<TX, false>, keys_smem<TX>());
    });
    if (a.bptr) bwd_band_keys_kernel<TX, true><<<grid, kBandThreads, keys_smem<TX>(), s>>>(a, W, X, P);
    else bwd_band_keys_kernel<TX, false><<<grid, kBandThreads, keys_smem<TX>(), s>>>(a, W, X, P);
}
template <typename TZ>
constexpr size_t sddmm_smem() {
    return kHeadDim * kWStride * sizeof(float) + 2 * kChunk * ZRow<TZ>::kStride * sizeof(TZ);
}
template <typename TG, typename TZ>
void band_sddmm(const BwdArgs& a, dim3 grid, cudaStream_t s, const TG* G, const TZ* Z, float* dA, float keep) {
    static std::once_flag once;
    std::call_once(once, [] {
        allow_smem(bwd_band_sddmm_kernel<TG, TZ, true>, sddmm_smem<TZ>());
        allow_smem(bwd_band_sddmm_kernel<TG, TZ, false>, sddmm_smem<TZ>());
    });
    if (a.bptr) bwd_band_sddmm_kernel<TG, TZ, true><<<grid, kBandThreads, sddmm_smem<TZ>(), s>>>(a, G, Z, dA, keep);
    else bwd_band_sddmm_kernel<TG, TZ, false><<<grid, kBandThreads, sddmm_smem<TZ>(), s>>>(a, G, Z, dA, keep);
}

// ---------------------------------------------------------------- CSR kernels
// (the edges outside the window runs; all edges without band kernels).  32 edges
// a round: the round's 32 operand rows are requested before the first is used, and
// the next round's edge indices and weights load while they are in flight.  The
// heavy rows (keys) -- the global rows' 3,500 edges outside their window, say --
// take a CTA each, its 8 warps an eighth of the edges each (partial sums added in
// warp order), at the start of the launch; the other rows a warp each, unit by unit.

// The item of CTA blockIdx.x (heavy) or of warp `warp` of it (light): unit u, row
// (key) i, and whether it is heavy.
__device__ __forceinline__ bool edge_item(const BwdArgs& a, const int32_t* order, int64_t heavy, int warp,
                                          int64_t& u, int64_t& i) {
    const int64_t hb = a.units * heavy;
    if ((int64_t)blockIdx.x < hb) {
        const int64_t rk = blockIdx.x / a.units;
        u = blockIdx.x - rk * a.units;
        i = order[rk];
        return true;
    }
    const int64_t item = ((int64_t)blockIdx.x - hb) * kBwdWarps + warp, rest = a.n - heavy;
    u = item / rest;
    i = order[heavy + (item - u * rest)];
    return false;
}
// A heavy item's warp takes the edges [v0, v1) of the len outside the run.
__device__ __forceinline__ void heavy_share(int64_t len, int warp, int64_t& v0, int64_t& v1) {
    const int64_t per = (len + kBwdWarps - 1) / kBwdWarps;
    v0 = per * warp < len ? per * warp : len;
    v1 = v0 + per < len ? v0 + per : len;
}

// sum over the edges v0 .. v1-1 outside the run (edge ids from at(v)) of w * X[row],
// lanes holding features 2l, 2l+1: ... row(v) / weight(v) give an edge's operand row
// and weight.
template <typename TX, class Row, class Weight>
__device__ __forceinline__ float2 edge_sum(int lane, int64_t v0, int64_t v1, const TX* Xu, Row row, Weight weight,
                                           float2 acc) {
    bool ok = v0 + lane < v1;
    float w_l = ok ? weight(v0 + lane) : 0.f;
    int32_t j_l = ok ? row(v0 + lane) : 0;
    for (int64_t vb = v0; vb < v1; vb += 32) {
        const int cnt = (v1 - vb) < 32 ? (int)(v1 - vb) : 32;
        float2 z[32];
#pragma unroll
        for (int t = 0; t < 32; ++t) {
            const int32_t j = __shfl_sync(0xffffffffu, j_l, t);
            z[t] = t < cnt ? load2(Xu + (size_t)j * kHeadDim) : make_float2(0.f, 0.f);
        }
        const float w_c = w_l;
        ok = vb + 32 + lane < v1;
        w_l = ok ? weight(vb + 32 + lane) : 0.f;
        j_l = ok ? row(vb + 32 + lane) : 0;
#pragma unroll
        for (int t = 0; t < 32; ++t) {
            const float w = __shfl_sync(0xffffffffu, w_c, t);
            acc.x = fmaf(w, z[t].x, acc.x);
            acc.y = fmaf(w, z[t].y, acc.y);
        }
    }
    return acc;
}

// A heavy item's total: the 8 warps' partial sums (in shared memory) added in warp
// order by warp 0, onto its initial value; false for the other warps.
__device__ __forceinline__ bool heavy_total(float2 (*part)[32], int warp, int lane, float2& acc) {
    part[warp][lane] = acc;
    __syncthreads();
    if (warp != 0) return false;
    float2 t = part[0][lane];
#pragma unroll
    for (int w = 1; w < kBwdWarps; ++w) { t.x += part[w][lane].x; t.y += part[w][lane].y; }
    acc = t;
    return true;
}


// ---- light rows (keys) by quarter-warps: 4 a warp, 32 a CTA after the heavy CTAs.
// Lane l of a quarter owns 8 features: 8l .. 8l+7 of bf16 operands (one 16-byte
// load per row), 4l .. 4l+3 and 32 + 4l .. +3 of fp32 ones (two); each quarter-warp
// reads whole 128-byte lines.  A batch of kQB edges (rows in flight per lane) at a
// time, the next batch's indices and weights loading meanwhile.
constexpr int kQItems = kBwdWarps * 4;

__device__ __forceinline__ bool quarter_item(const BwdArgs& a, const int32_t* order, int64_t heavy, int q,
                                             int64_t& u, int64_t& i) {
    const int64_t hb = a.units * heavy, rest = a.n - heavy;
    const int64_t item = ((int64_t)blockIdx.x - hb) * kQItems + q;
    if (rest <= 0 || item >= a.units * rest) return false;
    u = item / rest;
    i = order[heavy + (item - u * rest)];
    return true;
}
unsigned quarter_grid(const BwdArgs& a, int64_t heavy) {
    return (unsigned)(a.units * heavy + (a.units * (a.n - heavy) + kQItems - 1) / kQItems);
}

template <bool kWide>
__device__ __forceinline__ void load8(const float* row, int ql, float (&v)[8]) {
    const float4 x = *reinterpret_cast<const float4*>(row + (kWide ? 8 * ql : 4 * ql));
    const float4 y = *reinterpret_cast<const float4*>(row + (kWide ? 8 * ql + 4 : 32 + 4 * ql));
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w; v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
}
template <bool kWide>
__device__ __forceinline__ void load8(const __nv_bfloat16* row, int ql, float (&v)[8]) {
    uint2 x, y;
    if (kWide) {
        const uint4 w = *reinterpret_cast<const uint4*>(row + 8 * ql);
        x = make_uint2(w.x, w.y);
        y = make_uint2(w.z, w.w);
    } else {
        x = *reinterpret_cast<const uint2*>(row + 4 * ql);
        y = *reinterpret_cast<const uint2*>(row + 32 + 4 * ql);
    }
    v[0] = bf16lo(x.x); v[1] = bf16hi(x.x); v[2] = bf16lo(x.y); v[3] = bf16hi(x.y);
    v[4] = bf16lo(y.x); v[5] = bf16hi(y.x); v[6] = bf16lo(y.y); v[7] = bf16hi(y.y);
}
template <bool kWide>
__device__ __forceinline__ void store8(float* row, int ql, const float (&v)[8]) {
    *reinterpret_cast<float4*>(row + (kWide ? 8 * ql : 4 * ql)) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4*>(row + (kWide ? 8 * ql + 4 : 32 + 4 * ql)) = make_float4(v[4], v[5], v[6], v[7]);
}
template <bool kWide>
__device__ __forceinline__ void store8(__nv_bfloat16* row, int ql, const float (&v)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
        w[k] = *reinterpret_cast<const uint32_t*>(&h);
    }
    if (kWide) {
        *reinterpret_cast<uint4*>(row + 8 * ql) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
        *reinterpret_cast<uint2*>(row + 4 * ql) = make_uint2(w[0], w[1]);
        *reinterpret_cast<uint2*>(row + 32 + 4 * ql) = make_uint2(w[2], w[3]);
    }
}

// acc += sum over the edges 0 .. len-1 outside the run of weight(v) X[row(v)] (this
// lane's 8 features), in edge order.
template <typename TX, class Row, class Weight>
__device__ __forceinline__ void quarter_sum(int ql, unsigned qmask, int64_t len, const TX* Xu, Row row,
                                            Weight weight, float (&acc)[8]) {
    constexpr bool kWide = sizeof(TX) == 2;
    constexpr int kQB = kWide ? 8 : 4;
    int32_t jc = 0;
    float wc = 0.f;
    if (ql < kQB && ql < len) { jc = row(ql); wc = weight(ql); }
    for (int64_t vb = 0; vb < len; vb += kQB) {
        float x[kQB][8];
#pragma unroll
        for (int b = 0; b < kQB; ++b) {
            const int32_t j = __shfl_sync(qmask, jc, b, 8);
            if (vb + b < len) {
                load8<kWide>(Xu + (size_t)j * kHeadDim, ql, x[b]);
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) x[b][k] = 0.f;
            }
        }
        int32_t jn = 0;
        float wn = 0.f;
        if (ql < kQB && vb + kQB + ql < len) { jn = row(vb + kQB + ql); wn = weight(vb + kQB + ql); }
#pragma unroll
        for (int b = 0; b < kQB; ++b) {
            const float w = __shfl_sync(qmask, wc, b, 8);
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[k] = fmaf(w, x[b][k], acc[k]);
        }
        jc = jn;
        wc = wn;
    }
}

// Recomputed hop: Y[i] = (1 - alpha) (P[i] + sum_e A_e X[j]) + alpha V[i] (P: the
// band kernel's window sum, or null).
template <typename TX, typename TV>
__global__ void __launch_bounds__(kBwdWarps * 32)
bwd_hop_rows_kernel(BwdArgs a, const float* __restrict__ A, const TX* __restrict__ X,
                    const float* __restrict__ P, const TV* __restrict__ V, float* __restrict__ Y, float alpha) {
    __shared__ float2 part[kBwdWarps][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float keep = 1.f - alpha;
    int64_t u, i;
    if ((int64_t)blockIdx.x >= a.units * a.heavy_rows) {
        const int ql = lane & 7;
        const unsigned qmask = 0xFFu << (lane & 24);
        if (!quarter_item(a, a.row_order, a.heavy_rows, 4 * warp + (lane >> 3), u, i)) return;
        constexpr bool kWide = sizeof(TX) == 2;
        const size_t unit = (size_t)u * a.n * kHeadDim, row = unit + (size_t)i * kHeadDim;
        const float* Au = A + (size_t)u * a.nnz;
        const int64_t e0 = a.row_ptr[i], e1 = a.row_ptr[i + 1];
        int64_t s0, s1;
        row_run(a, i, e0, e1, s0, s1);
        float acc[8];
        if (P) load8<kWide>(P + row, ql, acc);
        else for (int k = 0; k < 8; ++k) acc[k] = 0.f;
        quarter_sum(ql, qmask, (e1 - e0) - (s1 - s0), X + unit,
                    [&](int64_t v) { return a.col[rest_pos(e0, v, s0, s1)]; },
                    [&](int64_t v) { return Au[rest_pos(e0, v, s0, s1)]; }, acc);
        float v[8], y[8];
        load8<kWide>(V + row, ql, v);
#pragma unroll
        for (int k = 0; k < 8; ++k) y[k] = fmaf(keep, acc[k], alpha * v[k]);
        store8<kWide>(Y + row, ql, y);
        return;
    }
    edge_item(a, a.row_order, a.heavy_rows, warp, u, i);
    const size_t unit = (size_t)u * a.n * kHeadDim;
    const float* Au = A + (size_t)u * a.nnz;
    const int64_t e0 = a.row_ptr[i], e1 = a.row_ptr[i + 1];
    int64_t s0, s1;
    row_run(a, i, e0, e1, s0, s1);
    const int64_t len = (e1 - e0) - (s1 - s0);
    int64_t v0, v1;
    heavy_share(len, warp, v0, v1);
    const size_t at = unit + (size_t)i * kHeadDim + 2 * lane;
    float2 acc = (P && warp == 0) ? load2(P + at) : make_float2(0.f, 0.f);
    acc = edge_sum(lane, v0, v1, X + unit + 2 * lane,
                   [&](int64_t v) { return a.col[rest_pos(e0, v, s0, s1)]; },
                   [&](int64_t v) { return Au[rest_pos(e0, v, s0, s1)]; }, acc);
    if (!heavy_total(part, warp, lane, acc)) return;
    const float2 v = load2(V + at);
    store2(Y + at, make_float2(fmaf(keep, acc.x, alpha * v.x), fmaf(keep, acc.y, alpha * v.y)));
}

// dA_e += keep * G[i] . Z[j] over the edges of row i (G: G_{k+1}, Z: Z_k; and, for
// the recomputed raw scores, G = Q, Z = K, keep = 1/8 on a zeroed A).
template <typename TG, typename TZ>
__global__ void __launch_bounds__(kBwdWarps * 32)
bwd_weight_grad_kernel(BwdArgs a, const TG* __restrict__ G, const TZ* __restrict__ Z,
                       float* __restrict__ dA, float keep) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int64_t u, i;
    if ((int64_t)blockIdx.x >= a.units * a.heavy_rows) {
        // a light row by a quarter-warp: kQB edges a batch, each edge's dot product
        // summed by its lanes' 8 features and then over the quarter (xor butterfly:
        // the same bits in every lane); the edge's own lane updates dA
        const int ql = lane & 7;
        const unsigned qmask = 0xFFu << (lane & 24);
        if (!quarter_item(a, a.row_order, a.heavy_rows, 4 * warp + (lane >> 3), u, i)) return;
        constexpr bool kWide = sizeof(TZ) == 2;
        constexpr int kQB = kWide ? 8 : 4;
        const size_t unit = (size_t)u * a.n * kHeadDim;
        const int64_t e0 = a.row_ptr[i], e1 = a.row_ptr[i + 1];
        int64_t s0, s1;
        row_run(a, i, e0, e1, s0, s1);
        const int64_t len = (e1 - e0) - (s1 - s0);
        float g[8];
        load8<kWide>(G + unit + (size_t)i * kHeadDim, ql, g);
        const TZ* Zu = Z + unit;
        float* dAu = dA + (size_t)u * a.nnz;
        bool okc = ql < kQB && ql < len;
        int64_t ec = rest_pos(e0, ql, s0, s1);
        int32_t jc = okc ? a.col[ec] : 0;
        for (int64_t vb = 0; vb < len; vb += kQB) {
            float z[kQB][8];
#pragma unroll
            for (int b = 0; b < kQB; ++b) {
                const int32_t j = __shfl_sync(qmask, jc, b, 8);
                if (vb + b < len) {
                    load8<kWide>(Zu + (size_t)j * kHeadDim, ql, z[b]);
                } else {
#pragma unroll
                    for (int k = 0; k < 8; ++k) z[b][k] = 0.f;
                }
            }
            const bool okn = ql < kQB && vb + kQB + ql < len;
            const int64_t en = rest_pos(e0, vb + kQB + ql, s0, s1);
            const int32_t jn = okn ? a.col[en] : 0;
            float mine = 0.f;
#pragma unroll
            for (int b = 0; b < kQB; ++b) {
                float d = g[0] * z[b][0];
#pragma unroll
                for (int k = 1; k < 8; ++k) d = fmaf(g[k], z[b][k], d);
                d += __shfl_xor_sync(qmask, d, 1, 8);
                d += __shfl_xor_sync(qmask, d, 2, 8);
                d += __shfl_xor_sync(qmask, d, 4, 8);
                if (ql == b) mine = d;
            }
            if (okc) dAu[ec] += keep * mine;
            okc = okn;
            ec = en;
            jc = jn;
        }
        return;
    }
    edge_item(a, a.row_order, a.heavy_rows, warp, u, i);
    const size_t unit = (size_t)u * a.n * kHeadDim;
    const int64_t e0 = a.row_ptr[i], e1 = a.row_ptr[i + 1];
    int64_t s0, s1;
    row_run(a, i, e0, e1, s0, s1);
    const int64_t len = (e1 - e0) - (s1 - s0);
    int64_t v0, v1;
    heavy_share(len, warp, v0, v1);
    const float2 g = load2(G + unit + (size_t)i * kHeadDim + 2 * lane);
    const TZ* Zu = Z + unit + 2 * lane;
    float* dAu = dA + (size_t)u * a.nnz;
    bool ok = v0 + lane < v1;
    int64_t e = rest_pos(e0, v0 + lane, s0, s1);
    int32_t j_l = ok ? a.col[e] : 0;
    for (int64_t vb = v0; vb < v1; vb += 32) {
        const int cnt = (v1 - vb) < 32 ? (int)(v1 - vb) : 32;
        float p[32];
#pragma unroll
        for (int t = 0; t < 32; ++t) {
            const int32_t j = __shfl_sync(0xffffffffu, j_l, t);
            const float2 z = t < cnt ? load2(Zu + (size_t)j * kHeadDim) : make_float2(0.f, 0.f);
            p[t] = fmaf(g.x, z.x, g.y * z.y);
        }
        const bool ok_c = ok;
        const int64_t e_c = e;
        ok = vb + 32 + lane < v1;
        e = rest_pos(e0, vb + 32 + lane, s0, s1);
        j_l = ok ? a.col[e] : 0;
        const float dot = warp_transpose_sum32(p, lane);             // edge vb + lane
        if (ok_c) dAu[e_c] += keep * dot;
    }
}

// Key j of the transposed hop: Gn[j] = keep * (P[j] + sum_{e = (i, j)} A_e G[i]);
// and dV_acc[j] = (first ? 0 : dV_acc[j]) + alpha G[j].  With dV_out set (k = 0),
// dV_out[j] = dV_acc[j] + alpha G[j] + Gn[j] in the I/O dtype and Gn is not written.
template <typename TG, typename TIo>
__global__ void __launch_bounds__(kBwdWarps * 32)
bwd_hop_t_kernel(BwdArgs a, const float* __restrict__ A, const float* __restrict__ At,
                 const TG* __restrict__ G, const float* __restrict__ P, float* __restrict__ Gn,
                 float* __restrict__ dV_acc, TIo* __restrict__ dV_out, float alpha, bool first) {
    __shared__ float2 part[kBwdWarps][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float keep = 1.f - alpha;
    int64_t u, j;
    if ((int64_t)blockIdx.x >= a.units * a.heavy_keys) {
        const int ql = lane & 7;
        const unsigned qmask = 0xFFu << (lane & 24);
        if (!quarter_item(a, a.key_order, a.heavy_keys, 4 * warp + (lane >> 3), u, j)) return;
        constexpr bool kWide = sizeof(TG) == 2;
        const size_t unit = (size_t)u * a.n * kHeadDim, row = unit + (size_t)j * kHeadDim;
        const float* Au = A + (size_t)u * a.nnz;
        const int64_t t0 = a.t_ptr[j], t1 = a.t_ptr[j + 1];
        int64_t s0, s1;
        key_run(a, j, t0, t1, s0, s1);
        float acc[8];
        if (P) load8<kWide>(P + row, ql, acc);
        else for (int k = 0; k < 8; ++k) acc[k] = 0.f;
        const float* Atj = At ? At + (size_t)u * a.nrest + a.trest[j] : nullptr;
        quarter_sum(ql, qmask, (t1 - t0) - (s1 - s0), G + unit,
                    [&](int64_t v) { return a.t_row[rest_pos(t0, v, s0, s1)]; },
                    [&](int64_t v) { return Atj ? Atj[v] : Au[a.t_edge[rest_pos(t0, v, s0, s1)]]; }, acc);
        float gj[8], dv[8], gn[8];
        load8<kWide>(G + row, ql, gj);
        if (first) for (int k = 0; k < 8; ++k) dv[k] = 0.f;
        else load8<kWide>(dV_acc + row, ql, dv);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            dv[k] = fmaf(alpha, gj[k], dv[k]);
            gn[k] = keep * acc[k];
        }
        if (dV_out) {
#pragma unroll
            for (int k = 0; k < 8; ++k) dv[k] += gn[k];
            store8<kWide>(dV_out + row, ql, dv);
        } else {
            store8<kWide>(dV_acc + row, ql, dv);
            store8<kWide>(Gn + row, ql, gn);
        }
        return;
    }
    edge_item(a, a.key_order, a.heavy_keys, warp, u, j);
    const size_t unit = (size_t)u * a.n * kHeadDim;
    const float* Au = A + (size_t)u * a.nnz;
    const int64_t t0 = a.t_ptr[j], t1 = a.t_ptr[j + 1];
    int64_t s0, s1;
    key_run(a, j, t0, t1, s0, s1);
    const int64_t len = (t1 - t0) - (s1 - s0);
    int64_t v0, v1;
    heavy_share(len, warp, v0, v1);
    const size_t at = unit + (size_t)j * kHeadDim + 2 * lane;
    float2 acc = (P && warp == 0) ? load2(P + at) : make_float2(0.f, 0.f);
    const float* Atj = At ? At + (size_t)u * a.nrest + a.trest[j] : nullptr;
    acc = edge_sum(lane, v0, v1, G + unit + 2 * lane,
                   [&](int64_t v) { return a.t_row[rest_pos(t0, v, s0, s1)]; },
                   [&](int64_t v) { return Atj ? Atj[v] : Au[a.t_edge[rest_pos(t0, v, s0, s1)]]; }, acc);
    if (!heavy_total(part, warp, lane, acc)) return;
    const float2 gj = load2(G + at);
    float2 dv = first ? make_float2(0.f, 0.f) : load2(dV_acc + at);
    dv.x = fmaf(alpha, gj.x, dv.x);
    dv.y = fmaf(alpha, gj.y, dv.y);
    const float2 gn = make_float2(keep * acc.x, keep * acc.y);
    if (dV_out) {
        store2(dV_out + at, make_float2(dv.x + gn.x, dv.y + gn.y));
    } else {
        store2(dV_acc + at, dv);
        store2(Gn + at, gn);
    }
}

// The weights of every key's incoming edges outside its window run, in key order:
// At[u][trest[j] + v] = A_e of the v-th such edge of key j, so that the transposed
// hops read them in sequence instead of through the edge ids.  Heavy keys take a
// CTA each (first), the others a warp each; kU loads in flight per thread.
unsigned weights_t_grid(const BwdArgs& a) {
    return (unsigned)(a.units * a.heavy_keys + (a.units * (a.n - a.heavy_keys) + kBwdWarps - 1) / kBwdWarps);
}
__global__ void __launch_bounds__(kBwdWarps * 32)
bwd_weights_t_kernel(BwdArgs a, const float* __restrict__ A, float* __restrict__ At) {
    constexpr int kU = 4;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t hb = a.units * a.heavy_keys;
    int64_t u, j;
    int first, stride;
    if ((int64_t)blockIdx.x < hb) {
        const int64_t rk = blockIdx.x / a.units;
        u = blockIdx.x - rk * a.units;
        j = a.key_order[rk];
        first = threadIdx.x;
        stride = kBwdWarps * 32;
    } else {
        const int64_t item = ((int64_t)blockIdx.x - hb) * kBwdWarps + warp, rest = a.n - a.heavy_keys;
        if (rest <= 0 || item >= a.units * rest) return;
        u = item / rest;
        j = a.key_order[a.heavy_keys + (item - u * rest)];
        first = lane;
        stride = 32;
    }
    const float* Au = A + (size_t)u * a.nnz;
    float* Atj = At + (size_t)u * a.nrest + a.trest[j];
    const int64_t t0 = a.t_ptr[j], t1 = a.t_ptr[j + 1];
    int64_t s0, s1;
    key_run(a, j, t0, t1, s0, s1);
    const int64_t len = (t1 - t0) - (s1 - s0);
    for (int64_t vb = first; vb < len; vb += (int64_t)kU * stride) {
        float w[kU];
#pragma unroll
        for (int q = 0; q < kU; ++q) {
            const int64_t v = vb + (int64_t)q * stride;
            w[q] = v < len ? Au[a.t_edge[rest_pos(t0, v, s0, s1)]] : 0.f;
        }
#pragma unroll
        for (int q = 0; q < kU; ++q) {
            const int64_t v = vb + (int64_t)q * stride;
            if (v < len) Atj[v] = w[q];
        }
    }
}

// Row i: the recomputed weights A_e = exp(s_e - m_i) / sum_t exp(s_t - m_i) from
// the raw scores s in A (in place), m_i the row's largest score.
__global__ void __launch_bounds__(kBwdWarps * 32)
bwd_scores_softmax_kernel(BwdArgs a, float* __restrict__ A) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * kBwdWarps + (threadIdx.x >> 5);
    if (gw >= a.units * a.n) return;
    int64_t u, i;
    warp_item(a, gw, a.row_order, a.heavy_rows, u, i);
    float* Au = A + (size_t)u * a.nnz;
    const int64_t e0 = a.row_ptr[i], e1 = a.row_ptr[i + 1];
    float m = -INFINITY;
    for (int64_t e = e0 + lane; e < e1; e += 32) m = fmaxf(m, Au[e]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float l = 0.f;
    for (int64_t e = e0 + lane; e < e1; e += 32) l += expf(Au[e] - m);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
    for (int64_t e = e0 + lane; e < e1; e += 32) Au[e] = expf(Au[e] - m) / l;
}

// Row i: dS_e = A_e (dA_e - sum_t A_t dA_t) * scale, in place over dA.
__global__ void __launch_bounds__(kBwdWarps * 32)
bwd_softmax_kernel(BwdArgs a, const float* __restrict__ A, float* __restrict__ dA) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * kBwdWarps + (threadIdx.x >> 5);
    if (gw >= a.units * a.n) return;
    int64_t u, i;
    warp_item(a, gw, a.row_order, a.heavy_rows, u, i);
    const float* Au = A + (size_t)u * a.nnz;
    float* dAu = dA + (size_t)u * a.nnz;
    const int64_t e0 = a.row_ptr[i], e1 = a.row_ptr[i + 1];
    float dot = 0.f;
    for (int64_t e = e0 + lane; e < e1; e += 32) dot = fmaf(Au[e], dAu[e], dot);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    for (int64_t e = e0 + lane; e < e1; e += 32) dAu[e] = Au[e] * (dAu[e] - dot) * kScale;
}

// Row i: out[i] = P[i] + sum_e W_e X[j] in the I/O dtype (dQ = dS K).
template <typename TIo>
__global__ void __launch_bounds__(kBwdWarps * 32)
bwd_rows_out_kernel(BwdArgs a, const float* __restrict__ W, const TIo* __restrict__ X,
                    const float* __restrict__ P, TIo* __restrict__ out) {
    __shared__ float2 part[kBwdWarps][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int64_t u, i;
    if ((int64_t)blockIdx.x >= a.units * a.heavy_rows) {
        const int ql = lane & 7;
        const unsigned qmask = 0xFFu << (lane & 24);
        if (!quarter_item(a, a.row_order, a.heavy_rows, 4 * warp + (lane >> 3), u, i)) return;
        constexpr bool kWide = sizeof(TIo) == 2;
        const size_t unit = (size_t)u * a.n * kHeadDim, row = unit + (size_t)i * kHeadDim;
        const float* Wu = W + (size_t)u * a.nnz;
        const int64_t e0 = a.row_ptr[i], e1 = a.row_ptr[i + 1];
        int64_t s0, s1;
        row_run(a, i, e0, e1, s0, s1);
        float acc[8];
        if (P) load8<kWide>(P + row, ql, acc);
        else for (int k = 0; k < 8; ++k) acc[k] = 0.f;
        quarter_sum(ql, qmask, (e1 - e0) - (s1 - s0), X + unit,
                    [&](int64_t v) { return a.col[rest_pos(e0, v, s0, s1)]; },
                    [&](int64_t v) { return Wu[rest_pos(e0, v, s0, s1)]; }, acc);
        store8<kWide>(out + row, ql, acc);
        return;
    }
    edge_item(a, a.row_order, a.heavy_rows, warp, u, i);
    const size_t unit = (size_t)u * a.n * kHeadDim;
    const float* Wu = W + (size_t)u * a.nnz;
    const int64_t e0 = a.row_ptr[i], e1 = a.row_ptr[i + 1];
    int64_t s0, s1;
    row_run(a, i, e0, e1, s0, s1);
    const int64_t len = (e1 - e0) - (s1 - s0);
    int64_t v0, v1;
    heavy_share(len, warp, v0, v1);
    const size_t at = unit + (size_t)i * kHeadDim + 2 * lane;
    float2 acc = (P && warp == 0) ? load2(P + at) : make_float2(0.f, 0.f);
    acc = edge_sum(lane, v0, v1, X + unit + 2 * lane,
                   [&](int64_t v) { return a.col[rest_pos(e0, v, s0, s1)]; },
                   [&](int64_t v) { return Wu[rest_pos(e0, v, s0, s1)]; }, acc);
    if (!heavy_total(part, warp, lane, acc)) return;
    store2(out + at, acc);
}

// Key j: dK_j = P[j] + sum_{e = (i, j)} dS_e Q[i] in the I/O dtype.
template <typename TIo>
__global__ void __launch_bounds__(kBwdWarps * 32)
bwd_dk_kernel(BwdArgs a, const float* __restrict__ dS, const TIo* __restrict__ Q,
              const float* __restrict__ P, TIo* __restrict__ dK) {
    __shared__ float2 part[kBwdWarps][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int64_t u, j;
    if ((int64_t)blockIdx.x >= a.units * a.heavy_keys) {
        const int ql = lane & 7;
        const unsigned qmask = 0xFFu << (lane & 24);
        if (!quarter_item(a, a.key_order, a.heavy_keys, 4 * warp + (lane >> 3), u, j)) return;
        constexpr bool kWide = sizeof(TIo) == 2;
        const size_t unit = (size_t)u * a.n * kHeadDim, row = unit + (size_t)j * kHeadDim;
        const float* dSu = dS + (size_t)u * a.nnz;
        const int64_t t0 = a.t_ptr[j], t1 = a.t_ptr[j + 1];
        int64_t s0, s1;
        key_run(a, j, t0, t1, s0, s1);
        float acc[8];
        if (P) load8<kWide>(P + row, ql, acc);
        else for (int k = 0; k < 8; ++k) acc[k] = 0.f;
        quarter_sum(ql, qmask, (t1 - t0) - (s1 - s0), Q + unit,
                    [&](int64_t v) { return a.t_row[rest_pos(t0, v, s0, s1)]; },
                    [&](int64_t v) { return dSu[a.t_edge[rest_pos(t0, v, s0, s1)]]; }, acc);
        store8<kWide>(dK + row, ql, acc);
        return;
    }
    edge_item(a, a.key_order, a.heavy_keys, warp, u, j);
    const size_t unit = (size_t)u * a.n * kHeadDim;
    const float* dSu = dS + (size_t)u * a.nnz;
    const int64_t t0 = a.t_ptr[j], t1 = a.t_ptr[j + 1];
    int64_t s0, s1;
    key_run(a, j, t0, t1, s0, s1);
    const int64_t len = (t1 - t0) - (s1 - s0);
    int64_t v0, v1;
    heavy_share(len, warp, v0, v1);
    const size_t at = unit + (size_t)j * kHeadDim + 2 * lane;
    float2 acc = (P && warp == 0) ? load2(P + at) : make_float2(0.f, 0.f);
    acc = edge_sum(lane, v0, v1, Q + unit + 2 * lane,
                   [&](int64_t v) { return a.t_row[rest_pos(t0, v, s0, s1)]; },
                   [&](int64_t v) { return dSu[a.t_edge[rest_pos(t0, v, s0, s1)]]; }, acc);
    if (!heavy_total(part, warp, lane, acc)) return;
    store2(dK + at, acc);
}

unsigned bwd_grid(const BwdArgs& a) {
    return (unsigned)((a.units * a.n + kBwdWarps - 1) / kBwdWarps);
}

int launched(const char* what) {
    const cudaError_t err = cudaGetLastError();
    return err == cudaSuccess ? DIFFUSER_OK : cuda_fail(err, what);
}

template <typename TIo>
int backward_typed(const BwdArgs& a, const CsrArgs& ca, const TIo* Q,
                   const TIo* K, const TIo* V, const TIo* dOut, int32_t dtype, int32_t hops,
                   float alpha, TIo* dQ, TIo* dK, TIo* dV, char* ws, const BwdLayout& L,
                   cudaStream_t stream) {
    const dim3 grid(bwd_grid(a)), block(kBwdWarps * 32);
    const dim3 qrgrid(quarter_grid(a, a.heavy_rows)), qkgrid(quarter_grid(a, a.heavy_keys));   // the products
    const bool band = a.wp0 != nullptr || a.bptr != nullptr;
    const dim3 bgrid((unsigned)(a.units * ((a.n + kTile - 1) / kTile)));
    const size_t io = (size_t)a.units * a.n * kHeadDim * sizeof(TIo);
    float* A = reinterpret_cast<float*>(ws + L.a);
    float* dA = reinterpret_cast<float*>(ws + L.da);
    float* dVacc = reinterpret_cast<float*>(ws + L.dv);
    float* P = band ? reinterpret_cast<float*>(ws + L.p) : nullptr;   // the band kernels' window sums
    float* At = a.trest ? reinterpret_cast<float*>(ws + L.at) : nullptr;   // key-ordered weights
    float* Gbuf[2] = {reinterpret_cast<float*>(ws + L.g[0]), reinterpret_cast<float*>(ws + L.g[1])};
    auto zstate = [&](int32_t k) { return reinterpret_cast<float*>(ws + L.z + (size_t)(k - 1) * L.z_stride); };
    cudaError_t err;
    int st;
    if (hops == 0) {
        // Z_K = V: dV = dOut, and nothing reaches the weights
        err = cudaMemcpyAsync(dV, dOut, io, cudaMemcpyDeviceToDevice, stream);
        if (err == cudaSuccess) err = cudaMemsetAsync(dQ, 0, io, stream);
        if (err == cudaSuccess) err = cudaMemsetAsync(dK, 0, io, stream);
        return err == cudaSuccess ? DIFFUSER_OK : cuda_fail(err, "backward with hops = 0");
    }
    // one launch scope per kernel (the launch counters and per-kernel events)
    auto hop = [&](auto&& launch) { LaunchScope scope(DIFFUSER_KERNEL_HOP, stream); launch(); };
    auto score = [&](auto&& launch) { LaunchScope scope(DIFFUSER_KERNEL_SCORE, stream); launch(); };
    // the forward's weights (on the band path: raw scores of the window runs as
    // tiles, of the other edges by the CSR kernel, then each row's softmax) and
    // states Z_1 .. Z_{K-1} (Z_0 is V)
    if (band) {
        err = cudaMemsetAsync(A, 0, (size_t)a.units * a.nnz * sizeof(float), stream);
        if (err != cudaSuccess) return cuda_fail(err, "clearing A");
        score([&] { band_sddmm<TIo, TIo>(a, bgrid, stream, Q, K, A, kScale); });
        score([&] { bwd_weight_grad_kernel<TIo, TIo><<<qrgrid, block, 0, stream>>>(a, Q, K, A, kScale); });
        score([&] { bwd_scores_softmax_kernel<<<grid, block, 0, stream>>>(a, A); });
        if ((st = launched("bwd_scores_softmax_kernel"))) return st;
        if (At) {
            score([&] { bwd_weights_t_kernel<<<weights_t_grid(a), block, 0, stream>>>(a, A, At); });
            if ((st = launched("bwd_weights_t_kernel"))) return st;
        }
    } else if ((st = launch_score_csr(ca, Q, K, dtype, A, stream))) {
        return st;
    }
    for (int32_t k = 1; k < hops; ++k) {
        if (k == 1) {
            if (band) hop([&] { band_rows(a, bgrid, stream, A, V, P); });
            hop([&] { bwd_hop_rows_kernel<TIo, TIo><<<qrgrid, block, 0, stream>>>(a, A, V, P, V, zstate(k), alpha); });
        } else {
            if (band) hop([&] { band_rows(a, bgrid, stream, A, zstate(k - 1), P); });
            hop([&] {
                bwd_hop_rows_kernel<float, TIo><<<qrgrid, block, 0, stream>>>(a, A, zstate(k - 1), P, V, zstate(k), alpha);
            });
        }
        if ((st = launched("bwd_hop_rows_kernel"))) return st;
    }
    err = cudaMemsetAsync(dA, 0, (size_t)a.units * a.nnz * sizeof(float), stream);
    if (err != cudaSuccess) return cuda_fail(err, "clearing dA");
    const float keep = 1.f - alpha;
    for (int32_t k = hops - 1; k >= 0; --k) {
        const bool top = (k == hops - 1);            // G_{k+1} is dOut itself
        float* Gn = Gbuf[k & 1];
        const float* Gf = Gbuf[(k + 1) & 1];         // G_{k+1} for k < hops - 1
        if (top && k == 0) {
            if (band) hop([&] { band_sddmm<TIo, TIo>(a, bgrid, stream, dOut, V, dA, keep); });
            hop([&] { bwd_weight_grad_kernel<TIo, TIo><<<qrgrid, block, 0, stream>>>(a, dOut, V, dA, keep); });
        } else if (top) {
            if (band)
                hop([&] { band_sddmm<TIo, float>(a, bgrid, stream, dOut, zstate(k), dA, keep); });
            hop([&] { bwd_weight_grad_kernel<TIo, float><<<qrgrid, block, 0, stream>>>(a, dOut, zstate(k), dA, keep); });
        } else if (k == 0) {
            if (band) hop([&] { band_sddmm<float, TIo>(a, bgrid, stream, Gf, V, dA, keep); });
            hop([&] { bwd_weight_grad_kernel<float, TIo><<<qrgrid, block, 0, stream>>>(a, Gf, V, dA, keep); });
        } else {
            if (band)
                hop([&] { band_sddmm<float, float>(a, bgrid, stream, Gf, zstate(k), dA, keep); });
            hop([&] { bwd_weight_grad_kernel<float, float><<<qrgrid, block, 0, stream>>>(a, Gf, zstate(k), dA, keep); });
        }
        if ((st = launched("bwd_weight_grad_kernel"))) return st;
        TIo* out = k == 0 ? dV : nullptr;
        if (top) {
            if (band) hop([&] { band_keys(a, bgrid, stream, A, dOut, P); });
            hop([&] {
                bwd_hop_t_kernel<TIo, TIo><<<qkgrid, block, 0, stream>>>(a, A, At, dOut, P, Gn, dVacc, out, alpha, true);
            });
        } else {
            if (band) hop([&] { band_keys(a, bgrid, stream, A, Gf, P); });
            hop([&] {
                bwd_hop_t_kernel<float, TIo><<<qkgrid, block, 0, stream>>>(a, A, At, Gf, P, Gn, dVacc, out, alpha, false);
            });
        }
        if ((st = launched("bwd_hop_t_kernel"))) return st;
    }
    score([&] { bwd_softmax_kernel<<<grid, block, 0, stream>>>(a, A, dA); });
    if (band) score([&] { band_rows(a, bgrid, stream, dA, K, P); });
    score([&] { bwd_rows_out_kernel<TIo><<<qrgrid, block, 0, stream>>>(a, dA, K, P, dQ); });
    if ((st = launched("bwd_rows_out_kernel"))) return st;
    if (band) score([&] { band_keys(a, bgrid, stream, dA, Q, P); });
    score([&] { bwd_dk_kernel<TIo><<<qkgrid, block, 0, stream>>>(a, dA, Q, P, dK); });
    return launched("bwd_dk_kernel");
}

}  // namespace

// The window runs of a token graph with a plain window: wp0[i], the CSR position
// of key lo(i) in row i, and tw0[j], the transposed-list position of row lo'(j)
// in key j's list (the same bounds as win_row / win_key).  False, and nothing
// kept, unless every run holds consecutive keys (rows).
bool window_runs(const diffuser_graph* g, const std::vector<int64_t>& t_ptr,
                 const std::vector<int32_t>& t_row, std::vector<int64_t>& wp0, std::vector<int64_t>& tw0) {
    if (g->kind != kTokenGraph || g->dilation != 1 || g->n < 1) return false;
    const int64_t n = g->n, r = g->r;
    wp0.assign((size_t)n, 0);
    tw0.assign((size_t)n, 0);
    for (int64_t i = 0; i < n; ++i) {
        const int64_t lo = i - r > 0 ? i - r : 0, hi = g->causal ? i : std::min(i + r, n - 1);
        const int32_t* b = g->h_col.data() + g->h_row_ptr[i];
        const int32_t* e = g->h_col.data() + g->h_row_ptr[i + 1];
        const int32_t* at = std::lower_bound(b, e, (int32_t)lo);
        if (e - at < hi - lo + 1) return false;
        for (int64_t k = 0; k <= hi - lo; ++k)
            if (at[k] != lo + k) return false;
        wp0[(size_t)i] = at - g->h_col.data();
    }
    for (int64_t j = 0; j < n; ++j) {
        const int64_t lo = g->causal ? j : (j - r > 0 ? j - r : 0), hi = std::min(j + r, n - 1);
        const int32_t* b = t_row.data() + t_ptr[(size_t)j];
        const int32_t* e = t_row.data() + t_ptr[(size_t)j + 1];
        const int32_t* at = std::lower_bound(b, e, (int32_t)lo);
        if (e - at < hi - lo + 1) return false;
        for (int64_t k = 0; k <= hi - lo; ++k)
            if (at[k] != lo + k) return false;
        tw0[(size_t)j] = at - t_row.data();
    }
    return true;
}

// The key-block runs of a block graph of 64-token blocks: every row of block row J
// holds the keys of its key blocks, ascending, each block as one run of 64 (the
// ragged last block fewer), the same for all its rows.  runs = [bptr (nb + 1) |
// bcol | btptr (nb + 1) | btrow | btpos]: block row J's key blocks, and for key
// block KB the row blocks holding it with its place in their lists.  False, and
// nothing kept, unless every row has exactly that form.
bool block_runs(const diffuser_graph* g, std::vector<int32_t>& runs) {
    if (g->kind != kBlockGraph || g->block != kTile || g->n < 1) return false;
    const int64_t n = g->n, nb = (n + kTile - 1) / kTile;
    std::vector<std::vector<int32_t>> allowed((size_t)nb);
    for (int64_t J = 0; J < nb; ++J) {
        const int64_t i = J * kTile;
        for (int64_t e = g->h_row_ptr[i]; e < g->h_row_ptr[i + 1]; ++e) {
            const int32_t kb = g->h_col[e] / kTile;
            if (allowed[(size_t)J].empty() || allowed[(size_t)J].back() != kb) allowed[(size_t)J].push_back(kb);
        }
        for (int64_t r = i; r < std::min(i + kTile, n); ++r) {
            int64_t e = g->h_row_ptr[r];
            for (int32_t kb : allowed[(size_t)J]) {
                const int64_t k0 = (int64_t)kb * kTile, k1 = std::min(k0 + kTile, n);
                for (int64_t j = k0; j < k1; ++j, ++e)
                    if (e >= g->h_row_ptr[r + 1] || g->h_col[e] != j) return false;
            }
            if (e != g->h_row_ptr[r + 1]) return false;
        }
    }
    std::vector<int32_t> bptr((size_t)nb + 1, 0), bcol, btptr((size_t)nb + 1, 0);
    for (int64_t J = 0; J < nb; ++J) {
        bcol.insert(bcol.end(), allowed[(size_t)J].begin(), allowed[(size_t)J].end());
        bptr[(size_t)J + 1] = (int32_t)bcol.size();
        for (int32_t kb : allowed[(size_t)J]) ++btptr[(size_t)kb + 1];
    }
    for (int64_t KB = 0; KB < nb; ++KB) btptr[(size_t)KB + 1] += btptr[(size_t)KB];
    std::vector<int32_t> btrow(bcol.size()), btpos(bcol.size());
    std::vector<int32_t> fill(btptr.begin(), btptr.end() - 1);
    for (int64_t J = 0; J < nb; ++J)
        for (size_t x = 0; x < allowed[(size_t)J].size(); ++x) {
            const int32_t at = fill[(size_t)allowed[(size_t)J][x]]++;
            btrow[(size_t)at] = (int32_t)J;
            btpos[(size_t)at] = (int32_t)x;
        }
    runs.clear();
    for (auto* v : {&bptr, &bcol, &btptr, &btrow, &btpos}) runs.insert(runs.end(), v->begin(), v->end());
    return true;
}

// The edges outside the window runs of a token graph with a plain window (its nnz
// less the window's pairs: row i's window holds the keys max(i - r, 0) ..
// min(i + r, n - 1), .. i when causal); 0 on other graphs.
int64_t window_rest(const diffuser_graph* g) {
    if (g->kind != kTokenGraph || g->dilation != 1) return 0;
    int64_t pairs = 0;
    for (int64_t i = 0; i < g->n; ++i) {
        const int64_t lo = i - g->r > 0 ? i - g->r : 0;
        const int64_t hi = g->causal ? i : std::min<int64_t>(i + g->r, g->n - 1);
        pairs += hi - lo + 1;
    }
    return g->nnz > pairs ? g->nnz - pairs : 0;
}

// The transposed graph (incoming edges of every key, rows ascending), built on
// the host from the CSR copy by a counting sort and uploaded (synchronously),
// with the window runs where the graph has them.  On failure the arrays
// allocated so far are freed and d_t_ptr stays null.
int build_transposed_graph(diffuser_graph* g) {
    const int64_t n = g->n, nnz = g->nnz;
    std::vector<int64_t> t_ptr(n + 1, 0);
    for (int64_t e = 0; e < nnz; ++e) ++t_ptr[g->h_col[e] + 1];
    for (int64_t j = 0; j < n; ++j) t_ptr[j + 1] += t_ptr[j];
    std::vector<int32_t> t_row(nnz > 0 ? nnz : 1);
    std::vector<int64_t> t_edge(nnz > 0 ? nnz : 1);
    std::vector<int64_t> fill(t_ptr.begin(), t_ptr.end() - 1);
    for (int64_t i = 0; i < n; ++i) {
        for (int64_t e = g->h_row_ptr[i]; e < g->h_row_ptr[i + 1]; ++e) {
            const int64_t at = fill[g->h_col[e]]++;
            t_row[at] = (int32_t)i;
            t_edge[at] = e;
        }
    }
    std::vector<int64_t> wp0, tw0;
    bool runs = window_runs(g, t_ptr, t_row, wp0, tw0);
    // where key j's incoming edges outside its window run start in the key-ordered
    // weights; their total must be the count the workspace was sized by
    std::vector<int64_t> trest;
    if (runs) {
        trest.assign((size_t)n + 1, 0);
        for (int64_t j = 0; j < n; ++j) {
            const int64_t lo = g->causal ? j : (j - g->r > 0 ? j - g->r : 0);
            const int64_t hi = std::min<int64_t>(j + g->r, n - 1);
            trest[(size_t)j + 1] = trest[(size_t)j] + (t_ptr[(size_t)j + 1] - t_ptr[(size_t)j]) - (hi - lo + 1);
        }
        if (trest[(size_t)n] != window_rest(g)) runs = false;
    }
    std::vector<int32_t> bruns;
    const bool blk = block_runs(g, bruns);
    // the heavy rows (keys): more than twice the mean edge count, heaviest first
    // (ties: ascending index), then the others in ascending order
    auto order_of = [&](auto len, std::vector<int32_t>& order) -> int64_t {
        std::vector<int32_t> heavy, light;
        for (int64_t i = 0; i < n; ++i) (len(i) * n > 2 * nnz ? heavy : light).push_back((int32_t)i);
        std::stable_sort(heavy.begin(), heavy.end(), [&](int32_t x, int32_t y) { return len(x) > len(y); });
        order = heavy;
        order.insert(order.end(), light.begin(), light.end());
        return (int64_t)heavy.size();
    };
    std::vector<int32_t> row_order, key_order;
    const int64_t heavy_rows = order_of([&](int64_t i) { return g->h_row_ptr[i + 1] - g->h_row_ptr[i]; }, row_order);
    const int64_t heavy_keys = order_of([&](int64_t j) { return t_ptr[(size_t)j + 1] - t_ptr[(size_t)j]; }, key_order);
    int64_t* d_ptr = nullptr;
    int32_t* d_row = nullptr;
    int64_t* d_edge = nullptr;
    int64_t* d_wp0 = nullptr;
    int64_t* d_tw0 = nullptr;
    int64_t* d_trest = nullptr;
    int32_t* d_orders = nullptr;             // [2][n]: row_order, key_order
    int32_t* d_bruns = nullptr;
    cudaError_t err = cudaMalloc(&d_ptr, sizeof(int64_t) * (n + 1));
    if (err == cudaSuccess) err = cudaMalloc(&d_orders, sizeof(int32_t) * 2 * (size_t)n);
    if (err == cudaSuccess)
        err = cudaMemcpy(d_orders, row_order.data(), sizeof(int32_t) * (size_t)n, cudaMemcpyHostToDevice);
    if (err == cudaSuccess)
        err = cudaMemcpy(d_orders + n, key_order.data(), sizeof(int32_t) * (size_t)n, cudaMemcpyHostToDevice);
    if (err == cudaSuccess) err = cudaMalloc(&d_row, sizeof(int32_t) * t_row.size());
    if (err == cudaSuccess) err = cudaMalloc(&d_edge, sizeof(int64_t) * t_edge.size());
    if (err == cudaSuccess)
        err = cudaMemcpy(d_ptr, t_ptr.data(), sizeof(int64_t) * (n + 1), cudaMemcpyHostToDevice);
    if (err == cudaSuccess)
        err = cudaMemcpy(d_row, t_row.data(), sizeof(int32_t) * t_row.size(), cudaMemcpyHostToDevice);
    if (err == cudaSuccess)
        err = cudaMemcpy(d_edge, t_edge.data(), sizeof(int64_t) * t_edge.size(), cudaMemcpyHostToDevice);
    if (runs) {
        if (err == cudaSuccess) err = cudaMalloc(&d_wp0, sizeof(int64_t) * (size_t)n);
        if (err == cudaSuccess) err = cudaMalloc(&d_tw0, sizeof(int64_t) * (size_t)n);
        if (err == cudaSuccess)
            err = cudaMemcpy(d_wp0, wp0.data(), sizeof(int64_t) * (size_t)n, cudaMemcpyHostToDevice);
        if (err == cudaSuccess)
            err = cudaMemcpy(d_tw0, tw0.data(), sizeof(int64_t) * (size_t)n, cudaMemcpyHostToDevice);
        if (err == cudaSuccess) err = cudaMalloc(&d_trest, sizeof(int64_t) * ((size_t)n + 1));
        if (err == cudaSuccess)
            err = cudaMemcpy(d_trest, trest.data(), sizeof(int64_t) * ((size_t)n + 1), cudaMemcpyHostToDevice);
    }
    if (blk) {
        if (err == cudaSuccess) err = cudaMalloc(&d_bruns, sizeof(int32_t) * bruns.size());
        if (err == cudaSuccess)
            err = cudaMemcpy(d_bruns, bruns.data(), sizeof(int32_t) * bruns.size(), cudaMemcpyHostToDevice);
    }
    if (err != cudaSuccess) {
        cudaFree(d_ptr);
        cudaFree(d_row);
        cudaFree(d_edge);
        cudaFree(d_wp0);
        cudaFree(d_tw0);
        cudaFree(d_trest);
        cudaFree(d_orders);
        cudaFree(d_bruns);
        return cuda_fail(err, "building the transposed graph");
    }
    g->d_orders = d_orders;
    g->d_bruns = d_bruns;
    g->bruns_blocks = blk ? ((int64_t)bruns.size() - 2 * ((n + kTile - 1) / kTile + 1)) / 3 : 0;   // bcol entries
    g->heavy_rows = heavy_rows;
    g->heavy_keys = heavy_keys;
    g->d_wp0 = d_wp0;
    g->d_tw0 = d_tw0;
    g->d_trest = d_trest;
    g->d_t_row = d_row;
    g->d_t_edge = d_edge;
    g->d_t_ptr = d_ptr;      // set last: non-null means the transposed graph is complete
    return DIFFUSER_OK;
}

int plan_backward_layout(const diffuser_graph* g, int64_t units, int32_t hops, BwdLayout* L) {
    // A, dA: [units][nnz] fp32; dV_acc, G (x2), the band kernels' window sums P,
    // Z_1 .. Z_{K-1}: [units][n][64] fp32; the weights outside the window runs in
    // key order: [units][nrest] fp32
    const int64_t nrest = window_rest(g);
    const double states = 4.0 + (hops > 1 ? hops - 1 : 0);
    const double need = (double)units * (2.0 * 4.0 * (double)g->nnz + 4.0 * (double)nrest +
                                         states * 4.0 * kHeadDim * (double)g->n);
    if (need > 4.0e18) return fail(DIFFUSER_ERR_OVERFLOW, "backward workspace size overflows size_t");
    auto al = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t U = (size_t)units, state = al(U * (size_t)g->n * kHeadDim * sizeof(float));
    const size_t edges = al(U * (size_t)g->nnz * sizeof(float));
    size_t off = 0;
    L->a = off; off += edges;
    L->da = off; off += edges;
    L->dv = off; off += state;
    L->g[0] = off; off += state;
    L->g[1] = off; off += state;
    L->p = off; off += state;
    L->at = off; off += al(U * (size_t)nrest * sizeof(float));
    L->nrest = nrest;
    L->z = off;
    L->z_stride = state;
    off += (hops > 1 ? (size_t)(hops - 1) : 0) * state;
    L->total = off;
    return DIFFUSER_OK;
}

int launch_backward_csr(const diffuser_graph* g, int64_t units, const void* Q, const void* K,
                        const void* V, const void* dOut, int32_t dtype, int32_t hops, float alpha,
                        void* dQ, void* dK, void* dV, char* ws, const BwdLayout& L, bool band,
                        cudaStream_t stream) {
    const bool runs = band && g->d_wp0 && g->d_tw0;
    const bool blk = band && g->d_bruns;
    const int64_t nb = (g->n + kTile - 1) / kTile, m = g->bruns_blocks;
    const int32_t* br = g->d_bruns;
    BwdArgs a{g->d_row_ptr, g->d_col, g->d_t_ptr, g->d_t_row, g->d_t_edge,
              runs ? g->d_wp0 : nullptr, runs ? g->d_tw0 : nullptr,
              blk ? br : nullptr, blk ? br + nb + 1 : nullptr, blk ? br + nb + 1 + m : nullptr,
              blk ? br + 2 * (nb + 1) + m : nullptr, blk ? br + 2 * (nb + 1) + 2 * m : nullptr,
              g->d_orders, g->d_orders + g->n,
              g->heavy_rows, g->heavy_keys, g->n, g->nnz, units, g->r, g->causal ? 1 : 0,
              runs && g->d_trest && L.nrest > 0 ? g->d_trest : nullptr, L.nrest};
    CsrArgs ca{g->d_row_ptr, g->d_col, g->n, g->nnz, units};
    if (dtype == DIFFUSER_DTYPE_BF16) {
        using T = __nv_bfloat16;
        return backward_typed<T>(a, ca, static_cast<const T*>(Q), static_cast<const T*>(K),
                                 static_cast<const T*>(V), static_cast<const T*>(dOut), dtype, hops,
                                 alpha, static_cast<T*>(dQ), static_cast<T*>(dK), static_cast<T*>(dV),
                                 ws, L, stream);
    }
    return backward_typed<float>(a, ca, static_cast<const float*>(Q), static_cast<const float*>(K),
                                 static_cast<const float*>(V), static_cast<const float*>(dOut), dtype,
                                 hops, alpha, static_cast<float*>(dQ), static_cast<float*>(dK),
                                 static_cast<float*>(dV), ws, L, stream);
}

}  // namespace dfs
