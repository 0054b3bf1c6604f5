// Scores and masked softmax for the band path ("Diffuser: modelling long
// sequences with multi-hop attention diffusion", eq S.1-S.5; "1.2.1 Static
// sparsity", eq 1-3), in four kernels:
//
//  * score_sparse_kernel: per row, the raw scores q_i.k_j/8 of the globals
//    outside the window (-inf inside it) and of the random extras, and their
//    maximum; a quarter-warp per row, each K row read as one 128-byte line,
//    8 dot products reduced across the quarter at once.  Per tile, the raw
//    scores of the global rows against the tile's keys with per-tile
//    (max, sum of exp).
//  * score_band_tc_kernel (tcgen05, persistent): S = Q K^T for a 128-row
//    tile against 64-key chunks of its window on bf16 tensor cores (fp32
//    accumulation in TMEM), in two passes over the chunks: the row maximum
//    m_i (band and sparse), then e = exp(s - m_i) written as the tile's
//    operand image, and the band part of the row sum.
//  * score_global_norm_kernel: merges the per-tile statistics into the global
//    rows' (max, 1/sum), normalizes their weights and writes each tile's
//    global-row operand image.
//  * score_finalize_kernel: a warp per row turns the sparse raw scores into
//    e = exp(s - m_i) (the out-of-window globals' as a tensor-core operand
//    image) and stores inv_l = 1 / (band sum + sparse sum).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "band_common.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace dfs {
namespace {

using band::bf16hi;
using band::bf16lo;
using band::kTileRows;

constexpr float kScale = 0.125f;   // 1/sqrt(64), exact

struct ScoreArgs {
    BandPlan plan;
    int64_t units;
    band::GraphRefs gr;
    band::Weights w;
    int* counters;      // [units] tile tickets
};

__device__ __forceinline__ void load_row64(const __nv_bfloat16* p, float (&x)[64]) {
    const uint4* v = reinterpret_cast<const uint4*>(p);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 w = __ldg(v + c);
        x[8 * c + 0] = bf16lo(w.x); x[8 * c + 1] = bf16hi(w.x);
        x[8 * c + 2] = bf16lo(w.y); x[8 * c + 3] = bf16hi(w.y);
        x[8 * c + 4] = bf16lo(w.z); x[8 * c + 5] = bf16hi(w.z);
        x[8 * c + 6] = bf16lo(w.w); x[8 * c + 7] = bf16hi(w.w);
    }
}


// ---------------------------------------------------------------- sparse scores
constexpr int kSparseThreads = 256;

// v[b] (b < 8) are this lane's partial sums of slot b; afterwards v[0] on
// lane l of the 8-lane group is the full sum of slot l (butterfly transpose).
__device__ __forceinline__ float reduce8_transpose(float (&v)[8], int ql, unsigned mask) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const bool up = ql & 4;
        const float send = up ? v[b] : v[b + 4];
        const float keep = up ? v[b + 4] : v[b];
        v[b] = keep + __shfl_xor_sync(mask, send, 4, 8);
    }
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        const bool up = ql & 2;
        const float send = up ? v[b] : v[b + 2];
        const float keep = up ? v[b + 2] : v[b];
        v[b] = keep + __shfl_xor_sync(mask, send, 2, 8);
    }
    const bool up = ql & 1;
    const float send = up ? v[0] : v[1];
    const float keep = up ? v[1] : v[0];
    return keep + __shfl_xor_sync(mask, send, 1, 8);
}

__device__ __forceinline__ void unpack8(const uint4& w, float (&x)[8]) {
    x[0] = bf16lo(w.x); x[1] = bf16hi(w.x); x[2] = bf16lo(w.y); x[3] = bf16hi(w.y);
    x[4] = bf16lo(w.z); x[5] = bf16hi(w.z); x[6] = bf16lo(w.w); x[7] = bf16hi(w.w);
}

__global__ void __launch_bounds__(kSparseThreads, 2)
score_sparse_kernel(ScoreArgs a, const __nv_bfloat16* __restrict__ Q,
                    const __nv_bfloat16* __restrict__ K) {
    __shared__ float4 sQG[kBandMaxGlobals * 16];   // q rows of the global positions (fp32)
    __shared__ float4 sKG[kBandMaxGlobals * 16];   // k rows of the global positions (fp32)
    __shared__ float scr[kBandMaxGlobals * kTileRows];   // the global rows' scores of this tile's keys
    const BandPlan& P = a.plan;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t u = blockIdx.x / P.tiles;
    const int tile = (int)(blockIdx.x - u * P.tiles);
    const int64_t i0 = (int64_t)tile * kTileRows;
    const int g = P.g;
    const __nv_bfloat16* Qu = Q + (size_t)u * P.n * kHeadDim;
    const __nv_bfloat16* Ku = K + (size_t)u * P.n * kHeadDim;
    for (int e = tid; e < g * 8; e += kSparseThreads) {
        const int sl = e >> 3, p = e & 7;
        const size_t off = (size_t)a.gr.globals[sl] * kHeadDim;
        float x[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(Qu + off) + p), x);
        sQG[sl * 16 + 2 * p] = make_float4(x[0], x[1], x[2], x[3]);
        sQG[sl * 16 + 2 * p + 1] = make_float4(x[4], x[5], x[6], x[7]);
        unpack8(__ldg(reinterpret_cast<const uint4*>(Ku + off) + p), x);
        sKG[sl * 16 + 2 * p] = make_float4(x[0], x[1], x[2], x[3]);
        sKG[sl * 16 + 2 * p + 1] = make_float4(x[4], x[5], x[6], x[7]);
    }
    __syncthreads();

    if (g > 0) {
        // (1) global rows x this tile's keys: thread t < 128 owns key j = i0 + t
        if (tid < kTileRows) {
            const int64_t j = i0 + tid;
            if (j < P.n) {
                float k[64];
                load_row64(Ku + (size_t)j * kHeadDim, k);
                for (int s = 0; s < g; ++s) {
                    float acc = 0.f;
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const float4 q = sQG[s * 16 + c];
                        acc = fmaf(q.x, k[4 * c], acc); acc = fmaf(q.y, k[4 * c + 1], acc);
                        acc = fmaf(q.z, k[4 * c + 2], acc); acc = fmaf(q.w, k[4 * c + 3], acc);
                    }
                    const float sc = acc * kScale;
                    a.w.A_gr[((size_t)u * g + s) * P.n + j] = sc;
                    scr[s * kTileRows + tid] = sc;
                }
            } else {
                for (int s = 0; s < g; ++s) scr[s * kTileRows + tid] = -INFINITY;
            }
        }
        __syncthreads();
        // per-tile (max, sum of exp) of each global row: one warp per row slot
        for (int s = warp; s < g; s += kSparseThreads / 32) {
            float m = -INFINITY;
            for (int t = lane; t < kTileRows; t += 32) m = fmaxf(m, scr[s * kTileRows + t]);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
            float l = 0.f;
            for (int t = lane; t < kTileRows; t += 32) {
                const float v = scr[s * kTileRows + t];
                l += v == -INFINITY ? 0.f : expf(v - m);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
            if (lane == 0) {
                float* st = a.w.sstat + (((size_t)u * P.tiles + tile) * g + s) * 2;
                st[0] = m;
                st[1] = l;
            }
        }
    }
    // (2) rows of this tile: quarter-warp qi owns rows 4 qi .. +3; lane ql holds
    //     features 8 ql .. +7 of q_i and reads the same 16 bytes of each k row
    const int ql = lane & 7, qi = 4 * warp + (lane >> 3);
    const unsigned qmask = 0xffu << (lane & 24);
    for (int mrow = 0; mrow < 4; ++mrow) {
        const int64_t i = i0 + 4 * qi + mrow;
        if (i >= P.n || a.gr.is_global[i]) continue;      // uniform within the quarter
        const int64_t lo = i - P.r < 0 ? 0 : i - P.r;
        const int64_t hi = i + P.r > P.n - 1 ? P.n - 1 : i + P.r;
        float q[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(Qu + (size_t)i * kHeadDim) + ql), q);
        float m = -INFINITY;
        float* wg = a.w.A_gc + ((size_t)u * P.n + i) * P.g_pad;
        for (int s0 = 0; s0 < g; s0 += 8) {
            float v[8];
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                const int sl = s0 + b < g ? s0 + b : 0;
                const float4 k0 = sKG[sl * 16 + 2 * ql], k1 = sKG[sl * 16 + 2 * ql + 1];
                v[b] = q[0] * k0.x + q[1] * k0.y + q[2] * k0.z + q[3] * k0.w +
                       q[4] * k1.x + q[5] * k1.y + q[6] * k1.z + q[7] * k1.w;
            }
            const float dot = reduce8_transpose(v, ql, qmask);   // slot s0 + ql
            const int sl = s0 + ql;
            if (sl < g) {
                const int64_t j = a.gr.globals[sl];
                const float sc = (j < lo || j > hi) ? dot * kScale : -INFINITY;   // -inf: inside the window
                wg[sl] = sc;
                m = fmaxf(m, sc);
            }
        }
        const int64_t e0 = a.gr.x_ptr[i], e1 = a.gr.x_ptr[i + 1];
        float* wx = a.w.A_x + (size_t)u * a.gr.nx;
        // 32 slots at a time: their columns loaded together (4 per lane), then four
        // batches of 8 k rows with the next batch's rows in flight during this one's math
        for (int64_t base = e0; base < e1; base += 32) {
            const int cnt = e1 - base < 32 ? (int)(e1 - base) : 32;
            int32_t jv[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) jv[k] = 8 * k + ql < cnt ? __ldg(a.gr.x_col + base + 8 * k + ql) : (int32_t)i;
            uint4 kr[2][8];
#pragma unroll
            for (int b = 0; b < 8; ++b)
                kr[0][b] = __ldg(reinterpret_cast<const uint4*>(
                                     Ku + (size_t)__shfl_sync(qmask, jv[0], b, 8) * kHeadDim) + ql);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (k < 3 && 8 * (k + 1) < cnt) {
#pragma unroll
                    for (int b = 0; b < 8; ++b)
                        kr[(k + 1) & 1][b] = __ldg(reinterpret_cast<const uint4*>(
                                                 Ku + (size_t)__shfl_sync(qmask, jv[k + 1], b, 8) * kHeadDim) + ql);
                }
                if (8 * k < cnt) {
                    float v[8];
#pragma unroll
                    for (int b = 0; b < 8; ++b) {
                        float kx[8];
                        unpack8(kr[k & 1][b], kx);
                        v[b] = q[0] * kx[0] + q[1] * kx[1] + q[2] * kx[2] + q[3] * kx[3] +
                               q[4] * kx[4] + q[5] * kx[5] + q[6] * kx[6] + q[7] * kx[7];
                    }
                    const float dot = reduce8_transpose(v, ql, qmask);   // slot base + 8 k + ql
                    if (8 * k + ql < cnt) {
                        const float sc = dot * kScale;
                        wx[base + 8 * k + ql] = sc;
                        m = fmaxf(m, sc);
                    }
                }
            }
        }
#pragma unroll
        for (int off = 4; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(qmask, m, off, 8));
        if (ql == 0) a.w.m_sparse[(size_t)u * P.n + i] = m;
    }
}

// A warp per row: e = exp(s - m_i) for the globals outside the window and the
// random extras (in place), and inv_l_i = 1 / (band sum + sparse sum).  On
// entry m_sparse holds m_i and inv_l the band part of the row sum.
__global__ void __launch_bounds__(256)
score_finalize_kernel(ScoreArgs a) {
    const BandPlan& P = a.plan;
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (gw >= a.units * P.n) return;
    const int64_t u = gw / P.n, i = gw - u * P.n;
    if (a.gr.is_global[i]) return;
    const size_t row = (size_t)u * P.n + i;
    const float m = a.w.m_sparse[row];
    float l = 0.f;
    if (lane < P.g16) {
        // the tile's out-of-window globals' operand image (hi, lo planes)
        const float e = lane < P.g ? expf(a.w.A_gc[row * P.g_pad + lane] - m) : 0.f;   // exp(-inf) = 0
        l += e;
        const int64_t tile = i / kTileRows;
        uint8_t* img = a.w.A_gcimg + (size_t)(u * P.tiles + tile) * 2 * band::gc_plane_bytes(P.g16) +
                       band::gc_offset((int)(i - tile * kTileRows), lane, P.g16);
        const __nv_bfloat16 hi = __float2bfloat16_rn(e);
        *reinterpret_cast<__nv_bfloat16*>(img) = hi;
        *reinterpret_cast<__nv_bfloat16*>(img + band::gc_plane_bytes(P.g16)) =
            __float2bfloat16_rn(e - __bfloat162float(hi));
    }
    const int64_t e0 = a.gr.x_ptr[i], e1 = a.gr.x_ptr[i + 1];
    float* wx = a.w.A_x + (size_t)u * a.gr.nx;
    for (int64_t e = e0 + lane; e < e1; e += 32) {
        const float v = expf(wx[e] - m);
        wx[e] = v;
        l += v;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
    if (lane == 0) a.w.inv_l[row] = 1.f / (a.w.inv_l[row] + l);
}

// ---------------------------------------------------------------- band scores (tcgen05)
// Persistent: one CTA per SM walks tiles round-robin.  Warp 0 loads Q tiles
// (two buffers) and K chunks (ring) by TMA; warp 1 issues the MMAs into a ring
// of TMEM S buffers; warps 2-3 normalize the global rows' weights of the tile's
// keys; warps 4-11 are row warps: warp w serves TMEM lane quadrant w % 4 and
// columns 32 ((w - 4) / 4) .. +31 of each 64-key S chunk.
constexpr int kBThreads = 384;
constexpr int kRowWarp0 = 4;
constexpr int kRowThreads = 256;
constexpr int kSChunk = 64;              // keys per chunk (MMA N)
constexpr int kKStages = 8;              // smem ring of K chunks (8 KB each)
constexpr int kSBufs = 8;                // TMEM S buffers (64 columns each)
constexpr int kBTmemCols = 512;
constexpr int kQBytes = kTileRows * kHeadDim * 2;
constexpr int kKBytes = kSChunk * kHeadDim * 2;
constexpr int kBSmemUsed = 1024 + 2 * kQBytes + kKStages * kKBytes + 2 * band::kChunkImageBytes +
                           2 * kRowThreads * 4 + 512;
// request at least 120 KB so that the shared memory alone keeps it to one CTA per SM
constexpr int kBSmemBytes = kBSmemUsed > 120 * 1024 ? kBSmemUsed : 120 * 1024;
constexpr float kLog2e = 1.4426950408889634f;

__global__ void __launch_bounds__(kBThreads, 1)
score_band_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     ScoreArgs a, int* status) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* sQ = smem;                                   // 2 x 16 KB
    uint8_t* sK = sQ + 2 * kQBytes;                       // kKStages x 8 KB
    uint8_t* sOut = sK + kKStages * kKBytes;                  // 2 x one chunk's weight image
    float* xch = reinterpret_cast<float*>(sOut + 2 * band::kChunkImageBytes);   // [2][256] row partials
    uint64_t* bars = reinterpret_cast<uint64_t*>(xch + 2 * kRowThreads);
    uint64_t* full_Q = bars;                  // [2]
    uint64_t* empty_Q = full_Q + 2;           // [2]
    uint64_t* full_K = empty_Q + 2;           // [kKStages]
    uint64_t* empty_K = full_K + kKStages;
    uint64_t* full_S = empty_K + kKStages;    // [kSBufs]
    uint64_t* empty_S = full_S + kSBufs;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(empty_S + kSBufs);

    const BandPlan& P = a.plan;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nc = P.chunks;                              // the tile's key chunks (from i0 - r64)
    const int per_tile = 2 * nc;                          // pass 1 (max), pass 2 (exp + write)
    const int64_t total_tiles = a.units * P.tiles;
    const int my_tiles = blockIdx.x < total_tiles
        ? (int)((total_tiles - 1 - blockIdx.x) / gridDim.x + 1) : 0;

    if (warp == 1) ptx::tmem_alloc(tmem_slot, kBTmemCols);
    if (tid == 0) {
        for (int s = 0; s < 2; ++s) { ptx::mbar_init(&full_Q[s], 1); ptx::mbar_init(&empty_Q[s], 1); }
        for (int s = 0; s < kKStages; ++s) { ptx::mbar_init(&full_K[s], 1); ptx::mbar_init(&empty_K[s], 1); }
        for (int s = 0; s < kSBufs; ++s) { ptx::mbar_init(&full_S[s], 1); ptx::mbar_init(&empty_S[s], kRowThreads); }
        ptx::fence_mbar_init();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            for (int lt = 0; lt < my_tiles; ++lt) {
                const int64_t tix = blockIdx.x + (int64_t)lt * gridDim.x;
                const int64_t u = tix / P.tiles;
                const int64_t i0 = (tix - u * P.tiles) * kTileRows;
                const int64_t jb = i0 - P.r64;
                const int qb = lt & 1;
                if (lt >= 2) ptx::mbar_wait(&empty_Q[qb], ((lt / 2) - 1) & 1, status);
                ptx::mbar_arrive_expect_tx(&full_Q[qb], kQBytes);
                ptx::tma_load_3d(sQ + qb * kQBytes, &tmQ, &full_Q[qb], 0, (int)i0, (int)u);
                for (int it = 0; it < per_tile; ++it) {
                    const int gi = lt * per_tile + it;
                    const int c = it % nc, s = gi % kKStages;
                    if (gi >= kKStages) ptx::mbar_wait(&empty_K[s], ((gi / kKStages) - 1) & 1, status);
                    ptx::mbar_arrive_expect_tx(&full_K[s], kKBytes);
                    ptx::tma_load_3d(sK + s * kKBytes, &tmK, &full_K[s], 0, (int)(jb + kSChunk * c), (int)u);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = ptx::mma_idesc(1, kSChunk);
            for (int lt = 0; lt < my_tiles; ++lt) {
                const int qb = lt & 1;
                ptx::mbar_wait(&full_Q[qb], (lt / 2) & 1, status);
                const uint32_t qa = ptx::smem_u32(sQ + qb * kQBytes);
                for (int it = 0; it < per_tile; ++it) {
                    const int gi = lt * per_tile + it;
                    const int s = gi % kKStages, b = gi % kSBufs;
                    ptx::mbar_wait(&full_K[s], (gi / kKStages) & 1, status);
                    if (gi >= kSBufs) ptx::mbar_wait(&empty_S[b], ((gi / kSBufs) - 1) & 1, status);
                    ptx::tc_fence_after();
                    const uint32_t kb = ptx::smem_u32(sK + s * kKBytes);
#pragma unroll
                    for (int ks = 0; ks < kHeadDim / 16; ++ks)
                        ptx::mma_bf16_ss(tmem + kSChunk * b, ptx::sw128_kmajor_desc(qa + 32 * ks),
                                         ptx::sw128_kmajor_desc(kb + 32 * ks), idesc, ks > 0);
                    ptx::mma_commit(&empty_K[s]);
                    ptx::mma_commit(&full_S[b]);
                }
                ptx::mma_commit(&empty_Q[qb]);
            }
            // drain the asynchronous commit arrivals before the CTA can exit
            const int total = my_tiles * per_tile;
            for (int s = 0; s < kKStages; ++s) {
                const int uses = (total - s + kKStages - 1) / kKStages;
                if (uses > 0) ptx::mbar_wait(&empty_K[s], (uses - 1) & 1, status);
            }
            for (int s = 0; s < 2; ++s) {
                const int uses = (my_tiles - s + 1) / 2;
                if (uses > 0) ptx::mbar_wait(&empty_Q[s], (uses - 1) & 1, status);
            }
        }
    } else if (warp < kRowWarp0) {
        // warps 2-3 have no role
    } else {
        const int rw = warp - kRowWarp0;          // 0..7
        const int quad = warp & 3, hcol = rw >> 2;
        const int t = quad * 32 + lane;           // row within the tile
        const int rtid = rw * 32 + lane;          // 0..255
        // the two warps of a TMEM lane quadrant own the same 32 rows: they meet
        // on barrier 2 + quad, and lane 0 of the first one issues their copies
        const int pair_bar = 2 + quad;
        const bool pair_leader = hcol == 0 && lane == 0;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const float a_sc = kLog2e * kScale;
        for (int lt = 0; lt < my_tiles; ++lt) {
            const int64_t tix = blockIdx.x + (int64_t)lt * gridDim.x;
            const int64_t u = tix / P.tiles;
            const int64_t i0 = (tix - u * P.tiles) * kTileRows;
            const int64_t jb = i0 - P.r64;
            const int64_t i = i0 + t;
            const bool row_ok = i < P.n && !a.gr.is_global[i < P.n ? i : 0];
            const int64_t lo = i - P.r < 0 ? 0 : i - P.r;
            const int64_t hi = i + P.r > P.n - 1 ? P.n - 1 : i + P.r;
            // this tile's weight image in global memory; a chunk's image is built
            // in shared memory (row t of a plane at 1024 (t / 8) + 128 (t % 8),
            // 16-byte slot q of the row at q ^ (t % 8)) and written by one bulk copy
            uint8_t* timg = reinterpret_cast<uint8_t*>(a.w.A_band) +
                            (size_t)(u * P.tiles + (i0 / kTileRows)) * P.chunks * band::kChunkImageBytes;
            const int trow = (t >> 3) * 1024 + (t & 7) * 128;
            float mraw = -INFINITY;               // max of the raw dot products q.k (unscaled)
            float m = 0.f, b2 = 0.f, lsum = 0.f;
            for (int it = 0; it < per_tile; ++it) {
                const int gi = lt * per_tile + it;
                const int b = gi % kSBufs, c = it % nc;
                const bool pass2 = it >= nc;
                if (it == nc) {
                    // both column halves of a row agree on the row maximum
                    xch[rtid] = mraw;
                    ptx::named_barrier_sync(pair_bar, 64);
                    const float other = xch[(rtid + 128) & 255];
                    const float ms = row_ok ? a.w.m_sparse[(size_t)u * P.n + i] : 0.f;
                    m = fmaxf(ms, fmaxf(mraw, other) * kScale);
                    b2 = m * kLog2e;
                    ptx::named_barrier_sync(pair_bar, 64);     // xch is reused below
                }
                ptx::mbar_wait(&full_S[b], (gi / kSBufs) & 1, status);
                __syncwarp();
                ptx::tc_fence_after();
                float sv[32];
                ptx::tmem_ld32(tmem + lane_base + kSChunk * b + 32 * hcol, sv);
                ptx::tc_fence_before();
                ptx::mbar_arrive(&empty_S[b]);
                const int64_t j0 = jb + kSChunk * c + 32 * hcol;
                const bool full_in = row_ok && j0 >= lo && j0 + 31 <= hi;
                const bool none_in = !row_ok || j0 > hi || j0 + 31 < lo;
                if (!pass2) {
                    if (full_in) {
#pragma unroll
                        for (int k = 0; k < 32; ++k) mraw = fmaxf(mraw, sv[k]);
                    } else if (!none_in) {
#pragma unroll
                        for (int k = 0; k < 32; ++k) {
                            const int64_t j = j0 + k;
                            if (j >= lo && j <= hi) mraw = fmaxf(mraw, sv[k]);
                        }
                    }
                } else {
                    // the staging buffer of this chunk is free once its previous bulk copy has read it
                    const int gs = lt * nc + c;           // pass-2 chunk count of this CTA
                    uint8_t* stg = sOut + (gs & 1) * band::kChunkImageBytes + trow;
                    if (pair_leader) ptx::bulk_wait_read<1>();
                    ptx::named_barrier_sync(pair_bar, 64);
                    float e[32];
                    if (!row_ok || none_in) {
#pragma unroll
                        for (int k = 0; k < 32; ++k) e[k] = 0.f;
                    } else if (full_in) {
#pragma unroll
                        for (int k = 0; k < 32; ++k) { e[k] = ptx::ex2_approx(fmaf(sv[k], a_sc, -b2)); lsum += e[k]; }
                    } else {
                        const int dlo = (int)(lo - j0), dhi = (int)(hi - j0);   // in-window keys k in [dlo, dhi]
#pragma unroll
                        for (int k = 0; k < 32; ++k) {
                            e[k] = (k >= dlo && k <= dhi) ? ptx::ex2_approx(fmaf(sv[k], a_sc, -b2)) : 0.f;
                            lsum += e[k];
                        }
                    }
#pragma unroll
                    for (int k8 = 0; k8 < 4; ++k8) {
                        uint32_t hw[4], lw[4];
#pragma unroll
                        for (int p2 = 0; p2 < 4; ++p2) {
                            const float x0 = e[8 * k8 + 2 * p2], x1 = e[8 * k8 + 2 * p2 + 1];
                            const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
                            const __nv_bfloat162 l =
                                __floats2bfloat162_rn(x0 - __low2float(h), x1 - __high2float(h));
                            hw[p2] = *reinterpret_cast<const uint32_t*>(&h);
                            lw[p2] = *reinterpret_cast<const uint32_t*>(&l);
                        }
                        const int slot = ((4 * hcol + k8) ^ (t & 7)) << 4;
                        *reinterpret_cast<uint4*>(stg + slot) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                        *reinterpret_cast<uint4*>(stg + band::kChunkPlaneBytes + slot) =
                            make_uint4(lw[0], lw[1], lw[2], lw[3]);
                    }
                    ptx::fence_proxy_async_smem();        // the pieces are visible to the bulk copy
                    ptx::named_barrier_sync(pair_bar, 64);
                    if (pair_leader) {
                        // rows 32 quad .. +31: 4 KB of each plane
                        const size_t qoff = (size_t)quad * 4096;
                        uint8_t* gdst = timg + (size_t)c * band::kChunkImageBytes + qoff;
                        const uint8_t* ssrc = sOut + (gs & 1) * band::kChunkImageBytes + qoff;
                        ptx::bulk_store(gdst, ssrc, 4096);
                        ptx::bulk_store(gdst + band::kChunkPlaneBytes, ssrc + band::kChunkPlaneBytes, 4096);
                        ptx::bulk_commit();
                    }
                }
            }
            // the row's maximum m_i and the band part of its sum (score_finalize_kernel adds the rest)
            xch[rtid] = lsum;
            ptx::named_barrier_sync(pair_bar, 64);
            if (hcol == 0 && row_ok) {
                a.w.inv_l[(size_t)u * P.n + i] = lsum + xch[rtid + 128];
                a.w.m_sparse[(size_t)u * P.n + i] = m;
            }
            ptx::named_barrier_sync(pair_bar, 64);     // xch is reused by the next tile
        }
        if (pair_leader) ptx::bulk_wait<0>();     // the last images are written before exit
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) ptx::tmem_dealloc(tmem, kBTmemCols);
}

// ---------------------------------------------------------------- global rows' weights
// One CTA per (unit, 128-key tile): A_gr = exp(s - max) / sum with the global
// rows' (max, 1/sum) from score_sparse_kernel, in place, and the tile's
// global-row operand image (hi / lo bf16; keys past n are 0).
__global__ void __launch_bounds__(256)
score_global_norm_kernel(ScoreArgs a) {
    __shared__ float2 st[kBandMaxGlobals];        // (max, 1 / sum) of each global row
    const BandPlan& P = a.plan;
    const int64_t u = blockIdx.x / P.tiles;
    const int64_t tile = blockIdx.x - u * P.tiles;
    const int64_t i0 = tile * kTileRows;
    // merge the per-tile (max, sum of exp) of every global row: 16 lanes per row,
    // each lane over tiles l, l + 16, ..., in a fixed order
    for (int s0 = 0; s0 < P.g; s0 += 16) {
        const int sl = s0 + (threadIdx.x >> 4), l = threadIdx.x & 15;
        const bool ok = sl < P.g;
        float M = -INFINITY;
        for (int tt = l; ok && tt < P.tiles; tt += 16)
            M = fmaxf(M, __ldg(a.w.sstat + (((size_t)u * P.tiles + tt) * P.g + sl) * 2));
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off, 16));
        float L = 0.f;
        for (int tt = l; ok && tt < P.tiles; tt += 16) {
            const float* sp = a.w.sstat + (((size_t)u * P.tiles + tt) * P.g + sl) * 2;
            const float mt = __ldg(sp);
            if (mt != -INFINITY) L += __ldg(sp + 1) * expf(mt - M);
        }
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off, 16);
        if (ok && l == 0) {
            st[sl] = make_float2(M, 1.f / L);
            if (tile == 0) {
                a.w.gstat[((size_t)u * P.g + sl) * 2] = M;
                a.w.gstat[((size_t)u * P.g + sl) * 2 + 1] = 1.f / L;
            }
        }
    }
    __syncthreads();
    uint8_t* gimg = a.w.A_gimg + (size_t)blockIdx.x * band::kGImgBytes;
    for (int e = threadIdx.x; e < P.g * kTileRows; e += blockDim.x) {
        const int sl = e / kTileRows, jj = e % kTileRows;
        float w = 0.f;
        if (i0 + jj < P.n) {
            const float gm = st[sl].x;
            const float ginv = st[sl].y;
            float* v = a.w.A_gr + ((size_t)u * P.g + sl) * P.n + i0 + jj;
            w = expf(*v - gm) * ginv;
            *v = w;
        }
        const int h = jj >> 6, k = jj & 63;
        const __nv_bfloat16 hi = __float2bfloat16_rn(w);
        const __nv_bfloat16 lo = __float2bfloat16_rn(w - __bfloat162float(hi));
        uint8_t* pe = gimg + h * 2 * band::kGImgPlaneBytes + (sl >> 3) * 1024 + (sl & 7) * 128 +
                      ((((k >> 3) ^ (sl & 7))) << 4) + (k & 7) * 2;
        *reinterpret_cast<__nv_bfloat16*>(pe) = hi;
        *reinterpret_cast<__nv_bfloat16*>(pe + band::kGImgPlaneBytes) = lo;
    }
}

// ---------------------------------------------------------------- weights -> CSR order
__global__ void __launch_bounds__(256)
band_to_csr_kernel(ScoreArgs a, const int64_t* __restrict__ row_ptr,
                   const int32_t* __restrict__ col, int64_t nnz, float* __restrict__ out) {
    const BandPlan& P = a.plan;
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (gw >= a.units * P.n) return;
    const int64_t u = gw / P.n, i = gw - u * P.n;
    const int64_t e0 = row_ptr[i], e1 = row_ptr[i + 1];
    float* o = out + (size_t)u * nnz;
    if (a.gr.is_global[i]) {
        const int s = a.gr.gslot[i];
        const float* Ag = a.w.A_gr + ((size_t)u * P.g + s) * P.n;
        for (int64_t e = e0 + lane; e < e1; e += 32) o[e] = Ag[col[e]];
        return;
    }
    const int64_t lo = i - P.r < 0 ? 0 : i - P.r;
    const int64_t hi = i + P.r > P.n - 1 ? P.n - 1 : i + P.r;
    const int64_t tile = i / kTileRows, t = i - tile * kTileRows;
    const int64_t jb = tile * kTileRows - P.r64;       // first key of the tile's chunk grid
    const float inv = a.w.inv_l[(size_t)u * P.n + i];
    const uint8_t* timg = reinterpret_cast<const uint8_t*>(a.w.A_band) +
                          (size_t)(u * P.tiles + tile) * P.chunks * band::kChunkImageBytes +
                          (t >> 3) * 1024 + (t & 7) * 128;
    const uint8_t* gcimg = a.w.A_gcimg + (size_t)(u * P.tiles + tile) * 2 * band::gc_plane_bytes(P.g16);
    const float* Ax = a.w.A_x + (size_t)u * a.gr.nx;
    int64_t xb = a.gr.x_ptr[i];
    // extras are the row's edges that are neither window nor global, in order
    for (int64_t base = e0; base < e1; base += 32) {
        const int64_t e = base + lane;
        const int64_t j = e < e1 ? col[e] : -1;
        const bool is_x = e < e1 && (j < lo || j > hi) && !a.gr.is_global[j < 0 ? 0 : j];
        const unsigned mask = __ballot_sync(0xffffffffu, is_x);
        const int rank = __popc(mask & ((1u << lane) - 1));
        if (e < e1) {
            float v;
            if (j >= lo && j <= hi) {
                const int64_t kk = j - jb;
                const uint8_t* pe = timg + (size_t)(kk >> 6) * band::kChunkImageBytes +
                                    ((((kk & 63) >> 3) ^ (t & 7)) << 4) + (kk & 7) * 2;
                v = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(pe)) +
                    __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(pe + band::kChunkPlaneBytes));
            }
            else if (a.gr.is_global[j]) {
                const uint8_t* pe = gcimg + band::gc_offset((int)t, a.gr.gslot[j], P.g16);
                v = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(pe)) +
                    __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(pe + band::gc_plane_bytes(P.g16)));
            }
            else v = Ax[xb + rank];
            o[e] = v * inv;
        }
        xb += __popc(mask);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

ScoreArgs make_args(const diffuser_graph* g, const BandPlan& p, int64_t units, char* ws,
                    const BandLayout& L) {
    ScoreArgs s;
    s.plan = p;
    s.units = units;
    s.gr = band_graph_refs(g);
    s.w = band_weights(ws, L);
    s.counters = reinterpret_cast<int*>(ws + L.counters);
    return s;
}

}  // namespace

int launch_band_scores(const diffuser_graph* g, const BandPlan& p, int64_t units, const void* Q,
                       const void* K, char* ws, const BandLayout& L, cudaStream_t stream) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(score_band_tc_kernel,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, kBSmemBytes);

    });
    if (attr_err != cudaSuccess) return cuda_fail(attr_err, "cudaFuncSetAttribute(scores)");
    cudaError_t err = cudaMemsetAsync(ws + L.counters, 0, (size_t)units * 4, stream);
    if (err != cudaSuccess) return cuda_fail(err, "clearing the tile counters");
    ScoreArgs a = make_args(g, p, units, ws, L);
    const auto* Qb = static_cast<const __nv_bfloat16*>(Q);
    const auto* Kb = static_cast<const __nv_bfloat16*>(K);
    const unsigned grid = (unsigned)(units * p.tiles);
    {
        LaunchScope scope(DIFFUSER_KERNEL_SCORE, stream);
        score_sparse_kernel<<<grid, kSparseThreads, 0, stream>>>(a, Qb, Kb);
    }
    if ((err = cudaGetLastError()) != cudaSuccess) return cuda_fail(err, "score_sparse_kernel");
    if (p.g > 0) {
        LaunchScope scope(DIFFUSER_KERNEL_SCORE, stream);
        score_global_norm_kernel<<<grid, 256, 0, stream>>>(a);
    }
    if ((err = cudaGetLastError()) != cudaSuccess) return cuda_fail(err, "score_global_norm_kernel");

    auto fn = encode_fn();
    if (!fn) return fail(DIFFUSER_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    CUtensorMap tmQ, tmK;
    const cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)p.n, (cuuint64_t)units};
    const cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)p.n * kHeadDim * 2};
    const cuuint32_t es[3] = {1, 1, 1};
    const cuuint32_t boxQ[3] = {(cuuint32_t)kHeadDim, (cuuint32_t)kTileRows, 1};
    const cuuint32_t boxK[3] = {(cuuint32_t)kHeadDim, (cuuint32_t)kSChunk, 1};
    CUresult r = fn(&tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(Q), dims, strides,
                    boxQ, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r == CUDA_SUCCESS)
        r = fn(&tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(K), dims, strides, boxK,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(DIFFUSER_ERR_CUDA, "cuTensorMapEncodeTiled (Q/K) failed: " + std::to_string((int)r));
    static int num_sms = 0;
    if (num_sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || num_sms < 1)
            num_sms = 1;
    }
    const unsigned pgrid = grid < (unsigned)num_sms ? grid : (unsigned)num_sms;
    {
        LaunchScope scope(DIFFUSER_KERNEL_SCORE, stream);
        score_band_tc_kernel<<<pgrid, kBThreads, kBSmemBytes, stream>>>(tmQ, tmK, a, g->d_status);
    }
    if ((err = cudaGetLastError()) != cudaSuccess) return cuda_fail(err, "score_band_tc_kernel");
    {
        LaunchScope scope(DIFFUSER_KERNEL_SCORE, stream);
        score_finalize_kernel<<<(unsigned)((units * p.n + 7) / 8), 256, 0, stream>>>(a);
    }
    if ((err = cudaGetLastError()) != cudaSuccess) return cuda_fail(err, "score_finalize_kernel");
    return DIFFUSER_OK;
}

int launch_band_to_csr(const diffuser_graph* g, const BandPlan& p, int64_t units, char* ws,
                       const BandLayout& L, float* A_out, cudaStream_t stream) {
    ScoreArgs a = make_args(g, p, units, ws, L);
    const unsigned grid = (unsigned)((units * p.n + 7) / 8);
    {
        LaunchScope scope(DIFFUSER_KERNEL_AUX, stream);
        band_to_csr_kernel<<<grid, 256, 0, stream>>>(a, g->d_row_ptr, g->d_col, g->nnz, A_out);
    }
    cudaError_t err = cudaGetLastError();
    return err == cudaSuccess ? DIFFUSER_OK : cuda_fail(err, "band_to_csr_kernel");
}

}  // namespace dfs
