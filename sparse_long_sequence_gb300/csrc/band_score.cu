// Scores and masked softmax for the band path ("Diffuser: modelling long
// sequences with multi-hop attention diffusion", eq S.1-S.5; "1.2.1 Static
// sparsity", eq 1-3), in two kernels:
//
//  * score_sparse_kernel (SIMT): per row, the raw scores q_i.k_j/8 of the
//    globals outside the window and of the random extras (one lane per key,
//    the 128-byte k_j row read whole), and their maximum; per tile, the raw
//    scores of the global rows against the tile's keys with per-tile
//    (max, sum of exp); the last tile of a unit merges those into the global
//    rows' (max, 1/sum).
//  * score_band_tc_kernel (tcgen05, persistent): S = Q K^T for a 128-row
//    tile against 64-key chunks of its window on bf16 tensor cores (fp32
//    accumulation in TMEM), in two passes over the chunks: the row maximum,
//    then e = exp(s - m) written into the band storage as a bf16 hi / lo
//    pair (zero outside the row's window) with the row sum; the
//    row threads then turn the row's sparse raw scores into e and store
//    inv_l = 1 / (band sum + sparse sum).
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

__device__ __forceinline__ float dot64(const float (&q)[64], const __nv_bfloat16* kp) {
    const uint4* v = reinterpret_cast<const uint4*>(kp);
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 w = __ldg(v + c);
        acc = fmaf(q[8 * c + 0], bf16lo(w.x), acc); acc = fmaf(q[8 * c + 1], bf16hi(w.x), acc);
        acc = fmaf(q[8 * c + 2], bf16lo(w.y), acc); acc = fmaf(q[8 * c + 3], bf16hi(w.y), acc);
        acc = fmaf(q[8 * c + 4], bf16lo(w.z), acc); acc = fmaf(q[8 * c + 5], bf16hi(w.z), acc);
        acc = fmaf(q[8 * c + 6], bf16lo(w.w), acc); acc = fmaf(q[8 * c + 7], bf16hi(w.w), acc);
    }
    return acc;
}

// ---------------------------------------------------------------- sparse scores
constexpr int kSparseThreads = 256;

__global__ void __launch_bounds__(kSparseThreads)
score_sparse_kernel(ScoreArgs a, const __nv_bfloat16* __restrict__ Q,
                    const __nv_bfloat16* __restrict__ K) {
    extern __shared__ float sm[];            // [g][65] global-row scores of this tile's keys
    __shared__ int ticket;
    const BandPlan& P = a.plan;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t u = blockIdx.x / P.tiles;
    const int tile = (int)(blockIdx.x - u * P.tiles);
    const int64_t i0 = (int64_t)tile * kTileRows;
    const int g = P.g;
    const __nv_bfloat16* Qu = Q + (size_t)u * P.n * kHeadDim;
    const __nv_bfloat16* Ku = K + (size_t)u * P.n * kHeadDim;

    if (g > 0) {
        // (1) global rows x this tile's keys: thread t < 128 owns key j = i0 + t
        float* scr = sm;                     // [g][kTileRows]
        if (tid < kTileRows) {
            const int64_t j = i0 + tid;
            if (j < P.n) {
                float k[64];
                load_row64(Ku + (size_t)j * kHeadDim, k);
                for (int s = 0; s < g; ++s) {
                    const float sc = dot64(k, Qu + (size_t)a.gr.globals[s] * kHeadDim) * kScale;
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
        __threadfence();
        __syncthreads();
        if (tid == 0) ticket = atomicAdd(&a.counters[u], 1);
        __syncthreads();
        if (ticket == P.tiles - 1) {
            __threadfence();
            for (int s = tid; s < g; s += kSparseThreads) {
                float M = -INFINITY;
                for (int tt = 0; tt < P.tiles; ++tt)
                    M = fmaxf(M, __ldcg(a.w.sstat + (((size_t)u * P.tiles + tt) * g + s) * 2));
                float L = 0.f;
                for (int tt = 0; tt < P.tiles; ++tt) {
                    const float* st = a.w.sstat + (((size_t)u * P.tiles + tt) * g + s) * 2;
                    const float mt = __ldcg(st);
                    if (mt != -INFINITY) L += __ldcg(st + 1) * expf(mt - M);
                }
                a.w.gstat[((size_t)u * g + s) * 2] = M;
                a.w.gstat[((size_t)u * g + s) * 2 + 1] = 1.f / L;
            }
            if (tid == 0) a.counters[u] = 0;
        }
    }
    // (2) rows of this tile, 16 per warp: globals outside the window + extras
    for (int rr = 0; rr < 16; ++rr) {
        const int64_t i = i0 + 16 * warp + rr;
        if (i >= P.n) break;
        if (a.gr.is_global[i]) continue;
        const int64_t lo = i - P.r < 0 ? 0 : i - P.r;
        const int64_t hi = i + P.r > P.n - 1 ? P.n - 1 : i + P.r;
        float q[64];
        load_row64(Qu + (size_t)i * kHeadDim, q);
        const int64_t e0 = a.gr.x_ptr[i], e1 = a.gr.x_ptr[i + 1];
        const int total = g + (int)(e1 - e0);
        float* wg = a.w.A_gc + ((size_t)u * P.n + i) * P.g_pad;
        float* wx = a.w.A_x + (size_t)u * a.gr.nx;
        float m = -INFINITY;
        for (int k = lane; k < total; k += 32) {
            if (k < g) {
                const int64_t j = a.gr.globals[k];
                float sc = 0.f;
                if (j < lo || j > hi) {
                    sc = dot64(q, Ku + (size_t)j * kHeadDim) * kScale;
                    m = fmaxf(m, sc);
                }
                wg[k] = sc;
            } else {
                const int64_t e = e0 + (k - g);
                const float sc = dot64(q, Ku + (size_t)a.gr.x_col[e] * kHeadDim) * kScale;
                wx[e] = sc;
                m = fmaxf(m, sc);
            }
        }
        for (int s = g + lane; s < P.g_pad; s += 32) wg[s] = 0.f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        if (lane == 0) a.w.m_sparse[(size_t)u * P.n + i] = m;
    }
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
constexpr int kBSmemUsed = 1024 + 2 * kQBytes + kKStages * kKBytes + 2 * kRowThreads * 4 + 512;
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
    float* xch = reinterpret_cast<float*>(sK + kKStages * kKBytes);   // [2][256] row partials
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
    } else if (warp == 2 || warp == 3) {
        // normalize the global rows' weights over each tile's keys:
        // A_gr = exp(s - max) / sum, with (max, 1/sum) from score_sparse_kernel;
        // also the tile's global-row operand image (hi / lo bf16, zero past n)
        for (int lt = 0; lt < my_tiles; ++lt) {
            const int64_t tix = blockIdx.x + (int64_t)lt * gridDim.x;
            const int64_t u = tix / P.tiles;
            const int64_t i0 = (tix - u * P.tiles) * kTileRows;
            const int64_t tkeys = P.n - i0 < kTileRows ? P.n - i0 : kTileRows;
            uint8_t* gimg = a.w.A_gimg + (size_t)tix * band::kGImgBytes;
            for (int e = tid - 64; e < P.g * kTileRows; e += 64) {
                const int sl = e / kTileRows, jj = e % kTileRows;
                float w = 0.f;
                if (jj < tkeys) {
                    const float gm = a.w.gstat[((size_t)u * P.g + sl) * 2];
                    const float ginv = a.w.gstat[((size_t)u * P.g + sl) * 2 + 1];
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
    } else {
        const int rw = warp - kRowWarp0;          // 0..7
        const int quad = warp & 3, hcol = rw >> 2;
        const int t = quad * 32 + lane;           // row within the tile
        const int rtid = rw * 32 + lane;          // 0..255
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
            // this tile's weight image; row t of a chunk's plane sits at
            // 1024 (t / 8) + 128 (t % 8), 16-byte slot q of the row at q ^ (t % 8)
            uint8_t* timg = reinterpret_cast<uint8_t*>(a.w.A_band) +
                            (size_t)(u * P.tiles + (i0 / kTileRows)) * P.chunks * band::kChunkImageBytes +
                            (t >> 3) * 1024 + (t & 7) * 128;
            float mraw = -INFINITY;               // max of the raw dot products q.k (unscaled)
            float m = 0.f, b2 = 0.f, lsum = 0.f;
            for (int it = 0; it < per_tile; ++it) {
                const int gi = lt * per_tile + it;
                const int b = gi % kSBufs, c = it % nc;
                const bool pass2 = it >= nc;
                if (it == nc) {
                    // both column halves of a row agree on the row maximum
                    xch[rtid] = mraw;
                    ptx::named_barrier_sync(1, kRowThreads);
                    const float other = xch[(rtid + 128) & 255];
                    const float ms = row_ok ? a.w.m_sparse[(size_t)u * P.n + i] : 0.f;
                    m = fmaxf(ms, fmaxf(mraw, other) * kScale);
                    b2 = m * kLog2e;
                    ptx::named_barrier_sync(1, kRowThreads);   // xch is reused below
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
                } else if (row_ok) {
                    float e[32];
                    if (full_in) {
#pragma unroll
                        for (int k = 0; k < 32; ++k) { e[k] = exp2f(fmaf(sv[k], a_sc, -b2)); lsum += e[k]; }
                    } else {
#pragma unroll
                        for (int k = 0; k < 32; ++k) {
                            const int64_t j = j0 + k;
                            e[k] = (j >= lo && j <= hi) ? exp2f(fmaf(sv[k], a_sc, -b2)) : 0.f;
                            lsum += e[k];
                        }
                    }
                    uint8_t* cimg = timg + (size_t)c * band::kChunkImageBytes;
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
                        *reinterpret_cast<uint4*>(cimg + slot) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                        *reinterpret_cast<uint4*>(cimg + band::kChunkPlaneBytes + slot) =
                            make_uint4(lw[0], lw[1], lw[2], lw[3]);
                    }
                }
            }
            // the row's sparse part (first column half) and the normalizer
            xch[rtid] = lsum;
            ptx::named_barrier_sync(1, kRowThreads);
            if (hcol == 0 && row_ok) {
                float l = lsum + xch[rtid + 128];
                float* wg = a.w.A_gc + ((size_t)u * P.n + i) * P.g_pad;
                for (int s2 = 0; s2 < P.g; ++s2) {
                    const int64_t j = a.gr.globals[s2];
                    const float e = (j < lo || j > hi) ? expf(wg[s2] - m) : 0.f;
                    wg[s2] = e;
                    l += e;
                }
                float* wx = a.w.A_x + (size_t)u * a.gr.nx;
                for (int64_t e = a.gr.x_ptr[i]; e < a.gr.x_ptr[i + 1]; ++e) {
                    const float v = expf(wx[e] - m);
                    wx[e] = v;
                    l += v;
                }
                a.w.inv_l[(size_t)u * P.n + i] = 1.f / l;
            }
            ptx::named_barrier_sync(1, kRowThreads);   // xch is reused by the next tile
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) ptx::tmem_dealloc(tmem, kBTmemCols);
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
    const float* Agc = a.w.A_gc + ((size_t)u * P.n + i) * P.g_pad;
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
            else if (a.gr.is_global[j]) v = Agc[a.gr.gslot[j]];
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
        if (attr_err == cudaSuccess)
            attr_err = cudaFuncSetAttribute(score_sparse_kernel,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            kBandMaxGlobals * kTileRows * (int)sizeof(float));
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
        score_sparse_kernel<<<grid, kSparseThreads, (size_t)p.g * kTileRows * sizeof(float),
                              stream>>>(a, Qb, Kb);
    }
    if ((err = cudaGetLastError()) != cudaSuccess) return cuda_fail(err, "score_sparse_kernel");

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
