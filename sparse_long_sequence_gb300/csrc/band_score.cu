// Scores and masked softmax for the band path ("Diffuser: modelling long
// sequences with multi-hop attention diffusion", eq S.1-S.5; "1.2.1 Static
// sparsity", eq 1-3), in four kernels:
//
//  * score_sparse_kernel: per row, the raw scores q_i.k_j/8 of the random
//    extras and their maximum; a quarter-warp per row, each K row read as one
//    128-byte line, 8 dot products reduced across the quarter at once.
//  * score_band_tc_kernel (tcgen05, persistent): S = Q K^T for a 128-row
//    tile against 64-key chunks of its window on bf16 tensor cores (fp32
//    accumulation in TMEM): the row maximum m_i.  For the attention-weights
//    export a second pass writes e = exp(s - m_i) as the tile's operand image
//    and the band part of the row sum; the forward skips it (its hop kernels
//    recompute the band weights from Q and K).  On the same tensor cores:
//    q_i.k_G for the globals outside each row's window (N = g16; their e as an
//    operand image) and q_G.k_j for the global rows against the tile's own
//    keys (raw scores).
//  * score_global_norm_kernel: per global row, its (max, 1/sum) over all keys,
//    the normalized weights, and its row of each tile's global-row operand
//    image.
//  * score_finalize_kernel (export only): a warp per row turns the extras' raw
//    scores into e = exp(s - m_i) and stores inv_l = 1 / (band + globals +
//    extras sum).  In the forward the first hop does this: its gather kernel
//    finishes the extras and its band kernel adds the band sum.
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
    const __nv_bfloat16* Q;
    const __nv_bfloat16* K;
    const uint8_t* Vpre;    // V, pulled into L2 for the first hop (null: not needed)
    size_t vbytes;
};

// ---------------------------------------------------------------- sparse scores
int sm_count_scores() {
    static int num_sms = 0;
    if (num_sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || num_sms < 1)
            num_sms = 1;
    }
    return num_sms;
}

constexpr int kSparseThreads = 256;
constexpr int kSparseBlocks = 2;         // CTAs per SM of the persistent sparse kernel

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

// Persistent, 8 warps per CTA.  The rows of all units are split evenly over the
// quarter-warps of the grid; a quarter walks its rows in windows of up to
// kSWinRows rows of one unit, as a sequence of batches of up to 8 slots of one
// row.  Batch b + 1's k rows (and q, if its row differs) load while batch b's
// dot products run, and batch b + 2's columns load meanwhile.  Lane l holds
// features 8 l .. 8 l + 7 of q and reads the same 16 bytes of each k row, so a
// load instruction reads whole 128-byte lines; the 8 partial dot products of a
// batch are reduced across the quarter at once.
constexpr int kSWinRows = 16;

__global__ void __launch_bounds__(kSparseThreads, kSparseBlocks)
score_sparse_kernel(ScoreArgs a, const __nv_bfloat16* __restrict__ Q,
                    const __nv_bfloat16* __restrict__ K) {
    __shared__ int sStart[32][kSWinRows + 1];     // per quarter: the window's row starts (unit-local slots)
    const BandPlan& P = a.plan;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ql = lane & 7, qi = 4 * warp + (lane >> 3);
    const unsigned qmask = 0xffu << (lane & 24);
    const int64_t nq = (int64_t)gridDim.x * 32, qg = (int64_t)blockIdx.x * 32 + qi;
    const int64_t rows_total = a.units * P.n;
    const int64_t R1 = (qg + 1) * rows_total / nq;
    int* ss = sStart[qi];
    for (int64_t Rw = qg * rows_total / nq; Rw < R1;) {
        const int64_t u = Rw / P.n;
        const int64_t iw = Rw - u * P.n;
        int64_t cnt64 = R1 - Rw;
        if (cnt64 > P.n - iw) cnt64 = P.n - iw;
        const int cnt = cnt64 < kSWinRows ? (int)cnt64 : kSWinRows;
        for (int m = ql; m <= cnt; m += 8) ss[m] = (int)a.gr.x_ptr[iw + m];
        __syncwarp(qmask);
        const uint4* Qu = reinterpret_cast<const uint4*>(Q + ((size_t)u * P.n + iw) * kHeadDim) + ql;
        const uint4* Ku = reinterpret_cast<const uint4*>(K + (size_t)u * P.n * kHeadDim) + ql;
        float* wx = a.w.A_x + (size_t)u * a.gr.nx;
        float* mx = a.w.m_sparse + (size_t)u * P.n + iw;
        // rows without extras (the global rows among them) have no maximum
        for (int m = ql; m < cnt; m += 8)
            if (ss[m + 1] == ss[m]) mx[m] = -INFINITY;
        // batch cursor: row r, first slot e; r == cnt past the end
        auto next = [&](int r, int e, int& r2, int& e2) {
            e2 = e + 8;
            r2 = r;
            if (e2 >= ss[r + 1]) {
                r2 = r + 1;
                while (r2 < cnt && ss[r2 + 1] == ss[r2]) ++r2;
                e2 = r2 < cnt ? ss[r2] : 0;
            }
        };
        int rA = 0;                               // the first row with extras
        while (rA < cnt && ss[rA + 1] == ss[rA]) ++rA;
        int eA = rA < cnt ? ss[rA] : 0;
        if (rA < cnt) {
            int rB, eB;
            next(rA, eA, rB, eB);
            auto cols = [&](int r, int e) -> int32_t {       // this lane's column of batch (r, e)
                return (r < cnt && e + ql < ss[r + 1]) ? __ldg(a.gr.x_col + e + ql) : 0;
            };
            // Slots past a row's end (and the batch after the last) read k row 0 of
            // the unit: their dot products land on lanes whose results are not stored.
            const int32_t jA = cols(rA, eA);
            int32_t jB = cols(rB, eB);
            uint4 qA = __ldg(Qu + (size_t)rA * 8);
            uint4 qB = rB < cnt ? __ldg(Qu + (size_t)rB * 8) : qA;
            uint4 kA[8], kB[8];
#pragma unroll
            for (int b = 0; b < 8; ++b) kA[b] = __ldcg(Ku + (size_t)__shfl_sync(qmask, jA, b, 8) * 8);
            float mrow = -INFINITY;               // this lane's running max of row rA
            // one batch: batch B's k rows load into kn while batch A's (in kc) are
            // used; the two arrays swap roles from one batch to the next
            auto step = [&](uint4 (&kc)[8], uint4 (&kn)[8]) {
                int rC, eC;
                if (rB < cnt) next(rB, eB, rC, eC); else { rC = cnt; eC = 0; }
                const int32_t jC = cols(rC, eC);
                const uint4 qC = (rC < cnt && rC != rB) ? __ldg(Qu + (size_t)rC * 8) : qB;
#pragma unroll
                for (int b = 0; b < 8; ++b) kn[b] = __ldcg(Ku + (size_t)__shfl_sync(qmask, jB, b, 8) * 8);
                // batch A: 8 partial dot products (pairs of features on packed FMAs;
                // bf16 products are exact in fp32), reduced across the quarter
                const float2 q01 = make_float2(bf16lo(qA.x), bf16hi(qA.x));
                const float2 q23 = make_float2(bf16lo(qA.y), bf16hi(qA.y));
                const float2 q45 = make_float2(bf16lo(qA.z), bf16hi(qA.z));
                const float2 q67 = make_float2(bf16lo(qA.w), bf16hi(qA.w));
                float v[8];
#pragma unroll
                for (int b = 0; b < 8; ++b) {
                    const uint4 k = kc[b];
                    float2 p = __fmul2_rn(q01, make_float2(bf16lo(k.x), bf16hi(k.x)));
                    p = __ffma2_rn(q23, make_float2(bf16lo(k.y), bf16hi(k.y)), p);
                    p = __ffma2_rn(q45, make_float2(bf16lo(k.z), bf16hi(k.z)), p);
                    p = __ffma2_rn(q67, make_float2(bf16lo(k.w), bf16hi(k.w)), p);
                    v[b] = p.x + p.y;
                }
                const float dot = reduce8_transpose(v, ql, qmask);   // slot eA + ql
                if (eA + ql < ss[rA + 1]) {
                    const float sc = dot * kScale;
                    wx[eA + ql] = sc;
                    mrow = fmaxf(mrow, sc);
                }
                if (rB != rA) {
                    // row rA ends with this batch
#pragma unroll
                    for (int off = 4; off > 0; off >>= 1) mrow = fmaxf(mrow, __shfl_xor_sync(qmask, mrow, off, 8));
                    if (ql == 0) mx[rA] = mrow;
                    mrow = -INFINITY;
                }
                rA = rB; eA = eB; qA = qB;
                rB = rC; eB = eC; qB = qC; jB = jC;
            };
            while (rA < cnt) {
                step(kA, kB);
                if (rA >= cnt) break;
                step(kB, kA);
            }
        }
        __syncwarp(qmask);                        // the window's smem is rewritten next
        Rw += cnt;
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
constexpr int kSBufs = 5;                // TMEM S buffers (64 columns each), columns 0..319
constexpr int kGcCol0 = 320;             // q_i . k_G (out-of-window globals): 2 x 32 columns
constexpr int kGrCol0 = 384;             // q_G . k_j of the tile's own keys: 2 chunks x 64 columns
constexpr int kGBufBytes = kBandMaxGlobals * 128;   // k or q rows of the globals (bf16, 128-byte swizzle)
constexpr int kBTmemCols = 512;
constexpr int kQBytes = kTileRows * kHeadDim * 2;
constexpr int kKBytes = kSChunk * kHeadDim * 2;
// the globals' q rows (the A operand of the global rows' scores; its descriptor
// spans 16 KB, so the buffers sit in front of larger ones) and k rows, 2 of each
constexpr int kBSmemUsed = 1024 + 2 * kQBytes + 2 * 2 * kGBufBytes + kKStages * kKBytes +
                           2 * band::kChunkImageBytes + 2 * kRowThreads * 4 + 512 + 4 * kBandMaxGlobals;
// request at least 120 KB so that the shared memory alone keeps it to one CTA per SM
constexpr int kBSmemBytes = kBSmemUsed > 120 * 1024 ? kBSmemUsed : 120 * 1024;
constexpr float kLog2e = 1.4426950408889634f;

// The two warps of TMEM lane quadrant 0 (lanes = global slots s): the global
// rows' raw scores against the tile's own keys (half hcol: keys i0 + 64 hcol
// .. +63), stored in A_gr.
__device__ __forceinline__ void global_row_scores(const ScoreArgs& a, int64_t u, int64_t i0, int lt, int hcol,
                                                  int lane, uint32_t tmem, uint64_t* full_GR,
                                                  uint64_t* empty_GR, int* status) {
    const BandPlan& P = a.plan;
    ptx::mbar_wait(full_GR, lt & 1, status);
    __syncwarp();
    ptx::tc_fence_after();
    float v0[32], v1[32];
    ptx::tmem_ld32(tmem + kGrCol0 + kSChunk * hcol, v0);
    ptx::tmem_ld32(tmem + kGrCol0 + kSChunk * hcol + 32, v1);
    ptx::tc_fence_before();
    ptx::mbar_arrive(empty_GR);
    const int64_t jb = i0 + kSChunk * hcol;
    if (lane < P.g && jb < P.n) {
        float* dst = a.w.A_gr + ((size_t)u * P.g + lane) * P.n + jb;
        if (jb + kSChunk <= P.n && (P.n & 3) == 0) {
#pragma unroll
            for (int c = 0; c < 8; ++c)
                reinterpret_cast<float4*>(dst)[c] = make_float4(v0[4 * c] * kScale, v0[4 * c + 1] * kScale,
                                                                v0[4 * c + 2] * kScale, v0[4 * c + 3] * kScale);
#pragma unroll
            for (int c = 0; c < 8; ++c)
                reinterpret_cast<float4*>(dst + 32)[c] = make_float4(v1[4 * c] * kScale, v1[4 * c + 1] * kScale,
                                                                     v1[4 * c + 2] * kScale, v1[4 * c + 3] * kScale);
        } else {
            const int nk = (int)(P.n - jb < kSChunk ? P.n - jb : kSChunk);
#pragma unroll
            for (int k = 0; k < 32; ++k) if (k < nk) dst[k] = v0[k] * kScale;
#pragma unroll
            for (int k = 0; k < 32; ++k) if (32 + k < nk) dst[32 + k] = v1[k] * kScale;
        }
    }
}

// kImages: two passes over the chunks (the row maximum, then e = exp(s - m)
// written as the tile's operand images, and the band part of the row sum).
// Without: one pass, the row maximum alone (the hop kernels recompute the band
// weights and the first hop adds up their sum).  The out-of-window globals'
// weights and the global rows' raw scores are written either way.
template <bool kImages>
__global__ void __launch_bounds__(kBThreads, 1)
score_band_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     ScoreArgs a, int* status) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* sQ = smem;                                   // 2 x 16 KB
    uint8_t* sQG = sQ + 2 * kQBytes;                      // 2 x the globals' q rows
    uint8_t* sKG = sQG + 2 * kGBufBytes;                  // 2 x the globals' k rows
    uint8_t* sK = sKG + 2 * kGBufBytes;                   // kKStages x 8 KB
    uint8_t* sOut = sK + kKStages * kKBytes;                  // 2 x one chunk's weight image
    float* xch = reinterpret_cast<float*>(sOut + 2 * band::kChunkImageBytes);   // [2][256] row partials
    uint64_t* bars = reinterpret_cast<uint64_t*>(xch + 2 * kRowThreads);
    uint64_t* full_Q = bars;                  // [2]
    uint64_t* empty_Q = full_Q + 2;           // [2]
    uint64_t* full_K = empty_Q + 2;           // [kKStages]
    uint64_t* empty_K = full_K + kKStages;
    uint64_t* full_S = empty_K + kKStages;    // [kSBufs]
    uint64_t* empty_S = full_S + kSBufs;
    uint64_t* full_G = empty_S + kSBufs;      // [2] the globals' q and k rows staged
    uint64_t* empty_G = full_G + 2;           // [2]
    uint64_t* full_GR = empty_G + 2;          // the global rows' scores of the tile are in TMEM
    uint64_t* empty_GR = full_GR + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(empty_GR + 1);
    int* sGpos = reinterpret_cast<int*>(tmem_slot + 2);            // the global positions

    const BandPlan& P = a.plan;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nc = P.chunks;                              // the tile's key chunks (from i0 - r64)
    const int per_tile = kImages ? 2 * nc : nc;           // pass 1 (max) [, pass 2 (exp + write)]
    const int64_t total_tiles = a.units * P.tiles;
    const int my_tiles = blockIdx.x < total_tiles
        ? (int)((total_tiles - 1 - blockIdx.x) / gridDim.x + 1) : 0;
    const bool has_g = P.g > 0;
    const int c0 = P.r64 / kSChunk;                       // chunks c0, c0 + 1: the tile's own keys

    if (warp == 1) ptx::tmem_alloc(tmem_slot, kBTmemCols);
    if (tid == 0) {
        for (int s = 0; s < 2; ++s) { ptx::mbar_init(&full_Q[s], 1); ptx::mbar_init(&empty_Q[s], 1); }
        for (int s = 0; s < kKStages; ++s) { ptx::mbar_init(&full_K[s], 1); ptx::mbar_init(&empty_K[s], 1); }
        // the row warps release an S buffer once per warp (lane 0, after the warp has synced)
        for (int s = 0; s < kSBufs; ++s) { ptx::mbar_init(&full_S[s], 1); ptx::mbar_init(&empty_S[s], kRowThreads / 32); }
        for (int s = 0; s < 2; ++s) { ptx::mbar_init(&full_G[s], 1); ptx::mbar_init(&empty_G[s], 1); }
        ptx::mbar_init(full_GR, 1);
        ptx::mbar_init(empty_GR, 64);
        ptx::fence_mbar_init();
    }
    if (tid < kBandMaxGlobals) sGpos[tid] = tid < P.g ? a.gr.globals[tid] : 0;
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // (the whole warp runs the loop; the elected lane issues the copies)
        for (int lt = 0; lt < my_tiles; ++lt) {
            const int64_t tix = blockIdx.x + (int64_t)lt * gridDim.x;
            const int64_t u = tix / P.tiles;
            const int64_t i0 = (tix - u * P.tiles) * kTileRows;
            const int64_t jb = i0 - P.r64;
            const int qb = lt & 1;
            if (lt >= 2) ptx::mbar_wait(&empty_Q[qb], ((lt / 2) - 1) & 1, status);
            __syncwarp();
            if (ptx::elect_one()) {
                ptx::mbar_arrive_expect_tx(&full_Q[qb], kQBytes);
                ptx::tma_load_3d(sQ + qb * kQBytes, &tmQ, &full_Q[qb], 0, (int)i0, (int)u);
            }
            for (int it = 0; it < per_tile; ++it) {
                const int gi = lt * per_tile + it;
                const int c = it % nc, s = gi % kKStages;
                if (gi >= kKStages) ptx::mbar_wait(&empty_K[s], ((gi / kKStages) - 1) & 1, status);
                __syncwarp();
                if (ptx::elect_one()) {
                    ptx::mbar_arrive_expect_tx(&full_K[s], kKBytes);
                    ptx::tma_load_3d(sK + s * kKBytes, &tmK, &full_K[s], 0, (int)(jb + kSChunk * c), (int)u);
                }
            }
        }
    } else if (warp == 1) {
        // (the whole warp runs the loop; the elected lane issues each instruction)
        {
            constexpr uint32_t idesc = ptx::mma_idesc(1, kSChunk);
            const uint32_t idesc_gc = ptx::mma_idesc(1, P.g16 > 0 ? P.g16 : 16);
            for (int lt = 0; lt < my_tiles; ++lt) {
                const int qb = lt & 1;
                ptx::mbar_wait(&full_Q[qb], (lt / 2) & 1, status);
                const uint32_t qa = ptx::smem_u32(sQ + qb * kQBytes);
                const uint32_t qg = ptx::smem_u32(sQG + qb * kGBufBytes);
                if (has_g) {
                    // q_i . k_G for the tile's rows (N = g16) into columns kGcCol0 + 32 (lt & 1)
                    ptx::mbar_wait(&full_G[qb], (lt / 2) & 1, status);
                    __syncwarp();
                    ptx::tc_fence_after();
                    const uint32_t kg = ptx::smem_u32(sKG + qb * kGBufBytes);
#pragma unroll
                    for (int ks = 0; ks < kHeadDim / 16; ++ks)
                        if (ptx::elect_one())
                            ptx::mma_bf16_ss(tmem + kGcCol0 + 32 * qb, ptx::sw128_kmajor_desc(qa + 32 * ks),
                                             ptx::sw128_kmajor_desc(kg + 32 * ks), idesc_gc, ks > 0);
                }
                for (int it = 0; it < per_tile; ++it) {
                    const int gi = lt * per_tile + it;
                    const int s = gi % kKStages, b = gi % kSBufs;
                    ptx::mbar_wait(&full_K[s], (gi / kKStages) & 1, status);
                    if (gi >= kSBufs) ptx::mbar_wait(&empty_S[b], ((gi / kSBufs) - 1) & 1, status);
                    __syncwarp();
                    ptx::tc_fence_after();
                    const uint32_t kb = ptx::smem_u32(sK + s * kKBytes);
#pragma unroll
                    for (int ks = 0; ks < kHeadDim / 16; ++ks)
                        if (ptx::elect_one())
                            ptx::mma_bf16_ss(tmem + kSChunk * b, ptx::sw128_kmajor_desc(qa + 32 * ks),
                                             ptx::sw128_kmajor_desc(kb + 32 * ks), idesc, ks > 0);
                    const int h = it - c0;
                    if (has_g && (h == 0 || h == 1)) {
                        // q_G . k_j for the tile's own keys (the global rows' scores):
                        // rows 0..g-1 of an M = 128 operand whose other rows are not used
                        if (h == 0 && lt >= 1) ptx::mbar_wait(empty_GR, (lt - 1) & 1, status);
                        __syncwarp();
                        ptx::tc_fence_after();
#pragma unroll
                        for (int ks = 0; ks < kHeadDim / 16; ++ks)
                            if (ptx::elect_one())
                                ptx::mma_bf16_ss(tmem + kGrCol0 + kSChunk * h, ptx::sw128_kmajor_desc(qg + 32 * ks),
                                                 ptx::sw128_kmajor_desc(kb + 32 * ks), idesc, ks > 0);
                        if (h == 1 && ptx::elect_one()) {
                            ptx::mma_commit(full_GR);
                            ptx::mma_commit(&empty_G[qb]);
                        }
                    }
                    if (ptx::elect_one()) {
                        ptx::mma_commit(&empty_K[s]);
                        ptx::mma_commit(&full_S[b]);
                    }
                }
                if (ptx::elect_one()) ptx::mma_commit(&empty_Q[qb]);
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
                if (has_g && uses > 0) ptx::mbar_wait(&empty_G[s], (uses - 1) & 1, status);
            }
        }
    } else if (warp == 2) {
        // the globals' q rows (A operand of the global rows' scores) and k rows
        // (B operand of the out-of-window globals' scores) of the tile's unit,
        // 128-byte swizzled: row s, 16-byte piece c at s * 128 + (c ^ (s % 8)) * 16
        if (has_g) {
            for (int lt = 0; lt < my_tiles; ++lt) {
                const int64_t tix = blockIdx.x + (int64_t)lt * gridDim.x;
                const int64_t u = tix / P.tiles;
                const int qb = lt & 1;
                if (lt >= 2) ptx::mbar_wait(&empty_G[qb], ((lt / 2) - 1) & 1, status);
                for (int e = lane; e < kBandMaxGlobals * 8; e += 32) {
                    const int sl = e >> 3, cch = e & 7;
                    uint4 qv = make_uint4(0u, 0u, 0u, 0u), kv = qv;
                    if (sl < P.g) {
                        const size_t off = ((size_t)u * P.n + a.gr.globals[sl]) * kHeadDim;
                        qv = __ldg(reinterpret_cast<const uint4*>(a.Q + off) + cch);
                        kv = __ldg(reinterpret_cast<const uint4*>(a.K + off) + cch);
                    }
                    const int o = sl * 128 + ((cch ^ (sl & 7)) << 4);
                    *reinterpret_cast<uint4*>(sQG + qb * kGBufBytes + o) = qv;
                    *reinterpret_cast<uint4*>(sKG + qb * kGBufBytes + o) = kv;
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&full_G[qb]);
            }
        }
    } else if (warp < kRowWarp0) {
        // warp 3: pull V into L2 (32 KB pieces round-robin over the CTAs) for the
        // first hop's gathers and band tiles, which read it right after this kernel
        if (a.Vpre && lane == 0) {
            constexpr size_t kPiece = 32768;
            for (size_t off = (size_t)blockIdx.x * kPiece; off < a.vbytes; off += (size_t)gridDim.x * kPiece) {
                const size_t len = a.vbytes - off < kPiece ? a.vbytes - off : kPiece;
                ptx::bulk_prefetch_l2(a.Vpre + off, (uint32_t)len);
            }
        }
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
            int64_t lo, hi;
            band::window_of(P, i, lo, hi);
            // this tile's weight image in global memory; a chunk's image is built
            // in shared memory (row t of a plane at 1024 (t / 8) + 128 (t % 8),
            // 16-byte slot q of the row at q ^ (t % 8)) and written by one bulk copy
            uint8_t* timg = reinterpret_cast<uint8_t*>(a.w.A_band) +
                            (size_t)(u * P.tiles + (i0 / kTileRows)) * P.chunks * band::kChunkImageBytes;
            const int trow = (t >> 3) * 1024 + (t & 7) * 128;
            float mraw = -INFINITY;               // max of the raw dot products q.k (unscaled)
            float m = 0.f, b2 = 0.f, lsum = 0.f;
            // the extras' maximum from score_sparse_kernel, loaded now so that its
            // latency passes under the tile's chunks (this row is rewritten only at the
            // tile's end, by this thread)
            const float ms_pre = row_ok ? a.w.m_sparse[(size_t)u * P.n + i] : 0.f;
            // both column halves of a row agree on the row maximum (band, the
            // out-of-window globals, and the extras from score_sparse_kernel)
            auto transition = [&]() {
                xch[rtid] = mraw;
                ptx::named_barrier_sync(pair_bar, 64);
                const float other = xch[(rtid + 128) & 255];
                m = fmaxf(ms_pre, fmaxf(mraw, other) * kScale);
                if (has_g) {
                    float gs[32];
                    ptx::tmem_ld32(tmem + lane_base + kGcCol0 + 32 * (lt & 1), gs);
#pragma unroll
                    for (int sl = 0; sl < kBandMaxGlobals; ++sl) {
                        if (sl < P.g) {
                            const int64_t j = sGpos[sl];
                            if (row_ok && band::reads_global_outside(P, j, lo, hi))
                                m = fmaxf(m, gs[sl] * kScale);
                        }
                    }
                    if (quad == 0) global_row_scores(a, u, i0, lt, hcol, lane, tmem, full_GR, empty_GR, status);
                }
                b2 = m * kLog2e;
                ptx::named_barrier_sync(pair_bar, 64);     // xch is reused below
            };
            for (int it = 0; it < per_tile; ++it) {
                const int gi = lt * per_tile + it;
                const int b = gi % kSBufs, c = it % nc;
                const bool pass2 = it >= nc;
                if (kImages && it == nc) transition();
                ptx::mbar_wait(&full_S[b], (gi / kSBufs) & 1, status);
                __syncwarp();
                ptx::tc_fence_after();
                float sv[32];
                ptx::tmem_ld32(tmem + lane_base + kSChunk * b + 32 * hcol, sv);
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&empty_S[b]);
                const int64_t j0 = jb + kSChunk * c + 32 * hcol;
                const bool full_in = row_ok && j0 >= lo && j0 + 31 <= hi;
                const bool none_in = !row_ok || j0 > hi || j0 + 31 < lo;
                if (!pass2) {
                    // four independent maxima (the max is exact in any order), then combined
                    float m4[4] = {mraw, -INFINITY, -INFINITY, -INFINITY};
                    if (full_in) {
#pragma unroll
                        for (int k = 0; k < 32; ++k) m4[k & 3] = fmaxf(m4[k & 3], sv[k]);
                    } else if (!none_in) {
                        const int dlo = (int)(lo - j0), dhi = (int)(hi - j0);   // in-window keys k in [dlo, dhi]
#pragma unroll
                        for (int k = 0; k < 32; ++k)
                            if (k >= dlo && k <= dhi) m4[k & 3] = fmaxf(m4[k & 3], sv[k]);
                    }
                    mraw = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
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
            if (!kImages) transition();
            if (has_g) {
                // the out-of-window globals: e = exp(s - m) as the tile's operand image
                // (this half's slots 8 hcol .. +7 and 16 + 8 hcol .. +7; 0 inside the window)
                float gs[32];
                ptx::tmem_ld32(tmem + lane_base + kGcCol0 + 32 * (lt & 1), gs);
                uint8_t* img = a.w.A_gcimg + (size_t)tix * 2 * band::gc_plane_bytes(P.g16);
#pragma unroll
                for (int q8 = 0; q8 < kBandMaxGlobals / 8; ++q8) {
                    if ((q8 & 1) != hcol || 8 * q8 >= P.g16) continue;
                    uint32_t hw[4], lw[4];
#pragma unroll
                    for (int p2 = 0; p2 < 4; ++p2) {
                        float x[2];
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2) {
                            const int sl = 8 * q8 + 2 * p2 + h2;
                            const int64_t j = sGpos[sl < P.g ? sl : 0];
                            x[h2] = (row_ok && sl < P.g && band::reads_global_outside(P, j, lo, hi))
                                        ? ptx::ex2_approx(fmaf(gs[sl], a_sc, -b2)) : 0.f;
                            lsum += x[h2];
                        }
                        const __nv_bfloat162 hh = __floats2bfloat162_rn(x[0], x[1]);
                        const __nv_bfloat162 ll =
                            __floats2bfloat162_rn(x[0] - __low2float(hh), x[1] - __high2float(hh));
                        hw[p2] = *reinterpret_cast<const uint32_t*>(&hh);
                        lw[p2] = *reinterpret_cast<const uint32_t*>(&ll);
                    }
                    uint8_t* pe = img + band::gc_offset(t, 8 * q8, P.g16);
                    *reinterpret_cast<uint4*>(pe) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                    *reinterpret_cast<uint4*>(pe + band::gc_plane_bytes(P.g16)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                }
            }
            // the row's maximum m_i and the band and globals' part of its sum
            // (score_finalize_kernel adds the extras)
            xch[rtid] = lsum;
            ptx::named_barrier_sync(pair_bar, 64);
            if (hcol == 0 && row_ok) {
                a.w.inv_l[(size_t)u * P.n + i] = lsum + xch[rtid + 128];
                a.w.m_sparse[(size_t)u * P.n + i] = m;
            }
            ptx::named_barrier_sync(pair_bar, 64);     // xch is reused by the next tile
        }
        if (kImages && pair_leader) ptx::bulk_wait<0>();     // the last images are written before exit
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) ptx::tmem_dealloc(tmem, kBTmemCols);
}

// ---------------------------------------------------------------- global rows' weights
// One CTA per (unit, global row s): the row's max and sum of exp over the keys
// it reads (all n; on the causal graph 0 .. its own position), by fixed-order
// tree reductions, then A_gr = exp(s - max) / sum in place and row s of every
// tile's global-row operand image (hi / lo bf16; keys it does not read are 0).
constexpr int kNormThreads = 256;

__global__ void __launch_bounds__(kNormThreads)
score_global_norm_kernel(ScoreArgs a) {
    __shared__ float red[kNormThreads / 32];
    const BandPlan& P = a.plan;
    const int64_t u = blockIdx.x / P.g;
    const int sl = (int)(blockIdx.x - u * P.g);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float* row = a.w.A_gr + ((size_t)u * P.g + sl) * P.n;
    const int64_t nread = P.causal ? (int64_t)a.gr.globals[sl] + 1 : P.n;   // keys 0 .. nread-1
    float mx = -INFINITY;
    for (int64_t j = tid; j < nread; j += kNormThreads) mx = fmaxf(mx, row[j]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    mx = red[0];
#pragma unroll
    for (int w = 1; w < kNormThreads / 32; ++w) mx = fmaxf(mx, red[w]);
    __syncthreads();
    float l = 0.f;
    for (int64_t j = tid; j < nread; j += kNormThreads) l += expf(row[j] - mx);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
    if (lane == 0) red[warp] = l;
    __syncthreads();
    l = 0.f;
#pragma unroll
    for (int w = 0; w < kNormThreads / 32; ++w) l += red[w];
    const float inv = 1.f / l;
    if (tid == 0) {
        a.w.gstat[((size_t)u * P.g + sl) * 2] = mx;
        a.w.gstat[((size_t)u * P.g + sl) * 2 + 1] = inv;
    }
    const int64_t nkeys = (int64_t)P.tiles * kTileRows;
    for (int64_t j = tid; j < nkeys; j += kNormThreads) {
        float w = 0.f;
        if (j < nread) w = expf(row[j] - mx) * inv;
        if (j < P.n) row[j] = w;
        const int64_t tile = j / kTileRows;
        const int jj = (int)(j - tile * kTileRows), h = jj >> 6, k = jj & 63;
        uint8_t* pe = a.w.A_gimg + (size_t)(u * P.tiles + tile) * band::kGImgBytes + h * 2 * band::kGImgPlaneBytes +
                      (sl >> 3) * 1024 + (sl & 7) * 128 + ((((k >> 3) ^ (sl & 7))) << 4) + (k & 7) * 2;
        const __nv_bfloat16 hi = __float2bfloat16_rn(w);
        *reinterpret_cast<__nv_bfloat16*>(pe) = hi;
        *reinterpret_cast<__nv_bfloat16*>(pe + band::kGImgPlaneBytes) = __float2bfloat16_rn(w - __bfloat162float(hi));
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
    int64_t lo, hi;
    band::window_of(P, i, lo, hi);
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
    s.Q = nullptr;
    s.K = nullptr;
    s.Vpre = nullptr;
    s.vbytes = 0;
    return s;
}

}  // namespace

int launch_band_scores(const diffuser_graph* g, const BandPlan& p, int64_t units, const void* Q,
                       const void* K, const void* V, char* ws, const BandLayout& L, bool weights_out,
                       cudaStream_t stream) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(score_band_tc_kernel<true>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, kBSmemBytes);
        if (attr_err == cudaSuccess)
            attr_err = cudaFuncSetAttribute(score_band_tc_kernel<false>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize, kBSmemBytes);
    });
    if (attr_err != cudaSuccess) return cuda_fail(attr_err, "cudaFuncSetAttribute(scores)");
    cudaError_t err;
    ScoreArgs a = make_args(g, p, units, ws, L);
    const auto* Qb = static_cast<const __nv_bfloat16*>(Q);
    const auto* Kb = static_cast<const __nv_bfloat16*>(K);
    a.Q = Qb;
    a.K = Kb;
    a.Vpre = static_cast<const uint8_t*>(V);
    a.vbytes = V ? (size_t)units * p.n * kHeadDim * 2 : 0;
    const unsigned grid = (unsigned)(units * p.tiles);
    {
        LaunchScope scope(DIFFUSER_KERNEL_SCORE, stream);
        score_sparse_kernel<<<(unsigned)(sm_count_scores() * kSparseBlocks), kSparseThreads, 0, stream>>>(a, Qb, Kb);
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
    const int num_sms = sm_count_scores();
    const unsigned pgrid = grid < (unsigned)num_sms ? grid : (unsigned)num_sms;
    {
        LaunchScope scope(DIFFUSER_KERNEL_SCORE, stream);
        if (weights_out)
            score_band_tc_kernel<true><<<pgrid, kBThreads, kBSmemBytes, stream>>>(tmQ, tmK, a, g->d_status);
        else
            score_band_tc_kernel<false><<<pgrid, kBThreads, kBSmemBytes, stream>>>(tmQ, tmK, a, g->d_status);
    }
    if ((err = cudaGetLastError()) != cudaSuccess) return cuda_fail(err, "score_band_tc_kernel");
    if (p.g > 0) {
        LaunchScope scope(DIFFUSER_KERNEL_SCORE, stream);
        score_global_norm_kernel<<<(unsigned)(units * p.g), kNormThreads, 0, stream>>>(a);
    }
    if ((err = cudaGetLastError()) != cudaSuccess) return cuda_fail(err, "score_global_norm_kernel");
    if (!weights_out) return DIFFUSER_OK;
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
