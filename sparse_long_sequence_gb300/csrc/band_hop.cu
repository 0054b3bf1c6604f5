// Diffusion hops of the band path (token graphs, bf16 I/O), over the weight
// layout described in band_common.cuh (unnormalized e_ij plus 1/l_i).
// Row i's stored window starts on a multiple of 4 keys, so the 32 keys of a
// chunk are eight 16-byte pieces of the row's storage: each row thread
// streams its own pieces with cp.async (de-skewing for free) and no two
// threads share a shared-memory slot.
//
// Hop Z_{k+1} = (1-alpha) A Z_k + alpha V ("Diffuser...", sec 2.4 eq S.7):
//   band:    tcgen05 MMA, M = 128 rows, N = 64 features, K = 32 keys per chunk,
//            3xTF32 split (hi = operand as stored, which the tensor core
//            truncates to tf32; lo = operand - trunc(operand)):
//            e_hi*Z_hi + e_hi*Z_lo + e_lo*Z_hi, fp32 accumulation in TMEM.
//   gcol, extras: warp-cooperative gathers of 256-byte Z_k rows, fp32 FMA
//            (hop_sparse_kernel, into a per-row partial).
//   global rows:  every tile adds its keys' share; the last tile of a unit
//            sums the shares (fixed order) and writes the global rows.
//   epilogue: z_i = (1 - alpha) * inv_l_i * (band_i + partial_i) + alpha * V_i.
// Z_k lives in three fp32 planes: row-major (for gathers) and transposed
// raw/lo planes (the K-major B operand of the MMA).
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
using band::tf32_trunc;
constexpr int kChunkKeys = 32;
// One CTA per SM: with two co-resident CTAs of this kernel, stale shared-memory
// tiles were observed in the first chunk of some tiles, so the kernel claims a
// whole SM (its shared memory alone rules out a second CTA) and uses the room
// for deeper pipelines.
// warps 0-7: A splitters (two per TMEM lane quadrant, 16 columns each),
// warps 8-11: epilogue, warp 12: TMA producer, warp 13: MMA issuer
constexpr int kThreads = 448;
constexpr int kSplitThreads = 256;
constexpr int kEpiWarp0 = 8, kTmaWarp = 12, kMmaWarp = 13;
constexpr int kAStages = 6;              // per-thread cp.async ring of A chunks (16 KB per stage)
constexpr int kZStages = 4;              // smem stages of Z^T hi+lo (16 KB each)
constexpr int kAccCols = 128;            // two 64-column accumulators (double-buffered tiles)
constexpr int kTStages = 6;              // TMEM stages of A hi+lo (64 columns each)
constexpr int kTmemCols = 512;
constexpr int kPStride = 68;             // floats per row of the gather partial buffer
constexpr int kAStageBytes = kTileRows * kChunkKeys * 4;
constexpr int kZPlaneBytes = kHeadDim * kChunkKeys * 4;
constexpr int kSmemBytes = 1024 + kAStages * kAStageBytes + kZStages * 2 * kZPlaneBytes +
                           kTileRows * kPStride * 4 + 256;
static_assert(kSmemBytes > 116 * 1024, "must exclude a second CTA per SM");
static_assert(kAccCols + 64 * kTStages <= kTmemCols, "TMEM columns");


struct HopArgs {
    BandPlan plan;
    int64_t units;
    float alpha;
    const uint8_t* is_global;
    const int32_t* globals;
    const int64_t* x_ptr;
    const int32_t* x_col;
    int64_t nx;
    const float* A_gc;
    const float* A_x;
    const float* A_gr;    // normalized global-row weights [units][g][n]
    const float* inv_l;   // [units][n]
    const void* Zr_in;    // hop 0: V (bf16); otherwise fp32 row-major Z_k
    const __nv_bfloat16* V;
    float* Zr_out;
    float* Zt_out;
    float* Ztl_out;
    __nv_bfloat16* out;   // last hop
    float* gpart;         // [units][tiles][g][64]
    int* counters;        // [units]
    int* status;
    float* Psum;          // [units][n][64]: gathered part of (A Z_k) per row
    const float* A_band;  // band weights, units x band_unit bytes
};

__device__ __forceinline__ void fma4(float4& acc, float w, const float4& z) {
    acc.x = fmaf(w, z.x, acc.x);
    acc.y = fmaf(w, z.y, acc.y);
    acc.z = fmaf(w, z.z, acc.z);
    acc.w = fmaf(w, z.w, acc.w);
}

template <bool kHop0, bool kLast>
__global__ void __launch_bounds__(kThreads, 1)
hop_band_kernel(const __grid_constant__ CUtensorMap tmZt, const __grid_constant__ CUtensorMap tmZl,
                HopArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* sA = smem;                                          // kAStages x 16 KB
    uint8_t* sZ = sA + kAStages * kAStageBytes;                  // kZStages x (hi 8 KB, lo 8 KB)
    float* sP = reinterpret_cast<float*>(sZ + kZStages * 2 * kZPlaneBytes);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sP + kTileRows * kPStride);
    uint64_t* full_tA = bars;
    uint64_t* empty_tA = full_tA + kTStages;
    uint64_t* full_Z = empty_tA + kTStages;
    uint64_t* empty_Z = full_Z + kZStages;
    uint64_t* acc_full = empty_Z + kZStages;                     // [2]
    uint64_t* acc_empty = acc_full + 2;                          // [2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);

    const BandPlan& P = a.plan;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int chunks = P.chunks;
    const int64_t total_tiles = a.units * P.tiles;
    // tiles of this CTA: blockIdx.x, blockIdx.x + gridDim.x, ...
    const int my_tiles = blockIdx.x < total_tiles
        ? (int)((total_tiles - 1 - blockIdx.x) / gridDim.x + 1) : 0;

    if (warp == kMmaWarp) ptx::tmem_alloc(tmem_slot, kTmemCols);
    if (tid == 0) {
        for (int s = 0; s < kTStages; ++s) { ptx::mbar_init(&full_tA[s], kSplitThreads); ptx::mbar_init(&empty_tA[s], 1); }
        for (int s = 0; s < kZStages; ++s) { ptx::mbar_init(&full_Z[s], 1); ptx::mbar_init(&empty_Z[s], 1); }
        for (int s = 0; s < 2; ++s) { ptx::mbar_init(&acc_full[s], 1); ptx::mbar_init(&acc_empty[s], 128); }
        ptx::fence_mbar_init();
    }
    if (warp == kTmaWarp && lane == 0) {
        ptx::prefetch_tensormap(&tmZt);
        if (!kHop0) ptx::prefetch_tensormap(&tmZl);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kTmaWarp) {
        // ---------------- TMA producer
        if (lane == 0) {
            for (int lt = 0; lt < my_tiles; ++lt) {
                const int64_t tix = blockIdx.x + (int64_t)lt * gridDim.x;
                const int64_t u = tix / P.tiles;
                const int64_t i0 = (tix - u * P.tiles) * kTileRows;
                const int64_t jb = i0 - P.r_up;
                for (int c = 0; c < chunks; ++c) {
                    const int gc = lt * chunks + c;
                    const int sz = gc % kZStages;
                    if (gc >= kZStages) ptx::mbar_wait(&empty_Z[sz], ((gc / kZStages) - 1) & 1, a.status);
                    uint8_t* zdst = sZ + sz * 2 * kZPlaneBytes;
                    ptx::mbar_arrive_expect_tx(&full_Z[sz], kHop0 ? kZPlaneBytes : 2 * kZPlaneBytes);
                    const int key = (int)(jb + kChunkKeys * c);
                    ptx::tma_load_3d(zdst, &tmZt, &full_Z[sz], key, 0, (int)u);
                    if (!kHop0) ptx::tma_load_3d(zdst + kZPlaneBytes, &tmZl, &full_Z[sz], key, 0, (int)u);
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issuer: accumulator lt & 1 of TMEM columns [64 (lt & 1), +64)
        if (lane == 0) {
            constexpr uint32_t idesc = ptx::mma_idesc(2, kHeadDim);
            for (int lt = 0; lt < my_tiles; ++lt) {
                const int ab = lt & 1;
                if (lt >= 2) ptx::mbar_wait(&acc_empty[ab], ((lt / 2) - 1) & 1, a.status);
                ptx::tc_fence_after();
                const uint32_t dacc = tmem + 64 * ab;
                for (int c = 0; c < chunks; ++c) {
                    const int gc = lt * chunks + c;
                    const int ta = gc % kTStages, sz = gc % kZStages;
                    ptx::mbar_wait(&full_tA[ta], (gc / kTStages) & 1, a.status);
                    ptx::mbar_wait(&full_Z[sz], (gc / kZStages) & 1, a.status);
                    ptx::tc_fence_after();
                    const uint32_t zhi = ptx::smem_u32(sZ + sz * 2 * kZPlaneBytes);
                    const uint32_t zlo = zhi + kZPlaneBytes;
#pragma unroll
                    for (int k = 0; k < kChunkKeys / 8; ++k) {
                        const uint32_t a_hi = tmem + kAccCols + 64 * ta + 8 * k;
                        const uint32_t a_lo = a_hi + 32;
                        const uint64_t bhi = ptx::sw128_kmajor_desc(zhi + 32 * k);
                        ptx::mma_tf32_ts(dacc, a_hi, bhi, idesc, (c | k) != 0);
                        if (!kHop0) ptx::mma_tf32_ts(dacc, a_hi, ptx::sw128_kmajor_desc(zlo + 32 * k), idesc, 1);
                        ptx::mma_tf32_ts(dacc, a_lo, bhi, idesc, 1);
                    }
                    ptx::mma_commit(&empty_tA[ta]);
                    ptx::mma_commit(&empty_Z[sz]);
                }
                ptx::mma_commit(&acc_full[ab]);
            }
            // Drain: the commits arrive asynchronously when the MMAs finish.  Wait
            // for the last phase of every empty barrier so that no arrival can land
            // in this shared memory after the CTA exits.
            const int total = my_tiles * chunks;
            for (int s = 0; s < kTStages; ++s) {
                const int uses = (total - s + kTStages - 1) / kTStages;
                if (uses > 0) ptx::mbar_wait(&empty_tA[s], (uses - 1) & 1, a.status);
            }
            for (int s = 0; s < kZStages; ++s) {
                const int uses = (total - s + kZStages - 1) / kZStages;
                if (uses > 0) ptx::mbar_wait(&empty_Z[s], (uses - 1) & 1, a.status);
            }
        }
    } else if (warp < kEpiWarp0) {
        // ---------------- A splitters.  Warp w serves TMEM lane quadrant w % 4 (rows
        // 32 (w % 4) .. +31) and columns 16 (w / 4) .. +15 of every 32-key chunk.
        // Each thread streams its own 64-byte share of its row's stored window
        // with cp.async into its slot of a ring (zero fill outside the row's
        // storage), then writes the masked hi / lo split into the TMEM A stage.
        // Only the thread itself reads its slot: cp.async.wait_group is the only
        // synchronization the copies need.
        const int quad = warp & 3, hcol = warp >> 2;
        const int t = quad * 32 + lane;          // row within the tile
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        // this thread's four 16-byte pieces inside a stage (row t, columns 16 hcol ..)
        const uint32_t slot0 = ptx::smem_u32(sA) + t * 128;
        uint32_t piece_off[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) piece_off[q] = (uint32_t)(((4 * hcol + q) ^ (t & 7)) << 4);
        const int wbase = 16 * hcol - 4 * (t / 4);   // window column of the thread's first key, chunk 0
        // copy cursor: chunk (cl, cc) of this CTA's tile sequence, advanced one chunk per refill
        int cl = 0, cc = 0, cslot = 0;
        const float* crow = nullptr;
        bool crow_ok = false;
        auto set_row = [&](int lx) {
            const int64_t tix = blockIdx.x + (int64_t)lx * gridDim.x;
            const int64_t u = tix / P.tiles;
            const int64_t i = (tix - u * P.tiles) * kTileRows + t;
            crow_ok = i < P.n;
            crow = a.A_band + (size_t)u * (P.band_unit / 4) + (size_t)(crow_ok ? i : 0) * P.W;
        };
        auto issue = [&]() {
            if (cl < my_tiles) {
                const int w0 = wbase + kChunkKeys * cc;
                const uint32_t dst = slot0 + (uint32_t)(cslot * kAStageBytes);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int w = w0 + 4 * q;
                    const bool ok = crow_ok && w >= 0 && w < P.W;
                    ptx::cp_async16(dst + piece_off[q], ok ? crow + w : crow, ok ? 16 : 0);
                }
                if (++cc == chunks) {
                    cc = 0;
                    if (++cl < my_tiles) set_row(cl);
                }
                if (++cslot == kAStages) cslot = 0;
            }
            ptx::cp_async_commit();
        };
        if (my_tiles > 0) set_row(0);
        for (int gx = 0; gx < kAStages; ++gx) issue();
        int rslot = 0, ta = 0;                   // smem slot and TMEM stage of chunk gc
        int gc = 0;
        for (int lt = 0; lt < my_tiles; ++lt) {
            const int64_t tix = blockIdx.x + (int64_t)lt * gridDim.x;
            const int64_t u = tix / P.tiles;
            const int64_t i0 = (tix - u * P.tiles) * kTileRows;
            const int64_t i = i0 + t;
            const bool row_ok = i < P.n && !a.is_global[i < P.n ? i : 0];
            const int64_t lo_key = i - P.r < 0 ? 0 : i - P.r;
            const int64_t hi_key = i + P.r > P.n - 1 ? P.n - 1 : i + P.r;
            // keys of this thread's columns relative to lo_key / hi_key, chunk 0
            const int jrel_lo = (int)(i0 - P.r_up + 16 * hcol - lo_key);
            const int jrel_hi = (int)(hi_key - (i0 - P.r_up + 16 * hcol));
            for (int c = 0; c < chunks; ++c, ++gc) {
                ptx::cp_async_wait<kAStages - 1>();
                float hi[16], lo[16];
                const uint8_t* rowp = sA + rslot * kAStageBytes + t * 128;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 x = *reinterpret_cast<const float4*>(rowp + piece_off[q]);
                    hi[4 * q + 0] = x.x; hi[4 * q + 1] = x.y; hi[4 * q + 2] = x.z; hi[4 * q + 3] = x.w;
                }
                // first key of the segment minus lo_key, and hi_key minus it
                const int d_lo = jrel_lo + kChunkKeys * c;
                const int d_hi = jrel_hi - kChunkKeys * c;
                if (!(row_ok && d_lo >= 0 && d_hi >= 15)) {
                    // partly (or not at all) inside the row's window
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        hi[k] = (row_ok && d_lo + k >= 0 && k <= d_hi) ? hi[k] : 0.f;
                }
#pragma unroll
                for (int k = 0; k < 16; ++k) lo[k] = hi[k] - tf32_trunc(hi[k]);
                if (gc >= kTStages) ptx::mbar_wait(&empty_tA[ta], ((gc / kTStages) - 1) & 1, a.status);
                __syncwarp();   // lanes leave the spin at different times; tcgen05.st is warp-collective
                ptx::tc_fence_after();
                const uint32_t col = tmem + lane_base + kAccCols + 64 * ta + 16 * hcol;
                ptx::tmem_st16x2(col, hi, col + 32, lo);
                ptx::tc_fence_before();
                ptx::mbar_arrive(&full_tA[ta]);
                issue();                         // refill the slot just read (its data are in TMEM now)
                if (++rslot == kAStages) rslot = 0;
                if (++ta == kTStages) ta = 0;
            }
        }
        ptx::cp_async_wait<0>();
    } else {
        // ---------------- epilogue: accumulator + gathered part, restart term, outputs
        const int q = warp - kEpiWarp0;          // TMEM lane quadrant and row block
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        for (int lt = 0; lt < my_tiles; ++lt) {
            const int64_t tix = blockIdx.x + (int64_t)lt * gridDim.x;
            const int64_t u = tix / P.tiles;
            const int64_t i0 = (tix - u * P.tiles) * kTileRows;
            // stage this block's gathered partial sums (coalesced) while the MMAs run
            for (int rr = 0; rr < 32; ++rr) {
                const int t = q * 32 + rr;
                const int64_t i = i0 + t;
                float2 pv = make_float2(0.f, 0.f);
                if (i < P.n)
                    pv = __ldg(reinterpret_cast<const float2*>(a.Psum + ((size_t)u * P.n + i) * kHeadDim) + lane);
                sP[t * kPStride + 2 * lane] = pv.x;
                sP[t * kPStride + 2 * lane + 1] = pv.y;
            }
            __syncwarp();
            const int ab = lt & 1;
            ptx::mbar_wait(&acc_full[ab], (lt / 2) & 1, a.status);
            __syncwarp();       // reconverge before the warp-collective tcgen05.ld
            ptx::tc_fence_after();
            const int t = q * 32 + lane;
            const int64_t i = i0 + t;
            const bool row_ok = i < P.n && !a.is_global[i < P.n ? i : 0];
            const float keep = (1.f - a.alpha) * (row_ok ? __ldg(a.inv_l + (size_t)u * P.n + i) : 0.f);
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                float d[32];
                ptx::tmem_ld32(tmem + lane_base + 64 * ab + 32 * half, d);
                if (half == 1) {
                    // both halves of this accumulator are in registers: hand it back
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(&acc_empty[ab]);
                }
                if (!row_ok) continue;
                const size_t row = ((size_t)u * P.n + i) * kHeadDim + 32 * half;
                const uint4* vp = reinterpret_cast<const uint4*>(a.V + row);
                float z[32];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 vv = __ldg(vp + c);
                    const uint32_t w4[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int k = 8 * c + 2 * e;
                        const float p0 = sP[t * kPStride + 32 * half + k];
                        const float p1 = sP[t * kPStride + 32 * half + k + 1];
                        z[k] = fmaf(keep, d[k] + p0, a.alpha * bf16lo(w4[e]));
                        z[k + 1] = fmaf(keep, d[k + 1] + p1, a.alpha * bf16hi(w4[e]));
                    }
                }
                if (kLast) {
                    uint4* op = reinterpret_cast<uint4*>(a.out + row);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t w4[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            __nv_bfloat162 h = __floats2bfloat162_rn(z[8 * c + 2 * e], z[8 * c + 2 * e + 1]);
                            w4[e] = *reinterpret_cast<uint32_t*>(&h);
                        }
                        op[c] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                } else {
                    float4* zr = reinterpret_cast<float4*>(a.Zr_out + row);
#pragma unroll
                    for (int c = 0; c < 8; ++c) zr[c] = make_float4(z[4 * c], z[4 * c + 1], z[4 * c + 2], z[4 * c + 3]);
                    const size_t tbase = ((size_t)u * kHeadDim + 32 * half) * P.nz + i;
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        a.Zt_out[tbase + (size_t)k * P.nz] = z[k];
                        a.Ztl_out[tbase + (size_t)k * P.nz] = z[k] - tf32_trunc(z[k]);
                    }
                }
            }
            __syncwarp();       // sP is restaged for the next tile
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) ptx::tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------- sparse part of a hop
// One CTA per (unit, 128-row block), 8 warps.  (1) The global rows: this
// block's keys contribute sum_j A_gr[s][j] Z_k[j]; the last block of a unit
// sums the shares in block order and writes Z_{k+1} of the global rows.
// (2) Every other row: the globals outside its window and its random extras,
// gathered as whole Z_k rows with several independent loads in flight, into
// Psum[u][i] (fp32), which the band kernel's epilogue adds.
constexpr int kSparseThreads = 256;
constexpr int kGatherBatch = 8;

// Row j of Z_k for unit u, 4 features per lane (hl = lane within a half-warp).
template <bool kHop0>
struct ZRows {
    const void* base;     // Z_k of this unit, offset to this lane's 4 features
    __device__ __forceinline__ ZRows(const HopArgs& a, int64_t u, int hl) {
        if constexpr (kHop0)
            base = static_cast<const __nv_bfloat16*>(a.Zr_in) + (size_t)u * a.plan.n * kHeadDim + 4 * hl;
        else
            base = static_cast<const float*>(a.Zr_in) + (size_t)u * a.plan.n * kHeadDim + 4 * hl;
    }
    __device__ __forceinline__ float4 operator()(int32_t j) const {
        if constexpr (kHop0) {
            const uint2 w = __ldg(reinterpret_cast<const uint2*>(
                static_cast<const __nv_bfloat16*>(base) + ((uint32_t)j << 6)));
            return make_float4(bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y));
        } else {
            return __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(base) +
                                                         ((uint32_t)j << 6)));
        }
    }
};

template <bool kHop0, bool kLast>
__global__ void __launch_bounds__(kSparseThreads, 4)
hop_sparse_kernel(HopArgs a) {
    extern __shared__ float red[];           // [8 warps][g][65] shares, then [g][64] Z rows of G
    __shared__ int ticket;
    const BandPlan& P = a.plan;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t u = blockIdx.x / P.tiles;
    const int tile = (int)(blockIdx.x - u * P.tiles);
    const int64_t i0 = (int64_t)tile * kTileRows;
    const int g = P.g;
    const int half = lane >> 4, hl = lane & 15;
    const unsigned hmask = 0xffffu << (16 * half);
    const ZRows<kHop0> zrow(a, u, hl);

    if (g > 0) {
        // (1) global rows: this warp's 16 keys j = i0 + 16 warp + jj; half-warp
        //     `half` takes keys jj = half, half + 2, ..., 4 features per lane
        const int64_t jbase = i0 + 16 * warp;
        float4 z[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int64_t j = jbase + 2 * k + half;
            z[k] = j < P.n ? zrow((int32_t)j) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int s = 0; s < g; ++s) {
            // lanes 0..15 fetch the 16 normalized weights of this warp's keys
            const int64_t jl = jbase + hl;
            const float wv = jl < P.n ? __ldg(a.A_gr + ((size_t)u * g + s) * P.n + jl) : 0.f;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < 8; ++k) fma4(acc, __shfl_sync(0xffffffffu, wv, 2 * k + half, 16), z[k]);
            // combine the two half-warps (even / odd keys)
            acc.x += __shfl_xor_sync(0xffffffffu, acc.x, 16);
            acc.y += __shfl_xor_sync(0xffffffffu, acc.y, 16);
            acc.z += __shfl_xor_sync(0xffffffffu, acc.z, 16);
            acc.w += __shfl_xor_sync(0xffffffffu, acc.w, 16);
            if (half == 0) {
                float* r = red + (warp * g + s) * 65 + 4 * hl;
                r[0] = acc.x; r[1] = acc.y; r[2] = acc.z; r[3] = acc.w;
            }
        }
        __syncthreads();
        float* part = a.gpart + (((size_t)u * P.tiles + tile) * g) * kHeadDim;
        for (int e = tid; e < g * kHeadDim; e += kSparseThreads) {
            const int s = e / kHeadDim, dd = e % kHeadDim;
            float sum = 0.f;
#pragma unroll
            for (int w8 = 0; w8 < 8; ++w8) sum += red[(w8 * g + s) * 65 + dd];
            part[e] = sum;
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) ticket = atomicAdd(&a.counters[u], 1);
        __syncthreads();
        if (ticket == P.tiles - 1) {
            __threadfence();
            const float keep = 1.f - a.alpha;
            for (int e = tid; e < g * kHeadDim; e += kSparseThreads) {
                const int s = e / kHeadDim, dd = e % kHeadDim;
                float sum = 0.f;
                for (int tt = 0; tt < P.tiles; ++tt)
                    sum += __ldcg(a.gpart + (((size_t)u * P.tiles + tt) * g + s) * kHeadDim + dd);
                const int64_t gi = a.globals[s];
                const size_t row = ((size_t)u * P.n + gi) * kHeadDim + dd;
                const float zz = fmaf(keep, sum, a.alpha * __bfloat162float(a.V[row]));
                if (kLast) {
                    a.out[row] = __float2bfloat16_rn(zz);
                } else {
                    a.Zr_out[row] = zz;
                    const size_t tr = ((size_t)u * kHeadDim + dd) * P.nz + gi;
                    a.Zt_out[tr] = zz;
                    a.Ztl_out[tr] = zz - tf32_trunc(zz);
                }
            }
            if (tid == 0) a.counters[u] = 0;
        }
        __syncthreads();
        // stage the Z_k rows of the global keys for the out-of-window global columns
        for (int e = tid; e < g * 16; e += kSparseThreads) {
            const int s = e >> 4, q = e & 15;
            const ZRows<kHop0> zq(a, u, q);
            reinterpret_cast<float4*>(red)[e] = zq(a.globals[s]);
        }
        __syncthreads();
    }
    // (2) rows of this block: each half-warp owns a row (16 lanes x 4 features);
    //     kGatherBatch gathers are issued before their FMAs.
    const float* ax = a.A_x + (size_t)u * a.nx;
    const float4* zg = reinterpret_cast<const float4*>(red) + hl;     // Z rows of G, this lane
    for (int rr = 0; rr < 16; rr += 2) {
        const int64_t i = i0 + 16 * warp + rr + half;
        const bool live = i < P.n && !a.is_global[i < P.n ? i : 0];
        if (!live) continue;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        // globals outside the window (weight 0 marks "inside the window")
        const float* wg = a.A_gc + ((size_t)u * P.n + i) * P.g_pad;
        for (int s0 = 0; s0 < g; s0 += 16) {
            const float wv = s0 + hl < g ? __ldg(wg + s0 + hl) : 0.f;
            const int cnt = g - s0 < 16 ? g - s0 : 16;
            for (int b = 0; b < cnt; ++b)
                fma4(acc, __shfl_sync(hmask, wv, b, 16), zg[(s0 + b) * 16]);
        }
        // random extras: (weight, column) pairs fetched 16 at a time; padded
        // slots carry weight 0 and column i, so every batch runs in full
        const int64_t e0 = a.x_ptr[i], e1 = a.x_ptr[i + 1];
        for (int64_t base = e0; base < e1; base += 16) {
            const int64_t e = base + hl;
            const float w_l = e < e1 ? __ldg(ax + e) : 0.f;
            const int32_t j_l = e < e1 ? __ldg(a.x_col + e) : (int32_t)i;
            const int cnt = (e1 - base) < 16 ? (int)(e1 - base) : 16;
            for (int t0 = 0; t0 < cnt; t0 += kGatherBatch) {
                float4 zz[kGatherBatch];
#pragma unroll
                for (int b = 0; b < kGatherBatch; ++b)
                    zz[b] = zrow(__shfl_sync(hmask, j_l, t0 + b, 16));
#pragma unroll
                for (int b = 0; b < kGatherBatch; ++b)
                    fma4(acc, __shfl_sync(hmask, w_l, t0 + b, 16), zz[b]);
            }
        }
        reinterpret_cast<float4*>(a.Psum + ((size_t)u * P.n + i) * kHeadDim)[hl] = acc;
    }
}

// V [units][n][64] bf16 -> transposed fp32 plane [units][64][nz] (Z_0 for the MMA)
__global__ void __launch_bounds__(256)
v_to_zt_kernel(const __nv_bfloat16* __restrict__ V, float* __restrict__ Zt, int64_t n, int64_t nz,
               int64_t units) {
    __shared__ float tile[32][65];
    const int64_t u = blockIdx.y;
    const int64_t j0 = (int64_t)blockIdx.x * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 8 warps
    for (int r = ty; r < 32; r += 8) {
        const int64_t j = j0 + r;
        if (j < n) {
            const __nv_bfloat162 h = reinterpret_cast<const __nv_bfloat162*>(
                V + ((size_t)u * n + j) * kHeadDim)[tx];
            tile[r][2 * tx] = __low2float(h);
            tile[r][2 * tx + 1] = __high2float(h);
        }
    }
    __syncthreads();
    for (int dd = ty; dd < kHeadDim; dd += 8) {
        const int64_t j = j0 + tx;
        if (j < n) Zt[((size_t)u * kHeadDim + dd) * nz + j] = tile[tx][dd];
    }
}

int encode(CUtensorMap* m, int rank, void* base, const cuuint64_t* dims, const cuuint64_t* strides,
           const cuuint32_t* box) {
    auto fn = band::tensor_map_encoder();
    if (!fn) return fail(DIFFUSER_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, rank, base, dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(DIFFUSER_ERR_CUDA, "cuTensorMapEncodeTiled failed: " + std::to_string((int)r));
    return DIFFUSER_OK;
}

template <bool kHop0, bool kLast>
int launch_hop(const CUtensorMap& tmZt, const CUtensorMap& tmZl, const HopArgs& a,
               cudaStream_t stream) {

    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(hop_band_kernel<kHop0, kLast>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (attr_err == cudaSuccess)
            attr_err = cudaFuncSetAttribute(hop_sparse_kernel<kHop0, kLast>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            8 * kBandMaxGlobals * 65 * (int)sizeof(float));
    });
    if (attr_err != cudaSuccess) return cuda_fail(attr_err, "cudaFuncSetAttribute(hop)");
    {
        LaunchScope scope(DIFFUSER_KERNEL_GATHER, stream);
        const size_t shmem = (size_t)8 * a.plan.g * 65 * sizeof(float);
        hop_sparse_kernel<kHop0, kLast><<<(unsigned)(a.units * a.plan.tiles), kSparseThreads,
                                          shmem, stream>>>(a);
    }
    cudaError_t serr = cudaGetLastError();
    if (serr != cudaSuccess) return cuda_fail(serr, "hop_sparse_kernel");
    static int num_sms = 0;
    if (num_sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || num_sms < 1)
            num_sms = 1;
    }
    const int64_t total_tiles = a.units * a.plan.tiles;
    dim3 grid((unsigned)(total_tiles < num_sms ? total_tiles : num_sms));
    {
        LaunchScope scope(DIFFUSER_KERNEL_HOP, stream);
        hop_band_kernel<kHop0, kLast><<<grid, kThreads, kSmemBytes, stream>>>(tmZt, tmZl, a);
    }
    cudaError_t err = cudaGetLastError();
    return err == cudaSuccess ? DIFFUSER_OK : cuda_fail(err, "hop_band_kernel");
}

}  // namespace

namespace band {
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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
}  // namespace band

band::GraphRefs band_graph_refs(const diffuser_graph* g) {
    return band::GraphRefs{g->d_is_global, g->d_gslot, g->d_globals, g->d_x_ptr, g->d_x_col, g->nx};
}

band::Weights band_weights(char* ws, const BandLayout& L) {
    band::Weights w;
    w.A_band = reinterpret_cast<float*>(ws + L.a_band);
    w.A_gc = reinterpret_cast<float*>(ws + L.a_gc);
    w.A_x = reinterpret_cast<float*>(ws + L.a_x);
    w.A_gr = reinterpret_cast<float*>(ws + L.a_gr);
    w.inv_l = reinterpret_cast<float*>(ws + L.inv_l);
    w.m_sparse = reinterpret_cast<float*>(ws + L.m_sparse);
    w.gstat = reinterpret_cast<float*>(ws + L.gstat);
    w.sstat = reinterpret_cast<float*>(ws + L.sstat);
    return w;
}

bool band_plan(const diffuser_graph* g, BandPlan* p) {
    if (g->kind != kTokenGraph || g->r < 8 || g->n_globals > kBandMaxGlobals) return false;
    p->n = g->n;
    p->r = g->r;
    p->r_up = (g->r + 3) / 4 * 4;
    p->W = (p->r_up + g->r + 4 + 3) / 4 * 4;
    p->g = g->n_globals;
    p->g_pad = (g->n_globals + 3) / 4 * 4;
    if (p->g_pad == 0) p->g_pad = 4;
    p->rows4 = (g->n + 3) / 4 * 4;
    p->nz = (g->n + 3) / 4 * 4;
    p->tiles = (int32_t)((g->n + kTileRows - 1) / kTileRows);
    p->chunks = (kTileRows + g->r + p->r_up + kChunkKeys - 1) / kChunkKeys;
    const size_t need = (size_t)p->rows4 * p->W * 4 + 8 * (size_t)p->r_up + 64;
    p->band_unit = (need + 1023) / 1024 * 1024;
    return true;
}

int plan_band_layout(const diffuser_graph* g, const BandPlan& p, int64_t units, BandLayout* L) {
    auto al = [](size_t x) { return (x + 1023) / 1024 * 1024; };
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off += al(bytes); return o; };
    const size_t U = (size_t)units;
    L->a_band = take(U * p.band_unit);
    L->a_gc = take(U * (size_t)p.n * p.g_pad * 4);
    L->a_x = take(U * (size_t)(g->nx > 0 ? g->nx : 1) * 4);
    L->a_gr = take(U * (size_t)(p.g > 0 ? p.g : 1) * p.n * 4);
    for (int s = 0; s < 2; ++s) {
        L->zr[s] = take(U * (size_t)p.n * kHeadDim * 4);
        L->zt[s] = take(U * (size_t)kHeadDim * p.nz * 4);
        L->ztl[s] = take(U * (size_t)kHeadDim * p.nz * 4);
    }
    L->gpart = take(U * (size_t)p.tiles * (p.g > 0 ? p.g : 1) * kHeadDim * 4);
    L->psum = take(U * (size_t)p.n * kHeadDim * 4);
    L->inv_l = take(U * (size_t)p.n * 4);
    L->m_sparse = take(U * (size_t)p.n * 4);
    L->gstat = take(U * (size_t)(p.g > 0 ? p.g : 1) * 2 * 4);
    L->sstat = take(U * (size_t)p.tiles * (p.g > 0 ? p.g : 1) * 2 * 4);
    L->counters = take(U * 4);
    L->total = off;
    return DIFFUSER_OK;
}

int launch_band_hops(const diffuser_graph* g, const BandPlan& p, int64_t units, const void* V,
                     int32_t hops, float alpha, void* out, char* ws, const BandLayout& L,
                     cudaStream_t stream) {
    cudaError_t err;
    float* zt0 = reinterpret_cast<float*>(ws + L.zt[0]);
    {
        dim3 grid((unsigned)((p.n + 31) / 32), (unsigned)units);
        LaunchScope scope(DIFFUSER_KERNEL_AUX, stream);
        v_to_zt_kernel<<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(V), zt0, p.n,
                                                 p.nz, units);
    }
    if ((err = cudaGetLastError()) != cudaSuccess) return cuda_fail(err, "v_to_zt_kernel");
    err = cudaMemsetAsync(ws + L.counters, 0, (size_t)units * 4, stream);
    if (err != cudaSuccess) return cuda_fail(err, "clearing the tile counters");

    // tensor maps of the two transposed Z planes (the MMA's B operand)
    CUtensorMap tmZt[2], tmZl[2];
    for (int s = 0; s < 2; ++s) {
        const cuuint64_t dims[3] = {(cuuint64_t)p.n, (cuuint64_t)kHeadDim, (cuuint64_t)units};
        const cuuint64_t strides[2] = {(cuuint64_t)p.nz * 4, (cuuint64_t)p.nz * 4 * kHeadDim};
        const cuuint32_t box[3] = {32, (cuuint32_t)kHeadDim, 1};
        int st = encode(&tmZt[s], 3, ws + L.zt[s], dims, strides, box);
        if (!st) st = encode(&tmZl[s], 3, ws + L.ztl[s], dims, strides, box);
        if (st) return st;
    }

    HopArgs a;
    a.plan = p;
    a.units = units;
    a.alpha = alpha;
    a.is_global = g->d_is_global;
    a.globals = g->d_globals;
    a.x_ptr = g->d_x_ptr;
    a.x_col = g->d_x_col;
    a.nx = g->nx;
    a.A_gc = reinterpret_cast<const float*>(ws + L.a_gc);
    a.A_x = reinterpret_cast<const float*>(ws + L.a_x);
    a.A_gr = reinterpret_cast<const float*>(ws + L.a_gr);
    a.inv_l = reinterpret_cast<const float*>(ws + L.inv_l);
    a.V = static_cast<const __nv_bfloat16*>(V);
    a.gpart = reinterpret_cast<float*>(ws + L.gpart);
    a.counters = reinterpret_cast<int*>(ws + L.counters);
    a.status = g->d_status;
    a.out = static_cast<__nv_bfloat16*>(out);
    a.Psum = reinterpret_cast<float*>(ws + L.psum);
    a.A_band = reinterpret_cast<const float*>(ws + L.a_band);
    for (int32_t k = 0; k < hops; ++k) {
        const int cur = k & 1, nxt = (k + 1) & 1;
        a.Zr_in = k == 0 ? V : static_cast<const void*>(ws + L.zr[cur]);
        a.Zr_out = reinterpret_cast<float*>(ws + L.zr[nxt]);
        a.Zt_out = reinterpret_cast<float*>(ws + L.zt[nxt]);
        a.Ztl_out = reinterpret_cast<float*>(ws + L.ztl[nxt]);
        const bool first = k == 0, last = k == hops - 1;
        int st;
        if (first && last) st = launch_hop<true, true>(tmZt[cur], tmZl[cur], a, stream);
        else if (first) st = launch_hop<true, false>(tmZt[cur], tmZl[cur], a, stream);
        else if (last) st = launch_hop<false, true>(tmZt[cur], tmZl[cur], a, stream);
        else st = launch_hop<false, false>(tmZt[cur], tmZl[cur], a, stream);
        if (st) return st;
    }
    return DIFFUSER_OK;
}

}  // namespace dfs
