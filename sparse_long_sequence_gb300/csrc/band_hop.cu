// Diffusion hops of the band path (token graphs, bf16 I/O).
//
// Hop Z_{k+1} = (1-alpha) A Z_k + alpha V ("Diffuser...", sec 2.4 eq S.7),
// two kernels per hop:
//   hop_gather_kernel: the random extras of every row not in G, into a
//            per-row partial P_i (whole Z_k rows gathered from L2).  The rows
//            are split over the quarter-warps of the grid; each walks
//            its rows' extras as one stream with several rows in flight, the
//            next slots' indices loading meanwhile; every load instruction
//            reads whole 128-byte lines.  Hops after the first also sum the
//            global rows of Z_k from the previous hop's tile shares.
//   hop_band_kernel (persistent, 128-row tiles): the window part, on tcgen05
//            tensor cores.  The band weights are not stored: per 128-key chunk
//            the kernel recomputes S = Q_tile K_chunk^T (bf16 operands, fp32 in
//            TMEM), turns it into e_ij = exp(s_ij - m_i) with the row maxima of
//            the score pass (0 outside the window), and writes e as bf16 hi + lo
//            (each the bf16 rounding of what is left) over the scores in tensor
//            memory as the A operand of the second MMA: e_hi*[Z_hi | Z_lo] (N = 128)
//            + e_lo*Z_hi (N = 64), fp32 accumulation in TMEM; the e_lo*Z_lo term
//            (below 2^-16 of the product) is the only one left out.  Re-reading
//            the weights from HBM on every hop would cost 4 bytes per edge; the
//            recomputation costs one exp per edge and a small MMA.  The globals
//            outside each row's window are one more K step into the same
//            accumulator (their stored weights' operand image [128 x g16]
//            against the global keys' Z_k rows).  The global rows (full rows
//            of A) ride along: on the chunk(s) that hold the tile's own keys,
//            the same Z_k tiles also multiply the global rows' weights of those
//            keys (a 32-row operand image) into a second accumulator, and each
//            tile writes that share.  Epilogue:
//            z_i = (1 - alpha) * inv_l_i * (band_i + P_i) + alpha * V_i,
//            written as the next [hi | lo] bf16 row and fp32 row, or as the
//            bf16 output.  The first hop also adds up the band part of each
//            row sum and completes inv_l.
// On the causal graph ("Diffuser...", sec 2.6) the window is [i - r, i], a
// tile's key chunks end at its last row, and the gather splits its rows by
// cost (late rows keep more draws) instead of by count.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <mutex>
#include <new>
#include <vector>

#include "band_common.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace dfs {
namespace {

using band::bf16hi;
using band::bf16lo;
using band::kChunkKeys;
using band::kTileRows;
// warp 0: TMA producer of Q and K, warp 1: score MMAs, warp 2: the weights'
// MMAs, warp 3: producer of Z_k, the globals' weight images and the global
// keys' Z_k rows, warps 4-19: the band weights of each chunk (warp w serves
// TMEM lane quadrant w % 4 and keys 16 ((w - 4) / 4) .. +15), warps 20-23: the
// tiles' epilogues (lane quadrant w % 4, all features).  One CTA per SM.
constexpr int kThreads = 768;
constexpr int kTmaWarp = 0, kSMmaWarp = 1, kPvMmaWarp = 2, kZWarp = 3;
constexpr int kSoftWarp0 = 4, kSoftThreads = 512, kSoftWarps = kSoftThreads / 32;   // band weights
constexpr int kEpiWarp0 = 20, kEpiWarps = 4;                                      // epilogue
constexpr int kEpiRowFloats = 68;        // an epilogue staging row (64 features, padded against bank conflicts)
constexpr int kSlices = kSoftWarps / 4;  // weight warps per TMEM lane quadrant (16 keys each)
constexpr int kQBytes = kTileRows * kHeadDim * 2;     // a Q tile, bf16 [128][64]
constexpr int kCK = 2 * kChunkKeys;    // keys per pipeline chunk (two 64-key halves of the key grid)
constexpr int kKBytes = kCK * kHeadDim * 2;           // a K chunk, bf16 [128][64]
constexpr int kSBufs = 2;                // pipeline slots (chunk g uses slot g % 2)
// Chunk g uses slot b = g % kSBufs of everything: its K stage (16 KB), its score /
// weight buffer (128 TMEM columns) and its Z stage (hi tile + lo tile, 32 KB),
// with one barrier per slot and event: full_K (K landed), full_S (scores
// written, K read), full_P (weights written by the 16 weight warps and Z
// landed), pv_done (the weights' MMAs are done: buffer and Z stage free).
// TMEM: the accumulator D in columns [0, 128) ([0,64) P Z_hi, [64,128) P_hi Z_lo)
constexpr int kGlobCol0 = 128;           // the global rows' accumulator, columns [128, 256)
constexpr int kSCol0 = 256;              // score / weight buffers, columns 256 + 128 b
// In buffer b, keys 16 s .. +15 of the chunk hold fp32 scores in columns 16 s .. +15;
// the weight warp of those keys overwrites them with the bf16 pairs of its weights,
// hi in columns 16 s .. +7 and lo in 16 s + 8 .. +15 (the A operand of K step s).
constexpr int kTmemCols = 512;
constexpr int kZTileBytes = kCK * 128;   // a chunk's Z_k rows, one 64-feature half (hi or lo)
constexpr int kZStageBytes = 2 * kZTileBytes;
constexpr float kScale = 0.125f;         // 1/sqrt(64)
constexpr float kLog2e = 1.4426950408889634f;
// Shared memory of a launch.  The global rows' operand image comes first: its
// descriptors span 16 KB past their start (rows 32..127 read whatever
// follows; those rows are not used).  Then 2 Q tiles, the K, Z and weight-image
// rings, the out-of-window globals' weight image (hi, lo; g16 slots) and their
// Z_k rows as an MN-major B tile (hi, lo), the row-sum exchange, barriers.
// The CTA's tiles as a shared-memory table (filled once, read by every role).
constexpr int kMaxCtaTiles = 192;         // the launch keeps each CTA at or below this many tiles
struct TileEntry { int32_t u, t; int16_t c_lo, c_hi; };
__host__ __device__ constexpr int band_smem_bytes(int g16) {
    return 1024 + band::kGImgBytes + 2 * kQBytes + kSBufs * (kKBytes + kZStageBytes) +
           2 * kTileRows * (g16 > 0 ? g16 : 16) * 2 + 2 * (g16 > 0 ? g16 : 16) * 128 +
           2 * kSoftThreads * 4 + 4 * 32 * kEpiRowFloats * 4 + 4 * 32 * 4 + 4 * 32 * kHeadDim * 2 +
           kMaxCtaTiles * (int)sizeof(TileEntry) + 16 + 512;
}
constexpr int kSmemBytesMax = band_smem_bytes(16) > band_smem_bytes(kBandMaxGlobals)
                                  ? band_smem_bytes(16) : band_smem_bytes(kBandMaxGlobals);
static_assert(kSmemBytesMax <= 227 * 1024, "shared memory per CTA");
static_assert(band_smem_bytes(0) > 116 * 1024, "must exclude a second CTA per SM");

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
    float* A_x;                  // extras' weights (raw scores on entry to the first hop)
    const uint8_t* A_gimg;       // global-row weight images [units][tiles] (kGImgBytes each)
    float* inv_l;                // [units][n] (the first hop's gather completes it)
    const float* m_sparse;       // [units][n] row maxima m_i
    const __nv_bfloat16* V;
    const uint8_t* A_gcimg;      // out-of-window globals' weight images [units][tiles][hi | lo]
    const float* Zf_in;          // Z_k as fp32 rows [n][64] (hops after the first)
    __nv_bfloat16* Z_out;        // Z_{k+1} ([n][hi 64 | lo 64]), all hops but the last
    float* Zf_out;               // Z_{k+1} as fp32 rows [n][64], all hops but the last
    __nv_bfloat16* out;          // the last hop's output [n][64]
    float* Psum;                 // [units][n][64] sparse partial of the rows not in G
    float* gpart;                // [units][tiles][g][64] the global rows' shares, per tile
    __nv_bfloat16* Zk_hilo;      // Z_k as [n][hi | lo] rows and
    float* Zk_f;                 // as fp32 rows: the gather of hops after the first writes
                                 // Z_k's global rows there (from the previous hop's shares)
    int* status;
    const int32_t* deal_ptr;     // [CTAs + 1] each CTA's range of deal_tiles (null: snake order)
    const int32_t* deal_tiles;   // the dealt tiles, u * tiles + t
};

// acc[0..3] += w * (z0, z1) with packed pairs (the same rounding as fmaf per element)
__device__ __forceinline__ void ffma8(float2 (&acc)[4], float w, const float4& z0, const float4& z1) {
    const float2 ww = make_float2(w, w);
    acc[0] = __ffma2_rn(ww, make_float2(z0.x, z0.y), acc[0]);
    acc[1] = __ffma2_rn(ww, make_float2(z0.z, z0.w), acc[1]);
    acc[2] = __ffma2_rn(ww, make_float2(z1.x, z1.y), acc[2]);
    acc[3] = __ffma2_rn(ww, make_float2(z1.z, z1.w), acc[3]);
}

// acc += w * one gathered row piece: 8 bf16 (kBf16) or 2 x 4 fp32 as raw words
template <bool kBf16>
__device__ __forceinline__ void ffma_row(float2 (&acc)[4], float w, const uint4 (&z)[kBf16 ? 1 : 2]) {
    if constexpr (kBf16) {
        const uint4 h = z[0];
        ffma8(acc, w, make_float4(bf16lo(h.x), bf16hi(h.x), bf16lo(h.y), bf16hi(h.y)),
              make_float4(bf16lo(h.z), bf16hi(h.z), bf16lo(h.w), bf16hi(h.w)));
    } else {
        ffma8(acc, w,
              make_float4(__uint_as_float(z[0].x), __uint_as_float(z[0].y), __uint_as_float(z[0].z),
                          __uint_as_float(z[0].w)),
              make_float4(__uint_as_float(z[1].x), __uint_as_float(z[1].y), __uint_as_float(z[1].z),
                          __uint_as_float(z[1].w)));
    }
}

// One float4 (features 4 fq .. 4 fq + 3) of global row s of unit u in the next
// state: (1 - alpha) * (the tiles' shares sum_j A_gr[s][j] Z[j]) + alpha * V,
// from the shares `gpart` that a band hop kernel wrote; written as [hi | lo]
// bf16 and fp32 row pieces (zhl, zf) or as the output.  L = 1 or 8 lanes
// (ql = 0 .. L-1, converged, mask qmask) compute it together, in a fixed order:
// lane ql adds the shares of tiles ql, ql + L, ... in turn, then the L partial
// sums are added pairwise; lane 0 writes.  Eight lanes when a unit has at least
// kCoopTiles tiles (more loads in flight per output), one lane otherwise.
constexpr int kCoopTiles = 16;
template <bool kOut>
__device__ __forceinline__ void global_row_out(const HopArgs& a, const float* gpart, int64_t u, int s,
                                               int fq, int L, int ql, unsigned qmask,
                                               __nv_bfloat16* zhl, float* zf) {
    const BandPlan& P = a.plan;
    const size_t tstride = (size_t)P.g * (kHeadDim / 4);  // float4s from one share to the next
    const int nshares = P.tiles;                          // one per tile
    const float4* src = reinterpret_cast<const float4*>(gpart) + (size_t)u * nshares * tstride +
                        (size_t)s * (kHeadDim / 4) + fq;
    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int t0 = ql; t0 < nshares; t0 += 8 * L) {
        float4 v[8];
#pragma unroll
        for (int b = 0; b < 8; ++b)
            v[b] = t0 + L * b < nshares ? __ldg(src + (size_t)(t0 + L * b) * tstride)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            sum.x += v[b].x; sum.y += v[b].y; sum.z += v[b].z; sum.w += v[b].w;
        }
    }
    for (int off = 1; off < L; off <<= 1) {
        sum.x += __shfl_xor_sync(qmask, sum.x, off, 8);
        sum.y += __shfl_xor_sync(qmask, sum.y, off, 8);
        sum.z += __shfl_xor_sync(qmask, sum.z, off, 8);
        sum.w += __shfl_xor_sync(qmask, sum.w, off, 8);
    }
    if (ql != 0) return;
    const float keep = 1.f - a.alpha;
    const int64_t gi = a.globals[s];
    const size_t vrow = ((size_t)u * P.n + gi) * kHeadDim + 4 * fq;
    const uint2 vv = __ldg(reinterpret_cast<const uint2*>(a.V + vrow));
    float z[4] = {fmaf(keep, sum.x, a.alpha * bf16lo(vv.x)), fmaf(keep, sum.y, a.alpha * bf16hi(vv.x)),
                  fmaf(keep, sum.z, a.alpha * bf16lo(vv.y)), fmaf(keep, sum.w, a.alpha * bf16hi(vv.y))};
    if (kOut) {
        const __nv_bfloat162 h0 = __floats2bfloat162_rn(z[0], z[1]);
        const __nv_bfloat162 h1 = __floats2bfloat162_rn(z[2], z[3]);
        *reinterpret_cast<uint2*>(a.out + vrow) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1));
    } else {
        uint32_t hw[2], lw[2];
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            const __nv_bfloat162 hh = __floats2bfloat162_rn(z[2 * p], z[2 * p + 1]);
            const __nv_bfloat162 ll =
                __floats2bfloat162_rn(z[2 * p] - __low2float(hh), z[2 * p + 1] - __high2float(hh));
            hw[p] = *reinterpret_cast<const uint32_t*>(&hh);
            lw[p] = *reinterpret_cast<const uint32_t*>(&ll);
        }
        __nv_bfloat16* zr = zhl + ((size_t)u * P.n + gi) * (2 * kHeadDim) + 4 * fq;
        *reinterpret_cast<uint2*>(zr) = make_uint2(hw[0], hw[1]);
        *reinterpret_cast<uint2*>(zr + kHeadDim) = make_uint2(lw[0], lw[1]);
        *reinterpret_cast<float4*>(zf + vrow) = make_float4(z[0], z[1], z[2], z[3]);
    }
}

// The output's global rows after the last hop: L lanes per float4 (global_row_out).
__global__ void __launch_bounds__(256) hop_global_out_kernel(HopArgs a) {
    const int64_t per_unit = (int64_t)a.plan.g * (kHeadDim / 4);
    const int L = a.plan.tiles >= kCoopTiles ? 8 : 1;
    const int64_t tix = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t idx = L == 8 ? tix >> 3 : tix;   // the same for the L lanes of an output
    if (idx >= a.units * per_unit) return;
    const int64_t u = idx / per_unit;
    const int rem = (int)(idx - u * per_unit);
    global_row_out<true>(a, a.gpart, u, rem >> 4, rem & 15, L, L == 8 ? (int)(threadIdx.x & 7) : 0,
                         L == 8 ? 0xFFu << (threadIdx.x & 24) : 0u, nullptr, nullptr);
}

// ---------------------------------------------------------------- the CTAs' tiles
// A tile's 128-key chunks c (keys i0 - r64 + 128 c .. +127) that hold at least one
// key in 0 .. n-1: c_lo .. c_hi (the others would only add zeros).
__host__ __device__ __forceinline__ void chunk_range(const BandPlan& P, int nc, int64_t i0, int& c_lo,
                                                     int& c_hi) {
    const int64_t below = (int64_t)P.r64 - i0 - (kCK - 1);     // chunk c lies below key 0 iff 128 c < below
    c_lo = below > 0 ? (int)((below + kCK - 1) / kCK) : 0;
    const int64_t last = (P.n - (i0 - P.r64) - 1) / kCK;       // the last chunk with a key below n
    c_hi = last < nc - 1 ? (int)last : nc - 1;
}

// The tile position (0 .. tiles-1) of rank p when the positions are ordered by
// falling chunk count: the interior positions (all nc chunks in range) in order,
// then the edge positions (the first and last few of a unit), heavier first.
__host__ __device__ int tile_position(const BandPlan& P, int nc, int p) {
    const int64_t tl = P.r64 > kCK - 1 ? ((int64_t)P.r64 - (kCK - 1) + kCK - 1) / kCK : 0;
    const int64_t rnum = P.n + P.r64 - 1 - (int64_t)kCK * (nc - 1);
    int64_t tr = rnum >= 0 ? rnum / kCK : -1;
    if (tr > P.tiles - 1) tr = P.tiles - 1;
    if (tl > tr) return p;                                      // no interior: natural order
    const int ni = (int)(tr - tl + 1);
    if (p < ni) return (int)tl + p;
    // merge the left edge (tl - 1 down to 0) and the right edge (tr + 1 up) by
    // falling chunk count, left first on ties
    auto count = [&](int64_t t) { int lo, hi; chunk_range(P, nc, t * kTileRows, lo, hi); return hi - lo; };
    int64_t li = tl - 1, ri = tr + 1;
    for (int q = p - ni;; --q) {
        const bool has_l = li >= 0, has_r = ri < P.tiles;
        const bool take_l = has_l && (!has_r || count(li) >= count(ri));
        const int64_t t = take_l ? li : ri;
        if (q == 0 || (!has_l && !has_r)) return (int)t;
        if (take_l) --li; else ++ri;
    }
}

// The launch's items k = 0 .. units * tiles - 1, heaviest first: every unit's
// interior tiles, unit by unit (so that CTAs running at the same time mostly hold
// neighbouring tiles, which share K and Z_k chunks in L2), then the edge tiles,
// heavier positions first (tile_position), unit by unit within a position.
__host__ __device__ __forceinline__ void band_item(const BandPlan& P, int64_t units, int nc, int64_t k,
                                                   int64_t& u, int& t) {
    const int64_t tl = P.r64 > kCK - 1 ? ((int64_t)P.r64 - (kCK - 1) + kCK - 1) / kCK : 0;
    const int64_t rnum = P.n + P.r64 - 1 - (int64_t)kCK * (nc - 1);
    int64_t tr = rnum >= 0 ? rnum / kCK : -1;
    if (tr > P.tiles - 1) tr = P.tiles - 1;
    const int64_t ni = tl <= tr ? tr - tl + 1 : 0;
    if (k < units * ni) { u = k / ni; t = (int)(tl + (k - u * ni)); }
    else { const int64_t k2 = k - units * ni, pr = ni + k2 / units; u = k2 - (k2 / units) * units; t = tile_position(P, nc, (int)pr); }
}

// Without a deal table the CTAs take the items in snake order over the rounds
// (round r: CTA b gets item r G + b, or r G + G - 1 - b when r is odd), so that the
// light edge tiles fill the last rounds; with one (band_deal), CTA b takes the
// tiles listed for it.
struct TileInfo { int64_t tix, u, i0; int c_lo, c_hi; };
__device__ __forceinline__ int cta_tile_count(int64_t total_tiles) {
    const int64_t G = gridDim.x, b = blockIdx.x, R = total_tiles / G, rem = total_tiles - R * G;
    return (int)(R + ((R & 1) == 0 ? (b < rem ? 1 : 0) : (b >= G - rem ? 1 : 0)));
}
__device__ __forceinline__ TileInfo cta_tile(const BandPlan& P, int64_t units, int nc, int lt) {
    const int64_t G = gridDim.x, b = blockIdx.x;
    const int64_t k = (int64_t)lt * G + ((lt & 1) ? G - 1 - b : b);
    TileInfo ti;
    int t;
    band_item(P, units, nc, k, ti.u, t);
    ti.tix = ti.u * P.tiles + t;
    ti.i0 = (int64_t)t * kTileRows;
    chunk_range(P, nc, ti.i0, ti.c_lo, ti.c_hi);
    return ti;
}

// ---------------------------------------------------------------- band part of a hop
// The band weights are recomputed here on every hop from Q and K rather than
// read back: per 64-key chunk, S = Q_tile K_chunk^T on the tensor cores (the
// same MMA as the score kernel, so the same values), e = exp(s - m_i) with the
// row maxima the score kernel stored (0 outside the window), written as the
// bf16 hi / lo operand image in shared memory, then D += P Z_k as before.  The
// first hop also adds up each row's band sum and completes inv_l.
template <bool kHop0, bool kLast>
__global__ void __launch_bounds__(kThreads, 1)
hop_band_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmZ, HopArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const int g16 = a.plan.g16, g16s = g16 > 0 ? g16 : 16;
    uint8_t* sGA = smem;                                         // global rows' image(s), 16 KB
    uint8_t* sQ = sGA + band::kGImgBytes;                        // 2 x 16 KB
    uint8_t* sK = sQ + 2 * kQBytes;                              // kSBufs x 16 KB
    uint8_t* sZ = sK + kSBufs * kKBytes;                         // kSBufs x (hi 16 KB, lo 16 KB)
    uint8_t* sGC = sZ + kSBufs * kZStageBytes;                   // out-of-window globals' weights
    uint8_t* sZG = sGC + 2 * kTileRows * g16s * 2;               // Z_k rows of the global keys
    float* xch = reinterpret_cast<float*>(sZG + 2 * g16s * 128);  // [2][256] row-sum halves
    float* sEpi = xch + 2 * kSoftThreads;                        // [4][32][68] epilogue staging
    float* sEpiKeep = sEpi + 4 * 32 * kEpiRowFloats;             // [4][32]
    __nv_bfloat16* sEpiV = reinterpret_cast<__nv_bfloat16*>(sEpiKeep + 4 * 32);   // [4][32][64] V rows
    TileEntry* sTile = reinterpret_cast<TileEntry*>(sEpiV + 4 * 32 * kHeadDim);   // [kMaxCtaTiles]
    int* sTotal = reinterpret_cast<int*>(sTile + kMaxCtaTiles);         // this CTA's chunk count
    uint64_t* bars = reinterpret_cast<uint64_t*>(sTotal + 4);
    uint64_t* full_Q = bars;                                     // [2]
    uint64_t* empty_Q = full_Q + 2;                              // [2]
    uint64_t* full_K = empty_Q + 2;                              // [kSBufs]
    uint64_t* full_S = full_K + kSBufs;                          // [kSBufs]
    uint64_t* full_P = full_S + kSBufs;                          // [kSBufs] keys 0-63 weighted + Z landed
    uint64_t* full_P1 = full_P + kSBufs;                         // [kSBufs] keys 64-127 weighted
    uint64_t* pv_done = full_P1 + kSBufs;                        // [kSBufs]
    uint64_t* acc_full = pv_done + kSBufs;
    uint64_t* acc_empty = acc_full + 1;
    uint64_t* glob_empty = acc_empty + 1;  // the global rows' accumulator has been read
    uint64_t* full_G = glob_empty + 1;     // [gbufs] the global rows' image of tile lt, buffer lt % gbufs
    uint64_t* empty_G = full_G + 2;        // [gbufs]
    uint64_t* full_GC = empty_G + 2;       // the image by bulk copy + the staged Z rows
    uint64_t* empty_GC = full_GC + 1;
    // first hop: the band sums of a quadrant's rows, from its weight warps to its
    // epilogue warp, double-buffered by tile parity: [quad][parity]
    uint64_t* xch_full = empty_GC + 1;                           // [4][2], kSlices arrivals
    uint64_t* xch_empty = xch_full + 8;                          // [4][2], 1 arrival
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xch_empty + 8);

    const BandPlan& P = a.plan;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // The global rows' image of a tile: four planes (two 64-key halves x hi, lo) of 32
    // rows in global memory.  With at most 16 global rows only the planes' first 16
    // rows are copied, into two 8 KB buffers used by alternate tiles, so that a tile's
    // image loads while the previous tile's global MMAs run; with more, one 16 KB
    // buffer.  (The MMA reads 128 A rows: rows past the copied ones fall on other
    // shared-memory data and reach only accumulator rows that are never read.)
    const int gbufs = P.g <= 16 ? 2 : 1;
    const int gplane = P.g <= 16 ? band::kGImgPlaneBytes / 2 : band::kGImgPlaneBytes;   // bytes per plane
    const int nc = P.chunks / 2;                 // 128-key chunks of a tile (the key grid has an even count)
    const int c0 = P.r64 / kCK;                  // the chunk of the tile's first own key
    const bool has_g = P.g > 0;
    const int gc_plane = band::gc_plane_bytes(g16);
    const int64_t total_tiles = a.units * P.tiles;
    // this CTA's tiles: its list in the deal table, or the snake order (cta_tile)
    const int my_tiles = a.deal_ptr ? a.deal_ptr[blockIdx.x + 1] - a.deal_ptr[blockIdx.x]
                                    : cta_tile_count(total_tiles);
    for (int lt = tid; lt < my_tiles && lt < kMaxCtaTiles; lt += kThreads) {
        if (a.deal_ptr) {
            const int32_t tix = a.deal_tiles[a.deal_ptr[blockIdx.x] + lt];
            const int32_t u = tix / P.tiles, t = tix - u * P.tiles;
            int lo, hi;
            chunk_range(P, nc, (int64_t)t * kTileRows, lo, hi);
            sTile[lt] = TileEntry{u, t, (int16_t)lo, (int16_t)hi};
        } else {
            const TileInfo ti = cta_tile(P, a.units, nc, lt);
            sTile[lt] = TileEntry{(int32_t)ti.u, (int32_t)(ti.i0 / kTileRows), (int16_t)ti.c_lo,
                                  (int16_t)ti.c_hi};
        }
    }

    if (warp == kSMmaWarp) ptx::tmem_alloc(tmem_slot, kTmemCols);
    if (tid == 0) {
        for (int s = 0; s < 2; ++s) { ptx::mbar_init(&full_Q[s], 1); ptx::mbar_init(&empty_Q[s], 1); }
        // the weight warps arrive once per warp (lane 0, after the warp has synced)
        for (int s = 0; s < kSBufs; ++s) {
            ptx::mbar_init(&full_K[s], 1);
            ptx::mbar_init(&full_S[s], 1);
            ptx::mbar_init(&full_P[s], kSoftWarps + 1);          // + the Z producer's arrival (with its bytes)
            ptx::mbar_init(&full_P1[s], kSoftWarps);
            ptx::mbar_init(&pv_done[s], 1);
        }
        ptx::mbar_init(acc_full, 1);
        ptx::mbar_init(acc_empty, kEpiWarps);
        ptx::mbar_init(glob_empty, 1);
        for (int s = 0; s < 2; ++s) { ptx::mbar_init(&full_G[s], 1); ptx::mbar_init(&empty_G[s], 1); }
        ptx::mbar_init(full_GC, 1 + kEpiWarps);  // the image's bytes + each epilogue warp's staged rows
        ptx::mbar_init(empty_GC, 1);
        for (int s = 0; s < 8; ++s) { ptx::mbar_init(&xch_full[s], kSlices); ptx::mbar_init(&xch_empty[s], 1); }
        ptx::fence_mbar_init();
    }
    if (warp == kTmaWarp && lane == 0) {
        ptx::prefetch_tensormap(&tmQ);
        ptx::prefetch_tensormap(&tmK);
        ptx::prefetch_tensormap(&tmZ);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // this CTA's chunk count (for the drains), summed from the table by every thread
    int total = 0;
    for (int lt = 0; lt < my_tiles; ++lt) total += sTile[lt].c_hi - sTile[lt].c_lo + 1;
    // tile lt of this CTA from the table
    auto tile = [&](int lt) {
        const TileEntry e = sTile[lt];
        TileInfo ti;
        ti.u = e.u;
        ti.tix = (int64_t)e.u * P.tiles + e.t;
        ti.i0 = (int64_t)e.t * kTileRows;
        ti.c_lo = e.c_lo;
        ti.c_hi = e.c_hi;
        return ti;
    };

    if (warp == kTmaWarp) {
        // ---------------- TMA producer of the score operands: the Q tile and the K
        // chunks (keys of the chunk grid jb = i0 - r64 ..; outside 0..n-1 they load
        // as zeros), in the order the score MMAs use them.
        // (the whole warp runs the loop; the elected lane issues the copies)
        {
            const uint64_t pol_keep = ptx::l2_evict_last();      // re-read by neighbouring tiles
            int g = 0, b = 0, ph = 0;                             // running chunk, slot, phase
            for (int lt = 0; lt < my_tiles; ++lt) {
                const TileInfo ti = tile(lt);
                const int qb = lt & 1;
                if (lt >= 2) ptx::mbar_wait(&empty_Q[qb], ((lt / 2) - 1) & 1, a.status);
                __syncwarp();
                if (ptx::elect_one()) {
                    ptx::mbar_arrive_expect_tx(&full_Q[qb], kQBytes);
                    ptx::tma_load_3d_hint(sQ + qb * kQBytes, &tmQ, &full_Q[qb], 0, (int)ti.i0, (int)ti.u, pol_keep);
                }
                for (int c = ti.c_lo; c <= ti.c_hi; ++c, ++g) {
                    // stage b is free once the scores of chunk g - kSBufs are written
                    if (g >= kSBufs) ptx::mbar_wait(&full_S[b], ph ^ 1, a.status);
                    __syncwarp();
                    if (ptx::elect_one()) {
                        ptx::mbar_arrive_expect_tx(&full_K[b], kKBytes);
                        ptx::tma_load_3d_hint(sK + b * kKBytes, &tmK, &full_K[b], 0,
                                              (int)(ti.i0 - P.r64 + kCK * c), (int)ti.u, pol_keep);
                    }
                    if (++b == kSBufs) { b = 0; ph ^= 1; }
                }
            }
        }
    } else if (warp == kZWarp) {
        // ---------------- producer of the weights' MMA operands (whole warp; lane 0
        // issues the copies): per tile the globals' images and the global keys'
        // Z_k rows, per chunk the Z_k rows, in the order the MMAs use them.
        const uint64_t pol_once = ptx::l2_evict_first(), pol_keep = ptx::l2_evict_last();
        int g = 0;                                                // running chunk
        for (int lt = 0; lt < my_tiles; ++lt) {
            const TileInfo ti = tile(lt);
            if (has_g) {
                // the global rows' image of this tile's keys, needed from chunk c0 on
                const int gb = lt % gbufs, gk = lt / gbufs;
                if (lt >= gbufs) ptx::mbar_wait(&empty_G[gb], (gk - 1) & 1, a.status);
                if (lane == 0) {
                    uint8_t* gdst = sGA + gb * (band::kGImgBytes / 2);
                    const uint8_t* gsrc = a.A_gimg + (size_t)ti.tix * band::kGImgBytes;
                    ptx::mbar_arrive_expect_tx(&full_G[gb], 4 * gplane);
                    for (int pl = 0; pl < 4; ++pl)
                        ptx::bulk_load_hint(gdst + pl * gplane, gsrc + pl * band::kGImgPlaneBytes, gplane,
                                            &full_G[gb], pol_once);
                }
            }
            for (int c = ti.c_lo; c <= ti.c_hi; ++c, ++g) {
                const int key = (int)(ti.i0 - P.r64 + kCK * c);
                const int b = g % kSBufs;
                // stage b is free once the weights' MMAs of chunk g - kSBufs are done; the
                // copy completes on the chunk's full_P barrier
                if (g >= kSBufs) ptx::mbar_wait(&pv_done[b], ((g / kSBufs) - 1) & 1, a.status);
                if (lane == 0) {
                    uint8_t* zdst = sZ + b * kZStageBytes;
                    ptx::mbar_arrive_expect_tx(&full_P[b], kHop0 ? kZTileBytes : 2 * kZTileBytes);
                    ptx::tma_load_3d_hint(zdst, &tmZ, &full_P[b], 0, key, (int)ti.u, pol_keep);
                    if (!kHop0)
                        ptx::tma_load_3d_hint(zdst + kZTileBytes, &tmZ, &full_P[b], kHeadDim, key, (int)ti.u,
                                              pol_keep);
                }
                __syncwarp();
            }
        }
    } else if (warp == kSMmaWarp) {
        // ---------------- score MMAs: S[b] = Q_tile K_chunk^T (both K-major,
        // 128-byte swizzle), as far ahead of the weights as the TMEM buffers allow:
        // buffer b is free once the weights' MMAs of its previous chunk are done
        // (the whole warp runs the loop; the elected lane issues each instruction)
        {
            constexpr uint32_t idesc_s = ptx::mma_idesc(1, kCK);
            // descriptors advance by (byte offset >> 4) in their address field
            const uint64_t qdesc0 = ptx::sw128_kmajor_desc(ptx::smem_u32(sQ));
            const uint64_t kdesc0 = ptx::sw128_kmajor_desc(ptx::smem_u32(sK));
            int g = 0, b = 0, ph = 0;                             // running chunk, slot, phase
            for (int lt = 0; lt < my_tiles; ++lt) {
                const TileInfo ti = tile(lt);
                const int qb = lt & 1;
                ptx::mbar_wait(&full_Q[qb], (lt >> 1) & 1, a.status);
                const uint64_t qd = qdesc0 + (uint64_t)(qb * (kQBytes >> 4));
                for (int c = ti.c_lo; c <= ti.c_hi; ++c, ++g) {
                    ptx::mbar_wait(&full_K[b], ph, a.status);
                    if (g >= kSBufs) ptx::mbar_wait(&pv_done[b], ph ^ 1, a.status);
                    __syncwarp();
                    ptx::tc_fence_after();
                    const uint64_t kd = kdesc0 + (uint64_t)(b * (kKBytes >> 4));
                    const uint32_t dS = tmem + kSCol0 + kCK * b;
#pragma unroll
                    for (int ks = 0; ks < kHeadDim / 16; ++ks)
                        if (ptx::elect_one()) ptx::mma_bf16_ss(dS, qd + 2 * ks, kd + 2 * ks, idesc_s, ks > 0);
                    if (ptx::elect_one()) ptx::mma_commit(&full_S[b]);   // also frees K stage b
                    if (c == ti.c_hi && ptx::elect_one()) ptx::mma_commit(&empty_Q[qb]);
                    if (++b == kSBufs) { b = 0; ph ^= 1; }
                }
            }
            // Drain: the commits arrive asynchronously when the MMAs finish; wait for
            // the last phase of each so that none lands in shared memory after exit.
            for (int s = 0; s < kSBufs; ++s) {
                const int uses = (total - s + kSBufs - 1) / kSBufs;
                if (uses > 0) ptx::mbar_wait(&full_S[s], (uses - 1) & 1, a.status);
            }
            for (int s = 0; s < 2; ++s) {
                const int uses = (my_tiles - s + 1) / 2;
                if (uses > 0) ptx::mbar_wait(&empty_Q[s], (uses - 1) & 1, a.status);
            }
        }
    } else if (warp == kPvMmaWarp) {
        // ---------------- the weights' MMAs, chunk by chunk as the weight images are
        // written: D += P_hi [Z_hi | Z_lo] + P_lo Z_hi, the globals and global rows
        // (the whole warp runs the loop; the elected lane issues each instruction)
        {
            constexpr uint32_t idesc64 = ptx::mma_idesc_bf16_bmn(64);
            constexpr uint32_t idesc128 = ptx::mma_idesc_bf16_bmn(128);
            const uint32_t dacc = tmem;
            // descriptors advance by (byte offset >> 4) in their address field
            const uint64_t zdesc0 = ptx::sw128_mnmajor_desc(ptx::smem_u32(sZ), kZTileBytes);
            const uint64_t gdesc0 = ptx::sw128_kmajor_desc(ptx::smem_u32(sGA));
            int sp = 0, pph = 0;                                  // running slot, phase
            for (int lt = 0; lt < my_tiles; ++lt) {
                const TileInfo ti = tile(lt);
                {
                    // the previous tile's accumulators have been read
                    if (lt >= 1) ptx::mbar_wait(acc_empty, (lt - 1) & 1, a.status);
                    __syncwarp();
                    ptx::tc_fence_after();
                    if (has_g) {
                        // the globals outside each row's window: [128 x g16] x [g16 x (hi | lo)]
                        ptx::mbar_wait(full_GC, lt & 1, a.status);
                        __syncwarp();
                        ptx::tc_fence_after();
                        const uint32_t gch = ptx::smem_u32(sGC), gcl = gch + gc_plane;
                        const uint32_t zg = ptx::smem_u32(sZG);
                        for (int ks = 0; ks < g16 / 16; ++ks) {
                            const uint64_t bdesc = ptx::sw128_mnmajor_desc(zg + 2048 * ks, g16 * 128);
                            if (ptx::elect_one())
                                ptx::mma_bf16_ss(dacc, ptx::noswz_kmajor_desc(gch + 256 * ks, 128, 16 * g16),
                                                 bdesc, kHop0 ? idesc64 : idesc128, ks != 0);
                            if (ptx::elect_one())
                                ptx::mma_bf16_ss(dacc, ptx::noswz_kmajor_desc(gcl + 256 * ks, 128, 16 * g16),
                                                 bdesc, idesc64, 1);
                        }
                        if (ptx::elect_one()) ptx::mma_commit(empty_GC);
                    }
                }
              for (int c = ti.c_lo; c <= ti.c_hi; ++c) {
                ptx::mbar_wait(&full_P[sp], pph, a.status);          // keys 0-63 weighted, Z stage landed
                __syncwarp();
                ptx::tc_fence_after();
                const uint32_t pbuf = tmem + kSCol0 + kCK * sp;   // K step ks: hi 16 ks, lo 16 ks + 8
                const uint64_t zd = zdesc0 + (uint64_t)(sp * (kZStageBytes >> 4));
#pragma unroll
                for (int ks = 0; ks < kCK / 16; ++ks) {
                    if (ks == kCK / 32) {
                        ptx::mbar_wait(&full_P1[sp], pph, a.status);    // keys 64-127 weighted
                        __syncwarp();
                        ptx::tc_fence_after();
                    }
                    const uint64_t bdesc = zd + (uint64_t)(128 * ks);     // 16 keys = 2048 bytes on
                    if (ptx::elect_one())
                        ptx::mma_bf16_ts(dacc, pbuf + 16 * ks, bdesc, kHop0 ? idesc64 : idesc128,
                                         has_g || c != ti.c_lo || ks != 0);
                    if (ptx::elect_one()) ptx::mma_bf16_ts(dacc, pbuf + 16 * ks + 8, bdesc, idesc64, 1);
                }
                // the chunk(s) holding the tile's own keys: c0, and c0 + 1 when r64 is an
                // odd multiple of 64 and that chunk is in range (a ragged last tile may end
                // before it); the image is released after the last of them
                const int glob_last = ((P.r64 % kCK) != 0 && c0 + 1 <= ti.c_hi) ? c0 + 1 : c0;
                if (has_g && (c == c0 || c == glob_last)) {
                    // the global rows x this tile's own keys i0 .. i0 + 127 (same Z_k
                    // stage): K step ks of this chunk holds keys 128 c + 16 ks - r64 on
                    // from i0, in 64-key half h of the image at its K step kk
                    const uint32_t dglob = tmem + kGlobCol0;
                    const int rel0 = kCK * c - P.r64;
#pragma unroll 1
                    for (int ks = 0; ks < kCK / 16; ++ks) {
                        const int rel = rel0 + 16 * ks;
                        if (rel < 0 || rel >= kTileRows) continue;
                        if (rel == 0) {
                            // the image is in shared memory and the previous tile's
                            // accumulator has been read
                            ptx::mbar_wait(&full_G[lt % gbufs], (lt / gbufs) & 1, a.status);
                            if (lt >= 1) ptx::mbar_wait(glob_empty, (lt - 1) & 1, a.status);
                            __syncwarp();
                            ptx::tc_fence_after();
                        }
                        const int h = rel >> 6, kk = (rel & 63) >> 4;
                        const uint64_t ghi = gdesc0 + (uint64_t)((((lt % gbufs) * (band::kGImgBytes / 2) + h * 2 * gplane) >> 4) +
                                                                 2 * kk);
                        const uint64_t glo = ghi + (uint64_t)(gplane >> 4);
                        const uint64_t bdesc = zd + (uint64_t)(128 * ks);
                        if (ptx::elect_one()) ptx::mma_bf16_ss(dglob, ghi, bdesc, kHop0 ? idesc64 : idesc128, rel != 0);
                        if (ptx::elect_one()) ptx::mma_bf16_ss(dglob, glo, bdesc, idesc64, 1);
                    }
                    if (c == glob_last && ptx::elect_one()) ptx::mma_commit(&empty_G[lt % gbufs]);
                }
                if (ptx::elect_one()) ptx::mma_commit(&pv_done[sp]);
                if (c == ti.c_hi && ptx::elect_one()) ptx::mma_commit(acc_full);
                if (++sp == kSBufs) { sp = 0; pph ^= 1; }
              }
            }
            for (int s = 0; s < kSBufs; ++s) {
                const int uses = (total - s + kSBufs - 1) / kSBufs;
                if (uses > 0) ptx::mbar_wait(&pv_done[s], (uses - 1) & 1, a.status);
            }
            if (has_g && my_tiles > 0) {
                for (int gb = 0; gb < gbufs; ++gb) {
                    const int uses = (my_tiles - gb + gbufs - 1) / gbufs;
                    if (uses > 0) ptx::mbar_wait(&empty_G[gb], (uses - 1) & 1, a.status);
                }
                ptx::mbar_wait(empty_GC, (my_tiles - 1) & 1, a.status);
            }
        }
    } else if (warp >= kSoftWarp0 && warp < kEpiWarp0) {
        // ---------------- band weights: thread <-> row t = 32 quad + lane of the tile,
        // keys 16 slice .. +15 of both 64-key halves of each chunk.
        const int quad = warp & 3;
        const int slice = (warp - kSoftWarp0) >> 2;       // keys 16 slice .. +15 of each half
        const int stid = tid - kSoftWarp0 * 32;           // 0..511
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const int t = quad * 32 + lane;
        const float a_sc = kLog2e * kScale;
        // this row of tile lt: its window lo..hi as offsets from the tile's key grid
        // origin i0 - r64 (an empty window, hi < 0 <= lo, for a global row or a row
        // past the end), b2 = m_i log2(e), and the tile's chunk range: few registers,
        // as the weight code needs most of them
        struct Row { int lo, hi; float b2; int c_lo, c_hi; };
        auto row_of = [&](int lt) {
            Row w;
            const TileInfo ti = tile(lt);
            const int64_t u = ti.u, i0 = ti.i0;
            w.c_lo = ti.c_lo;
            w.c_hi = ti.c_hi;
            const int64_t i = i0 + t;
            const bool ok = i < P.n && !a.is_global[i < P.n ? i : 0];
            int64_t lo, hi;
            band::window_of(P, i, lo, hi);
            const int64_t jb = i0 - P.r64;
            w.lo = ok ? (int)(lo - jb) : 1 << 30;
            w.hi = ok ? (int)(hi - jb) : -1;
            w.b2 = ok ? __ldg(a.m_sparse + (size_t)u * P.n + i) * kLog2e : 0.f;
            return w;
        };
        // e = exp(s - m_i) for this row's 16 keys j0 .. j0 + 15 (offsets from the key
        // grid origin) inside its window, else 0, as hi and lo bf16 pairs (two keys
        // per TMEM column)
        auto weights16 = [&](const uint32_t (&r)[16], const Row& row, int j0, float& lsum,
                             uint32_t (&hw)[8], uint32_t (&lw)[8]) {
            const bool full_in = j0 >= row.lo && j0 + 15 <= row.hi;
            const bool none_in = j0 > row.hi || j0 + 15 < row.lo;
            if (none_in) {
#pragma unroll
                for (int p2 = 0; p2 < 8; ++p2) { hw[p2] = 0u; lw[p2] = 0u; }
                return;
            }
            // pair by pair (few live registers): the scaling as one packed fma (the same
            // roundings as fmaf); at a window edge the keys outside it are set to 0
            const float2 sc = make_float2(a_sc, a_sc), nb = make_float2(-row.b2, -row.b2);
            auto pair = [&](int p2, float x0, float x1) {
                if (kHop0) { lsum += x0; lsum += x1; }
                const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
                const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - __low2float(h), x1 - __high2float(h));
                hw[p2] = *reinterpret_cast<const uint32_t*>(&h);
                lw[p2] = *reinterpret_cast<const uint32_t*>(&l);
            };
            if (full_in) {
#pragma unroll
                for (int p2 = 0; p2 < 8; ++p2) {
                    const float2 y = __ffma2_rn(make_float2(__uint_as_float(r[2 * p2]), __uint_as_float(r[2 * p2 + 1])),
                                                sc, nb);
                    pair(p2, ptx::ex2_approx(y.x), ptx::ex2_approx(y.y));
                }
            } else {
                const int dlo = row.lo - j0, dhi = row.hi - j0;       // in-window keys k in [dlo, dhi]
#pragma unroll
                for (int p2 = 0; p2 < 8; ++p2) {
                    const float2 y = __ffma2_rn(make_float2(__uint_as_float(r[2 * p2]), __uint_as_float(r[2 * p2 + 1])),
                                                sc, nb);
                    const float x0 = (2 * p2 >= dlo && 2 * p2 <= dhi) ? ptx::ex2_approx(y.x) : 0.f;
                    const float x1 = (2 * p2 + 1 >= dlo && 2 * p2 + 1 <= dhi) ? ptx::ex2_approx(y.y) : 0.f;
                    pair(p2, x0, x1);
                }
            }
        };
        Row row = my_tiles > 0 ? row_of(0) : Row{};
        Row next_row = row;
        float lsum = 0.f;
        int lt = 0, c = row.c_lo, sb = 0, sph = 0;         // running tile, chunk, slot, phase
        for (int g = 0; g < total; ++g) {
            if (c == row.c_hi && lt + 1 < my_tiles) next_row = row_of(lt + 1);
            // this warp's columns of buffer sb: keys 16 slice .. +15 of both 64-key
            // halves, the scores, then (in place) the weights
            ptx::mbar_wait(&full_S[sb], sph, a.status);
            __syncwarp();
            ptx::tc_fence_after();
            const uint32_t col = tmem + lane_base + kSCol0 + kCK * sb + 16 * slice;
            uint32_t ra[16], rb[16];
            ptx::tmem_ld16_issue(col, ra);
            ptx::tmem_ld16_issue(col + kChunkKeys, rb);
            ptx::tmem_ld_wait16(ra);
            ptx::tmem_ld_wait16(rb);
            const int j0 = kCK * c + 16 * slice;
            {
                uint32_t hw[8], lw[8];
                weights16(ra, row, j0, lsum, hw, lw);
                __syncwarp();   // reconverge before the warp-collective tcgen05.st
                ptx::tmem_st16_hilo(col, hw, lw);                 // hi in columns +0..7, lo in +8..15
            }
            // the first 64 keys' weights are in: their MMAs may start while the
            // second half is computed
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&full_P[sb]);
            {
                uint32_t hw[8], lw[8];
                weights16(rb, row, j0 + kChunkKeys, lsum, hw, lw);
                __syncwarp();
                ptx::tmem_st16_hilo(col + kChunkKeys, hw, lw);
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&full_P1[sb]);
            if (kHop0 && c == row.c_hi) {
                // the row's band sum (this slice) for the epilogue warp of the quadrant;
                // the buffer of this parity is free once that warp has read tile lt - 2's
                const int xb = quad * 2 + (lt & 1);
                if (lt >= 2) ptx::mbar_wait(&xch_empty[xb], ((lt / 2) - 1) & 1, a.status);
                xch[(lt & 1) * kSoftThreads + stid] = lsum;
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&xch_full[xb]);
            }
            if (++sb == kSBufs) { sb = 0; sph ^= 1; }
            if (++c > row.c_hi && ++lt < my_tiles) {
                row = next_row;
                c = row.c_lo;
                lsum = 0.f;
            }
        }
    } else if (warp >= kEpiWarp0) {
        // ---------------- epilogue: the warp of lane quadrant q reads rows 32 q .. +31
        // of the accumulator (thread <-> row), stages them in shared memory, then
        // walks the rows two at a time with half a warp per row (lane: 4
        // features) so that every global load and store covers whole lines.
        const int quad = warp & 3;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const int t = quad * 32 + lane;
        float* st = sEpi + quad * (32 * kEpiRowFloats);                    // [32 rows][68]
        float* sk = sEpiKeep + quad * 32;                                  // keep of each row (< 0: skip)
        __nv_bfloat16* sv = sEpiV + quad * 32 * kHeadDim;                   // [32 rows][64] V
        const int hr = lane >> 4, f4 = lane & 15;                          // row of the pair, feature quad
        // The out-of-window globals of tile lt: their weights' image by bulk copy, and
        // the global keys' Z_k rows as an MN-major B tile (key row s: hi 128 bytes,
        // lo g16 * 128 bytes on; 16-byte chunk c at (c ^ (s % 8)) * 16; rows past g
        // are zero), staged a tile ahead of the MMAs that read them.
        auto stage_gc = [&](int lt) {
            const TileInfo ti = tile(lt);
            const int64_t tix = ti.tix, u = ti.u;
            if (quad == 0 && lane == 0) {
                ptx::mbar_arrive_expect_tx(full_GC, 2 * gc_plane);
                ptx::bulk_load_hint(sGC, a.A_gcimg + (size_t)tix * 2 * gc_plane, 2 * gc_plane, full_GC,
                                    ptx::l2_evict_first());
            }
            // the key rows' hi and lo halves, as asynchronous copies from Z_k's hi | lo
            // rows (V, whose lo part is zero, on the first hop); 16 pieces per row
            for (int e = t; e < g16 * 16; e += kEpiWarps * 32) {
                const int sl = e >> 4, half = (e >> 3) & 1, cch = e & 7;
                uint8_t* dst = sZG + half * g16 * 128 + sl * 128 + ((cch ^ (sl & 7)) << 4);
                if (sl < P.g && !(kHop0 && half)) {
                    const size_t row = (size_t)u * P.n + a.globals[sl];
                    if (kHop0) ptx::cp_async16(dst, a.V + row * kHeadDim + 8 * cch);
                    else ptx::cp_async16(dst, a.Zk_hilo + row * (2 * kHeadDim) + half * kHeadDim + 8 * cch);
                } else {
                    *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            ptx::cp_async_commit();
        };
        // this thread's copies have landed: visible to the MMAs, and the warp signals
        auto stage_gc_done = [&]() {
            ptx::cp_async_wait_all();
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(full_GC);
        };
        if (has_g && my_tiles > 0) {
            stage_gc(0);
            stage_gc_done();
        }
        for (int lt = 0; lt < my_tiles; ++lt) {
            {
                // this quadrant's rows of Psum into its staging rows and of V into its V
                // rows, as asynchronous copies issued before the accumulator is waited
                // for (the tile's MMAs hide their latency); the accumulator is added to
                // the Psum rows below.  Lanes 0-15 copy one 256-byte Psum row, lanes
                // 16-31 the next; a 128-byte V row takes 8 lanes.
                const TileInfo tp = tile(lt);
                const size_t ub = (size_t)tp.u * P.n;
#pragma unroll
                for (int it = 0; it < 16; ++it) {
                    const int idx = it * 32 + lane, r = idx >> 4, c = idx & 15;
                    const int64_t ir = tp.i0 + quad * 32 + r;
                    if (ir < P.n)
                        ptx::cp_async16(st + r * kEpiRowFloats + 4 * c, a.Psum + (ub + ir) * kHeadDim + 4 * c);
                }
#pragma unroll
                for (int it = 0; it < 8; ++it) {
                    const int idx = it * 32 + lane, r = idx >> 3, c = idx & 7;
                    const int64_t ir = tp.i0 + quad * 32 + r;
                    if (ir < P.n)
                        ptx::cp_async16(sv + r * kHeadDim + 8 * c, a.V + (ub + ir) * kHeadDim + 8 * c);
                }
                ptx::cp_async_commit();
            }
            if (has_g && lt + 1 < my_tiles) {
                ptx::mbar_wait(empty_GC, lt & 1, a.status);      // tile lt's globals' MMAs are done
                stage_gc(lt + 1);
            }
            const TileInfo ti = tile(lt);
            const int64_t u = ti.u, i0 = ti.i0;
            const int64_t i = i0 + t;
            const bool row_ok = i < P.n && !a.is_global[i < P.n ? i : 0];
            const size_t urow = (size_t)u * P.n + (row_ok ? i : 0);
            float inv = row_ok ? __ldg(a.inv_l + urow) : 0.f;
            if (kHop0) {
                // the first hop completes the row sum: band halves (from the weight
                // warps) + the globals' and extras' part already in inv_l
                const int xb = quad * 2 + (lt & 1);
                ptx::mbar_wait(&xch_full[xb], (lt / 2) & 1, a.status);
                const float* xr = xch + (lt & 1) * kSoftThreads + t;        // slice s at xr[128 s]
                const float lband = ((xr[0] + xr[128]) + xr[256]) + xr[384];
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&xch_empty[xb]);
                inv = row_ok ? 1.f / (lband + inv) : 0.f;
                if (row_ok) a.inv_l[urow] = inv;
            }
            ptx::mbar_wait(acc_full, lt & 1, a.status);
            ptx::cp_async_wait_all();       // also the next tile's global key rows (stage_gc)
            if (has_g && lt + 1 < my_tiles) {
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(full_GC);
            }
            __syncwarp();       // reconverge before the warp-collective tcgen05.ld; the
                                // quadrant's Psum and V rows are in shared memory
            ptx::tc_fence_after();
            // the accumulator rows (D[0:64) + D[64:128)) added to them, two loads in
            // flight per wait
#pragma unroll
            for (int h = 0; h < 4; h += (kHop0 ? 2 : 1)) {
                uint32_t dr[32];
                if (kHop0) ptx::tmem_ld32_issue(tmem + lane_base + 16 * h, dr);
                else ptx::tmem_ld16x2_issue(tmem + lane_base + 16 * h, tmem + lane_base + kHeadDim + 16 * h, dr);
                ptx::tmem_ld_wait32(dr);
#pragma unroll
                for (int hh = 0; hh < (kHop0 ? 2 : 1); ++hh) {
                    float dh[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        dh[k] = kHop0 ? __uint_as_float(dr[16 * hh + k])
                                      : __uint_as_float(dr[k]) + __uint_as_float(dr[16 + k]);
                    float4* dst = reinterpret_cast<float4*>(st + lane * kEpiRowFloats + 16 * (h + hh));
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        const float4 p = dst[c4];
                        dst[c4] = make_float4(dh[4 * c4] + p.x, dh[4 * c4 + 1] + p.y, dh[4 * c4 + 2] + p.z,
                                              dh[4 * c4 + 3] + p.w);
                    }
                }
            }
            ptx::tc_fence_before();
            sk[lane] = row_ok ? (1.f - a.alpha) * inv : -1.f;
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(acc_empty);          // the accumulator D is read
            if (has_g && quad == 0) {
                // TMEM lanes 0..31 of the global accumulator are the global slots s:
                // this tile's share of the global rows (summed by global_row_out)
#pragma unroll
                for (int f = 0; f < 4; f += (kHop0 ? 2 : 1)) {
                    uint32_t gr[32];
                    if (kHop0) ptx::tmem_ld32_issue(tmem + kGlobCol0 + 16 * f, gr);
                    else ptx::tmem_ld16x2_issue(tmem + kGlobCol0 + 16 * f, tmem + kGlobCol0 + kHeadDim + 16 * f, gr);
                    ptx::tmem_ld_wait32(gr);
                    if (lane < P.g) {
#pragma unroll
                        for (int ff = 0; ff < (kHop0 ? 2 : 1); ++ff) {
                            float4* gp = reinterpret_cast<float4*>(
                                a.gpart + (((size_t)u * P.tiles + (i0 / kTileRows)) * P.g + lane) * kHeadDim +
                                16 * (f + ff));
#pragma unroll
                            for (int c4 = 0; c4 < 4; ++c4) {
                                float v[4];
#pragma unroll
                                for (int k = 0; k < 4; ++k)
                                    v[k] = kHop0 ? __uint_as_float(gr[16 * ff + 4 * c4 + k])
                                                 : __uint_as_float(gr[4 * c4 + k]) + __uint_as_float(gr[16 + 4 * c4 + k]);
                                gp[c4] = make_float4(v[0], v[1], v[2], v[3]);
                            }
                        }
                    }
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(glob_empty);
            }
            // rows r = 2 it + hr; this lane's features 4 f4 .. +3
            const size_t ubase = (size_t)u * P.n;
#pragma unroll 1
            for (int it0 = 0; it0 < 16; it0 += 4) {
                uint2 vv[4];
                float keep[4];
                size_t rr[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int r = 2 * (it0 + q) + hr;
                    keep[q] = sk[r];
                    rr[q] = ubase + (size_t)(i0 + quad * 32 + r);
                    if (keep[q] >= 0.f) vv[q] = reinterpret_cast<const uint2*>(sv + r * kHeadDim)[f4];
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (keep[q] < 0.f) continue;
                    const int r = 2 * (it0 + q) + hr;
                    const float4 dv = *reinterpret_cast<const float4*>(st + r * kEpiRowFloats + 4 * f4);   // D + Psum
                    float z[4] = {fmaf(keep[q], dv.x, a.alpha * bf16lo(vv[q].x)),
                                  fmaf(keep[q], dv.y, a.alpha * bf16hi(vv[q].x)),
                                  fmaf(keep[q], dv.z, a.alpha * bf16lo(vv[q].y)),
                                  fmaf(keep[q], dv.w, a.alpha * bf16hi(vv[q].y))};
                    const __nv_bfloat162 h0 = __floats2bfloat162_rn(z[0], z[1]);
                    const __nv_bfloat162 h1 = __floats2bfloat162_rn(z[2], z[3]);
                    const uint2 hv = make_uint2(*reinterpret_cast<const uint32_t*>(&h0),
                                                *reinterpret_cast<const uint32_t*>(&h1));
                    if (kLast) {
                        reinterpret_cast<uint2*>(a.out + rr[q] * kHeadDim)[f4] = hv;
                    } else {
                        const __nv_bfloat162 l0 = __floats2bfloat162_rn(z[0] - __low2float(h0), z[1] - __high2float(h0));
                        const __nv_bfloat162 l1 = __floats2bfloat162_rn(z[2] - __low2float(h1), z[3] - __high2float(h1));
                        __nv_bfloat16* zr = a.Z_out + rr[q] * (2 * kHeadDim);
                        reinterpret_cast<uint2*>(zr)[f4] = hv;
                        reinterpret_cast<uint2*>(zr + kHeadDim)[f4] =
                            make_uint2(*reinterpret_cast<const uint32_t*>(&l0), *reinterpret_cast<const uint32_t*>(&l1));
                        reinterpret_cast<float4*>(a.Zf_out + rr[q] * kHeadDim)[f4] =
                            make_float4(z[0], z[1], z[2], z[3]);
                    }
                }
            }
            __syncwarp();       // the staging rows are rewritten by the next tile
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kSMmaWarp) ptx::tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------- sparse part of a hop
// Persistent, 8 warps per CTA.  The rows of all units are split over the
// quarter-warps of the grid in contiguous ranges: of equal row count on the
// bidirectional graph (random extras per row vary little, so equal rows are
// equal work; global rows carry none), and of equal cost on the causal graph,
// where a row keeps only the draws that land before it, so late rows carry
// far more extras than early ones (a row costs kRowCost plus its extras).
// A quarter walks its rows in windows of up to kWinRows rows of one unit,
// whose extras are one contiguous stretch of the extras list: it streams that
// stretch kB slots at a time (every slot's Z_k row in flight at once) while the
// indices and weights of the next kB slots load, one slot per lane, and reach
// the quarter by shuffles.
// On leaving a row it writes the row's sum P_i (zeros for a row without
// extras; nothing for a global row).  Lane l of a quarter owns features
// 4 l .. 4 l + 3 and 32 + 4 l .. 32 + 4 l + 3, so each load instruction reads
// whole 128-byte lines of the gathered rows.
constexpr int kGThreadsG = 256;
constexpr int kWinRows = 16;
constexpr int64_t kRowCost = 2;      // a row's fixed work (its P_i store, its window slots), in extras

// Causal graph: the first rows (over all units, u n + i) of quarters q and q + 1
// of nq, each the smallest row whose cost prefix u (kRowCost n + nx) +
// kRowCost i + x_ptr[i] reaches q / nq (resp. (q + 1) / nq) of the total.
// Monotone in q; q = nq gives units * n.  The quarter's 8 lanes run both
// searches together, 8 probes a round (about log9 n rounds of one load
// each).  All 8 lanes of the quarter must be converged here.  (The products
// stay far inside int64: nq < 2^15 and the total cost < 2^40.)
__device__ __forceinline__ void causal_row_range(const HopArgs& a, int64_t q, int64_t nq, int ql,
                                                 unsigned qmask, int shift, int64_t& R0,
                                                 int64_t& R1) {
    const int64_t n = a.plan.n;
    const int64_t per_unit = kRowCost * n + a.nx, total = a.units * per_unit;
    const int64_t t0 = q * total / nq, t1 = (q + 1) * total / nq;
    const int64_t u0 = t0 / per_unit, rem0 = t0 - u0 * per_unit;
    const int64_t u1 = t1 / per_unit, rem1 = t1 - u1 * per_unit;
    // the answer i lies in [lo, hi]; cost(i) >= rem is false below it, true from it on
    int64_t lo0 = 0, hi0 = n, lo1 = 0, hi1 = n;
    while (lo0 < hi0 || lo1 < hi1) {
        const int64_t p0 = lo0 + (hi0 - lo0) * (ql + 1) / 9;   // < hi0 while lo0 < hi0
        const int64_t p1 = lo1 + (hi1 - lo1) * (ql + 1) / 9;
        const bool f0 = lo0 < hi0 && kRowCost * p0 + __ldg(a.x_ptr + p0) >= rem0;
        const bool f1 = lo1 < hi1 && kRowCost * p1 + __ldg(a.x_ptr + p1) >= rem1;
        const unsigned b0 = (__ballot_sync(qmask, f0) >> shift) & 0xFFu;
        const unsigned b1 = (__ballot_sync(qmask, f1) >> shift) & 0xFFu;
        if (lo0 < hi0) {
            const int k = 8 - __popc(b0);                          // probes below the answer
            const int64_t plo = lo0 + (hi0 - lo0) * k / 9;         // probe k - 1 (if k > 0)
            const int64_t phi = lo0 + (hi0 - lo0) * (k + 1) / 9;   // probe k (if k < 8)
            if (k > 0) lo0 = plo + 1;
            if (k < 8) hi0 = phi;
        }
        if (lo1 < hi1) {
            const int k = 8 - __popc(b1);
            const int64_t plo = lo1 + (hi1 - lo1) * k / 9;
            const int64_t phi = lo1 + (hi1 - lo1) * (k + 1) / 9;
            if (k > 0) lo1 = plo + 1;
            if (k < 8) hi1 = phi;
        }
    }
    R0 = u0 * n + lo0;
    R1 = u1 * n + lo1;
}

template <bool kHop0, int kB, int kMinBlocks>
__global__ void __launch_bounds__(kGThreadsG, kMinBlocks)
hop_gather_kernel(HopArgs a) {
    static_assert(kB <= 8, "one slot per lane of a quarter");
    __shared__ int sStart[32][kWinRows + 1];      // per quarter: the window's row starts (unit-local slots)
    __shared__ float sMax[32][kWinRows];          // per quarter: the rows' m_i (first hop)
    __shared__ uint8_t sGlob[32][kWinRows];       // per quarter: the window's rows in G
    const BandPlan& P = a.plan;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ql = lane & 7;
    const int qi = 4 * warp + (lane >> 3);
    const unsigned qmask = 0xFFu << (lane & 24);  // this quarter's lanes
    const int64_t nq = (int64_t)gridDim.x * 32, q = (int64_t)blockIdx.x * 32 + qi;
    int64_t R0, R1;
    if (P.causal) {
        causal_row_range(a, q, nq, ql, qmask, lane & 24, R0, R1);
    } else {
        const int64_t rows_total = a.units * P.n;
        R0 = q * rows_total / nq;
        R1 = (q + 1) * rows_total / nq;
    }
    int* ss = sStart[qi];
    float* sm = sMax[qi];
    uint8_t* sg = sGlob[qi];
    if (!kHop0 && P.g > 0) {
        // Z_k of the global rows, from the previous hop's shares: one float4 per
        // quarter-warp (or per thread, global_row_out), spread over all CTAs (no
        // extra reads them: the extras exclude G)
        const int64_t per_unit = (int64_t)P.g * (kHeadDim / 4), total = a.units * per_unit;
        if (P.tiles >= kCoopTiles) {
            for (int64_t idx = (int64_t)qi * gridDim.x + blockIdx.x; idx < total;
                 idx += (int64_t)(kGThreadsG / 8) * gridDim.x) {
                const int64_t u = idx / per_unit;
                const int rem = (int)(idx - u * per_unit);
                global_row_out<false>(a, a.gpart, u, rem >> 4, rem & 15, 8, ql, qmask, a.Zk_hilo, a.Zk_f);
            }
        } else {
            for (int64_t idx = (int64_t)tid * gridDim.x + blockIdx.x; idx < total;
                 idx += (int64_t)blockDim.x * gridDim.x) {
                const int64_t u = idx / per_unit;
                const int rem = (int)(idx - u * per_unit);
                global_row_out<false>(a, a.gpart, u, rem >> 4, rem & 15, 1, 0, 0u, a.Zk_hilo, a.Zk_f);
            }
        }
        __syncwarp();     // reconverge: the quarters below synchronize only among themselves
    }
    for (int64_t Rw = R0; Rw < R1;) {
        const int64_t u = Rw / P.n;
        const int64_t iw = Rw - u * P.n;
        int64_t cnt64 = R1 - Rw;
        if (cnt64 > P.n - iw) cnt64 = P.n - iw;
        const int cnt = cnt64 < kWinRows ? (int)cnt64 : kWinRows;
        const size_t ubase = (size_t)u * P.n;
        // the window's row starts, global flags (and row maxima)
        for (int m = ql; m <= cnt; m += 8) {
            ss[m] = (int)a.x_ptr[iw + m];
            if (m < cnt) {
                sg[m] = a.is_global[iw + m];
                if (kHop0) sm[m] = a.m_sparse[ubase + iw + m];
            }
        }
        __syncwarp(qmask);
        const int sb = ss[0], se = ss[cnt];
        float* wq = a.A_x + (size_t)u * a.nx;
        // this lane's features of row j of Z_k: fp32 rows, features 4 ql .. +3 and
        // 32 + 4 ql .. +3 at zrow + 16 j (two 128-byte lines per quarter); the first
        // hop's bf16 V rows, features 8 ql .. +7 at vrow + 8 j (one line per quarter).
        // The accumulators hold the same features, in the same order.  The rows are
        // read past L1 (.cg): few of them are read twice by one SM.
        const uint4* zrow = reinterpret_cast<const uint4*>(a.Zf_in) + ubase * 16 + ql;
        const uint4* vrow = reinterpret_cast<const uint4*>(a.V) + ubase * 8 + ql;
        float4* prow = reinterpret_cast<float4*>(a.Psum) + ubase * 16 + (kHop0 ? 2 * ql : ql);
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
        int cur = 0;                              // window row being accumulated
        int nb = ss[1];                           // first slot past row cur
        // First hop only: the extras' weights arrive as raw scores s; each
        // becomes e = exp(s - m_i) (stored back for the later hops), and the
        // row's sum of e is added to inv_l_i (the globals' part of the sum on
        // entry; the band kernel adds the band part and inverts it).
        float mcur = kHop0 ? sm[0] : 0.f;
        float lsum = 0.f;
        // closes row cur: its partial P_i (and, first hop, inv_l_i)
        auto finish_row = [&]() {
            if (!sg[cur]) {
                float4* pr = prow + (size_t)(iw + cur) * 16;
                pr[0] = make_float4(acc[0].x, acc[0].y, acc[1].x, acc[1].y);
                pr[kHop0 ? 1 : 8] = make_float4(acc[2].x, acc[2].y, acc[3].x, acc[3].y);
                if (kHop0 && ql == 0) a.inv_l[ubase + iw + cur] += lsum;
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[k] = make_float2(0.f, 0.f);
            lsum = 0.f;
            ++cur;
        };
        // slot sb + ql's index and weight (slots past the window read row 0 with weight 0)
        int32_t jc = 0;
        float wc = 0.f;
        if (ql < kB && sb + ql < se) { jc = __ldg(a.x_col + sb + ql); wc = __ldg(wq + sb + ql); }
        for (int e0 = sb; e0 < se; e0 += kB) {
            int32_t jn = 0;
            float wn = 0.f;
            const int en = e0 + kB + ql;
            if (ql < kB && en < se) { jn = __ldg(a.x_col + en); wn = __ldg(wq + en); }
            uint4 zr[kB][kHop0 ? 1 : 2];
#pragma unroll
            for (int b = 0; b < kB; ++b) {
                const int j = __shfl_sync(qmask, jc, b, 8);
                if (kHop0) {
                    zr[b][0] = __ldcg(vrow + 8 * j);
                } else {
                    zr[b][0] = __ldcg(zrow + 16 * j);
                    zr[b][kHop0 ? 0 : 1] = __ldcg(zrow + 16 * j + 8);
                }
            }
            if (e0 + kB <= nb) {
                // the whole batch belongs to row cur
                if (kHop0) {
                    wc = expf(wc - mcur);
                    if (ql < kB) wq[e0 + ql] = wc;
                }
#pragma unroll
                for (int b = 0; b < kB; ++b) {
                    const float w = __shfl_sync(qmask, wc, b, 8);
                    if (kHop0) lsum += w;
                    ffma_row<kHop0>(acc, w, zr[b]);
                }
            } else {
#pragma unroll
                for (int b = 0; b < kB; ++b) {
                    const int e = e0 + b;
                    if (e < se) {
                        while (e >= nb) {
                            finish_row();
                            nb = ss[cur < cnt ? cur + 1 : cnt];
                            if (kHop0) mcur = sm[cur];
                        }
                        float w = __shfl_sync(qmask, wc, b, 8);
                        if (kHop0) {
                            w = expf(w - mcur);
                            if (ql == b) wq[e] = w;
                            lsum += w;
                        }
                        ffma_row<kHop0>(acc, w, zr[b]);
                    }
                }
            }
            jc = jn;
            wc = wn;
        }
        // the rows left (the last one, and any without extras)
        while (cur < cnt) finish_row();
        __syncwarp(qmask);                        // the window's smem is rewritten next
        Rw += cnt;
    }
}

// the gather configuration: slots in flight per quarter-warp (hops after the
// first, the first hop), CTAs per SM
constexpr int kGatherBatch = 5, kGatherBatch0 = 8, kGatherBlocks = 3;

// bf16 tensor map over rows of `row_elems` elements: box of 64 elements x box_rows rows
int encode_rows(CUtensorMap* m, const void* base, int64_t n, int64_t units, int row_elems,
                int box_rows = kChunkKeys) {
    auto fn = band::tensor_map_encoder();
    if (!fn) return fail(DIFFUSER_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    const cuuint64_t dims[3] = {(cuuint64_t)row_elems, (cuuint64_t)n, (cuuint64_t)units};
    const cuuint64_t strides[2] = {(cuuint64_t)row_elems * 2, (cuuint64_t)n * row_elems * 2};
    const cuuint32_t box[3] = {(cuuint32_t)kHeadDim, (cuuint32_t)box_rows, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(DIFFUSER_ERR_CUDA, "cuTensorMapEncodeTiled failed: " + std::to_string((int)r));
    return DIFFUSER_OK;
}

int sm_count() {
    static int num_sms = 0;
    if (num_sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || num_sms < 1)
            num_sms = 1;
    }
    return num_sms;
}

// One CTA per SM, or more (in waves) when an SM's share would exceed the tile table.
int64_t band_ctas(int64_t total_tiles) {
    const int64_t sms = sm_count();
    int64_t ctas = total_tiles < sms ? total_tiles : sms;
    if ((total_tiles + ctas - 1) / ctas > kMaxCtaTiles) ctas = (total_tiles + kMaxCtaTiles - 1) / kMaxCtaTiles;
    return ctas;
}

template <bool kHop0, bool kLast>
int launch_hop(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmZ, const HopArgs& a,
               cudaStream_t stream) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(hop_band_kernel<kHop0, kLast>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytesMax);
    });
    if (attr_err != cudaSuccess) return cuda_fail(attr_err, "cudaFuncSetAttribute(hop)");
    const int sms = sm_count();
    const int64_t total_tiles = a.units * a.plan.tiles;
    {
        LaunchScope scope(DIFFUSER_KERNEL_GATHER, stream);
        hop_gather_kernel<kHop0, kHop0 ? kGatherBatch0 : kGatherBatch, kGatherBlocks>
            <<<(unsigned)(sms * kGatherBlocks), kGThreadsG, 0, stream>>>(a);
    }
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return cuda_fail(err, "hop_gather_kernel");
    dim3 grid((unsigned)band_ctas(total_tiles));
    {
        LaunchScope scope(DIFFUSER_KERNEL_HOP, stream);
        hop_band_kernel<kHop0, kLast><<<grid, kThreads, band_smem_bytes(a.plan.g16), stream>>>(tmQ, tmK, tmZ, a);
    }
    err = cudaGetLastError();
    if (err != cudaSuccess) return cuda_fail(err, "hop_band_kernel");
    if (kLast && a.plan.g > 0) {
        LaunchScope scope(DIFFUSER_KERNEL_GATHER, stream);
        const int64_t outs = a.units * a.plan.g * (kHeadDim / 4);
        const int64_t threads = a.plan.tiles >= kCoopTiles ? 8 * outs : outs;
        hop_global_out_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, stream>>>(a);
    }
    err = cudaGetLastError();
    return err == cudaSuccess ? DIFFUSER_OK : cuda_fail(err, "hop_global_out_kernel");
}

// A tile's cost in the deal: 2 per 128-key chunk and 1 for the tile's own
// hand-offs (a tile boundary costs about half a chunk's period).
int64_t band_tile_cost(const BandPlan& P, int nc, int t) {
    int lo, hi;
    chunk_range(P, nc, (int64_t)t * kTileRows, lo, hi);
    return 2 * (int64_t)(hi - lo + 1) + 1;
}

}  // namespace

// The deal tables of a graph's band path, one per (units, CTAs); never evicted, as
// a captured replay of a forward holds the pointers it was launched with.
struct BandDeals {
    struct Entry {
        int64_t units;
        int64_t ctas;
        int32_t* d_ptr;
        int32_t* d_tiles;
    };
    std::mutex mu;
    std::vector<Entry> entries;
};

BandDeals* create_band_deals() { return new (std::nothrow) BandDeals(); }

void destroy_band_deals(BandDeals* d) {
    if (!d) return;
    for (auto& e : d->entries) {
        cudaFree(e.d_ptr);
        cudaFree(e.d_tiles);
    }
    delete d;
}

namespace {

constexpr size_t kMaxBandDeals = 4;

// The snake order over the rounds gives every CTA ceil or floor of tiles / CTAs
// tiles; when that does not divide, the CTAs with one tile more get their share
// of heavy tiles as well (4 interior tiles and 2 edge tiles, where 3 and 3 would
// do).  Starting from the snake deal, the busiest CTA repeatedly trades a tile for
// a lighter one of the least busy CTA (or hands it one) while that lowers the
// larger of the two loads.  Each CTA then takes its tiles in item order (heaviest
// first, neighbouring tiles together).  Where no trade helps, the launch keeps the
// snake order (a null table).  Built on the first launch for (units, CTAs), outside
// stream capture; while the caller's stream is capturing, after
// kMaxBandDeals tables, or when a CTA's list would not fit its table, the kernel
// deals in snake order instead.
void band_deal(const diffuser_graph* g, const BandPlan& P, int64_t units, int64_t ctas,
               cudaStream_t stream, HopArgs& a) {
    a.deal_ptr = nullptr;
    a.deal_tiles = nullptr;
    BandDeals* D = g->band_deals;
    if (!D || ctas < 2) return;
    std::lock_guard<std::mutex> lk(D->mu);
    for (const auto& e : D->entries)
        if (e.units == units && e.ctas == ctas) {
            a.deal_ptr = e.d_ptr;
            a.deal_tiles = e.d_tiles;
            return;
        }
    if (D->entries.size() >= kMaxBandDeals) return;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) return;
    const int64_t total = units * (int64_t)P.tiles;
    if (total > INT32_MAX) return;
    const int nc = P.chunks / 2;
    std::vector<int64_t> pos_cost((size_t)P.tiles);
    for (int t = 0; t < P.tiles; ++t) pos_cost[(size_t)t] = band_tile_cost(P, nc, t);
    std::vector<int32_t> tile_of((size_t)total);
    std::vector<int64_t> cost((size_t)total);
    std::vector<std::vector<int64_t>> lists((size_t)ctas);   // items k per CTA
    std::vector<int64_t> load((size_t)ctas, 0);
    for (int64_t k = 0; k < total; ++k) {
        int64_t u;
        int t;
        band_item(P, units, nc, k, u, t);
        tile_of[(size_t)k] = (int32_t)(u * P.tiles + t);
        cost[(size_t)k] = pos_cost[(size_t)t];
        const int64_t r = k / ctas, q = k - r * ctas, b = (r & 1) ? ctas - 1 - q : q;
        lists[(size_t)b].push_back(k);
        load[(size_t)b] += cost[(size_t)k];
    }
    int64_t trades = 0;
    for (int64_t iter = 0; iter < 4 * ctas; ++iter, ++trades) {
        const size_t M = (size_t)(std::max_element(load.begin(), load.end()) - load.begin());
        const size_t B = (size_t)(std::min_element(load.begin(), load.end()) - load.begin());
        if (M == B) break;
        // the best trade: hand over x (y = none) or swap x for a lighter y
        int64_t best = load[M];
        long bx = -1, by = -1;
        for (size_t ix = 0; ix < lists[M].size(); ++ix) {
            const int64_t cx = cost[(size_t)lists[M][ix]];
            if (lists[B].size() < (size_t)kMaxCtaTiles) {
                const int64_t worst = std::max(load[M] - cx, load[B] + cx);
                if (worst < best) { best = worst; bx = (long)ix; by = -1; }
            }
            for (size_t iy = 0; iy < lists[B].size(); ++iy) {
                const int64_t d = cx - cost[(size_t)lists[B][iy]];
                if (d <= 0) continue;
                const int64_t worst = std::max(load[M] - d, load[B] + d);
                if (worst < best) { best = worst; bx = (long)ix; by = (long)iy; }
            }
        }
        if (bx < 0) break;
        const int64_t kx = lists[M][(size_t)bx];
        lists[M].erase(lists[M].begin() + bx);
        load[M] -= cost[(size_t)kx];
        if (by >= 0) {
            const int64_t ky = lists[B][(size_t)by];
            lists[B].erase(lists[B].begin() + by);
            load[B] -= cost[(size_t)ky];
            lists[M].push_back(ky);
            load[M] += cost[(size_t)ky];
        }
        lists[B].push_back(kx);
        load[B] += cost[(size_t)kx];
    }
    if (trades == 0) {                                // the snake order itself: no table
        D->entries.push_back({units, ctas, nullptr, nullptr});
        return;
    }
    std::vector<int32_t> ptr((size_t)ctas + 1, 0), tiles;
    tiles.reserve((size_t)total);
    for (int64_t b = 0; b < ctas; ++b) {
        auto& l = lists[(size_t)b];
        if (l.size() > (size_t)kMaxCtaTiles) return;
        std::sort(l.begin(), l.end());
        for (int64_t k : l) tiles.push_back(tile_of[(size_t)k]);
        ptr[(size_t)b + 1] = (int32_t)tiles.size();
    }
    int32_t *dp = nullptr, *dt = nullptr;
    cudaError_t err = cudaMalloc(&dp, sizeof(int32_t) * ptr.size());
    if (err == cudaSuccess) err = cudaMalloc(&dt, sizeof(int32_t) * tiles.size());
    if (err == cudaSuccess) err = cudaMemcpy(dp, ptr.data(), sizeof(int32_t) * ptr.size(), cudaMemcpyHostToDevice);
    if (err == cudaSuccess)
        err = cudaMemcpy(dt, tiles.data(), sizeof(int32_t) * tiles.size(), cudaMemcpyHostToDevice);
    if (err != cudaSuccess) {
        cudaFree(dp);
        cudaFree(dt);
        cudaGetLastError();                           // the snake order serves instead
        return;
    }
    D->entries.push_back({units, ctas, dp, dt});
    a.deal_ptr = dp;
    a.deal_tiles = dt;
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
    w.A_band = reinterpret_cast<__nv_bfloat16*>(ws + L.a_band);
    w.A_gc = reinterpret_cast<float*>(ws + L.a_gc);
    w.A_gcimg = reinterpret_cast<uint8_t*>(ws + L.a_gcimg);
    w.A_x = reinterpret_cast<float*>(ws + L.a_x);
    w.A_gr = reinterpret_cast<float*>(ws + L.a_gr);
    w.A_gimg = reinterpret_cast<uint8_t*>(ws + L.a_gimg);
    w.inv_l = reinterpret_cast<float*>(ws + L.inv_l);
    w.m_sparse = reinterpret_cast<float*>(ws + L.m_sparse);
    w.gstat = reinterpret_cast<float*>(ws + L.gstat);
    return w;
}

bool band_plan(const diffuser_graph* g, BandPlan* p) {
    if (g->kind != kTokenGraph || g->dilation != 1 || g->r < 8 || g->n_globals > kBandMaxGlobals)
        return false;
    p->n = g->n;
    p->r = g->r;
    p->causal = g->causal ? 1 : 0;
    p->r64 = (g->r + kChunkKeys - 1) / kChunkKeys * kChunkKeys;
    p->g = g->n_globals;
    p->g_pad = (g->n_globals + 3) / 4 * 4;
    if (p->g_pad == 0) p->g_pad = 4;
    p->g16 = (g->n_globals + 15) / 16 * 16;
    p->tiles = (int32_t)((g->n + kTileRows - 1) / kTileRows);
    // keys i0 - r64 .. i0 + 127 + (the window's upper radius: r, or 0 when causal),
    // in an even number of 64-key chunks (the hop kernel takes them in pairs)
    const int64_t up = g->causal ? 0 : g->r;
    p->chunks = (int32_t)((p->r64 + kTileRows + up + kChunkKeys - 1) / kChunkKeys);
    p->chunks += p->chunks & 1;
    p->band_unit = (size_t)p->tiles * p->chunks * band::kChunkImageBytes;
    return true;
}

int plan_band_layout(const diffuser_graph* g, const BandPlan& p, int64_t units, BandLayout* L) {
    auto al = [](size_t x) { return (x + 1023) / 1024 * 1024; };
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off += al(bytes); return o; };
    const size_t U = (size_t)units;
    const size_t gg = p.g > 0 ? (size_t)p.g : 1;
    L->a_band = take(U * p.band_unit);
    L->a_gc = take(U * (size_t)p.n * p.g_pad * 4);
    L->a_gcimg = take(U * (size_t)p.tiles * 2 * band::gc_plane_bytes(p.g16 > 0 ? p.g16 : 16));
    L->a_x = take(U * (size_t)(g->nx > 0 ? g->nx : 1) * 4);
    L->a_gr = take(U * gg * p.n * 4);
    L->a_gimg = take(U * (size_t)p.tiles * band::kGImgBytes);
    for (int s = 0; s < 2; ++s) L->z[s] = take(U * (size_t)p.n * 2 * kHeadDim * 2);
    for (int s = 0; s < 2; ++s) L->zf[s] = take(U * (size_t)p.n * kHeadDim * 4);
    L->psum = take(U * (size_t)p.n * kHeadDim * 4);
    L->gpart = take(U * (size_t)p.tiles * gg * kHeadDim * 4);
    L->inv_l = take(U * (size_t)p.n * 4);
    L->m_sparse = take(U * (size_t)p.n * 4);
    L->gstat = take(U * gg * 2 * 4);
    L->total = off;
    return DIFFUSER_OK;
}

int launch_band_hops(const diffuser_graph* g, const BandPlan& p, int64_t units, const void* Q,
                     const void* K, const void* V, int32_t hops, float alpha, void* out, char* ws,
                     const BandLayout& L, cudaStream_t stream) {
    // tensor maps: Q tiles and K chunks (the scores), and the B operand of the
    // weights' MMA: V ([n][64]) for hop 0, then the Z_k rows ([n][hi | lo])
    CUtensorMap tmQ, tmK, tmV, tmZ[2];
    int st = encode_rows(&tmQ, Q, p.n, units, kHeadDim, kTileRows);
    if (!st) st = encode_rows(&tmK, K, p.n, units, kHeadDim, kCK);
    if (!st) st = encode_rows(&tmV, V, p.n, units, kHeadDim, kCK);
    for (int s = 0; s < 2 && !st; ++s) st = encode_rows(&tmZ[s], ws + L.z[s], p.n, units, 2 * kHeadDim, kCK);
    if (st) return st;

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
    a.A_x = reinterpret_cast<float*>(ws + L.a_x);
    a.m_sparse = reinterpret_cast<const float*>(ws + L.m_sparse);
    a.A_gimg = reinterpret_cast<const uint8_t*>(ws + L.a_gimg);
    a.inv_l = reinterpret_cast<float*>(ws + L.inv_l);
    a.Psum = reinterpret_cast<float*>(ws + L.psum);
    a.A_gcimg = reinterpret_cast<const uint8_t*>(ws + L.a_gcimg);
    a.V = static_cast<const __nv_bfloat16*>(V);
    a.gpart = reinterpret_cast<float*>(ws + L.gpart);
    a.status = g->d_status;
    a.out = static_cast<__nv_bfloat16*>(out);
    band_deal(g, p, units, band_ctas(units * p.tiles), stream, a);
    // Z_{k+1} of hop k lives in z[k & 1]; hop k reads Z_k (V for k = 0)
    for (int32_t k = 0; k < hops; ++k) {
        const bool first = k == 0, last = k == hops - 1;
        a.Z_out = reinterpret_cast<__nv_bfloat16*>(ws + L.z[k & 1]);
        a.Zf_in = first ? nullptr : reinterpret_cast<const float*>(ws + L.zf[(k - 1) & 1]);
        a.Zf_out = reinterpret_cast<float*>(ws + L.zf[k & 1]);
        a.Zk_hilo = first ? nullptr : reinterpret_cast<__nv_bfloat16*>(ws + L.z[(k - 1) & 1]);
        a.Zk_f = first ? nullptr : reinterpret_cast<float*>(ws + L.zf[(k - 1) & 1]);
        const CUtensorMap& tm = first ? tmV : tmZ[(k - 1) & 1];
        if (first && last) st = launch_hop<true, true>(tmQ, tmK, tm, a, stream);
        else if (first) st = launch_hop<true, false>(tmQ, tmK, tm, a, stream);
        else if (last) st = launch_hop<false, true>(tmQ, tmK, tm, a, stream);
        else st = launch_hop<false, false>(tmQ, tmK, tm, a, stream);
        if (st) return st;
    }
    return DIFFUSER_OK;
}

}  // namespace dfs
