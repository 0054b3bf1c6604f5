// Block-sparse path: the BigBird ITC block graph with 64-token blocks, bf16
// I/O ("1.2.1 Static sparsity: Longformer, BigBird and sliding windows", sec 2
// eq 13 and the 12-block example; "038 BigBird: keeping long-sequence
// information paths with sparse connections", sec 2: block row J reads its
// window blocks, the global blocks and its random blocks; the global block
// rows read every block).  Every allowed block pair is a dense 64 x 64 piece
// of the score matrix and of A, so both contractions run on the tcgen05
// tensor cores:
//
//  * A tile is 128 rows: block rows J0 = 2T and J1 = 2T + 1.  Its key blocks
//    are the union of the two rows' allowed blocks, ascending, taken two at a
//    time as 128-key chunks (kb0, kb1) with a 2 x 2 mask: which of the two
//    block rows each key block is allowed for.  The lists are built once per
//    graph on the host from the graph's own CSR (every token of a block row
//    has the same neighbour set, so the first token's row gives the blocks).
//  * the score pass: S = Q_tile K_chunk^T per chunk (bf16 operands, fp32
//    accumulation in tensor memory); each row's maximum over its allowed keys
//    (the row softmax, "Diffuser: modelling long sequences with multi-hop
//    attention diffusion", eq S.1-S.5): m_i on the base-2 exponent scale.  The
//    first hop adds up each row's weights and stores inv_l_i = 1 / l_i.
//  * block_hop_kernel (one launch per hop, eq S.7): S again for every chunk
//    (the same MMAs, so the same values), e_ij = 2^(s_ij log2(e) / 8 - m_i) on
//    the allowed keys (0 elsewhere) written over the scores as bf16 hi + lo
//    (hi = e rounded to bf16, lo = the remainder rounded to bf16), then
//    D += e_hi [Z_hi | Z_lo] + e_lo Z_hi on the tensor cores with Z_k held as
//    bf16 hi + lo rows; the e_lo Z_lo term (below 2^-16 of the product) is the
//    only one left out.  Epilogue: z_i = (1 - alpha) inv_l_i D_i + alpha V_i,
//    written as the next [hi | lo] row, or as the bf16 output after the last
//    hop.  Storing A instead would cost 4 bytes per edge per hop of HBM
//    traffic; the recomputation costs one exp per edge and a K = 64 MMA.  The
//    first hop's weight warps also add up each row's weights (fp32, before the
//    split) and hand the four key slices' sums to the epilogue, which stores
//    inv_l_i for the later hops.
//
// Roles (24 warps, one CTA per SM, persistent over a per-CTA tile table):
// warp 0 loads Q tiles and K chunks (TMA), warp 1 issues the score MMAs,
// warp 2 the weights' MMAs, warp 3 loads the Z_k chunks, warps 4-19 turn
// scores into weights (warp w: TMEM lane quadrant w % 4, keys 16 ((w - 4) / 4)
// .. +15 of both 64-key halves), warps 20-23 are the epilogue (hop) or merge
// the four key slices' row maxima (score).  Every barrier wait is bounded
// (ptx::mbar_wait) and records a status instead of hanging.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <functional>
#include <mutex>
#include <queue>
#include <utility>
#include <vector>

#include "band_common.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace dfs {
namespace {

constexpr int kBlock = 64;                 // tokens per block (the only block size of this path)
constexpr int kTile = 128;                 // rows per tile: two block rows
constexpr int kCK = 128;                   // keys per chunk: two key blocks
constexpr int kThreads = 768;
constexpr int kTmaWarp = 0, kSMmaWarp = 1, kPvMmaWarp = 2, kZWarp = 3;
constexpr int kSoftWarp0 = 4, kSoftWarps = 16, kSlices = 4;
constexpr int kEpiWarp0 = 20, kEpiWarps = 4;
constexpr int kEpiRowFloats = 68;          // staging row, padded against bank conflicts
constexpr int kQBytes = kTile * kHeadDim * 2;       // 16 KB
constexpr int kKBytes = kCK * kHeadDim * 2;         // 16 KB (two 64-row boxes)
constexpr int kHalfBytes = kBlock * kHeadDim * 2;   // 8 KB: one key block of K or of a Z half
constexpr int kZTileBytes = kCK * 128;              // one 64-feature half (hi or lo) of a chunk
constexpr int kZStageBytes = 2 * kZTileBytes;
constexpr int kSlots = 3;                  // pipeline slots (chunk g uses slot g % 3)
constexpr int kSCol0 = 128;                // score / weight buffers: columns 128 + 128 b
constexpr int kTmemCols = 512;             // D in [0, 128)
constexpr int kMaxCtaTiles = 256;
constexpr float kLog2eScale = 1.4426950408889634f * 0.125f;   // log2(e) / sqrt(64)

// Launch modes: bit 0 a hop (else the score pass), bit 1 the first hop (reads
// V, whose lo part is zero), bit 2 the last hop (writes the output)
enum Mode { kScore = 0, kHopMid = 1, kHopFirst = 3, kHopLast = 5, kHopOnly = 7 };

struct TileEntry { int32_t u, t, c0, c1; };      // unit, tile position, chunks [c0, c1)

struct BlockArgs {
    int64_t n;
    int64_t units;
    int32_t tiles;                 // tile positions per unit
    const int32_t* chunks;         // [total][4]: kb0, kb1, mask bits, 0
    const int32_t* tile_ptr;       // [tiles + 1] chunk range of each position
    const int32_t* order;          // [tiles] positions by falling chunk count
    const int32_t* deal_ptr;       // [CTAs + 1] each CTA's range of deal_items (null: snake order)
    const int32_t* deal_items;     // launch items k (position rank k / units, unit k % units)
    float* mb2;                    // [units][n] row max of s log2(e) / 8 over the allowed keys
    float* inv_l;                  // [units][n] 1 / sum of 2^(s log2(e) / 8 - mb2) (first hop)
    const __nv_bfloat16* V;        // [units][n][64]
    __nv_bfloat16* Z_out;          // [units][n][hi 64 | lo 64], all hops but the last
    __nv_bfloat16* out;            // the last hop's output [units][n][64]
    float alpha;
    int* status;
};

__host__ __device__ constexpr int block_smem_bytes() {
    return 1024 + 2 * kQBytes + kSlots * (kKBytes + kZStageBytes) + 4 * 32 * kEpiRowFloats * 4 +
           4 * 32 * 4 + 2 * kSlices * kTile * 4 +
           kMaxCtaTiles * (int)sizeof(TileEntry) + 512;
}
static_assert(block_smem_bytes() <= 227 * 1024, "shared memory per CTA");
static_assert(block_smem_bytes() > 116 * 1024, "must exclude a second CTA per SM");

// Item k of the launch (position rank k / units, unit k % units).  With a deal
// table (built on the host, see block_deal) each CTA takes its listed items;
// without one the items go to the CTAs heaviest first in snake order over the
// rounds (round r: CTA b gets item r G + b, or r G + G - 1 - b when r is odd).
__device__ __forceinline__ int cta_tile_count(int64_t total) {
    const int64_t G = gridDim.x, b = blockIdx.x, R = total / G, rem = total - R * G;
    return (int)(R + ((R & 1) == 0 ? (b < rem ? 1 : 0) : (b >= G - rem ? 1 : 0)));
}

template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
block_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
             const __grid_constant__ CUtensorMap tmZ, BlockArgs a) {
    constexpr bool kHop = (kMode & 1) != 0;
    constexpr bool kHop0 = (kMode & 2) != 0;
    constexpr bool kLast = (kMode & 4) != 0;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* sQ = smem;                                          // 2 x 16 KB
    uint8_t* sK = sQ + 2 * kQBytes;                              // kSlots x 16 KB
    uint8_t* sZ = sK + kSlots * kKBytes;                         // kSlots x (hi 16 KB, lo 16 KB)
    float* sEpi = reinterpret_cast<float*>(sZ + kSlots * kZStageBytes);   // [4][32][68]
    float* sKeep = sEpi + 4 * 32 * kEpiRowFloats;                // [4][32]
    float* xch = sKeep + 4 * 32;                                 // [2][kSlices][128] row maxima / sums
    TileEntry* sTile = reinterpret_cast<TileEntry*>(xch + 2 * kSlices * kTile);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sTile + kMaxCtaTiles);
    uint64_t* full_Q = bars;                  // [2]
    uint64_t* empty_Q = full_Q + 2;           // [2]
    uint64_t* full_K = empty_Q + 2;           // [kSlots]
    uint64_t* full_S = full_K + kSlots;       // [kSlots] scores written (also frees the K stage)
    uint64_t* full_P = full_S + kSlots;       // [kSlots] hop: key block 0 weighted + Z landed
    uint64_t* full_P1 = full_P + kSlots;      // [kSlots] hop: key block 1 weighted
    uint64_t* slot_free = full_P1 + kSlots;   // [kSlots] hop: weights' MMAs done; score: S read
    uint64_t* acc_full = slot_free + kSlots;
    uint64_t* acc_empty = acc_full + 1;
    uint64_t* xch_full = acc_empty + 1;       // [4][2] a quadrant's slices wrote their row maxima
                                              // (score) or row sums (first hop)
    uint64_t* xch_empty = xch_full + 8;       // [4][2] the epilogue warp has read them
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xch_empty + 8);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t total_items = a.units * a.tiles;
    const int my_tiles = a.deal_ptr ? a.deal_ptr[blockIdx.x + 1] - a.deal_ptr[blockIdx.x]
                                    : cta_tile_count(total_items);
    for (int lt = tid; lt < my_tiles && lt < kMaxCtaTiles; lt += kThreads) {
        const int64_t G = gridDim.x, b = blockIdx.x;
        const int64_t k = a.deal_ptr ? (int64_t)a.deal_items[a.deal_ptr[b] + lt]
                                     : (int64_t)lt * G + ((lt & 1) ? G - 1 - b : b);
        const int64_t rank = k / a.units, u = k - rank * a.units;
        const int t = a.order[rank];
        sTile[lt] = TileEntry{(int32_t)u, t, a.tile_ptr[t], a.tile_ptr[t + 1]};
    }
    if (warp == kSMmaWarp) ptx::tmem_alloc(tmem_slot, kTmemCols);
    if (tid == 0) {
        for (int s = 0; s < 2; ++s) { ptx::mbar_init(&full_Q[s], 1); ptx::mbar_init(&empty_Q[s], 1); }
        for (int s = 0; s < kSlots; ++s) {
            ptx::mbar_init(&full_K[s], 1);
            ptx::mbar_init(&full_S[s], 1);
            ptx::mbar_init(&full_P[s], kSoftWarps + 1);   // the weight warps + the Z copies' arrival
            ptx::mbar_init(&full_P1[s], kSoftWarps);
            ptx::mbar_init(&slot_free[s], kHop ? 1 : kSoftWarps);
        }
        ptx::mbar_init(acc_full, 1);
        ptx::mbar_init(acc_empty, kEpiWarps);
        for (int s = 0; s < 8; ++s) { ptx::mbar_init(&xch_full[s], kSlices); ptx::mbar_init(&xch_empty[s], 1); }
        ptx::fence_mbar_init();
    }
    if (warp == kTmaWarp && lane == 0) {
        ptx::prefetch_tensormap(&tmQ);
        ptx::prefetch_tensormap(&tmK);
        if (kHop) ptx::prefetch_tensormap(&tmZ);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // the set-up above reads only the graph's lists; everything below may touch what
    // the previous launch on the stream reads or writes
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    int total = 0;                                   // this CTA's chunks
    for (int lt = 0; lt < my_tiles; ++lt) total += sTile[lt].c1 - sTile[lt].c0;
    auto chunk = [&](int c) { return reinterpret_cast<const int4*>(a.chunks)[c]; };

    if (warp == kTmaWarp) {
        // ---------------- Q tiles and K chunks (two 64-key boxes each), in MMA order
        // (the whole warp runs the loop; the elected lane issues the copies)
        {
            const uint64_t pol_keep = ptx::l2_evict_last();
            int g = 0, b = 0, ph = 0;
            for (int lt = 0; lt < my_tiles; ++lt) {
                const TileEntry te = sTile[lt];
                const int qb = lt & 1;
                if (lt >= 2) ptx::mbar_wait(&empty_Q[qb], ((lt / 2) - 1) & 1, a.status);
                __syncwarp();
                if (ptx::elect_one()) {
                    ptx::mbar_arrive_expect_tx(&full_Q[qb], kQBytes);
                    ptx::tma_load_3d_hint(sQ + qb * kQBytes, &tmQ, &full_Q[qb], 0, te.t * kTile, te.u, pol_keep);
                }
                for (int c = te.c0; c < te.c1; ++c, ++g) {
                    const int4 ch = chunk(c);
                    if (g >= kSlots) ptx::mbar_wait(&full_S[b], ph ^ 1, a.status);
                    __syncwarp();
                    if (ptx::elect_one()) {
                        ptx::mbar_arrive_expect_tx(&full_K[b], kKBytes);
                        ptx::tma_load_3d_hint(sK + b * kKBytes, &tmK, &full_K[b], 0, ch.x * kBlock, te.u, pol_keep);
                        ptx::tma_load_3d_hint(sK + b * kKBytes + kHalfBytes, &tmK, &full_K[b], 0, ch.y * kBlock,
                                              te.u, pol_keep);
                    }
                    if (++b == kSlots) { b = 0; ph ^= 1; }
                }
            }
        }
    } else if (warp == kZWarp) {
        // ---------------- Z_k chunks (hop): the two key blocks' hi rows, and lo rows after hop 0
        // (the whole warp runs the loop; the elected lane issues the copies)
        if (kHop) {
            const uint64_t pol_keep = ptx::l2_evict_last();
            int g = 0;
            for (int lt = 0; lt < my_tiles; ++lt) {
                const TileEntry te = sTile[lt];
                for (int c = te.c0; c < te.c1; ++c, ++g) {
                    const int4 ch = chunk(c);
                    const int b = g % kSlots;
                    if (g >= kSlots) ptx::mbar_wait(&slot_free[b], ((g / kSlots) - 1) & 1, a.status);
                    __syncwarp();
                    if (ptx::elect_one()) {
                        uint8_t* zdst = sZ + b * kZStageBytes;
                        ptx::mbar_arrive_expect_tx(&full_P[b], kHop0 ? 2 * kHalfBytes : 4 * kHalfBytes);
                        ptx::tma_load_3d_hint(zdst, &tmZ, &full_P[b], 0, ch.x * kBlock, te.u, pol_keep);
                        ptx::tma_load_3d_hint(zdst + kHalfBytes, &tmZ, &full_P[b], 0, ch.y * kBlock, te.u, pol_keep);
                        if (!kHop0) {
                            ptx::tma_load_3d_hint(zdst + kZTileBytes, &tmZ, &full_P[b], kHeadDim, ch.x * kBlock,
                                                  te.u, pol_keep);
                            ptx::tma_load_3d_hint(zdst + kZTileBytes + kHalfBytes, &tmZ, &full_P[b], kHeadDim,
                                                  ch.y * kBlock, te.u, pol_keep);
                        }
                    }
                }
            }
        }
    } else if (warp == kSMmaWarp) {
        // ---------------- score MMAs S[b] = Q_tile K_chunk^T (K-major, 128-byte swizzle)
        // (the whole warp runs the loop; the elected lane issues each instruction)
        {
            constexpr uint32_t idesc_s = ptx::mma_idesc(1, kCK);
            const uint64_t qdesc0 = ptx::sw128_kmajor_desc(ptx::smem_u32(sQ));
            const uint64_t kdesc0 = ptx::sw128_kmajor_desc(ptx::smem_u32(sK));
            int g = 0, b = 0, ph = 0;
            for (int lt = 0; lt < my_tiles; ++lt) {
                const TileEntry te = sTile[lt];
                const int qb = lt & 1;
                ptx::mbar_wait(&full_Q[qb], (lt >> 1) & 1, a.status);
                const uint64_t qd = qdesc0 + (uint64_t)(qb * (kQBytes >> 4));
                for (int c = te.c0; c < te.c1; ++c, ++g) {
                    ptx::mbar_wait(&full_K[b], ph, a.status);
                    if (g >= kSlots) ptx::mbar_wait(&slot_free[b], ph ^ 1, a.status);
                    __syncwarp();
                    ptx::tc_fence_after();
                    const uint64_t kd = kdesc0 + (uint64_t)(b * (kKBytes >> 4));
                    const uint32_t dS = tmem + kSCol0 + kCK * b;
#pragma unroll
                    for (int ks = 0; ks < kHeadDim / 16; ++ks)
                        if (ptx::elect_one()) ptx::mma_bf16_ss(dS, qd + 2 * ks, kd + 2 * ks, idesc_s, ks > 0);
                    if (ptx::elect_one()) ptx::mma_commit(&full_S[b]);
                    if (c == te.c1 - 1 && ptx::elect_one()) ptx::mma_commit(&empty_Q[qb]);
                    if (++b == kSlots) { b = 0; ph ^= 1; }
                }
            }
            // drain: the last commit of each barrier lands before the CTA exits
            for (int s = 0; s < kSlots; ++s) {
                const int uses = (total - s + kSlots - 1) / kSlots;
                if (uses > 0) ptx::mbar_wait(&full_S[s], (uses - 1) & 1, a.status);
            }
            for (int s = 0; s < 2; ++s) {
                const int uses = (my_tiles - s + 1) / 2;
                if (uses > 0) ptx::mbar_wait(&empty_Q[s], (uses - 1) & 1, a.status);
            }
        }
    } else if (warp == kPvMmaWarp) {
        // ---------------- weights' MMAs (hop): D += e_hi [Z_hi | Z_lo] + e_lo Z_hi
        // (the whole warp runs the loop; the elected lane issues each instruction)
        if (kHop) {
            constexpr uint32_t idesc64 = ptx::mma_idesc_bf16_bmn(64);
            constexpr uint32_t idesc128 = ptx::mma_idesc_bf16_bmn(128);
            const uint64_t zdesc0 = ptx::sw128_mnmajor_desc(ptx::smem_u32(sZ), kZTileBytes);
            int sp = 0, pph = 0;
            for (int lt = 0; lt < my_tiles; ++lt) {
                const TileEntry te = sTile[lt];
                if (lt >= 1) ptx::mbar_wait(acc_empty, (lt - 1) & 1, a.status);
                __syncwarp();
                ptx::tc_fence_after();
                for (int c = te.c0; c < te.c1; ++c) {
                    ptx::mbar_wait(&full_P[sp], pph, a.status);
                    __syncwarp();
                    ptx::tc_fence_after();
                    const uint32_t pbuf = tmem + kSCol0 + kCK * sp;   // K step ks: hi 16 ks, lo 16 ks + 8
                    const uint64_t zd = zdesc0 + (uint64_t)(sp * (kZStageBytes >> 4));
#pragma unroll
                    for (int ks = 0; ks < kCK / 16; ++ks) {
                        if (ks == kCK / 32) {
                            ptx::mbar_wait(&full_P1[sp], pph, a.status);    // key block 1 weighted
                            __syncwarp();
                            ptx::tc_fence_after();
                        }
                        const uint64_t bdesc = zd + (uint64_t)(128 * ks);   // 16 keys = 2048 bytes on
                        if (ptx::elect_one())
                            ptx::mma_bf16_ts(tmem, pbuf + 16 * ks, bdesc, kHop0 ? idesc64 : idesc128,
                                             c != te.c0 || ks != 0);
                        if (ptx::elect_one()) ptx::mma_bf16_ts(tmem, pbuf + 16 * ks + 8, bdesc, idesc64, 1);
                    }
                    if (ptx::elect_one()) ptx::mma_commit(&slot_free[sp]);
                    if (c == te.c1 - 1 && ptx::elect_one()) ptx::mma_commit(acc_full);
                    if (++sp == kSlots) { sp = 0; pph ^= 1; }
                }
            }
            for (int s = 0; s < kSlots; ++s) {
                const int uses = (total - s + kSlots - 1) / kSlots;
                if (uses > 0) ptx::mbar_wait(&slot_free[s], (uses - 1) & 1, a.status);
            }
        }
    } else if (warp >= kSoftWarp0 && warp < kEpiWarp0) {
        // ---------------- scores -> weights (hop) or row statistics (score); thread <->
        // row t = 32 quad + lane of the tile, keys 16 slice .. +15 of both key blocks
        const int quad = warp & 3;
        const int slice = (warp - kSoftWarp0) >> 2;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const int t = quad * 32 + lane;
        const int rh = t >> 6;                       // 0: block row J0, 1: block row J1
        int lt = 0, sb = 0, sph = 0;
        TileEntry te = my_tiles > 0 ? sTile[0] : TileEntry{0, 0, 0, 0};
        int c = te.c0;
        int64_t urow = 0;
        bool row_ok = false;
        float b2 = 0.f;                              // hop: this row's m_i
        float m = -INFINITY;                         // score: running max
        float lsum = 0.f;                            // first hop: this slice's part of the row sum
        auto enter_tile = [&]() {
            const int64_t i = (int64_t)te.t * kTile + t;
            row_ok = i < a.n;
            urow = (size_t)te.u * a.n + (row_ok ? i : 0);
            if (kHop) b2 = row_ok ? __ldg(a.mb2 + urow) : 0.f;
            m = -INFINITY;
            lsum = 0.f;
        };
        // this slice's value of the row (max or sum) for the quadrant's epilogue warp at
        // the tile's last chunk; the buffer of this parity is free once that warp has
        // read tile lt - 2's
        auto hand_over = [&](float v) {
            const int xb = quad * 2 + (lt & 1);
            if (lt >= 2) ptx::mbar_wait(&xch_empty[xb], ((lt / 2) - 1) & 1, a.status);
            xch[((lt & 1) * kSlices + slice) * kTile + t] = v;
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&xch_full[xb]);
        };
        if (my_tiles > 0) enter_tile();
        for (int g = 0; g < total; ++g) {
            const int4 ch = chunk(c);
            ptx::mbar_wait(&full_S[sb], sph, a.status);
            __syncwarp();
            ptx::tc_fence_after();
            const uint32_t col = tmem + lane_base + kSCol0 + kCK * sb + 16 * slice;
            uint32_t ra[16], rb[16];
            ptx::tmem_ld16_issue(col, ra);
            ptx::tmem_ld16_issue(col + kBlock, rb);
            ptx::tmem_ld_wait16(ra);
            ptx::tmem_ld_wait16(rb);
            // keys of this slice in the two blocks; allowed for this row's block row, inside 0..n-1
            const int64_t j0 = (int64_t)ch.x * kBlock + 16 * slice, j1 = (int64_t)ch.y * kBlock + 16 * slice;
            const bool on0 = row_ok && ((ch.z >> rh) & 1), on1 = row_ok && ((ch.z >> (2 + rh)) & 1);
            const int lim0 = on0 ? (int)min((int64_t)16, a.n - j0) : 0;   // keys k < lim are in
            const int lim1 = on1 ? (int)min((int64_t)16, a.n - j1) : 0;
            if constexpr (!kHop) {
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&slot_free[sb]);       // the scores are in registers
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    if (k < lim0) m = fmaxf(m, __uint_as_float(ra[k]) * kLog2eScale);
                    if (k < lim1) m = fmaxf(m, __uint_as_float(rb[k]) * kLog2eScale);
                }
                if (c == te.c1 - 1) hand_over(m);
            } else {
                uint32_t hw[8], lw[8];
                auto split = [&](float x0, float x1, int p2) {
                    if (kHop0) lsum += x0 + x1;
                    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
                    const __nv_bfloat162 lo = __floats2bfloat162_rn(x0 - __low2float(h), x1 - __high2float(h));
                    hw[p2] = *reinterpret_cast<const uint32_t*>(&h);
                    lw[p2] = *reinterpret_cast<const uint32_t*>(&lo);
                };
                // lim is the same for the whole warp except in a ragged last tile: a key
                // block is allowed for all 16 keys (no per-key select, the scaling as
                // packed pairs) or for none (no exps), and only a block cut by the
                // sequence end takes the general path
                auto weights = [&](const uint32_t (&r)[16], int lim) {
                    if (lim >= 16) {
                        const float2 sc = make_float2(kLog2eScale, kLog2eScale), nb = make_float2(-b2, -b2);
#pragma unroll
                        for (int p2 = 0; p2 < 8; ++p2) {
                            const float2 y = __ffma2_rn(make_float2(__uint_as_float(r[2 * p2]), __uint_as_float(r[2 * p2 + 1])),
                                                        sc, nb);
                            split(ptx::ex2_approx(y.x), ptx::ex2_approx(y.y), p2);
                        }
                    } else if (lim <= 0) {
#pragma unroll
                        for (int p2 = 0; p2 < 8; ++p2) { hw[p2] = 0u; lw[p2] = 0u; }
                    } else {
#pragma unroll
                        for (int p2 = 0; p2 < 8; ++p2) {
                            const int k0 = 2 * p2, k1 = 2 * p2 + 1;
                            const float x0 = k0 < lim ? ptx::ex2_approx(fmaf(__uint_as_float(r[k0]), kLog2eScale, -b2)) : 0.f;
                            const float x1 = k1 < lim ? ptx::ex2_approx(fmaf(__uint_as_float(r[k1]), kLog2eScale, -b2)) : 0.f;
                            split(x0, x1, p2);
                        }
                    }
                };
                weights(ra, lim0);
                __syncwarp();       // reconverge before the warp-collective tcgen05.st
                ptx::tmem_st16_hilo(col, hw, lw);
                // key block 0's weights are in: its MMAs may start while block 1's are computed
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&full_P[sb]);
                weights(rb, lim1);
                __syncwarp();
                ptx::tmem_st16_hilo(col + kBlock, hw, lw);
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&full_P1[sb]);
                if (kHop0 && c == te.c1 - 1) hand_over(lsum);
            }
            if (++sb == kSlots) { sb = 0; sph ^= 1; }
            if (++c == te.c1 && ++lt < my_tiles) {
                te = sTile[lt];
                c = te.c0;
                enter_tile();
            }
        }
    } else if (warp >= kEpiWarp0) {
        const int quad = warp & 3;
        const int t = quad * 32 + lane;
        // the four key slices' values of row t of tile lt (max or sum), in slice order
        auto take_over = [&](int lt, bool is_max) {
            const int xb = quad * 2 + (lt & 1);
            ptx::mbar_wait(&xch_full[xb], (lt / 2) & 1, a.status);
            const float* xs = xch + (lt & 1) * kSlices * kTile + t;
            const float v = is_max ? fmaxf(fmaxf(xs[0], xs[kTile]), fmaxf(xs[2 * kTile], xs[3 * kTile]))
                                   : ((xs[0] + xs[kTile]) + xs[2 * kTile]) + xs[3 * kTile];
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&xch_empty[xb]);
            return v;
        };
        if constexpr (!kHop) {
            // ---------------- merge of the four slices' maxima: the row's m_i
            for (int lt = 0; lt < my_tiles; ++lt) {
                const TileEntry te = sTile[lt];
                const float mm = take_over(lt, true);
                const int64_t i = (int64_t)te.t * kTile + t;
                if (i < a.n) a.mb2[(size_t)te.u * a.n + i] = mm;
            }
        } else {
            // ---------------- epilogue: accumulator rows -> shared staging -> half a warp
            // per row, every global load and store covering whole lines
            const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
            float* st = sEpi + quad * (32 * kEpiRowFloats);
            float* sk = sKeep + quad * 32;
            const int hr = lane >> 4, f4 = lane & 15;
            for (int lt = 0; lt < my_tiles; ++lt) {
                const TileEntry te = sTile[lt];
                const int64_t i0 = (int64_t)te.t * kTile;
                {
                    // this quadrant's V rows (4 KB, contiguous) pulled into L2 now: the
                    // write loop below reads them after the tile's MMAs
                    const int64_t r0 = i0 + quad * 32;
                    const int64_t nr = a.n - r0 < 32 ? a.n - r0 : 32;
                    if (lane == 0 && nr > 0)
                        ptx::bulk_prefetch_l2(a.V + ((size_t)te.u * a.n + r0) * kHeadDim,
                                              (uint32_t)nr * kHeadDim * 2);
                }
                const int64_t i = i0 + t;
                const bool row_ok = i < a.n;
                const size_t urow = (size_t)te.u * a.n + (row_ok ? i : 0);
                float inv;
                if (kHop0) {
                    // the first hop completes the row sum from the four slices' parts
                    const float l = take_over(lt, false);
                    inv = row_ok ? 1.f / l : 0.f;
                    if (row_ok) a.inv_l[urow] = inv;
                } else {
                    inv = row_ok ? __ldg(a.inv_l + urow) : 0.f;
                }
                ptx::mbar_wait(acc_full, lt & 1, a.status);
                __syncwarp();       // reconverge for tcgen05.ld
                ptx::tc_fence_after();
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
                        for (int c4 = 0; c4 < 4; ++c4)
                            dst[c4] = make_float4(dh[4 * c4], dh[4 * c4 + 1], dh[4 * c4 + 2], dh[4 * c4 + 3]);
                    }
                }
                ptx::tc_fence_before();
                sk[lane] = row_ok ? (1.f - a.alpha) * inv : -1.f;
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(acc_empty);
                const size_t ubase = (size_t)te.u * a.n;
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
                        // V from global memory (L2): its latency is off the MMAs' path
                        if (keep[q] >= 0.f) vv[q] = __ldg(reinterpret_cast<const uint2*>(a.V + rr[q] * kHeadDim) + f4);
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (keep[q] < 0.f) continue;
                        const int r = 2 * (it0 + q) + hr;
                        const float4 dv = *reinterpret_cast<const float4*>(st + r * kEpiRowFloats + 4 * f4);
                        const float z[4] = {fmaf(keep[q], dv.x, a.alpha * band::bf16lo(vv[q].x)),
                                            fmaf(keep[q], dv.y, a.alpha * band::bf16hi(vv[q].x)),
                                            fmaf(keep[q], dv.z, a.alpha * band::bf16lo(vv[q].y)),
                                            fmaf(keep[q], dv.w, a.alpha * band::bf16hi(vv[q].y))};
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
                        }
                    }
                }
                __syncwarp();       // the staging rows are rewritten by the next tile
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kSMmaWarp) ptx::tmem_dealloc(tmem, kTmemCols);
}

// bf16 tensor map over [units][n][row_elems] with a box of 64 elements x box_rows rows
int encode_map(CUtensorMap* m, const void* base, int64_t n, int64_t units, int row_elems, int box_rows) {
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

int num_sms() {
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
            sms = 1;
    }
    return sms;
}

// CTAs of a launch over `total` items: one per SM, more when the snake dealing
// would give a CTA more items than its table holds
int64_t block_ctas(int64_t total) {
    int64_t ctas = total < num_sms() ? total : num_sms();
    if ((total + ctas - 1) / ctas > kMaxCtaTiles) ctas = (total + kMaxCtaTiles - 1) / kMaxCtaTiles;
    return ctas;
}

template <int kMode>
int launch_block(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmZ,
                 const BlockArgs& a, cudaStream_t stream) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(block_kernel<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        block_smem_bytes());
    });
    if (attr_err != cudaSuccess) return cuda_fail(attr_err, "cudaFuncSetAttribute(block kernel)");
    const int64_t ctas = block_ctas(a.units * a.tiles);
    {
        LaunchScope scope(kMode == kScore ? DIFFUSER_KERNEL_SCORE : DIFFUSER_KERNEL_HOP, stream);
        const cudaError_t e = launch_pdl(block_kernel<kMode>, dim3((unsigned)ctas), dim3(kThreads),
                                         (size_t)block_smem_bytes(), stream, tmQ, tmK, tmZ, a);
        if (e != cudaSuccess) return cuda_fail(e, "block_kernel");
    }
    const cudaError_t err = cudaGetLastError();
    return err == cudaSuccess ? DIFFUSER_OK : cuda_fail(err, "block_kernel");
}

}  // namespace

bool block_eligible(const diffuser_graph* g) {
    return g->kind == kBlockGraph && g->block == kBlock && g->d_blk_chunks != nullptr;
}

// The deal tables of a graph, one per (units, CTAs); never evicted, as a captured
// replay of a forward holds the pointers it was launched with.
struct BlockDeals {
    struct Entry {
        int64_t units;
        int64_t ctas;
        int32_t* d_ptr;
        int32_t* d_items;
    };
    std::mutex mu;
    std::vector<Entry> entries;
};

void destroy_block_deals(BlockDeals* d) {
    if (!d) return;
    for (auto& e : d->entries) {
        cudaFree(e.d_ptr);
        cudaFree(e.d_items);
    }
    delete d;
}

// The tiles' key-block lists from the host CSR: block row J's allowed blocks are
// the distinct blocks of its first token's row (all its tokens share them).
int build_block_tiles(diffuser_graph* g) {
    if (g->kind != kBlockGraph || g->block != kBlock) return DIFFUSER_OK;
    const int64_t nb = (g->n + kBlock - 1) / kBlock;
    if (nb > (int64_t(1) << 24)) return DIFFUSER_OK;            // beyond the chunk records' range
    const int64_t tiles = (g->n + kTile - 1) / kTile;
    std::vector<std::vector<int32_t>> allowed(nb);
    for (int64_t J = 0; J < nb; ++J) {
        const int64_t i = J * kBlock;
        for (int64_t e = g->h_row_ptr[i]; e < g->h_row_ptr[i + 1]; ++e) {
            const int32_t kb = g->h_col[e] / kBlock;
            if (allowed[J].empty() || allowed[J].back() != kb) allowed[J].push_back(kb);
        }
    }
    std::vector<int32_t> chunks, tile_ptr(tiles + 1, 0);
    std::vector<uint8_t> bits(nb);
    for (int64_t t = 0; t < tiles; ++t) {
        std::fill(bits.begin(), bits.end(), 0);
        for (int rh = 0; rh < 2; ++rh) {
            const int64_t J = 2 * t + rh;
            if (J < nb)
                for (int32_t kb : allowed[J]) bits[kb] |= (uint8_t)(1 << rh);
        }
        std::vector<int32_t> list;
        for (int64_t kb = 0; kb < nb; ++kb)
            if (bits[kb]) list.push_back((int32_t)kb);
        for (size_t q = 0; q < list.size(); q += 2) {
            const int32_t kb0 = list[q];
            const bool pair = q + 1 < list.size();
            const int32_t kb1 = pair ? list[q + 1] : kb0;      // odd count: repeat, masked off
            const int32_t m = bits[kb0] | (pair ? bits[kb1] << 2 : 0);
            chunks.insert(chunks.end(), {kb0, kb1, m, 0});
        }
        tile_ptr[t + 1] = (int32_t)(chunks.size() / 4);
    }
    std::vector<int32_t> order(tiles);
    for (int64_t t = 0; t < tiles; ++t) order[t] = (int32_t)t;
    std::stable_sort(order.begin(), order.end(), [&](int32_t x, int32_t y) {
        return tile_ptr[x + 1] - tile_ptr[x] > tile_ptr[y + 1] - tile_ptr[y];
    });
    int32_t *d_chunks = nullptr, *d_ptr = nullptr, *d_order = nullptr;
    cudaError_t err = cudaMalloc(&d_chunks, sizeof(int32_t) * chunks.size());
    if (err == cudaSuccess) err = cudaMalloc(&d_ptr, sizeof(int32_t) * tile_ptr.size());
    if (err == cudaSuccess) err = cudaMalloc(&d_order, sizeof(int32_t) * order.size());
    if (err == cudaSuccess)
        err = cudaMemcpy(d_chunks, chunks.data(), sizeof(int32_t) * chunks.size(), cudaMemcpyHostToDevice);
    if (err == cudaSuccess)
        err = cudaMemcpy(d_ptr, tile_ptr.data(), sizeof(int32_t) * tile_ptr.size(), cudaMemcpyHostToDevice);
    if (err == cudaSuccess)
        err = cudaMemcpy(d_order, order.data(), sizeof(int32_t) * order.size(), cudaMemcpyHostToDevice);
    if (err != cudaSuccess) {
        cudaFree(d_chunks);
        cudaFree(d_ptr);
        cudaFree(d_order);
        return cuda_fail(err, "uploading the block tiles' key lists");
    }
    g->d_blk_tile_ptr = d_ptr;
    g->d_blk_order = d_order;
    g->h_blk_tile_ptr = tile_ptr;
    g->h_blk_order = order;
    if (!g->blk_deals) g->blk_deals = new BlockDeals();
    g->blk_tiles = (int32_t)tiles;
    g->blk_chunks = (int64_t)(chunks.size() / 4);
    g->d_blk_chunks = d_chunks;            // set last: non-null means the lists are complete
    return DIFFUSER_OK;
}

namespace {

constexpr size_t kMaxDeals = 4;

// The launch's items dealt heaviest first, each to the CTA with the fewest chunks so
// far (ties: the lowest index): a position with many more key blocks than the rest
// (the global block rows read all of them) then shares its CTA with fewer light
// tiles, where the snake order gives every CTA the same number of items.  Built on
// the first launch for (units, CTAs), outside stream capture; while the caller's
// stream is capturing, after kMaxDeals tables, or when a CTA's list would not fit
// its table, the kernel deals in snake order instead.
void block_deal(const diffuser_graph* g, int64_t units, int64_t ctas, cudaStream_t stream, BlockArgs& a) {
    a.deal_ptr = nullptr;
    a.deal_items = nullptr;
    BlockDeals* D = g->blk_deals;
    if (!D) return;
    std::lock_guard<std::mutex> lk(D->mu);
    for (const auto& e : D->entries)
        if (e.units == units && e.ctas == ctas) {
            a.deal_ptr = e.d_ptr;
            a.deal_items = e.d_items;
            return;
        }
    if (D->entries.size() >= kMaxDeals) return;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) return;
    const int64_t total = units * (int64_t)g->blk_tiles;
    if (total > INT32_MAX || (int64_t)g->h_blk_order.size() != g->blk_tiles) return;
    using Load = std::pair<int64_t, int64_t>;        // (chunks so far, CTA)
    std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
    for (int64_t b = 0; b < ctas; ++b) heap.push({0, b});
    std::vector<std::vector<int32_t>> lists((size_t)ctas);
    for (int64_t k = 0; k < total; ++k) {            // chunk counts fall with k
        const int32_t t = g->h_blk_order[(size_t)(k / units)];
        const int64_t size = g->h_blk_tile_ptr[(size_t)t + 1] - g->h_blk_tile_ptr[(size_t)t];
        const Load top = heap.top();
        heap.pop();
        lists[(size_t)top.second].push_back((int32_t)k);
        heap.push({top.first + size, top.second});
    }
    std::vector<int32_t> ptr((size_t)ctas + 1, 0), items;
    items.reserve((size_t)total);
    for (int64_t b = 0; b < ctas; ++b) {
        if (lists[(size_t)b].size() > (size_t)kMaxCtaTiles) return;
        items.insert(items.end(), lists[(size_t)b].begin(), lists[(size_t)b].end());
        ptr[(size_t)b + 1] = (int32_t)items.size();
    }
    int32_t *dp = nullptr, *di = nullptr;
    cudaError_t err = cudaMalloc(&dp, sizeof(int32_t) * ptr.size());
    if (err == cudaSuccess) err = cudaMalloc(&di, sizeof(int32_t) * items.size());
    if (err == cudaSuccess) err = cudaMemcpy(dp, ptr.data(), sizeof(int32_t) * ptr.size(), cudaMemcpyHostToDevice);
    if (err == cudaSuccess)
        err = cudaMemcpy(di, items.data(), sizeof(int32_t) * items.size(), cudaMemcpyHostToDevice);
    if (err != cudaSuccess) {
        cudaFree(dp);
        cudaFree(di);
        cudaGetLastError();                           // the snake order serves instead
        return;
    }
    D->entries.push_back({units, ctas, dp, di});
    a.deal_ptr = dp;
    a.deal_items = di;
}

}  // namespace

int plan_block_layout(const diffuser_graph* g, int64_t units, BlockLayout* L) {
    auto al = [](size_t x) { return (x + 1023) / 1024 * 1024; };
    const size_t U = (size_t)units;
    size_t off = 0;
    for (int s = 0; s < 2; ++s) { L->z[s] = off; off += al(U * (size_t)g->n * 2 * kHeadDim * 2); }
    L->mb2 = off; off += al(U * (size_t)g->n * 4);
    L->inv_l = off; off += al(U * (size_t)g->n * 4);
    L->total = off;
    return DIFFUSER_OK;
}

namespace {

BlockArgs block_args(const diffuser_graph* g, int64_t units, char* ws, const BlockLayout& L) {
    BlockArgs a;
    a.n = g->n;
    a.units = units;
    a.tiles = g->blk_tiles;
    a.chunks = g->d_blk_chunks;
    a.tile_ptr = g->d_blk_tile_ptr;
    a.order = g->d_blk_order;
    a.deal_ptr = nullptr;
    a.deal_items = nullptr;
    a.mb2 = reinterpret_cast<float*>(ws + L.mb2);
    a.inv_l = reinterpret_cast<float*>(ws + L.inv_l);
    a.V = nullptr;
    a.out = nullptr;
    a.alpha = 0.f;
    a.status = g->d_status;
    a.Z_out = nullptr;
    return a;
}

}  // namespace

int launch_block_scores(const diffuser_graph* g, int64_t units, const void* Q, const void* K, char* ws,
                        const BlockLayout& L, cudaStream_t stream) {
    CUtensorMap tmQ, tmK;
    int st = encode_map(&tmQ, Q, g->n, units, kHeadDim, kTile);
    if (!st) st = encode_map(&tmK, K, g->n, units, kHeadDim, kBlock);
    if (st) return st;
    BlockArgs a = block_args(g, units, ws, L);
    block_deal(g, units, block_ctas(units * g->blk_tiles), stream, a);
    return launch_block<kScore>(tmQ, tmK, tmK, a, stream);     // the score pass loads no Z
}

int launch_block_hops(const diffuser_graph* g, int64_t units, const void* Q, const void* K,
                      const void* V, int32_t hops, float alpha, void* out, char* ws,
                      const BlockLayout& L, cudaStream_t stream) {
    CUtensorMap tmQ, tmK, tmV, tmZ[2];
    int st = encode_map(&tmQ, Q, g->n, units, kHeadDim, kTile);
    if (!st) st = encode_map(&tmK, K, g->n, units, kHeadDim, kBlock);
    if (!st) st = encode_map(&tmV, V, g->n, units, kHeadDim, kBlock);
    for (int s = 0; s < 2 && !st; ++s) st = encode_map(&tmZ[s], ws + L.z[s], g->n, units, 2 * kHeadDim, kBlock);
    if (st) return st;
    BlockArgs a = block_args(g, units, ws, L);
    block_deal(g, units, block_ctas(units * g->blk_tiles), stream, a);
    a.V = static_cast<const __nv_bfloat16*>(V);
    a.out = static_cast<__nv_bfloat16*>(out);
    a.alpha = alpha;
    // Z_{k+1} of hop k lives in z[k & 1]; hop k reads Z_k (V for k = 0)
    for (int32_t k = 0; k < hops; ++k) {
        const bool first = k == 0, last = k == hops - 1;
        a.Z_out = reinterpret_cast<__nv_bfloat16*>(ws + L.z[k & 1]);
        const CUtensorMap& tm = first ? tmV : tmZ[(k - 1) & 1];
        if (first && last) st = launch_block<kHopOnly>(tmQ, tmK, tm, a, stream);
        else if (first) st = launch_block<kHopFirst>(tmQ, tmK, tm, a, stream);
        else if (last) st = launch_block<kHopLast>(tmQ, tmK, tm, a, stream);
        else st = launch_block<kHopMid>(tmQ, tmK, tm, a, stream);
        if (st) return st;
    }
    return DIFFUSER_OK;
}

int launch_block_forward(const diffuser_graph* g, int64_t units, const void* Q, const void* K,
                         const void* V, int32_t hops, float alpha, void* out, char* ws,
                         const BlockLayout& L, cudaStream_t stream) {
    int st = launch_block_scores(g, units, Q, K, ws, L, stream);
    return st ? st : launch_block_hops(g, units, Q, K, V, hops, alpha, out, ws, L, stream);
}

}  // namespace dfs
