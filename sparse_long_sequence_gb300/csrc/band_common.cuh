// Shared pieces of the band path (token graphs, bf16 I/O): kernel argument
// blocks and small device helpers used by the score and hop kernels.
//
// Weight layout of one (batch, head) unit u ("Diffuser: modelling long
// sequences with multi-hop attention diffusion", sec 2.2 / 2.4: score once,
// aggregate K times).  The weights are stored unnormalized, e_ij =
// exp(s_ij - m_i), together with inv_l_i = 1 / sum_j e_ij, so that
// A_ij = e_ij * inv_l_i ("1.2.1 Static sparsity", eq 3):
//   band   [tiles][chunks][hi | lo][128 rows x 64 keys] bf16: tile T holds
//                      rows 128 T .. +127 against keys of the chunk grid
//                      jb + 64 c + k, jb = 128 T - r64, as the exact
//                      shared-memory image of the tensor-core A operand
//                      (K-major, 128-byte swizzle: row t at 1024 (t / 8) +
//                      128 (t % 8), 16-byte slot q at q ^ (t % 8)); e_ij =
//                      hi + lo (hi = e rounded to bf16, lo = the remainder
//                      rounded to bf16) for |i-j| <= r, 0 <= j < n, else 0
//   gcol   [n][g_pad]  slot s <-> key G[s]: raw scores (-inf inside row i's window)
//   gcimg  [tiles][hi | lo][128 rows x g16 slots] bf16: e of those scores
//                      (0 inside the window and for slots past g), as the
//                      tensor-core A operand image (K-major, no swizzle:
//                      8-row x 16-byte core matrices, the next 8 slots 128
//                      bytes on, the next 8 rows 16 g16 bytes on); g16 = g
//                      rounded up to 16
//   extra  [nx]        e of the random edges outside window and G, CSR order
//   inv_l  [n]         per-row normalizer of the rows not in G
//   grow   [g][n]      the global rows' weights A_ij (raw scores until the
//                      global-row norm kernel normalizes them with
//   gstat  [g][2]      their (row max, 1 / row sum of exp(s - max)))
//   gimg   [tiles][2][hi | lo][32 rows x 64 keys] bf16: the normalized
//                      global-row weights of tile T's own keys 128 T .. +127
//                      (two 64-key halves), as the tensor-core A operand
//                      image (rows s < g; keys past n are 0)
// The hop state Z_k is kept twice: as [n][hi 64 | lo 64] bf16 rows (Z = hi +
// lo), the B operand of the band MMA, and as [n][64] fp32 rows, the source of
// the random-edge row gathers.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>

#include "internal.h"

namespace dfs {
namespace band {

constexpr int kTileRows = 128;
constexpr int kChunkKeys = 64;
constexpr int kChunkPlaneBytes = kTileRows * kChunkKeys * 2;      // one bf16 plane of a chunk
constexpr int kChunkImageBytes = 2 * kChunkPlaneBytes;            // hi + lo
constexpr int kGImgRows = 32;                                      // the global rows' operand rows
constexpr int kGImgPlaneBytes = kGImgRows * kChunkKeys * 2;        // 4 KB
constexpr int kGImgBytes = 2 * 2 * kGImgPlaneBytes;                // 2 halves x (hi, lo): 16 KB

// the out-of-window globals' operand image of a tile: one plane holds 128 rows
// x g16 bf16 slots; byte offset of (row t, slot s) within a plane
__host__ __device__ constexpr int gc_plane_bytes(int g16) { return kTileRows * g16 * 2; }
__host__ __device__ constexpr int gc_offset(int t, int s, int g16) {
    return (t >> 3) * (16 * g16) + (t & 7) * 16 + (s >> 3) * 128 + (s & 7) * 2;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Window [lo, hi] of row i: [i - r, i + r] cut to [0, n), or [i - r, i] on the
// causal graph (the r+1 history positions; "1.2.1 Static sparsity", sec 1.1).
__device__ __forceinline__ void window_of(const BandPlan& P, int64_t i, int64_t& lo, int64_t& hi) {
    const int64_t up = P.causal ? 0 : P.r;
    lo = i - P.r < 0 ? 0 : i - P.r;
    hi = i + up > P.n - 1 ? P.n - 1 : i + up;
}

// Whether a non-global row with window [lo, hi] reads the global at j through
// the out-of-window globals' weights: j outside the window and, on the causal
// graph, not after the row (Diffuser notes sec 2.6: A lower-triangular).
__device__ __forceinline__ bool reads_global_outside(const BandPlan& P, int64_t j, int64_t lo,
                                                     int64_t hi) {
    return j < lo || (j > hi && !P.causal);
}

// Pointers into the band layout of the workspace (see plan_band_layout).
struct Weights {
    __nv_bfloat16* A_band;   // units x band_unit bytes
    float* A_gc;       // [units][n][g_pad]
    float* A_x;        // [units][nx]
    float* A_gr;       // [units][g][n] global-row weights (raw scores before normalization)
    uint8_t* A_gimg;   // [units][tiles] global-row weight images (kGImgBytes each)
    uint8_t* A_gcimg;  // [units][tiles] out-of-window global weight images (gc_image_bytes each)
    float* inv_l;      // [units][n]
    float* m_sparse;   // [units][n] max raw score over a row's gcol + extras
    float* gstat;      // [units][g][2]
};

struct GraphRefs {
    const uint8_t* is_global;
    const int32_t* gslot;
    const int32_t* globals;
    const int64_t* x_ptr;
    const int32_t* x_col;
    int64_t nx;
};

// Driver entry point of cuTensorMapEncodeTiled (null if unavailable).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

}  // namespace band

band::GraphRefs band_graph_refs(const diffuser_graph* g);
band::Weights band_weights(char* ws, const BandLayout& L);

}  // namespace dfs
