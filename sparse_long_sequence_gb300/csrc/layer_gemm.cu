// The projections around the diffusion module ("Diffuser: modelling long
// sequences with multi-hop attention diffusion", sec 2.1: per head Q = X W_Q,
// K = X W_K, V = X W_V; sec 2.4 and Fig S.3: the heads' outputs Z_K are
// concatenated and projected by W_O), as dense GEMMs on the tcgen05 tensor
// cores: bf16 operands, fp32 accumulation in tensor memory, bf16 results.
//
// One kernel, C[128 x 256 tile] = A . B^T with both operands K-major (the
// nn.Linear weight layout [out][in]):
//  * the Q/K/V projection: A = X [B][n][D] (a 3-d map, K = D), B = W_qkv
//    [3 H d][D]; the epilogue scatters column j = s H d + h d + f of token
//    (b, i) into tensor s (Q, K, V) at [b][h][i][f];
//  * the output projection: A = the heads' outputs Z [B][H][n][d] through a
//    4-d map whose K blocks are the heads (the concatenation costs nothing),
//    B = W_O [D][H d]; the epilogue writes Y [B][n][D].
// A 128-token tile lies inside one batch item.  Ragged edges (n, N, K) load
// as zeros through the tensor maps and are not stored.
//
// Roles (6 warps, one persistent CTA per SM taking tiles blockIdx.x,
// blockIdx.x + gridDim.x, ...): warp 0 loads the A and B stages (TMA, a
// 4-stage ring that runs on across tiles), warp 1 allocates tensor memory and
// issues the MMAs (M = 128, N = 256, K = 16 per instruction) into one of two
// 256-column accumulators, warps 2-5 read the other accumulator (lane quadrant
// w % 4) and store bf16, so a tile's epilogue overlaps the next tile's MMAs.
// Every barrier wait is bounded and records a status instead of hanging.
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

constexpr int kTM = 128, kTN = 256, kTK = 64;      // tile and K step (64 bf16 = one 128-byte row)
constexpr int kStages = 4;
constexpr int kABytes = kTM * kTK * 2;             // 16 KB
constexpr int kBBytes = kTN * kTK * 2;             // 32 KB
constexpr int kGemmThreads = 192;
constexpr int kEpiWarp0 = 2;                       // warps 0 TMA, 1 MMA, 2..5 epilogue
static_assert(kGemmThreads == 32 * (kEpiWarp0 + 4), "four epilogue warps, one per lane quadrant");
constexpr int kGemmSmem = 1024 + kStages * (kABytes + kBBytes) + 256;   // + barriers
static_assert(kGemmSmem <= 227 * 1024, "shared memory per CTA");

enum ProjMode { kQkv = 0, kOut = 1 };

struct GemmArgs {
    int64_t n;             // tokens per batch item
    int32_t B, H, D;       // batch, heads, model width
    int32_t N;             // output columns: 3 H d (projection) or D (output)
    int32_t k_blocks;      // K steps of 64
    int32_t m_tiles;       // 128-token tiles per batch item
    int32_t n_tiles;       // 256-column tiles
    __nv_bfloat16* q;      // projection outputs [B][H][n][64]
    __nv_bfloat16* k;
    __nv_bfloat16* v;
    __nv_bfloat16* y;      // output projection [B][n][D]
    int* status;
};

struct GemmTile { int b, i0, n0; };

// tile t: tokens i0 .. i0 + 127 of batch item b, columns n0 .. n0 + 255; consecutive
// tiles share a column block (the weights' tile stays in L2)
__device__ __forceinline__ GemmTile gemm_tile(const GemmArgs& a, int64_t t) {
    GemmTile g;
    g.i0 = (int)(t % a.m_tiles) * kTM;
    g.b = (int)((t / a.m_tiles) % a.B);
    g.n0 = (int)(t / ((int64_t)a.m_tiles * a.B)) * kTN;
    return g;
}

template <int kMode>
__global__ void __launch_bounds__(kGemmThreads, 1)
proj_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, GemmArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = sA + kStages * kABytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + kStages * kBBytes);   // [kStages]
    uint64_t* empty = full + kStages;                                        // [kStages]
    uint64_t* acc_full = empty + kStages;                                    // [2]
    uint64_t* acc_empty = acc_full + 2;                                      // [2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t total_tiles = (int64_t)a.m_tiles * a.B * a.n_tiles;
    const int my_tiles = blockIdx.x < total_tiles
        ? (int)((total_tiles - 1 - blockIdx.x) / gridDim.x + 1) : 0;
    auto tile = [&](int lt) { return gemm_tile(a, blockIdx.x + (int64_t)lt * gridDim.x); };

    if (warp == 1) ptx::tmem_alloc(tmem_slot, 2 * kTN);
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) { ptx::mbar_init(&full[s], 1); ptx::mbar_init(&empty[s], 1); }
        for (int s = 0; s < 2; ++s) { ptx::mbar_init(&acc_full[s], 1); ptx::mbar_init(&acc_empty[s], 4); }
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmB);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // (the whole warp runs the loop; the elected lane issues the copies)
        const uint64_t pol_a = ptx::l2_evict_first(), pol_b = ptx::l2_evict_last();
        int g = 0;                                           // running K step over this CTA's tiles
        for (int lt = 0; lt < my_tiles; ++lt) {
            const GemmTile tl = tile(lt);
            for (int kb = 0; kb < a.k_blocks; ++kb, ++g) {
                const int s = g % kStages;
                if (g >= kStages) ptx::mbar_wait(&empty[s], ((g / kStages) - 1) & 1, a.status);
                __syncwarp();
                if (ptx::elect_one()) {
                    ptx::mbar_arrive_expect_tx(&full[s], kABytes + kBBytes);
                    if constexpr (kMode == kQkv)
                        ptx::tma_load_3d_hint(sA + s * kABytes, &tmA, &full[s], kb * kTK, tl.i0, tl.b, pol_a);
                    else
                        ptx::tma_load_4d_hint(sA + s * kABytes, &tmA, &full[s], 0, tl.i0, kb, tl.b, pol_a);
                    ptx::tma_load_2d_hint(sB + s * kBBytes, &tmB, &full[s], kb * kTK, tl.n0, pol_b);
                }
            }
        }
    } else if (warp == 1) {
        // (the whole warp runs the loop; the elected lane issues each instruction)
        {
            constexpr uint32_t idesc = ptx::mma_idesc(1, kTN);
            const uint64_t adesc0 = ptx::sw128_kmajor_desc(ptx::smem_u32(sA));
            const uint64_t bdesc0 = ptx::sw128_kmajor_desc(ptx::smem_u32(sB));
            int g = 0;
            for (int lt = 0; lt < my_tiles; ++lt) {
                const int buf = lt & 1;
                // the epilogue has read this accumulator's previous tile
                if (lt >= 2) ptx::mbar_wait(&acc_empty[buf], ((lt / 2) - 1) & 1, a.status);
                __syncwarp();
                ptx::tc_fence_after();
                const uint32_t dacc = tmem + buf * kTN;
                for (int kb = 0; kb < a.k_blocks; ++kb, ++g) {
                    const int s = g % kStages;
                    ptx::mbar_wait(&full[s], (g / kStages) & 1, a.status);
                    __syncwarp();
                    ptx::tc_fence_after();
                    const uint64_t ad = adesc0 + (uint64_t)(s * (kABytes >> 4));
                    const uint64_t bd = bdesc0 + (uint64_t)(s * (kBBytes >> 4));
#pragma unroll
                    for (int ks = 0; ks < kTK / 16; ++ks)
                        if (ptx::elect_one()) ptx::mma_bf16_ss(dacc, ad + 2 * ks, bd + 2 * ks, idesc, kb > 0 || ks > 0);
                    if (ptx::elect_one()) ptx::mma_commit(&empty[s]);
                }
                if (ptx::elect_one()) ptx::mma_commit(&acc_full[buf]);
            }
            // drain: the last commits land before the CTA exits
            for (int s = 0; s < kStages; ++s) {
                const int uses = (g - s + kStages - 1) / kStages;
                if (uses > 0) ptx::mbar_wait(&empty[s], (uses - 1) & 1, a.status);
            }
        }
    } else {
        // epilogue: thread <-> tile row t (lane quadrant warp % 4), 32 columns per load
        const int quad = warp & 3;
        const int t = quad * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        for (int lt = 0; lt < my_tiles; ++lt) {
            const GemmTile tl = tile(lt);
            const int b = tl.b, n0 = tl.n0, buf = lt & 1;
            const int64_t i = tl.i0 + t;
            ptx::mbar_wait(&acc_full[buf], (lt / 2) & 1, a.status);
            __syncwarp();
            ptx::tc_fence_after();
            uint4 w[4];
#pragma unroll 1
            for (int c0 = 0; c0 < kTN; c0 += 32) {
                uint32_t r[32];
                ptx::tmem_ld32_issue(tmem + lane_base + buf * kTN + c0, r);
                ptx::tmem_ld_wait32(r);
                if (c0 + 32 == kTN) {
                    // the accumulator is read: the MMAs of the tile after next may overwrite it
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(&acc_empty[buf]);
                }
                const int j0 = n0 + c0;                  // a multiple of 32: one head's half row
                if (i >= a.n || j0 >= a.N) continue;
                uint32_t* wp = reinterpret_cast<uint32_t*>(w);
#pragma unroll
                for (int p = 0; p < 16; ++p) {
                    const __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(r[2 * p]), __uint_as_float(r[2 * p + 1]));
                    wp[p] = *reinterpret_cast<const uint32_t*>(&h);
                }
                uint4* dst;
                if constexpr (kMode == kQkv) {
                    const int hd = a.H * kHeadDim;
                    const int s = j0 / hd, rem = j0 - s * hd, h = rem / kHeadDim, f0 = rem - h * kHeadDim;
                    __nv_bfloat16* base = s == 0 ? a.q : (s == 1 ? a.k : a.v);
                    dst = reinterpret_cast<uint4*>(base + (((size_t)b * a.H + h) * a.n + i) * kHeadDim + f0);
                } else {
                    dst = reinterpret_cast<uint4*>(a.y + ((size_t)b * a.n + i) * a.D + j0);
                }
                if (kMode == kOut && j0 + 32 > a.N) {
                    // a ragged last column block: element by element
                    const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(w);
                    __nv_bfloat16* d = reinterpret_cast<__nv_bfloat16*>(dst);
                    for (int q = 0; q < a.N - j0; ++q) d[q] = e[q];
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q) dst[q] = w[q];
                }
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) ptx::tmem_dealloc(tmem, 2 * kTN);
}

int encode(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
           const cuuint32_t* box) {
    auto fn = band::tensor_map_encoder();
    if (!fn) return fail(DIFFUSER_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    const cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box,
                    es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(DIFFUSER_ERR_CUDA, "cuTensorMapEncodeTiled failed: " + std::to_string((int)r));
    return DIFFUSER_OK;
}

template <int kMode>
int launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a, cudaStream_t stream) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(proj_gemm_kernel<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        kGemmSmem);
    });
    if (attr_err != cudaSuccess) return cuda_fail(attr_err, "cudaFuncSetAttribute(projection GEMM)");
    const int64_t tiles = (int64_t)a.m_tiles * a.B * a.n_tiles;
    if (tiles > INT32_MAX) return fail(DIFFUSER_ERR_OVERFLOW, "projection GEMM too large");
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) sms = 1;
    const int64_t grid = tiles < sms ? tiles : sms;      // one persistent CTA per SM
    {
        LaunchScope scope(DIFFUSER_KERNEL_AUX, stream);
        proj_gemm_kernel<kMode><<<(unsigned)grid, kGemmThreads, kGemmSmem, stream>>>(tmA, tmB, a);
    }
    const cudaError_t err = cudaGetLastError();
    return err == cudaSuccess ? DIFFUSER_OK : cuda_fail(err, "proj_gemm_kernel");
}

}  // namespace

int check_layer_shape(int64_t B, int64_t n, int32_t D, int32_t H, int32_t d) {
    if (B < 1 || n < 1 || H < 1 || D < 1 || B > INT32_MAX || n > INT32_MAX || H > 4096)
        return fail(DIFFUSER_ERR_INVALID_ARG, "B, n, H, D out of range");
    if (d != kHeadDim) return fail(DIFFUSER_ERR_UNSUPPORTED, "head width d must be 64");
    if (D % 8 != 0 || D > (1 << 16))
        return fail(DIFFUSER_ERR_UNSUPPORTED, "the model width D must be a multiple of 8, at most 65536");
    return DIFFUSER_OK;
}

int launch_qkv_projection(const void* X, const void* Wqkv, int64_t B, int64_t n, int32_t D, int32_t H,
                          void* Q, void* K, void* V, int* status, cudaStream_t stream) {
    CUtensorMap tmA, tmB;
    const cuuint64_t adims[3] = {(cuuint64_t)D, (cuuint64_t)n, (cuuint64_t)B};
    const cuuint64_t astr[2] = {(cuuint64_t)D * 2, (cuuint64_t)n * D * 2};
    const cuuint32_t abox[3] = {kTK, kTM, 1};
    const int32_t N = 3 * H * kHeadDim;
    const cuuint64_t bdims[2] = {(cuuint64_t)D, (cuuint64_t)N};
    const cuuint64_t bstr[1] = {(cuuint64_t)D * 2};
    const cuuint32_t bbox[2] = {kTK, kTN};
    int st = encode(&tmA, X, 3, adims, astr, abox);
    if (!st) st = encode(&tmB, Wqkv, 2, bdims, bstr, bbox);
    if (st) return st;
    GemmArgs a{};
    a.n = n;
    a.B = (int32_t)B;
    a.H = H;
    a.D = D;
    a.N = N;
    a.k_blocks = (D + kTK - 1) / kTK;
    a.m_tiles = (int32_t)((n + kTM - 1) / kTM);
    a.n_tiles = (N + kTN - 1) / kTN;
    a.q = static_cast<__nv_bfloat16*>(Q);
    a.k = static_cast<__nv_bfloat16*>(K);
    a.v = static_cast<__nv_bfloat16*>(V);
    a.status = status;
    return launch_gemm<kQkv>(tmA, tmB, a, stream);
}

int launch_output_projection(const void* Z, const void* Wo, int64_t B, int64_t n, int32_t D, int32_t H,
                             void* Y, int* status, cudaStream_t stream) {
    CUtensorMap tmA, tmB;
    const cuuint64_t adims[4] = {(cuuint64_t)kHeadDim, (cuuint64_t)n, (cuuint64_t)H, (cuuint64_t)B};
    const cuuint64_t astr[3] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)n * kHeadDim * 2,
                                (cuuint64_t)H * n * kHeadDim * 2};
    const cuuint32_t abox[4] = {kTK, kTM, 1, 1};
    const int32_t Kd = H * kHeadDim;
    const cuuint64_t bdims[2] = {(cuuint64_t)Kd, (cuuint64_t)D};
    const cuuint64_t bstr[1] = {(cuuint64_t)Kd * 2};
    const cuuint32_t bbox[2] = {kTK, kTN};
    int st = encode(&tmA, Z, 4, adims, astr, abox);
    if (!st) st = encode(&tmB, Wo, 2, bdims, bstr, bbox);
    if (st) return st;
    GemmArgs a{};
    a.n = n;
    a.B = (int32_t)B;
    a.H = H;
    a.D = D;
    a.N = D;
    a.k_blocks = H;                          // one K step per head
    a.m_tiles = (int32_t)((n + kTM - 1) / kTM);
    a.n_tiles = (D + kTN - 1) / kTN;
    a.y = static_cast<__nv_bfloat16*>(Y);
    a.status = status;
    return launch_gemm<kOut>(tmA, tmB, a, stream);
}

}  // namespace dfs
