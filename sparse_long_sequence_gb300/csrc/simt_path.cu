// CSR SIMT path: general over any graph, fp32 arithmetic throughout.  It is
// the path for fp32 I/O (whose error budget rules out tf32 tensor cores) and
// for graphs without a fast layout, and the reference implementation the
// tensor-core kernels are checked against on the device.
//
//  * score_csr_kernel: one warp per (unit, row), 32 edges per round.  Lane l
//    holds features 2l, 2l+1 of q_i; for each edge of the round the warp reads
//    the key row k_j whole (each lane its two features, one coalesced line per
//    row), every lane forms its two-feature part of each of the 32 dot
//    products, and a butterfly over the lanes leaves edge t's score with lane t.
//    Each lane keeps an online (max, sum) pair over its edges; the pairs are
//    merged across the warp, then each lane normalises the weights it wrote.
//    ("Diffuser: modelling long sequences with multi-hop attention
//    diffusion", eq S.1-S.5; "1.2.1 Static sparsity", eq 1-3.)
//  * hop_csr_kernel: one warp per (unit, row).  Lanes own two of the 64
//    features; for each edge the warp reads one 256-byte (fp32) or 128-byte
//    (bf16) row of Z_k, coalesced, and accumulates A_ij * Z_k[j]; the
//    restart term is fused:  dst_i = (1 - alpha) acc + alpha V_i
//    (same Diffuser notes, sec 2.4 eq S.7).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "internal.h"

namespace dfs {
namespace {

constexpr int kWarpsPerBlock = 8;

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <typename T> struct Pair;
template <> struct Pair<float> {
    static __device__ __forceinline__ float2 load(const float* p) {
        return *reinterpret_cast<const float2*>(p);
    }
};
template <> struct Pair<__nv_bfloat16> {
    static __device__ __forceinline__ float2 load(const __nv_bfloat16* p) {
        uint32_t w = *reinterpret_cast<const uint32_t*>(p);
        return make_float2(bf16lo(w), bf16hi(w));
    }
};


template <bool kBf16>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
score_csr_kernel(CsrArgs a, const void* __restrict__ Q, const void* __restrict__ K,
                 float* __restrict__ A) {
    using T = typename std::conditional<kBf16, __nv_bfloat16, float>::type;
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    if (gw >= a.units * a.n) return;
    const int64_t u = gw / a.n, i = gw - u * a.n;
    const size_t unit = (size_t)u * a.n * kHeadDim;
    const T* Ku = static_cast<const T*>(K) + unit + 2 * lane;
    float* Au = A + (size_t)u * a.nnz;
    const float2 q = Pair<T>::load(static_cast<const T*>(Q) + unit + (size_t)i * kHeadDim + 2 * lane);
    const float scale = 0.125f;  // 1/sqrt(64), exact
    const int64_t e0 = a.row_ptr[i], e1 = a.row_ptr[i + 1];

    float m = -INFINITY, l = 0.f;
    for (int64_t base = e0; base < e1; base += 32) {
        const int64_t e = base + lane;
        const int32_t j_l = e < e1 ? a.col[e] : 0;
        const int cnt = (e1 - base) < 32 ? (int)(e1 - base) : 32;
        float p[32];        // all 32 key rows requested before the first is used
#pragma unroll
        for (int t = 0; t < 32; ++t) {
            const int32_t j = __shfl_sync(0xffffffffu, j_l, t);
            const float2 kv = t < cnt ? Pair<T>::load(Ku + (size_t)j * kHeadDim) : make_float2(0.f, 0.f);
            p[t] = fmaf(q.x, kv.x, q.y * kv.y);
        }
        const float s = warp_transpose_sum32(p, lane) * scale;     // edge base + lane
        if (e < e1) {
            Au[e] = s;
            if (s > m) { l = l * expf(m - s) + 1.f; m = s; }
            else       { l += expf(s - m); }
        }
    }
    // merge the per-lane (max, sum) pairs
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        float m2 = __shfl_xor_sync(0xffffffffu, m, off);
        float l2 = __shfl_xor_sync(0xffffffffu, l, off);
        float mm = fmaxf(m, m2);
        float a1 = (m == -INFINITY) ? 0.f : l * expf(m - mm);
        float a2 = (m2 == -INFINITY) ? 0.f : l2 * expf(m2 - mm);
        m = mm;
        l = a1 + a2;
    }
    for (int64_t e = e0 + lane; e < e1; e += 32) Au[e] = expf(Au[e] - m) / l;
}

__device__ __forceinline__ void store_pair(float* p, float2 v) {
    *reinterpret_cast<float2*>(p) = v;
}
__device__ __forceinline__ void store_pair(__nv_bfloat16* p, float2 v) {
    *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(v.x, v.y);
}

template <typename TSrc, typename TV, typename TDst>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
hop_csr_kernel(CsrArgs a, const float* __restrict__ A, const TSrc* __restrict__ src,
               const TV* __restrict__ V, TDst* __restrict__ dst, float alpha) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    if (gw >= a.units * a.n) return;
    const int64_t u = gw / a.n, i = gw - u * a.n;
    const size_t unit = (size_t)u * a.n * kHeadDim;
    const TSrc* Z = src + unit + 2 * lane;
    const float* Au = A + (size_t)u * a.nnz;
    const int64_t e0 = a.row_ptr[i], e1 = a.row_ptr[i + 1];

    // 32 edges per round: all 32 rows of Z_k are requested before the first is
    // used (a long row, such as a global row, is latency-bound otherwise); the
    // sum still runs in edge order
    float2 acc = make_float2(0.f, 0.f);
    for (int64_t base = e0; base < e1; base += 32) {
        const int64_t e = base + lane;
        const float a_l = e < e1 ? Au[e] : 0.f;
        const int32_t j_l = e < e1 ? a.col[e] : 0;
        const int cnt = (e1 - base) < 32 ? (int)(e1 - base) : 32;
        float2 z[32];
#pragma unroll
        for (int t = 0; t < 32; ++t) {
            const int32_t j = __shfl_sync(0xffffffffu, j_l, t);
            z[t] = t < cnt ? Pair<TSrc>::load(Z + (size_t)j * kHeadDim) : make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int t = 0; t < 32; ++t) {
            const float w = __shfl_sync(0xffffffffu, a_l, t);
            acc.x = fmaf(w, z[t].x, acc.x);
            acc.y = fmaf(w, z[t].y, acc.y);
        }
    }
    const float2 v = Pair<TV>::load(V + unit + (size_t)i * kHeadDim + 2 * lane);
    const float keep = 1.f - alpha;
    float2 r = make_float2(fmaf(keep, acc.x, alpha * v.x), fmaf(keep, acc.y, alpha * v.y));
    store_pair(dst + unit + (size_t)i * kHeadDim + 2 * lane, r);
}

unsigned grid_for(const CsrArgs& a) {
    return (unsigned)((a.units * a.n + kWarpsPerBlock - 1) / kWarpsPerBlock);
}

template <typename TIo>
int hop_dispatch(const CsrArgs& a, const float* A, const void* src, bool src_is_io,
                 const void* V, void* dst, bool dst_is_io, float alpha, cudaStream_t stream) {
    const TIo* v = static_cast<const TIo*>(V);
    dim3 grid(grid_for(a)), block(kWarpsPerBlock * 32);
    LaunchScope scope(DIFFUSER_KERNEL_HOP, stream);
    if (src_is_io && dst_is_io)
        hop_csr_kernel<TIo, TIo, TIo><<<grid, block, 0, stream>>>(
            a, A, static_cast<const TIo*>(src), v, static_cast<TIo*>(dst), alpha);
    else if (src_is_io)
        hop_csr_kernel<TIo, TIo, float><<<grid, block, 0, stream>>>(
            a, A, static_cast<const TIo*>(src), v, static_cast<float*>(dst), alpha);
    else if (dst_is_io)
        hop_csr_kernel<float, TIo, TIo><<<grid, block, 0, stream>>>(
            a, A, static_cast<const float*>(src), v, static_cast<TIo*>(dst), alpha);
    else
        hop_csr_kernel<float, TIo, float><<<grid, block, 0, stream>>>(
            a, A, static_cast<const float*>(src), v, static_cast<float*>(dst), alpha);
    cudaError_t err = cudaGetLastError();
    return err == cudaSuccess ? DIFFUSER_OK : cuda_fail(err, "hop_csr_kernel");
}

}  // namespace

int launch_score_csr(const CsrArgs& a, const void* Q, const void* K, int32_t dtype, float* A,
                     cudaStream_t stream) {
    dim3 grid(grid_for(a)), block(kWarpsPerBlock * 32);
    {
        LaunchScope scope(DIFFUSER_KERNEL_SCORE, stream);
        if (dtype == DIFFUSER_DTYPE_BF16)
            score_csr_kernel<true><<<grid, block, 0, stream>>>(a, Q, K, A);
        else
            score_csr_kernel<false><<<grid, block, 0, stream>>>(a, Q, K, A);
    }
    cudaError_t err = cudaGetLastError();
    return err == cudaSuccess ? DIFFUSER_OK : cuda_fail(err, "score_csr_kernel");
}

int launch_hop_csr(const CsrArgs& a, const float* A, const void* src, bool src_is_io,
                   const void* V, void* dst, bool dst_is_io, int32_t dtype, float alpha,
                   cudaStream_t stream) {
    if (dtype == DIFFUSER_DTYPE_BF16)
        return hop_dispatch<__nv_bfloat16>(a, A, src, src_is_io, V, dst, dst_is_io, alpha, stream);
    return hop_dispatch<float>(a, A, src, src_is_io, V, dst, dst_is_io, alpha, stream);
}

}  // namespace dfs
