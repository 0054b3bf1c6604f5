// Backward pass on the CSR path: the gradients dQ, dK, dV of <dOut, Z_K>
// ("Diffuser: modelling long sequences with multi-hop attention diffusion",
// sec 2.6: training runs the same unrolled K-hop recursion, and the gradient
// flows back through every round of aggregation into the weights and from
// there into the scores).  fp32 arithmetic throughout; any graph, either I/O
// dtype.  With G_K = dOut, after recomputing A and Z_1 .. Z_{K-1} with the
// forward's own kernels, for k = K-1 .. 0:
//
//  * bwd_weight_grad_kernel (warp per row i, 32 edges per round; lane l holds
//    features 2l, 2l+1 of G_{k+1}[i] and reads the same two features of every
//    edge's Z_k row, one coalesced line per row; a butterfly over the lanes
//    leaves edge t's dot product with lane t):
//    dA_e += (1 - alpha) G_{k+1}[i] . Z_k[j]  for e = (i, j);
//  * bwd_hop_t_kernel (warp per key j over its incoming edges, the transposed
//    graph; lanes own feature pairs):  G_k[j] = (1 - alpha) sum_e A_e G_{k+1}[i],
//    and dV_acc[j] += alpha G_{k+1}[j]; at k = 0 it writes dV = dV_acc + G_0
//    instead of G_0 (Z_0 = V).
//
// then the softmax and the scores:
//
//  * bwd_softmax_dq_kernel (warp per row i):  dS_e = A_e (dA_e - sum_t A_t dA_t)
//    / sqrt(64), stored over dA, and dQ_i = sum_e dS_e k_j;
//  * bwd_dk_kernel (warp per key j over its incoming edges):  dK_j = sum_e dS_e q_i.
//
// Every sum runs in a fixed order (edges ascending within a row; incoming
// edges by ascending row within a key), so the result is deterministic.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

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
    int64_t n, nnz, units;
};

// dA_e += keep * G[i] . Z[j] over the edges of row i (G: G_{k+1}, Z: Z_k).
template <typename TG, typename TZ>
__global__ void __launch_bounds__(kBwdWarps * 32)
bwd_weight_grad_kernel(BwdArgs a, const TG* __restrict__ G, const TZ* __restrict__ Z,
                       float* __restrict__ dA, float keep) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * kBwdWarps + (threadIdx.x >> 5);
    if (gw >= a.units * a.n) return;
    const int64_t u = gw / a.n, i = gw - u * a.n;
    const size_t unit = (size_t)u * a.n * kHeadDim;
    const int64_t e0 = a.row_ptr[i], e1 = a.row_ptr[i + 1];
    const float2 g = load2(G + unit + (size_t)i * kHeadDim + 2 * lane);
    const TZ* Zu = Z + unit + 2 * lane;
    float* dAu = dA + (size_t)u * a.nnz;
    for (int64_t base = e0; base < e1; base += 32) {
        const int64_t e = base + lane;
        const int32_t j_l = e < e1 ? a.col[e] : 0;
        const int cnt = (e1 - base) < 32 ? (int)(e1 - base) : 32;
        float p[32];        // all 32 rows requested before the first is used
#pragma unroll
        for (int t = 0; t < 32; ++t) {
            const int32_t j = __shfl_sync(0xffffffffu, j_l, t);
            const float2 z = t < cnt ? load2(Zu + (size_t)j * kHeadDim) : make_float2(0.f, 0.f);
            p[t] = fmaf(g.x, z.x, g.y * z.y);
        }
        const float dot = warp_transpose_sum32(p, lane);             // edge base + lane
        if (e < e1) dAu[e] += keep * dot;
    }
}

// Key j of the transposed hop: Gn[j] = keep * sum_{e = (i, j)} A_e G[i]; and
// dV_acc[j] = (first ? 0 : dV_acc[j]) + alpha G[j].  With dV_out set (k = 0),
// dV_out[j] = dV_acc[j] + alpha G[j] + Gn[j] in the I/O dtype and Gn is not written.
template <typename TG, typename TIo>
__global__ void __launch_bounds__(kBwdWarps * 32)
bwd_hop_t_kernel(BwdArgs a, const float* __restrict__ A, const TG* __restrict__ G,
                 float* __restrict__ Gn, float* __restrict__ dV_acc, TIo* __restrict__ dV_out,
                 float alpha, bool first) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * kBwdWarps + (threadIdx.x >> 5);
    if (gw >= a.units * a.n) return;
    const int64_t u = gw / a.n, j = gw - u * a.n;
    const size_t unit = (size_t)u * a.n * kHeadDim;
    const TG* Gu = G + unit + 2 * lane;
    const float* Au = A + (size_t)u * a.nnz;
    const int64_t t0 = a.t_ptr[j], t1 = a.t_ptr[j + 1];
    float2 acc = make_float2(0.f, 0.f);
    for (int64_t base = t0; base < t1; base += 32) {
        const int64_t t = base + lane;
        const float w_l = t < t1 ? Au[a.t_edge[t]] : 0.f;
        const int32_t i_l = t < t1 ? a.t_row[t] : 0;
        const int cnt = (t1 - base) < 32 ? (int)(t1 - base) : 32;
        float2 gv[32];        // all 32 rows requested before the first is used
#pragma unroll
        for (int s = 0; s < 32; ++s) {
            const int32_t i = __shfl_sync(0xffffffffu, i_l, s);
            gv[s] = s < cnt ? load2(Gu + (size_t)i * kHeadDim) : make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int s = 0; s < 32; ++s) {
            const float w = __shfl_sync(0xffffffffu, w_l, s);
            acc.x = fmaf(w, gv[s].x, acc.x);
            acc.y = fmaf(w, gv[s].y, acc.y);
        }
    }
    const float keep = 1.f - alpha;
    const size_t at = unit + (size_t)j * kHeadDim + 2 * lane;
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

// Row i: dS_e = A_e (dA_e - sum_t A_t dA_t) * scale in place over dA, then
// dQ_i = sum_e dS_e K[j] in the I/O dtype.
template <typename TIo>
__global__ void __launch_bounds__(kBwdWarps * 32)
bwd_softmax_dq_kernel(BwdArgs a, const float* __restrict__ A, float* __restrict__ dA,
                      const TIo* __restrict__ K, TIo* __restrict__ dQ) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * kBwdWarps + (threadIdx.x >> 5);
    if (gw >= a.units * a.n) return;
    const int64_t u = gw / a.n, i = gw - u * a.n;
    const size_t unit = (size_t)u * a.n * kHeadDim;
    const float* Au = A + (size_t)u * a.nnz;
    float* dAu = dA + (size_t)u * a.nnz;
    const int64_t e0 = a.row_ptr[i], e1 = a.row_ptr[i + 1];
    float dot = 0.f;
    for (int64_t e = e0 + lane; e < e1; e += 32) dot = fmaf(Au[e], dAu[e], dot);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    const TIo* Ku = K + unit + 2 * lane;
    float2 acc = make_float2(0.f, 0.f);
    for (int64_t base = e0; base < e1; base += 32) {
        const int64_t e = base + lane;
        float ds_l = 0.f;
        int32_t j_l = 0;
        if (e < e1) {
            ds_l = Au[e] * (dAu[e] - dot) * kScale;
            dAu[e] = ds_l;
            j_l = a.col[e];
        }
        const int cnt = (e1 - base) < 32 ? (int)(e1 - base) : 32;
        float2 kv[32];        // all 32 rows requested before the first is used
#pragma unroll
        for (int s = 0; s < 32; ++s) {
            const int32_t j = __shfl_sync(0xffffffffu, j_l, s);
            kv[s] = s < cnt ? load2(Ku + (size_t)j * kHeadDim) : make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int s = 0; s < 32; ++s) {
            const float w = __shfl_sync(0xffffffffu, ds_l, s);
            acc.x = fmaf(w, kv[s].x, acc.x);
            acc.y = fmaf(w, kv[s].y, acc.y);
        }
    }
    store2(dQ + unit + (size_t)i * kHeadDim + 2 * lane, acc);
}

// Key j: dK_j = sum_{e = (i, j)} dS_e Q[i] in the I/O dtype.
template <typename TIo>
__global__ void __launch_bounds__(kBwdWarps * 32)
bwd_dk_kernel(BwdArgs a, const float* __restrict__ dS, const TIo* __restrict__ Q,
              TIo* __restrict__ dK) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * kBwdWarps + (threadIdx.x >> 5);
    if (gw >= a.units * a.n) return;
    const int64_t u = gw / a.n, j = gw - u * a.n;
    const size_t unit = (size_t)u * a.n * kHeadDim;
    const float* dSu = dS + (size_t)u * a.nnz;
    const TIo* Qu = Q + unit + 2 * lane;
    const int64_t t0 = a.t_ptr[j], t1 = a.t_ptr[j + 1];
    float2 acc = make_float2(0.f, 0.f);
    for (int64_t base = t0; base < t1; base += 32) {
        const int64_t t = base + lane;
        const float w_l = t < t1 ? dSu[a.t_edge[t]] : 0.f;
        const int32_t i_l = t < t1 ? a.t_row[t] : 0;
        const int cnt = (t1 - base) < 32 ? (int)(t1 - base) : 32;
        float2 qv[32];        // all 32 rows requested before the first is used
#pragma unroll
        for (int s = 0; s < 32; ++s) {
            const int32_t i = __shfl_sync(0xffffffffu, i_l, s);
            qv[s] = s < cnt ? load2(Qu + (size_t)i * kHeadDim) : make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int s = 0; s < 32; ++s) {
            const float w = __shfl_sync(0xffffffffu, w_l, s);
            acc.x = fmaf(w, qv[s].x, acc.x);
            acc.y = fmaf(w, qv[s].y, acc.y);
        }
    }
    store2(dK + unit + (size_t)j * kHeadDim + 2 * lane, acc);
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
    const size_t io = (size_t)a.units * a.n * kHeadDim * sizeof(TIo);
    float* A = reinterpret_cast<float*>(ws + L.a);
    float* dA = reinterpret_cast<float*>(ws + L.da);
    float* dVacc = reinterpret_cast<float*>(ws + L.dv);
    float* Gbuf[2] = {reinterpret_cast<float*>(ws + L.g[0]), reinterpret_cast<float*>(ws + L.g[1])};
    auto zstate = [&](int32_t k) { return reinterpret_cast<float*>(ws + L.z + (size_t)(k - 1) * L.z_stride); };
    cudaError_t err;
    if (hops == 0) {
        // Z_K = V: dV = dOut, and nothing reaches the weights
        err = cudaMemcpyAsync(dV, dOut, io, cudaMemcpyDeviceToDevice, stream);
        if (err == cudaSuccess) err = cudaMemsetAsync(dQ, 0, io, stream);
        if (err == cudaSuccess) err = cudaMemsetAsync(dK, 0, io, stream);
        return err == cudaSuccess ? DIFFUSER_OK : cuda_fail(err, "backward with hops = 0");
    }
    // the forward's weights and states Z_1 .. Z_{K-1} (Z_0 is V)
    int st = launch_score_csr(ca, Q, K, dtype, A, stream);
    for (int32_t k = 1; k < hops && st == DIFFUSER_OK; ++k)
        st = launch_hop_csr(ca, A, k == 1 ? static_cast<const void*>(V) : zstate(k - 1), k == 1, V,
                            zstate(k), false, dtype, alpha, stream);
    if (st != DIFFUSER_OK) return st;
    err = cudaMemsetAsync(dA, 0, (size_t)a.units * a.nnz * sizeof(float), stream);
    if (err != cudaSuccess) return cuda_fail(err, "clearing dA");
    const float keep = 1.f - alpha;
    for (int32_t k = hops - 1; k >= 0; --k) {
        const bool top = (k == hops - 1);            // G_{k+1} is dOut itself
        float* Gn = Gbuf[k & 1];
        const float* Gf = Gbuf[(k + 1) & 1];         // G_{k+1} for k < hops - 1
        {
            LaunchScope scope(DIFFUSER_KERNEL_HOP, stream);
            if (top && k == 0)
                bwd_weight_grad_kernel<TIo, TIo><<<grid, block, 0, stream>>>(a, dOut, V, dA, keep);
            else if (top)
                bwd_weight_grad_kernel<TIo, float><<<grid, block, 0, stream>>>(a, dOut, zstate(k), dA, keep);
            else if (k == 0)
                bwd_weight_grad_kernel<float, TIo><<<grid, block, 0, stream>>>(a, Gf, V, dA, keep);
            else
                bwd_weight_grad_kernel<float, float><<<grid, block, 0, stream>>>(a, Gf, zstate(k), dA, keep);
        }
        if ((st = launched("bwd_weight_grad_kernel"))) return st;
        {
            LaunchScope scope(DIFFUSER_KERNEL_HOP, stream);
            TIo* out = k == 0 ? dV : nullptr;
            if (top)
                bwd_hop_t_kernel<TIo, TIo><<<grid, block, 0, stream>>>(a, A, dOut, Gn, dVacc, out, alpha, true);
            else
                bwd_hop_t_kernel<float, TIo><<<grid, block, 0, stream>>>(a, A, Gf, Gn, dVacc, out, alpha, false);
        }
        if ((st = launched("bwd_hop_t_kernel"))) return st;
    }
    {
        LaunchScope scope(DIFFUSER_KERNEL_SCORE, stream);
        bwd_softmax_dq_kernel<TIo><<<grid, block, 0, stream>>>(a, A, dA, K, dQ);
    }
    if ((st = launched("bwd_softmax_dq_kernel"))) return st;
    {
        LaunchScope scope(DIFFUSER_KERNEL_SCORE, stream);
        bwd_dk_kernel<TIo><<<grid, block, 0, stream>>>(a, dA, Q, dK);
    }
    return launched("bwd_dk_kernel");
}

}  // namespace

// The transposed graph (incoming edges of every key, rows ascending), built on
// the host from the CSR copy by a counting sort and uploaded (synchronously).
// On failure the arrays allocated so far are freed and d_t_ptr stays null.
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
    int64_t* d_ptr = nullptr;
    int32_t* d_row = nullptr;
    int64_t* d_edge = nullptr;
    cudaError_t err = cudaMalloc(&d_ptr, sizeof(int64_t) * (n + 1));
    if (err == cudaSuccess) err = cudaMalloc(&d_row, sizeof(int32_t) * t_row.size());
    if (err == cudaSuccess) err = cudaMalloc(&d_edge, sizeof(int64_t) * t_edge.size());
    if (err == cudaSuccess)
        err = cudaMemcpy(d_ptr, t_ptr.data(), sizeof(int64_t) * (n + 1), cudaMemcpyHostToDevice);
    if (err == cudaSuccess)
        err = cudaMemcpy(d_row, t_row.data(), sizeof(int32_t) * t_row.size(), cudaMemcpyHostToDevice);
    if (err == cudaSuccess)
        err = cudaMemcpy(d_edge, t_edge.data(), sizeof(int64_t) * t_edge.size(), cudaMemcpyHostToDevice);
    if (err != cudaSuccess) {
        cudaFree(d_ptr);
        cudaFree(d_row);
        cudaFree(d_edge);
        return cuda_fail(err, "building the transposed graph");
    }
    g->d_t_row = d_row;
    g->d_t_edge = d_edge;
    g->d_t_ptr = d_ptr;      // set last: non-null means the transposed graph is complete
    return DIFFUSER_OK;
}

int plan_backward_layout(const diffuser_graph* g, int64_t units, int32_t hops, BwdLayout* L) {
    // A, dA: [units][nnz] fp32; dV_acc, G (x2), Z_1 .. Z_{K-1}: [units][n][64] fp32
    const double states = 3.0 + (hops > 1 ? hops - 1 : 0);
    const double need = (double)units * (2.0 * 4.0 * (double)g->nnz +
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
    L->z = off;
    L->z_stride = state;
    off += (hops > 1 ? (size_t)(hops - 1) : 0) * state;
    L->total = off;
    return DIFFUSER_OK;
}

int launch_backward_csr(const diffuser_graph* g, int64_t units, const void* Q, const void* K,
                        const void* V, const void* dOut, int32_t dtype, int32_t hops, float alpha,
                        void* dQ, void* dK, void* dV, char* ws, const BwdLayout& L,
                        cudaStream_t stream) {
    BwdArgs a{g->d_row_ptr, g->d_col, g->d_t_ptr, g->d_t_row, g->d_t_edge, g->n, g->nnz, units};
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
