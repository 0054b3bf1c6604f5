// diffuser_forward_no_alloc: the forward pass for callers that must not
// allocate device memory while it runs -- for example code running inside a
// CUDA stream capture, a real-time serving loop whose memory is fixed at
// start-up, or a host framework that owns every allocation and forbids
// cudaMalloc/cudaFree (and allocating library calls) on its hot path.
//
// Instead of a caller-provided workspace, the intermediate weights A and the
// hop state Z_k live in one fixed-size array in device global memory that the
// library defines at file scope.  Every GPU that loads the library holds that
// array until the process exits.  It runs the general CSR kernels (the same
// score and hop kernels as diffuser_forward's CSR path).
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"

namespace dfs {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;   // 32 MiB per device
constexpr int kMaxDevices = 64;

// The scratch array.  In host code this symbol is only a stand-in: its device
// address must be fetched with cudaGetSymbolAddress on each device.
__device__ __align__(256) unsigned char g_no_alloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device, looked up once
// per device (on the first call made with that device current).
int scratch_for_current_device(void** ptr) {
    int dev = -1;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return cuda_fail(err, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(DIFFUSER_ERR_UNSUPPORTED, "device index beyond the supported range");
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        err = cudaGetSymbolAddress(&p, g_no_alloc_scratch);
        if (err != cudaSuccess) return cuda_fail(err, "cudaGetSymbolAddress(scratch)");
        g_scratch_ptr[dev] = p;
    }
    *ptr = g_scratch_ptr[dev];
    return DIFFUSER_OK;
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

}  // namespace
}  // namespace dfs

using namespace dfs;

extern "C" {

size_t diffuser_no_alloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

int diffuser_forward_no_alloc(const void* Q, const void* K, const void* V, int32_t dtype,
                              int64_t B, int64_t H, int32_t d, const diffuser_graph* g,
                              int32_t hops, float alpha, void* out, diffuser_stream stream) {
    try {
        if (!g) return fail(DIFFUSER_ERR_INVALID_ARG, "graph is NULL");
        if (B < 1 || H < 1) return fail(DIFFUSER_ERR_INVALID_ARG, "B and H must be >= 1");
        if (d != kHeadDim) return fail(DIFFUSER_ERR_UNSUPPORTED, "head width d must be 64");
        if (dtype != DIFFUSER_DTYPE_FP32 && dtype != DIFFUSER_DTYPE_BF16)
            return fail(DIFFUSER_ERR_UNSUPPORTED, "dtype must be FP32 or BF16");
        if (!Q || !K || !V || !out) return fail(DIFFUSER_ERR_INVALID_ARG, "a tensor pointer is NULL");
        if ((reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K) |
             reinterpret_cast<uintptr_t>(V) | reinterpret_cast<uintptr_t>(out)) & 15)
            return fail(DIFFUSER_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
        if (hops < 0) return fail(DIFFUSER_ERR_INVALID_ARG, "hops must be >= 0");
        if (!(alpha >= 0.f && alpha <= 1.f))
            return fail(DIFFUSER_ERR_INVALID_ARG, "alpha must lie in [0, 1]");
        const size_t units = (size_t)B * (size_t)H;
        const size_t io = units * (size_t)g->n * kHeadDim * (dtype == DIFFUSER_DTYPE_BF16 ? 2 : 4);
        if (overlap(out, io, Q, io) || overlap(out, io, K, io))
            return fail(DIFFUSER_ERR_INVALID_ARG, "out overlaps Q or K");
        if (hops > 0 && overlap(out, io, V, io))
            return fail(DIFFUSER_ERR_INVALID_ARG, "out may alias V only when hops == 0");
        // scratch: A [units][nnz] fp32, then two fp32 hop-state buffers [units][n][64]
        const double a_bytes = (double)units * (double)g->nnz * 4.0;
        const double z_bytes = (double)units * (double)g->n * kHeadDim * 4.0;
        const double need = (double)round256((size_t)a_bytes) + 2.0 * (double)round256((size_t)z_bytes);
        if (need > (double)kNoAllocScratchBytes)
            return fail(DIFFUSER_ERR_WORKSPACE,
                        "problem too large for the no-allocation scratch: needs " +
                            std::to_string((long long)need) + " bytes, the fixed array holds " +
                            std::to_string((long long)kNoAllocScratchBytes));
        int dev = -1;
        cudaError_t err = cudaGetDevice(&dev);
        if (err != cudaSuccess) return cuda_fail(err, "cudaGetDevice");
        if (dev != g->device)
            return fail(DIFFUSER_ERR_INVALID_ARG, "the current device is not the graph's device");
        void* scratch = nullptr;
        int st = scratch_for_current_device(&scratch);
        if (st) return st;

        cudaStream_t s = stream;
        if (hops == 0) {
            if (out == V) return DIFFUSER_OK;
            err = cudaMemcpyAsync(out, V, io, cudaMemcpyDeviceToDevice, s);
            return err == cudaSuccess ? DIFFUSER_OK : cuda_fail(err, "copying V to out (hops = 0)");
        }
        char* base = static_cast<char*>(scratch);
        float* A = reinterpret_cast<float*>(base);
        float* zbuf[2] = {reinterpret_cast<float*>(base + round256((size_t)a_bytes)),
                          reinterpret_cast<float*>(base + round256((size_t)a_bytes) +
                                                   round256((size_t)z_bytes))};
        CsrArgs a{g->d_row_ptr, g->d_col, g->n, g->nnz, (int64_t)units};
        if ((st = launch_score_csr(a, Q, K, dtype, A, s))) return st;
        for (int32_t k = 0; k < hops; ++k) {
            const bool first = (k == 0), last = (k == hops - 1);
            const void* src = first ? V : zbuf[(k - 1) & 1];
            void* dst = last ? out : zbuf[k & 1];
            if ((st = launch_hop_csr(a, A, src, first, V, dst, last, dtype, alpha, s))) return st;
        }
        return DIFFUSER_OK;
    } catch (...) {
        return fail(DIFFUSER_ERR_ALLOC, "unexpected exception");
    }
}

}  // extern "C"
