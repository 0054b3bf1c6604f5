// diffuser_forward_no_alloc: the forward pass for callers that must not
// allocate device memory while it runs -- for example a serving loop whose
// device memory is fixed at start-up, or a host framework that owns every
// allocation and forbids cudaMalloc/cudaFree (and allocating library calls)
// on its hot path.
//
// Instead of a caller-provided workspace, the intermediate weights A and the
// hop state Z_k live in one fixed-size array in device global memory that the
// library defines at file scope.  Every GPU that loads the library holds that
// array until the process exits.  It runs the general CSR kernels with the
// same argument checks, workspace layout and hop sequence as
// diffuser_forward's CSR path.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <string>

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

}  // namespace
}  // namespace dfs

using namespace dfs;

extern "C" {

size_t diffuser_no_alloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

int diffuser_forward_no_alloc(const void* Q, const void* K, const void* V, int32_t dtype,
                              int64_t B, int64_t H, int32_t d, const diffuser_graph* g,
                              int32_t hops, float alpha, void* out, diffuser_stream stream) {
    try {
        int st = check_shape(g, B, H, d, dtype);
        if (st) return st;
        if (!Q || !K || !V || !out) return fail(DIFFUSER_ERR_INVALID_ARG, "a tensor pointer is NULL");
        if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(out))
            return fail(DIFFUSER_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
        if (hops < 0) return fail(DIFFUSER_ERR_INVALID_ARG, "hops must be >= 0");
        if (!(alpha >= 0.f && alpha <= 1.f))
            return fail(DIFFUSER_ERR_INVALID_ARG, "alpha must lie in [0, 1]");
        const size_t io = io_bytes(g, B, H, dtype);
        if (overlaps(out, io, Q, io) || overlaps(out, io, K, io))
            return fail(DIFFUSER_ERR_INVALID_ARG, "out overlaps Q or K");
        if (hops > 0 && overlaps(out, io, V, io))
            return fail(DIFFUSER_ERR_INVALID_ARG, "out may alias V only when hops == 0");
        // the CSR path's layout (A, then two hop-state buffers) inside the fixed array
        Layout L;
        if ((st = plan_layout(g, B, H, &L))) return st;
        if (L.total > kNoAllocScratchBytes)
            return fail(DIFFUSER_ERR_WORKSPACE,
                        "problem too large for the no-allocation scratch: needs " +
                            std::to_string(L.total) + " bytes, the fixed array holds " +
                            std::to_string(kNoAllocScratchBytes));
        if ((st = check_device(g))) return st;
        if ((st = check_status_word(g))) return st;
        void* scratch = nullptr;
        if ((st = scratch_for_current_device(&scratch))) return st;

        char* base = static_cast<char*>(scratch);
        CsrArgs a{g->d_row_ptr, g->d_col, g->n, g->nnz, B * H};
        if (hops == 0) return run_hops_csr(g, a, nullptr, V, dtype, 0, alpha, out, base, L, stream);
        float* A = reinterpret_cast<float*>(base + L.a_off);
        if ((st = launch_score_csr(a, Q, K, dtype, A, stream))) return st;
        return run_hops_csr(g, a, A, V, dtype, hops, alpha, out, base, L, stream);
    } catch (...) {
        return fail(DIFFUSER_ERR_ALLOC, "unexpected exception");
    }
}

}  // extern "C"
