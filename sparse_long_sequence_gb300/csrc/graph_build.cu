// Deterministic graph construction on the device: count -> exclusive scan ->
// fill, one thread per row.  Produces the deduplicated CSR (rows and columns
// ascending) that every kernel and the parity checks use.
//
// Token graph ("Diffuser: modelling long sequences with multi-hop attention
// diffusion", sec 2.2; "1.2.1 Static sparsity: Longformer, BigBird and
// sliding windows", sec 1.1 eq 5 and sec 1.2 eq 12):
//   i in G:  N(i) = {0..n-1}
//   else:    N(i) = window [i-r, i+r] cut to [0,n)  u  G  u  extras(i)
// where extras(i) are the random draws splitmix64(seed ^ (i*R + t)) mod n
// (or, for the uniform-spaced variant, the grid positions of row_draw) that
// fall outside the window and outside G, sorted and deduplicated.  The three
// parts are disjoint, so a row is a merge of three sorted lists.
//
// Causal token graph (Diffuser notes sec 2.6: A lower-triangular, every edge
// obeys j <= i; sliding-window page sec 1.1: the causal window holds the r+1
// history positions): the same sets cut to [0, i].  Each row's upper limit
// `last` is i instead of n-1; draws that land after i are dropped.
//
// Dilated token graph (sliding-window page, sec 1.2 eq 11): the window of row
// i is the progression i + k * dilation, |k| <= r; its rows are built by
// separate kernels that merge that progression, G and the row's draws.
//
// Block graph (same page, sec 2 eq 13; "038 BigBird", sec 2): allowed blocks
// of block row J are all blocks for J < gb, else [0, gb) u (window blocks u
// random blocks); the tokens of the allowed blocks, ascending.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace dfs {
namespace {

// SplitMix64 output function (Steele, Lea and Flood 2014): golden-ratio
// increment, then two xor-shift-multiply rounds and a final xor-shift.
__device__ __forceinline__ uint64_t splitmix64(uint64_t x) {
    uint64_t z = x + 0x9E3779B97F4A7C15ULL;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

// number of entries of the sorted array a[0..len) that are < x
__device__ __forceinline__ int32_t count_less(const int32_t* a, int32_t len, int64_t x) {
    int32_t lo = 0, hi = len;
    while (lo < hi) {
        int32_t mid = (lo + hi) >> 1;
        if (a[mid] < x) lo = mid + 1; else hi = mid;
    }
    return lo;
}

struct TokenParams {
    int64_t n;
    int32_t r, g, R;
    uint64_t seed;
    const int32_t* globals;
    const uint8_t* is_global;
    int32_t causal;
    int32_t uniform;     // 1: the R extras of a row sit on a uniform grid instead of random draws
};

// Extra t of row i: the random draw splitmix64(seed ^ (i R + t)) mod n, or on
// the uniform grid ("w uni.", Diffuser notes sec 4.5, Tab S.7; the spacing
// rule is not given): i + floor((2t + 1) n / (2R)) mod n, half a spacing on
// from i, spacing n / R around the ring of positions.
__device__ __forceinline__ int64_t row_draw(const TokenParams& p, int64_t i, int32_t t) {
    if (p.uniform) return (i + ((int64_t)(2 * t + 1) * p.n) / (2 * (int64_t)p.R)) % p.n;
    const uint64_t key = (uint64_t)i * (uint64_t)p.R + (uint64_t)t;
    return (int64_t)(splitmix64(p.seed ^ key) % (uint64_t)p.n);
}

// last column row i may read: i for the causal graph, else n-1
__device__ __forceinline__ int64_t row_last(const TokenParams& p, int64_t i) {
    return p.causal ? i : p.n - 1;
}

// window [lo, hi] of row i, cut to [0, last]
__device__ __forceinline__ void row_window(const TokenParams& p, int64_t i, int64_t& lo,
                                           int64_t& hi) {
    const int64_t last = row_last(p, i);
    lo = i - p.r < 0 ? 0 : i - p.r;
    hi = i + p.r > last ? last : i + p.r;
}

// Sorted, deduplicated random draws of row i that fall outside its window
// and outside G.  Returns their number; xs must hold R entries.
__device__ int32_t row_extras(const TokenParams& p, int64_t i, int64_t lo, int64_t hi,
                              int32_t* xs) {
    int32_t cnt = 0;
    for (int32_t t = 0; t < p.R; ++t) {
        const int64_t j = row_draw(p, i, t);
        if (j > row_last(p, i) || (j >= lo && j <= hi) || p.is_global[j]) continue;
        // insertion into the sorted prefix, dropping duplicates
        int32_t pos = cnt;
        while (pos > 0 && xs[pos - 1] > j) --pos;
        if (pos > 0 && xs[pos - 1] == j) continue;
        for (int32_t q = cnt; q > pos; --q) xs[q] = xs[q - 1];
        xs[pos] = (int32_t)j;
        ++cnt;
    }
    return cnt;
}

__global__ void token_count_kernel(TokenParams p, int64_t* counts) {
    extern __shared__ int32_t smem_xs[];
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= p.n) return;
    const int64_t last = row_last(p, i);
    if (p.is_global[i]) { counts[i] = last + 1; return; }
    int64_t lo, hi;
    row_window(p, i, lo, hi);
    int64_t c = hi - lo + 1;
    c += count_less(p.globals, p.g, lo) +
         (count_less(p.globals, p.g, last + 1) - count_less(p.globals, p.g, hi + 1));
    int32_t* xs = smem_xs + (size_t)threadIdx.x * p.R;
    c += row_extras(p, i, lo, hi, xs);
    counts[i] = c;
}

// Merge the entries of G and xs that lie in [from, to] into col, ascending.
__device__ int64_t merge_range(const int32_t* G, int32_t g, const int32_t* xs, int32_t nx,
                               int64_t from, int64_t to, int32_t* col) {
    int32_t a = count_less(G, g, from), a_end = count_less(G, g, to + 1);
    int32_t b = count_less(xs, nx, from), b_end = count_less(xs, nx, to + 1);
    int64_t w = 0;
    while (a < a_end || b < b_end) {
        if (b >= b_end || (a < a_end && G[a] < xs[b])) col[w++] = G[a++];
        else col[w++] = xs[b++];
    }
    return w;
}

__global__ void extras_count_kernel(TokenParams p, int64_t* counts) {
    extern __shared__ int32_t smem_xs[];
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= p.n) return;
    if (p.is_global[i]) { counts[i] = 0; return; }
    int64_t lo, hi;
    row_window(p, i, lo, hi);
    counts[i] = row_extras(p, i, lo, hi, smem_xs + (size_t)threadIdx.x * p.R);
}

__global__ void extras_fill_kernel(TokenParams p, const int64_t* x_ptr, int32_t* x_col) {
    extern __shared__ int32_t smem_xs[];
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= p.n || p.is_global[i]) return;
    int64_t lo, hi;
    row_window(p, i, lo, hi);
    int32_t* xs = smem_xs + (size_t)threadIdx.x * p.R;
    int32_t nx = row_extras(p, i, lo, hi, xs);
    for (int32_t q = 0; q < nx; ++q) x_col[x_ptr[i] + q] = xs[q];
}

__global__ void token_fill_kernel(TokenParams p, const int64_t* row_ptr, int32_t* col) {
    extern __shared__ int32_t smem_xs[];
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= p.n) return;
    int32_t* out = col + row_ptr[i];
    const int64_t last = row_last(p, i);
    if (p.is_global[i]) {
        for (int64_t j = 0; j <= last; ++j) out[j] = (int32_t)j;
        return;
    }
    int64_t lo, hi;
    row_window(p, i, lo, hi);
    int32_t* xs = smem_xs + (size_t)threadIdx.x * p.R;
    int32_t nx = row_extras(p, i, lo, hi, xs);
    int64_t w = merge_range(p.globals, p.g, xs, nx, 0, lo - 1, out);
    for (int64_t j = lo; j <= hi; ++j) out[w++] = (int32_t)j;
    merge_range(p.globals, p.g, xs, nx, hi + 1, last, out + w);
}

// ---- dilated token graph (sliding-window page, sec 1.2 eq 11) ----
// Row i's window is the progression i + k dil, |k| <= r, cut to [0, last]; a
// row is the merge of that progression, the globals up to last and the row's
// own draws up to last, each value entering once.  (dil = 1 graphs take the
// token kernels above.)

// Sorted, deduplicated random draws of row i that do not lie after `last`.
__device__ int32_t row_draws(const TokenParams& p, int64_t i, int64_t last, int32_t* xs) {
    int32_t cnt = 0;
    for (int32_t t = 0; t < p.R; ++t) {
        const int64_t j = row_draw(p, i, t);
        if (j > last) continue;
        int32_t pos = cnt;
        while (pos > 0 && xs[pos - 1] > j) --pos;
        if (pos > 0 && xs[pos - 1] == j) continue;
        for (int32_t q = cnt; q > pos; --q) xs[q] = xs[q - 1];
        xs[pos] = (int32_t)j;
        ++cnt;
    }
    return cnt;
}

// The merged row (written to out unless it is null); returns its length.
__device__ int64_t dilated_row(const TokenParams& p, int32_t dil, int64_t i, const int32_t* xs,
                               int32_t nx, int32_t* out) {
    const int64_t last = row_last(p, i);
    const int64_t kmin = -(i / dil < p.r ? i / dil : (int64_t)p.r);          // i + k dil >= 0
    const int64_t kmax = (last - i) / dil < p.r ? (last - i) / dil : (int64_t)p.r;   // <= last
    const int32_t a_end = count_less(p.globals, p.g, last + 1);
    const int64_t none = INT64_MAX;
    int64_t k = kmin, w = 0;
    int32_t a = 0, b = 0;
    for (;;) {
        const int64_t vw = k <= kmax ? i + k * dil : none;
        const int64_t vg = a < a_end ? (int64_t)p.globals[a] : none;
        const int64_t vx = b < nx ? (int64_t)xs[b] : none;
        int64_t v = vw < vg ? vw : vg;
        if (vx < v) v = vx;
        if (v == none) break;
        if (out) out[w] = (int32_t)v;
        ++w;
        if (vw == v) ++k;
        if (vg == v) ++a;
        if (vx == v) ++b;
    }
    return w;
}

__global__ void dilated_count_kernel(TokenParams p, int32_t dil, int64_t* counts) {
    extern __shared__ int32_t smem_xs[];
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= p.n) return;
    const int64_t last = row_last(p, i);
    if (p.is_global[i]) { counts[i] = last + 1; return; }
    int32_t* xs = smem_xs + (size_t)threadIdx.x * p.R;
    const int32_t nx = row_draws(p, i, last, xs);
    counts[i] = dilated_row(p, dil, i, xs, nx, nullptr);
}

__global__ void dilated_fill_kernel(TokenParams p, int32_t dil, const int64_t* row_ptr,
                                    int32_t* col) {
    extern __shared__ int32_t smem_xs[];
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= p.n) return;
    int32_t* out = col + row_ptr[i];
    const int64_t last = row_last(p, i);
    if (p.is_global[i]) {
        for (int64_t j = 0; j <= last; ++j) out[j] = (int32_t)j;
        return;
    }
    int32_t* xs = smem_xs + (size_t)threadIdx.x * p.R;
    const int32_t nx = row_draws(p, i, last, xs);
    dilated_row(p, dil, i, xs, nx, out);
}

struct BlockParams {
    int64_t n, nb;
    int32_t block, half, s, gb;
    uint64_t seed;
};

// Sorted, deduplicated allowed blocks >= gb of block row J >= gb (window and
// random blocks); blocks [0, gb) are allowed for every row in addition.
__device__ int32_t other_blocks(const BlockParams& p, int64_t J, int32_t* bl) {
    int32_t cnt = 0;
    auto insert = [&](int64_t b) {
        if (b < p.gb || b < 0 || b >= p.nb) return;
        int32_t pos = cnt;
        while (pos > 0 && bl[pos - 1] > b) --pos;
        if (pos > 0 && bl[pos - 1] == b) return;
        for (int32_t q = cnt; q > pos; --q) bl[q] = bl[q - 1];
        bl[pos] = (int32_t)b;
        ++cnt;
    };
    for (int64_t b = J - p.half; b <= J + p.half; ++b) insert(b);
    for (int32_t t = 0; t < p.s; ++t) {
        uint64_t key = (uint64_t)J * (uint64_t)p.s + (uint64_t)t;
        insert((int64_t)(splitmix64(p.seed ^ key) % (uint64_t)p.nb));
    }
    return cnt;
}

__device__ __forceinline__ int64_t block_len(const BlockParams& p, int64_t b) {
    int64_t start = b * p.block;
    int64_t end = start + p.block < p.n ? start + p.block : p.n;
    return end - start;
}

__global__ void block_count_kernel(BlockParams p, int64_t* counts) {
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= p.n) return;
    int64_t J = i / p.block;
    if (J < p.gb) { counts[i] = p.n; return; }
    int32_t bl[kMaxWindowBlocks + kMaxRandBlocks];
    int32_t cnt = other_blocks(p, J, bl);
    int64_t prefix = (int64_t)p.gb * p.block;
    int64_t c = prefix < p.n ? prefix : p.n;
    for (int32_t q = 0; q < cnt; ++q) c += block_len(p, bl[q]);
    counts[i] = c;
}

__global__ void block_fill_kernel(BlockParams p, const int64_t* row_ptr, int32_t* col) {
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= p.n) return;
    int32_t* out = col + row_ptr[i];
    int64_t J = i / p.block;
    if (J < p.gb) {
        for (int64_t j = 0; j < p.n; ++j) out[j] = (int32_t)j;
        return;
    }
    int32_t bl[kMaxWindowBlocks + kMaxRandBlocks];
    int32_t cnt = other_blocks(p, J, bl);
    int64_t w = 0;
    int64_t prefix = (int64_t)p.gb * p.block;
    if (prefix > p.n) prefix = p.n;
    for (int64_t j = 0; j < prefix; ++j) out[w++] = (int32_t)j;
    for (int32_t q = 0; q < cnt; ++q) {
        int64_t start = (int64_t)bl[q] * p.block;
        int64_t len = block_len(p, bl[q]);
        for (int64_t j = 0; j < len; ++j) out[w++] = (int32_t)(start + j);
    }
}

// Exclusive scan of counts[0..n) into row_ptr[0..n]; one block of 1024
// threads walks the array in chunks, carrying the running total.
__global__ void __launch_bounds__(1024) exclusive_scan_kernel(const int64_t* counts, int64_t n,
                                                              int64_t* row_ptr) {
    __shared__ int64_t warp_sums[32];
    __shared__ int64_t carry;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int64_t base = 0; base < n; base += 1024) {
        int64_t idx = base + threadIdx.x;
        int64_t v = idx < n ? counts[idx] : 0;
        int64_t x = v;  // inclusive scan within the warp
        for (int off = 1; off < 32; off <<= 1) {
            int64_t y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) warp_sums[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int64_t s = warp_sums[lane];
            for (int off = 1; off < 32; off <<= 1) {
                int64_t y = __shfl_up_sync(0xffffffffu, s, off);
                if (lane >= off) s += y;
            }
            warp_sums[lane] = s;  // inclusive over warps
        }
        __syncthreads();
        int64_t before = carry + (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
        if (idx < n) row_ptr[idx] = before;
        __syncthreads();
        if (threadIdx.x == 1023) carry = before + v;
        __syncthreads();
    }
    if (threadIdx.x == 0) row_ptr[n] = carry;
}

int scan_and_alloc(diffuser_graph* g, int64_t* d_counts, cudaStream_t stream) {
    cudaError_t err = cudaMalloc(&g->d_row_ptr, sizeof(int64_t) * (g->n + 1));
    if (err != cudaSuccess) return fail(DIFFUSER_ERR_ALLOC, "cudaMalloc(row_ptr) failed");
    {
        LaunchScope scope(DIFFUSER_KERNEL_BUILD, stream);
        exclusive_scan_kernel<<<1, 1024, 0, stream>>>(d_counts, g->n, g->d_row_ptr);
    }
    if ((err = cudaGetLastError()) != cudaSuccess) return cuda_fail(err, "exclusive_scan_kernel");
    int64_t nnz = 0;
    err = cudaMemcpyAsync(&nnz, g->d_row_ptr + g->n, sizeof(int64_t), cudaMemcpyDeviceToHost,
                          stream);
    if (err == cudaSuccess) err = cudaStreamSynchronize(stream);
    if (err != cudaSuccess) return cuda_fail(err, "reading nnz");
    if (nnz <= 0 || nnz > kMaxNnz)
        return fail(DIFFUSER_ERR_OVERFLOW, "edge count out of range: " + std::to_string(nnz));
    g->nnz = nnz;
    err = cudaMalloc(&g->d_col, sizeof(int32_t) * nnz);
    if (err != cudaSuccess) return fail(DIFFUSER_ERR_ALLOC, "cudaMalloc(col) failed");
    return DIFFUSER_OK;
}

// Extras list (random edges outside the window and G): count, scan, fill.
int build_extras(diffuser_graph* g, const TokenParams& p, unsigned blocks, int threads,
                 size_t shmem, int64_t* d_counts, cudaStream_t stream) {
    cudaError_t err;
    {
        LaunchScope scope(DIFFUSER_KERNEL_BUILD, stream);
        extras_count_kernel<<<blocks, threads, shmem, stream>>>(p, d_counts);
    }
    if ((err = cudaGetLastError()) != cudaSuccess) return cuda_fail(err, "extras_count_kernel");
    err = cudaMalloc(&g->d_x_ptr, sizeof(int64_t) * (g->n + 1));
    if (err != cudaSuccess) return fail(DIFFUSER_ERR_ALLOC, "cudaMalloc(x_ptr) failed");
    {
        LaunchScope scope(DIFFUSER_KERNEL_BUILD, stream);
        exclusive_scan_kernel<<<1, 1024, 0, stream>>>(d_counts, g->n, g->d_x_ptr);
    }
    if ((err = cudaGetLastError()) != cudaSuccess) return cuda_fail(err, "exclusive_scan_kernel");
    int64_t nx = 0;
    err = cudaMemcpyAsync(&nx, g->d_x_ptr + g->n, sizeof(int64_t), cudaMemcpyDeviceToHost, stream);
    if (err == cudaSuccess) err = cudaStreamSynchronize(stream);
    if (err != cudaSuccess) return cuda_fail(err, "reading the extras count");
    g->nx = nx;
    err = cudaMalloc(&g->d_x_col, sizeof(int32_t) * (nx > 0 ? nx : 1));
    if (err != cudaSuccess) return fail(DIFFUSER_ERR_ALLOC, "cudaMalloc(x_col) failed");
    {
        LaunchScope scope(DIFFUSER_KERNEL_BUILD, stream);
        extras_fill_kernel<<<blocks, threads, shmem, stream>>>(p, g->d_x_ptr, g->d_x_col);
    }
    if ((err = cudaGetLastError()) != cudaSuccess) return cuda_fail(err, "extras_fill_kernel");
    return DIFFUSER_OK;
}

int copy_csr_to_host(diffuser_graph* g, cudaStream_t stream) {
    g->h_row_ptr.resize(g->n + 1);
    g->h_col.resize(g->nnz);
    cudaError_t err = cudaMemcpyAsync(g->h_row_ptr.data(), g->d_row_ptr,
                                      sizeof(int64_t) * (g->n + 1), cudaMemcpyDeviceToHost, stream);
    if (err == cudaSuccess)
        err = cudaMemcpyAsync(g->h_col.data(), g->d_col, sizeof(int32_t) * g->nnz,
                              cudaMemcpyDeviceToHost, stream);
    if (err == cudaSuccess) err = cudaStreamSynchronize(stream);
    if (err != cudaSuccess) return cuda_fail(err, "copying the CSR to the host");
    return DIFFUSER_OK;
}

}  // namespace

int build_token_graph_device(diffuser_graph* g, cudaStream_t stream) {
    const int64_t n = g->n;
    cudaError_t err;
    std::vector<uint8_t> flags(n, 0);
    std::vector<int32_t> slots(n, -1);
    for (size_t s = 0; s < g->h_globals.size(); ++s) {
        flags[g->h_globals[s]] = 1;
        slots[g->h_globals[s]] = (int32_t)s;
    }
    err = cudaMalloc(&g->d_is_global, n);
    if (err != cudaSuccess) return fail(DIFFUSER_ERR_ALLOC, "cudaMalloc(is_global) failed");
    err = cudaMalloc(&g->d_gslot, sizeof(int32_t) * n);
    if (err != cudaSuccess) return fail(DIFFUSER_ERR_ALLOC, "cudaMalloc(gslot) failed");
    err = cudaMemcpyAsync(g->d_gslot, slots.data(), sizeof(int32_t) * n, cudaMemcpyHostToDevice,
                          stream);
    if (err != cudaSuccess) return cuda_fail(err, "uploading the global slots");
    err = cudaMalloc(&g->d_globals, sizeof(int32_t) * (g->n_globals > 0 ? g->n_globals : 1));
    if (err != cudaSuccess) return fail(DIFFUSER_ERR_ALLOC, "cudaMalloc(globals) failed");
    err = cudaMemcpyAsync(g->d_is_global, flags.data(), n, cudaMemcpyHostToDevice, stream);
    if (err == cudaSuccess && g->n_globals > 0)
        err = cudaMemcpyAsync(g->d_globals, g->h_globals.data(), sizeof(int32_t) * g->n_globals,
                              cudaMemcpyHostToDevice, stream);
    if (err != cudaSuccess) return cuda_fail(err, "uploading the global positions");

    int64_t* d_counts = nullptr;
    err = cudaMalloc(&d_counts, sizeof(int64_t) * n);
    if (err != cudaSuccess) return fail(DIFFUSER_ERR_ALLOC, "cudaMalloc(counts) failed");

    TokenParams p{n,        g->r,           g->n_globals,   g->rand_per_row,
                  g->seed,  g->d_globals,   g->d_is_global, g->causal ? 1 : 0, g->uniform};
    // per-thread scratch for the extras lives in shared memory; keep it <= 48 KB
    int threads = 128;
    while (threads > 1 && (size_t)threads * p.R * sizeof(int32_t) > 48 * 1024) threads >>= 1;
    size_t shmem = (size_t)threads * p.R * sizeof(int32_t);
    unsigned blocks = (unsigned)((n + threads - 1) / threads);
    int status = DIFFUSER_OK;
    {
        LaunchScope scope(DIFFUSER_KERNEL_BUILD, stream);
        token_count_kernel<<<blocks, threads, shmem, stream>>>(p, d_counts);
    }
    if ((err = cudaGetLastError()) != cudaSuccess) status = cuda_fail(err, "token_count_kernel");
    if (status == DIFFUSER_OK) status = scan_and_alloc(g, d_counts, stream);
    if (status == DIFFUSER_OK) {
        {
            LaunchScope scope(DIFFUSER_KERNEL_BUILD, stream);
            token_fill_kernel<<<blocks, threads, shmem, stream>>>(p, g->d_row_ptr, g->d_col);
        }
        if ((err = cudaGetLastError()) != cudaSuccess) status = cuda_fail(err, "token_fill_kernel");
    }
    if (status == DIFFUSER_OK) status = build_extras(g, p, blocks, threads, shmem, d_counts, stream);
    if (status == DIFFUSER_OK) status = copy_csr_to_host(g, stream);
    cudaFree(d_counts);
    return status;
}

int build_dilated_graph_device(diffuser_graph* g, cudaStream_t stream) {
    const int64_t n = g->n;
    cudaError_t err;
    std::vector<uint8_t> flags(n, 0);
    for (int32_t s : g->h_globals) flags[s] = 1;
    err = cudaMalloc(&g->d_is_global, n);
    if (err != cudaSuccess) return fail(DIFFUSER_ERR_ALLOC, "cudaMalloc(is_global) failed");
    err = cudaMalloc(&g->d_globals, sizeof(int32_t) * (g->n_globals > 0 ? g->n_globals : 1));
    if (err != cudaSuccess) return fail(DIFFUSER_ERR_ALLOC, "cudaMalloc(globals) failed");
    err = cudaMemcpyAsync(g->d_is_global, flags.data(), n, cudaMemcpyHostToDevice, stream);
    if (err == cudaSuccess && g->n_globals > 0)
        err = cudaMemcpyAsync(g->d_globals, g->h_globals.data(), sizeof(int32_t) * g->n_globals,
                              cudaMemcpyHostToDevice, stream);
    if (err != cudaSuccess) return cuda_fail(err, "uploading the global positions");
    int64_t* d_counts = nullptr;
    err = cudaMalloc(&d_counts, sizeof(int64_t) * n);
    if (err != cudaSuccess) return fail(DIFFUSER_ERR_ALLOC, "cudaMalloc(counts) failed");
    TokenParams p{n,       g->r,         g->n_globals,   g->rand_per_row,
                  g->seed, g->d_globals, g->d_is_global, g->causal ? 1 : 0, g->uniform};
    // per-thread scratch for the draws lives in shared memory; keep it <= 48 KB
    int threads = 128;
    while (threads > 1 && (size_t)threads * p.R * sizeof(int32_t) > 48 * 1024) threads >>= 1;
    const size_t shmem = (size_t)threads * p.R * sizeof(int32_t);
    const unsigned blocks = (unsigned)((n + threads - 1) / threads);
    int status = DIFFUSER_OK;
    {
        LaunchScope scope(DIFFUSER_KERNEL_BUILD, stream);
        dilated_count_kernel<<<blocks, threads, shmem, stream>>>(p, g->dilation, d_counts);
    }
    if ((err = cudaGetLastError()) != cudaSuccess) status = cuda_fail(err, "dilated_count_kernel");
    if (status == DIFFUSER_OK) status = scan_and_alloc(g, d_counts, stream);
    if (status == DIFFUSER_OK) {
        {
            LaunchScope scope(DIFFUSER_KERNEL_BUILD, stream);
            dilated_fill_kernel<<<blocks, threads, shmem, stream>>>(p, g->dilation, g->d_row_ptr,
                                                                     g->d_col);
        }
        if ((err = cudaGetLastError()) != cudaSuccess) status = cuda_fail(err, "dilated_fill_kernel");
    }
    if (status == DIFFUSER_OK) status = copy_csr_to_host(g, stream);
    cudaFree(d_counts);
    return status;
}

int build_block_graph_device(diffuser_graph* g, cudaStream_t stream) {
    const int64_t n = g->n;
    cudaError_t err;
    int64_t* d_counts = nullptr;
    err = cudaMalloc(&d_counts, sizeof(int64_t) * n);
    if (err != cudaSuccess) return fail(DIFFUSER_ERR_ALLOC, "cudaMalloc(counts) failed");
    BlockParams p{n, (n + g->block - 1) / g->block, g->block, (g->window_blocks - 1) / 2,
                  g->rand_blocks, g->global_blocks, g->seed};
    const int threads = 128;
    unsigned blocks = (unsigned)((n + threads - 1) / threads);
    int status = DIFFUSER_OK;
    {
        LaunchScope scope(DIFFUSER_KERNEL_BUILD, stream);
        block_count_kernel<<<blocks, threads, 0, stream>>>(p, d_counts);
    }
    if ((err = cudaGetLastError()) != cudaSuccess) status = cuda_fail(err, "block_count_kernel");
    if (status == DIFFUSER_OK) status = scan_and_alloc(g, d_counts, stream);
    if (status == DIFFUSER_OK) {
        {
            LaunchScope scope(DIFFUSER_KERNEL_BUILD, stream);
            block_fill_kernel<<<blocks, threads, 0, stream>>>(p, g->d_row_ptr, g->d_col);
        }
        if ((err = cudaGetLastError()) != cudaSuccess) status = cuda_fail(err, "block_fill_kernel");
    }
    if (status == DIFFUSER_OK) status = copy_csr_to_host(g, stream);
    cudaFree(d_counts);
    return status;
}

}  // namespace dfs
