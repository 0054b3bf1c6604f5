// Internal declarations of libdiffuser (host dispatch <-> kernels).  Not part
// of the public ABI; see include/diffuser.h for that.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <utility>
#include <string>
#include <vector>

#include "../../include/diffuser.h"

namespace dfs {

constexpr int kHeadDim = 64;          // d = d_h = d_v, fixed by the kernels
constexpr int32_t kMaxRandPerRow = 1024;
constexpr int32_t kMaxWindowBlocks = 63;
constexpr int32_t kMaxRandBlocks = 64;
constexpr int64_t kMaxNnz = int64_t(1) << 40;
constexpr int32_t kBandMaxGlobals = 32;   // the band path handles at most this many globals

enum GraphKind { kTokenGraph = 0, kBlockGraph = 1 };

// Geometry of the band path's decomposed weight layout (token graphs).
struct BandPlan {
    int64_t n;          // sequence length
    int32_t r;          // window radius
    int32_t causal;     // 1: causal graph (window [i - r, i]; a row reads globals g <= i only)
    int32_t r64;        // the radius rounded up to a multiple of 64 (start of a tile's key chunks)
    int32_t g, g_pad;   // number of globals, padded to a multiple of 4
    int32_t g16;        // g rounded up to 16 (the K of the out-of-window globals' MMA), 0 if g = 0
    int32_t tiles;      // 128-row tiles per unit
    int32_t chunks;     // 64-key chunks per tile (even)
    size_t band_unit;   // bytes of one unit's band weights (tiles x chunks x 32 KB)
};

// Byte offsets of the band path's workspace regions.
struct BandLayout {
    size_t a_band, a_gc, a_gcimg, a_x, a_gr, a_gimg;
    size_t z[2];        // hop state Z_k, [units][n][hi 64 | lo 64] bf16, ping-pong
    size_t zf[2];       // the same Z_k as fp32 rows [units][n][64] (row gathers)
    size_t psum;        // sparse partial of the rows not in G, [units][n][64] fp32
    size_t gpart, inv_l, m_sparse, gstat, total;
};

// Byte offsets of the backward pass's workspace regions (fp32 throughout).
struct BwdLayout {
    size_t a, da;       // weights A and their gradient dA (then dS), [units][nnz]
    size_t dv;          // the dV accumulator, [units][n][64]
    size_t g[2];        // G_k, the gradient reaching Z_k, ping-pong, [units][n][64]
    size_t p;           // the band kernels' window sums, [units][n][64]
    size_t at;          // the weights of the edges outside the keys' window runs in key order,
                        // [units][nrest] (token graphs with a plain window; nrest = 0 otherwise)
    int64_t nrest;
    size_t z, z_stride; // Z_1 .. Z_{K-1}, each [units][n][64]
    size_t total;
};

}  // namespace dfs

namespace dfs {
struct ReplayCache;
struct BlockDeals;
struct BandDeals;
}

struct diffuser_graph {
    int kind = dfs::kTokenGraph;
    int device = 0;
    int64_t n = 0;
    int64_t nnz = 0;
    // token graph parameters
    int32_t r = 0, n_globals = 0, rand_per_row = 0;
    bool causal = false;              // token graph cut to j <= i
    int32_t dilation = 1;             // token graph: spacing of the window's positions
    int32_t uniform = 0;              // token graph: extras on a uniform grid, not random draws
    // block graph parameters
    int32_t block = 0, window_blocks = 0, rand_blocks = 0, global_blocks = 0;
    uint64_t seed = 0;
    // device CSR
    int64_t* d_row_ptr = nullptr;
    int32_t* d_col = nullptr;
    int32_t* d_globals = nullptr;     // token graph: sorted global positions
    uint8_t* d_is_global = nullptr;   // token graph: per-position flag
    int32_t* d_gslot = nullptr;       // token graph: slot of a position in G, or -1
    // token graph, decomposed layout: random edges outside the window and G
    int64_t nx = 0;                   // number of such "extra" edges
    int64_t* d_x_ptr = nullptr;       // [n+1]
    int32_t* d_x_col = nullptr;       // [nx], ascending within a row
    // transposed graph (the backward pass): incoming edges of each key, rows ascending
    int64_t* d_t_ptr = nullptr;       // [n+1]
    int32_t* d_t_row = nullptr;       // [nnz] row i of each incoming edge
    int64_t* d_t_edge = nullptr;      // [nnz] its CSR edge id
    int64_t* d_wp0 = nullptr;         // [n] token graph, plain window: CSR position of row i's window run
    int64_t* d_tw0 = nullptr;         // [n] ... and transposed-list position of key j's (null otherwise)
    int64_t* d_trest = nullptr;       // [n+1] ... and where key j's incoming edges outside its run start
                                      //   in the key-ordered weights (null otherwise)
    int32_t* d_orders = nullptr;      // [2][n] the backward's row and key orders (heavy ones first)
    int64_t heavy_rows = 0, heavy_keys = 0;
    int32_t* d_bruns = nullptr;       // block graph, 64-token blocks: the backward's key-block runs
    int64_t bruns_blocks = 0;         // their entries (key blocks over all block rows)
    // status block written by kernels: the word (0 = ok) at [0], the device
    // address of h_status at byte 8 (a bounded wait that gives up writes both)
    // block graph with 64-token blocks: each 128-row tile's key blocks, paired into
    // 128-key chunks (block_path.cu)
    int32_t* d_blk_chunks = nullptr;  // [blk_chunks][4]: key blocks kb0, kb1, mask bits, 0
    int32_t* d_blk_tile_ptr = nullptr;   // [blk_tiles + 1]
    int32_t* d_blk_order = nullptr;   // [blk_tiles] tile positions by falling chunk count
    int32_t blk_tiles = 0;
    int64_t blk_chunks = 0;
    std::vector<int32_t> h_blk_tile_ptr, h_blk_order;   // host copies of the two lists above
    dfs::BlockDeals* blk_deals = nullptr;   // per (B H, CTAs): the tiles dealt to the CTAs (block_path.cu)
    dfs::BandDeals* band_deals = nullptr;   // the same for the band path's hop kernel (band_hop.cu)
    int* d_status = nullptr;
    int* h_status = nullptr;          // page-locked, mapped host mirror of the word
    dfs::ReplayCache* replay = nullptr;   // captured band-path forwards (see abi.cu)
    // host copy of the CSR
    std::vector<int64_t> h_row_ptr;
    std::vector<int32_t> h_col;
    std::vector<int32_t> h_globals;
};

namespace dfs {

// ---- status plumbing (abi.cu) -------------------------------------------------
int fail(int status, const std::string& msg);
int cuda_fail(cudaError_t err, const char* what);

// DIFFUSER_ERR_DEVICE when a kernel has reported a failure on g since the last
// reset (read from the host mirror of the status word: no synchronization).
int check_status_word(const diffuser_graph* g);

// ---- argument checks and the CSR path's workspace (abi.cu) ------------------
// CSR-path workspace: [A: units*nnz fp32][Z ping: units*n*64 fp32][Z pong: same],
// each region 256-byte aligned.
struct Layout {
    size_t a_off, z0_off, z1_off, total;
};
int plan_layout(const diffuser_graph* g, int64_t B, int64_t H, Layout* L);   // OVERFLOW-checked
int check_shape(const diffuser_graph* g, int64_t B, int64_t H, int32_t d, int32_t dtype);
int check_device(const diffuser_graph* g);
bool aligned16(const void* p);
size_t io_bytes(const diffuser_graph* g, int64_t B, int64_t H, int32_t dtype);
bool overlaps(const void* a, size_t na, const void* b, size_t nb);
struct CsrArgs;
// The hops over weights already in A (CSR order): Z_0 = V, the last hop writes
// out; hops = 0 copies V to out.  The hop state lives in ws at L's offsets.
int run_hops_csr(const diffuser_graph* g, const CsrArgs& a, const float* A, const void* V,
                 int32_t dtype, int32_t hops, float alpha, void* out, char* ws, const Layout& L,
                 cudaStream_t stream);

// ---- launch accounting and profiling (abi.cu) ------------------------------
// Brackets one kernel launch: counts it and, while a profile is open, records
// CUDA events around it on `stream`.
class LaunchScope {
  public:
    LaunchScope(diffuser_kernel_kind kind, cudaStream_t stream);
    ~LaunchScope();
    LaunchScope(const LaunchScope&) = delete;
    LaunchScope& operator=(const LaunchScope&) = delete;

  private:
    int slot_ = -1;
    int capture_slot_ = -1;
    cudaStream_t stream_;
};

// ---- graph construction kernels (graph_build.cu) ---------------------------
int build_token_graph_device(diffuser_graph* g, cudaStream_t stream);
int build_block_graph_device(diffuser_graph* g, cudaStream_t stream);
int build_dilated_graph_device(diffuser_graph* g, cudaStream_t stream);   // dilation > 1

// ---- CSR SIMT path (simt_path.cu) ------------------------------------------
#ifdef __CUDACC__
// Launch with programmatic dependent launch allowed: the kernel may be scheduled
// before the previous kernel on the stream completes, and must call
// ptx::griddep_wait before it touches memory that kernel reads or writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// v[k] of every lane of a full warp is one lane's share of value k (k < 32); on
// return, lane l holds the sum over the 32 lanes of value l.  A butterfly over the
// lane bits: at each of the 5 steps a lane keeps the half of its values whose index
// bit matches its own lane bit and adds its partner's copy of it (16 + 8 + 4 + 2 + 1
// shuffles).  The order of the additions is fixed: repeated calls give identical bits.
__device__ __forceinline__ float warp_transpose_sum32(float (&v)[32], int lane) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int k = 0; k < off; ++k) {
            const float send = upper ? v[k] : v[k + off];
            const float keep = upper ? v[k + off] : v[k];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    return v[0];
}
#endif

struct CsrArgs {
    const int64_t* row_ptr;
    const int32_t* col;
    int64_t n;
    int64_t nnz;
    int64_t units;   // B*H
};

// A[u][e] = masked row softmax of q_i.k_j / sqrt(64), CSR edge order.
int launch_score_csr(const CsrArgs& a, const void* Q, const void* K, int32_t dtype, float* A,
                     cudaStream_t stream);

// One PPR hop over CSR weights:  dst = (1-alpha) * A src + alpha * V.
//   src is the I/O dtype when src_is_io (hop 0 reads V), fp32 otherwise;
//   dst is the I/O dtype when dst_is_io (the last hop writes out), fp32 otherwise.
int launch_hop_csr(const CsrArgs& a, const float* A, const void* src, bool src_is_io,
                   const void* V, void* dst, bool dst_is_io, int32_t dtype, float alpha,
                   cudaStream_t stream);

// ---- backward pass (backward.cu): CSR path, either I/O dtype ----------------
int build_transposed_graph(diffuser_graph* g);   // from the host CSR copy
int plan_backward_layout(const diffuser_graph* g, int64_t units, int32_t hops, BwdLayout* L);
int launch_backward_csr(const diffuser_graph* g, int64_t units, const void* Q, const void* K,
                        const void* V, const void* dOut, int32_t dtype, int32_t hops, float alpha,
                        void* dQ, void* dK, void* dV, char* ws, const BwdLayout& L, bool band,
                        cudaStream_t stream);

// ---- block-sparse path (block_path.cu): block graphs of 64-token blocks, bf16 I/O
struct BlockLayout {
    size_t z[2];        // hop state Z_k, [units][n][hi 64 | lo 64] bf16, ping-pong
    size_t mb2, inv_l;  // per-row max (base-2 scale) and inverse sum, [units][n] fp32
    size_t total;
};
bool block_eligible(const diffuser_graph* g);
int build_block_tiles(diffuser_graph* g);      // from the host CSR copy; no-op for other graphs
void destroy_block_deals(BlockDeals* d);
BandDeals* create_band_deals();                // null on allocation failure (snake order then)
void destroy_band_deals(BandDeals* d);
int plan_block_layout(const diffuser_graph* g, int64_t units, BlockLayout* L);
// the score pass (row max and sum) and the hops; launch_block_forward runs both
int launch_block_scores(const diffuser_graph* g, int64_t units, const void* Q, const void* K, char* ws,
                        const BlockLayout& L, cudaStream_t stream);
int launch_block_hops(const diffuser_graph* g, int64_t units, const void* Q, const void* K,
                      const void* V, int32_t hops, float alpha, void* out, char* ws,
                      const BlockLayout& L, cudaStream_t stream);
int launch_block_forward(const diffuser_graph* g, int64_t units, const void* Q, const void* K,
                         const void* V, int32_t hops, float alpha, void* out, char* ws,
                         const BlockLayout& L, cudaStream_t stream);

// ---- the projections around the module (layer_gemm.cu): tcgen05 GEMMs, bf16 --
int check_layer_shape(int64_t B, int64_t n, int32_t D, int32_t H, int32_t d);
// Q, K, V [B][H][n][64] = per-head projections of X [B][n][D] by Wqkv [3 H 64][D]
int launch_qkv_projection(const void* X, const void* Wqkv, int64_t B, int64_t n, int32_t D, int32_t H,
                          void* Q, void* K, void* V, int* status, cudaStream_t stream);
// Y [B][n][D] = concat_h Z[b][h][i][:] projected by Wo [D][H 64]
int launch_output_projection(const void* Z, const void* Wo, int64_t B, int64_t n, int32_t D, int32_t H,
                             void* Y, int* status, cudaStream_t stream);

// ---- band path (band_score.cu, band_hop.cu): token graphs, bf16 I/O --------
bool band_plan(const diffuser_graph* g, BandPlan* p);   // false: graph not eligible
int plan_band_layout(const diffuser_graph* g, const BandPlan& p, int64_t units, BandLayout* L);
// Scores and softmax statistics.  weights_out: also the band weights as tile
// images and the finished row sums (the attention-weights export).  Without,
// the forward's state: row maxima, the out-of-window globals' weights and
// their part of the row sum in inv_l, the extras' raw scores and the global
// rows' weights; the first hop completes the rest (launch_band_hops follows).
// V (may be null) is only pulled into L2 for the first hop, under the score kernels.
int launch_band_scores(const diffuser_graph* g, const BandPlan& p, int64_t units, const void* Q,
                       const void* K, const void* V, char* ws, const BandLayout& L, bool weights_out,
                       cudaStream_t stream);
int launch_band_hops(const diffuser_graph* g, const BandPlan& p, int64_t units, const void* Q,
                     const void* K, const void* V, int32_t hops, float alpha, void* out, char* ws,
                     const BandLayout& L, cudaStream_t stream);
int launch_band_to_csr(const diffuser_graph* g, const BandPlan& p, int64_t units, char* ws,
                       const BandLayout& L, float* A_out, cudaStream_t stream);

}  // namespace dfs
