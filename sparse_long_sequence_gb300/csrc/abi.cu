// C ABI of libdiffuser: argument checks, graph objects, workspace layout,
// launch sequence, launch accounting and device-time profiling.  Every entry
// point returns a status and never lets a C++ exception out.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "internal.h"

namespace dfs {

namespace {
thread_local std::string g_last_error;

std::atomic<int64_t> g_launches[DIFFUSER_KERNEL_KINDS];
std::atomic<int> g_path{DIFFUSER_PATH_AUTO};

// ---- profiler: events recorded around launches while a profile is open ----
struct ProfileRecord {
    int kind;
    cudaEvent_t start, stop;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfileRecord> g_prof_records;
std::vector<cudaEvent_t> g_event_pool;

// ---- CUDA-graph capture: launches made while a capture context is set are
// counted there (and credited at each replay) instead of in the counters ----
struct CaptureCtx {
    int64_t launches[DIFFUSER_KERNEL_KINDS] = {0};
};
thread_local CaptureCtx* t_capture = nullptr;

cudaEvent_t take_event() {
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool mul_overflows(size_t a, size_t b, size_t* out) {
    if (a != 0 && b > SIZE_MAX / a) return true;
    *out = a * b;
    return false;
}
}  // namespace

int fail(int status, const std::string& msg) {
    g_last_error = msg;
    return status;
}

int cuda_fail(cudaError_t err, const char* what) {
    g_last_error = std::string(what) + ": " + cudaGetErrorString(err);
    return DIFFUSER_ERR_CUDA;
}

LaunchScope::LaunchScope(diffuser_kernel_kind kind, cudaStream_t stream) : stream_(stream) {
    if (t_capture) {
        t_capture->launches[kind] += 1;    // counted at each replay
        capture_slot_ = 0;
        return;
    }
    g_launches[kind].fetch_add(1, std::memory_order_relaxed);
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (!g_prof_on) return;
    cudaEvent_t a = take_event(), b = take_event();
    if (!a || !b) return;
    cudaEventRecord(a, stream);
    g_prof_records.push_back({(int)kind, a, b});
    slot_ = (int)g_prof_records.size() - 1;
}

LaunchScope::~LaunchScope() {
    if (capture_slot_ >= 0) return;
    if (slot_ < 0) return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (slot_ < (int)g_prof_records.size()) cudaEventRecord(g_prof_records[slot_].stop, stream_);
}

// ---- workspace layout ---------------------------------------------------------
int plan_layout(const diffuser_graph* g, int64_t B, int64_t H, Layout* L) {
    size_t units = (size_t)B * (size_t)H;
    size_t a_bytes, z_elems, z_bytes;
    if (mul_overflows(units, (size_t)g->nnz, &a_bytes) || mul_overflows(a_bytes, 4, &a_bytes) ||
        mul_overflows(units, (size_t)g->n * kHeadDim, &z_elems) ||
        mul_overflows(z_elems, 4, &z_bytes))
        return fail(DIFFUSER_ERR_OVERFLOW, "workspace size overflows size_t");
    L->a_off = 0;
    L->z0_off = align_up(a_bytes);
    L->z1_off = L->z0_off + align_up(z_bytes);
    L->total = L->z1_off + align_up(z_bytes);
    return DIFFUSER_OK;
}

int check_shape(const diffuser_graph* g, int64_t B, int64_t H, int32_t d, int32_t dtype) {
    if (!g) return fail(DIFFUSER_ERR_INVALID_ARG, "graph is NULL");
    if (B < 1 || H < 1 || B > (int64_t(1) << 31) || H > (int64_t(1) << 31))
        return fail(DIFFUSER_ERR_INVALID_ARG, "B and H must be >= 1");
    if (d != kHeadDim) return fail(DIFFUSER_ERR_UNSUPPORTED, "head width d must be 64");
    if (dtype != DIFFUSER_DTYPE_FP32 && dtype != DIFFUSER_DTYPE_BF16)
        return fail(DIFFUSER_ERR_UNSUPPORTED, "dtype must be FP32 or BF16");
    return DIFFUSER_OK;
}

int check_status_word(const diffuser_graph* g) {
    const int word = g->h_status ? *reinterpret_cast<const volatile int*>(g->h_status) : 0;
    if (word == 0) return DIFFUSER_OK;
    return fail(DIFFUSER_ERR_DEVICE, "a kernel on this graph reported status " + std::to_string(word) +
                                         " (results since the last reset are invalid; "
                                         "clear it with diffuser_graph_status(reset = 1))");
}

int check_device(const diffuser_graph* g) {
    int dev = -1;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return cuda_fail(err, "cudaGetDevice");
    if (dev != g->device)
        return fail(DIFFUSER_ERR_INVALID_ARG, "the current device is not the graph's device");
    return DIFFUSER_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

size_t io_bytes(const diffuser_graph* g, int64_t B, int64_t H, int32_t dtype) {
    return (size_t)B * H * g->n * kHeadDim * (dtype == DIFFUSER_DTYPE_BF16 ? 2 : 4);
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

int check_workspace_bytes(size_t need, void* ws, size_t ws_bytes) {
    if (!ws) return fail(DIFFUSER_ERR_WORKSPACE, "workspace is NULL");
    if (reinterpret_cast<uintptr_t>(ws) % kAlign)
        return fail(DIFFUSER_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if (ws_bytes < need)
        return fail(DIFFUSER_ERR_WORKSPACE, "workspace too small: need " +
                                                std::to_string(need) + " bytes");
    return DIFFUSER_OK;
}

int check_workspace(const Layout& L, void* ws, size_t ws_bytes) {
    return check_workspace_bytes(L.total, ws, ws_bytes);
}

// The band path (tensor-core window tiles) serves token graphs with bf16 I/O;
// everything else runs the CSR SIMT path.
bool use_band(const diffuser_graph* g, int32_t dtype, BandPlan* p) {
    if (g_path.load() == DIFFUSER_PATH_CSR) return false;
    if (dtype != DIFFUSER_DTYPE_BF16) return false;
    return band_plan(g, p);
}

// Workspace bytes: enough for the CSR layout and, where the graph and dtype
// are eligible, the band layout, so that the size does not depend on the
// selected path.
int workspace_need(const diffuser_graph* g, int64_t B, int64_t H, int32_t dtype, size_t* need) {
    Layout L;
    int st = plan_layout(g, B, H, &L);
    if (st) return st;
    *need = L.total;
    BandPlan bp;
    if (dtype == DIFFUSER_DTYPE_BF16 && band_plan(g, &bp)) {
        BandLayout BL;
        if ((st = plan_band_layout(g, bp, B * H, &BL))) return st;
        if (BL.total > *need) *need = BL.total;
    }
    if (dtype == DIFFUSER_DTYPE_BF16 && block_eligible(g)) {
        BlockLayout KL;
        if ((st = plan_block_layout(g, B * H, &KL))) return st;
        if (KL.total > *need) *need = KL.total;
    }
    return DIFFUSER_OK;
}

// The block-sparse tensor-core path serves block graphs of 64-token blocks with
// bf16 I/O (the general CSR path runs everything else).
bool use_block(const diffuser_graph* g, int32_t dtype) {
    if (g_path.load() == DIFFUSER_PATH_CSR) return false;
    return dtype == DIFFUSER_DTYPE_BF16 && block_eligible(g);
}

// The hops over weights already in A (CSR order): Z_0 = V, last hop -> out.
int run_hops_csr(const diffuser_graph* g, const CsrArgs& a, const float* A, const void* V,
                 int32_t dtype, int32_t hops, float alpha, void* out, char* ws, const Layout& L,
                 cudaStream_t stream) {
    if (hops == 0) {
        if (out == V) return DIFFUSER_OK;
        size_t bytes = io_bytes(g, a.units, 1, dtype);
        cudaError_t err = cudaMemcpyAsync(out, V, bytes, cudaMemcpyDeviceToDevice, stream);
        return err == cudaSuccess ? DIFFUSER_OK : cuda_fail(err, "copying V to out (hops = 0)");
    }
    float* zbuf[2] = {reinterpret_cast<float*>(ws + L.z0_off),
                      reinterpret_cast<float*>(ws + L.z1_off)};
    for (int32_t k = 0; k < hops; ++k) {
        const bool first = (k == 0), last = (k == hops - 1);
        const void* src = first ? V : zbuf[(k - 1) & 1];
        void* dst = last ? out : zbuf[k & 1];
        int st = launch_hop_csr(a, A, src, first, V, dst, last, dtype, alpha, stream);
        if (st != DIFFUSER_OK) return st;
    }
    return DIFFUSER_OK;
}

// ---- replay of captured band-path forwards ---------------------------------
// The second forward with the same pointers, shape, hops, alpha and path is
// captured on an internal stream into a CUDA graph; later ones replay it on
// the caller's stream (launch counts are credited per replay).  While a
// profile is open, and while the caller's stream is capturing its own graph,
// forwards launch their kernels directly.
// marks the keys of host-buffer forwards (whose replays include the copies)
constexpr int kHostPathKey = 1 << 8;

struct ReplayKey {
    const void *Q, *K, *V, *out, *ws;
    size_t ws_bytes;
    int64_t B, H;
    int32_t dtype, hops;
    float alpha;
    int path;
    bool operator==(const ReplayKey& o) const {
        return Q == o.Q && K == o.K && V == o.V && out == o.out && ws == o.ws && ws_bytes == o.ws_bytes &&
               B == o.B && H == o.H && dtype == o.dtype && hops == o.hops &&
               std::memcmp(&alpha, &o.alpha, sizeof(float)) == 0 && path == o.path;
    }
};

struct ReplayEntry {
    ReplayKey key{};
    uint64_t stamp = 0;
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    int64_t launches[DIFFUSER_KERNEL_KINDS] = {0};
};

struct ReplayCache {
    std::mutex mu;
    std::vector<ReplayEntry> entries;
    uint64_t clock = 0;
};

namespace {
constexpr size_t kReplayEntries = 4;
constexpr int kMaxReplayDevices = 64;
std::mutex g_capture_mu;
cudaStream_t g_capture_stream[kMaxReplayDevices] = {nullptr};

void destroy_entry(ReplayEntry& e) {
    if (e.exec) cudaGraphExecDestroy(e.exec);
    if (e.graph) cudaGraphDestroy(e.graph);
    e = ReplayEntry{};
}

cudaStream_t capture_stream(int dev) {
    if (dev < 0 || dev >= kMaxReplayDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_capture_mu);
    if (!g_capture_stream[dev] &&
        cudaStreamCreateWithFlags(&g_capture_stream[dev], cudaStreamNonBlocking) != cudaSuccess)
        g_capture_stream[dev] = nullptr;
    return g_capture_stream[dev];
}

int replay(ReplayEntry& e, cudaStream_t stream) {
    for (int k = 0; k < DIFFUSER_KERNEL_KINDS; ++k)
        g_launches[k].fetch_add(e.launches[k], std::memory_order_relaxed);
    cudaError_t err = cudaGraphLaunch(e.exec, stream);
    return err == cudaSuccess ? DIFFUSER_OK : cuda_fail(err, "cudaGraphLaunch(forward)");
}

// Captures `launch` (which enqueues the forward on the stream it is given) into
// e; false when capture or instantiation is not possible (nothing is kept).
template <class Launch>
bool capture(ReplayEntry& e, int dev, Launch&& launch) {
    cudaStream_t cs = capture_stream(dev);
    if (!cs) return false;
    CaptureCtx ctx;
    if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return false;
    t_capture = &ctx;
    const int st = launch(cs);
    t_capture = nullptr;
    cudaGraph_t graph = nullptr;
    const cudaError_t cerr = cudaStreamEndCapture(cs, &graph);
    auto drop = [&]() {
        if (graph) cudaGraphDestroy(graph);
        cudaGetLastError();
        return false;
    };
    if (st != DIFFUSER_OK || cerr != cudaSuccess || !graph) return drop();
    cudaGraphExec_t exec = nullptr;
    if (cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) return drop();
    e.graph = graph;
    e.exec = exec;
    for (int k = 0; k < DIFFUSER_KERNEL_KINDS; ++k) e.launches[k] = ctx.launches[k];
    return true;
}
}  // namespace

void destroy_replay_cache(ReplayCache* c) {
    if (!c) return;
    for (auto& e : c->entries) destroy_entry(e);
    delete c;
}

// The band-path forward through the replay cache of g.
template <class Launch>
int band_forward(const diffuser_graph* g, const ReplayKey& key, cudaStream_t stream, Launch&& launch) {
    ReplayCache* c = g->replay;
    // a caller capturing its own graph on this stream records the kernels themselves
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (!c || cudaStreamIsCapturing(stream, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone)
        return launch(stream);
    bool profiling;
    {
        std::lock_guard<std::mutex> lk(g_prof_mu);
        profiling = g_prof_on;
    }
    if (profiling) return launch(stream);          // per-kernel events need direct launches
    std::lock_guard<std::mutex> lk(c->mu);
    ++c->clock;
    for (auto& e : c->entries) {
        if (!(e.key == key)) continue;
        e.stamp = c->clock;
        if (e.exec) return replay(e, stream);
        // seen once before: capture this time (launches fall back to direct on failure)
        if (capture(e, g->device, launch)) return replay(e, stream);
        return launch(stream);
    }
    // first sighting: run directly and remember the key
    if (c->entries.size() >= kReplayEntries) {
        size_t old = 0;
        for (size_t k = 1; k < c->entries.size(); ++k)
            if (c->entries[k].stamp < c->entries[old].stamp) old = k;
        destroy_entry(c->entries[old]);
        c->entries.erase(c->entries.begin() + old);
    }
    ReplayEntry e;
    e.key = key;
    e.stamp = c->clock;
    c->entries.push_back(std::move(e));
    return launch(stream);
}

int forward_device(const void* Q, const void* K, const void* V, int32_t dtype, int64_t B,
                   int64_t H, int32_t d, const diffuser_graph* g, int32_t hops, float alpha,
                   void* out, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    int st = check_shape(g, B, H, d, dtype);
    if (st) return st;
    if (!Q || !K || !V || !out) return fail(DIFFUSER_ERR_INVALID_ARG, "a tensor pointer is NULL");
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(out))
        return fail(DIFFUSER_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
    if (hops < 0) return fail(DIFFUSER_ERR_INVALID_ARG, "hops must be >= 0");
    if (!(alpha >= 0.f && alpha <= 1.f))
        return fail(DIFFUSER_ERR_INVALID_ARG, "alpha must lie in [0, 1]");
    const size_t bytes = io_bytes(g, B, H, dtype);
    if (overlaps(out, bytes, Q, bytes) || overlaps(out, bytes, K, bytes))
        return fail(DIFFUSER_ERR_INVALID_ARG, "out overlaps Q or K");
    if (hops > 0 && overlaps(out, bytes, V, bytes))
        return fail(DIFFUSER_ERR_INVALID_ARG, "out may alias V only when hops == 0");
    size_t need = 0;
    if ((st = workspace_need(g, B, H, dtype, &need))) return st;
    if ((st = check_workspace_bytes(need, workspace, workspace_bytes))) return st;
    if ((st = check_device(g))) return st;
    if ((st = check_status_word(g))) return st;

    char* ws = static_cast<char*>(workspace);
    CsrArgs a{g->d_row_ptr, g->d_col, g->n, g->nnz, B * H};
    Layout L;
    if ((st = plan_layout(g, B, H, &L))) return st;
    if (hops == 0) return run_hops_csr(g, a, nullptr, V, dtype, 0, alpha, out, ws, L, stream);
    BandPlan bp;
    if (use_band(g, dtype, &bp)) {
        BandLayout BL;
        if ((st = plan_band_layout(g, bp, B * H, &BL))) return st;
        const ReplayKey key{Q, K, V, out, workspace, workspace_bytes, B, H, dtype, hops, alpha, g_path.load()};
        return band_forward(g, key, stream, [&](cudaStream_t s) {
            int r = launch_band_scores(g, bp, B * H, Q, K, V, ws, BL, false, s);
            if (!r) r = launch_band_hops(g, bp, B * H, Q, K, V, hops, alpha, out, ws, BL, s);
            return r;
        });
    }
    if (use_block(g, dtype)) {
        BlockLayout KL;
        if ((st = plan_block_layout(g, B * H, &KL))) return st;
        const ReplayKey key{Q, K, V, out, workspace, workspace_bytes, B, H, dtype, hops, alpha, g_path.load()};
        return band_forward(g, key, stream, [&](cudaStream_t s) {
            return launch_block_forward(g, B * H, Q, K, V, hops, alpha, out, ws, KL, s);
        });
    }
    float* A = reinterpret_cast<float*>(ws + L.a_off);
    if ((st = launch_score_csr(a, Q, K, dtype, A, stream))) return st;
    return run_hops_csr(g, a, A, V, dtype, hops, alpha, out, ws, L, stream);
}

// The side stream of the host-buffer forward that uploads V (one per device,
// created on first use and kept for the life of the process).
int upload_stream(int device, cudaStream_t* s) {
    static std::mutex mu;
    static cudaStream_t pool[16] = {};
    if (device < 0 || device >= 16) return fail(DIFFUSER_ERR_CUDA, "device index out of range");
    std::lock_guard<std::mutex> lock(mu);
    if (!pool[device]) {
        cudaError_t err = cudaStreamCreateWithFlags(&pool[device], cudaStreamNonBlocking);
        if (err != cudaSuccess) {
            pool[device] = nullptr;
            return cuda_fail(err, "upload stream");
        }
    }
    *s = pool[device];
    return DIFFUSER_OK;
}

// The device address of a pinned host buffer mapped into this device's address
// space, or nullptr.
void* mapped_host(void* p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

// Forward from host buffers on the band or block path: Q and K upload side by
// side (on the forward's stream and a side stream) and the score kernels start as
// soon as both are in; V then uploads on the side stream under the score kernels,
// and the hops wait for it.  When `out` is pinned and mapped, the last hop writes it
// in place (no download after the kernels); else it lands in dO and is copied back.
// With all four host buffers pinned, repeated calls replay the whole sequence
// (copies and kernels) as one captured graph, like the device-buffer forward.
// scores(dQ, dK, s) and run_hops(dQ, dK, dV, out, s) enqueue the path's kernels.
template <class Scores, class Hops>
int forward_host_overlapped(const void* Q, const void* K, const void* V, int64_t B, int64_t H,
                            const diffuser_graph* g, int32_t hops, float alpha, void* out, char* dQ,
                            char* dK, char* dV, char* dO, char* ws, size_t ws_bytes, size_t bytes,
                            cudaStream_t stream, Scores&& scores, Hops&& run_hops) {
    size_t need = 0;
    int st = workspace_need(g, B, H, DIFFUSER_DTYPE_BF16, &need);
    if (st) return st;
    if ((st = check_workspace_bytes(need, ws, ws_bytes))) return st;
    cudaStream_t up;
    if ((st = upload_stream(g->device, &up))) return st;
    void* out_dev = mapped_host(out);
    if (out_dev && !aligned16(out_dev)) out_dev = nullptr;
    const bool pinned = out_dev && mapped_host(const_cast<void*>(Q)) && mapped_host(const_cast<void*>(K)) &&
                        mapped_host(const_cast<void*>(V));
    cudaEvent_t ev[4] = {};
    cudaError_t err = cudaSuccess;
    for (int i = 0; i < 4 && err == cudaSuccess; ++i) err = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
    // ev[0]: entry on the stream (the uploads follow earlier work there); ev[1]: K is
    // in; ev[2]: Q and K are in; ev[3]: V is in.  V uploads after Q and K so that it
    // does not share the link with the uploads the score kernels wait for.
    auto enqueue = [&](cudaStream_t s) -> int {
        cudaError_t e = cudaEventRecord(ev[0], s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(up, ev[0], 0);
        if (e == cudaSuccess) e = cudaMemcpyAsync(dQ, Q, bytes, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaMemcpyAsync(dK, K, bytes, cudaMemcpyHostToDevice, up);
        if (e == cudaSuccess) e = cudaEventRecord(ev[1], up);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ev[1], 0);
        if (e == cudaSuccess) e = cudaEventRecord(ev[2], s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(up, ev[2], 0);
        if (e == cudaSuccess) e = cudaMemcpyAsync(dV, V, bytes, cudaMemcpyHostToDevice, up);
        if (e == cudaSuccess) e = cudaEventRecord(ev[3], up);
        if (e != cudaSuccess) return cuda_fail(e, "host-buffer forward (uploads)");
        int r = scores(dQ, dK, s);
        if (r) return r;
        if ((e = cudaStreamWaitEvent(s, ev[3], 0)) != cudaSuccess) return cuda_fail(e, "host-buffer forward");
        r = run_hops(dQ, dK, dV, out_dev ? out_dev : static_cast<void*>(dO), s);
        if (r) return r;
        if (!out_dev && (e = cudaMemcpyAsync(out, dO, bytes, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
            return cuda_fail(e, "device-to-host copy");
        return DIFFUSER_OK;
    };
    if (err != cudaSuccess) {
        st = cuda_fail(err, "host-buffer forward (events)");
    } else if (pinned) {
        const ReplayKey key{Q, K, V, out, ws, ws_bytes, B, H, DIFFUSER_DTYPE_BF16, hops, alpha,
                            g_path.load() | kHostPathKey};
        st = band_forward(g, key, stream, enqueue);
    } else {
        st = enqueue(stream);
    }
    for (int i = 0; i < 4; ++i)
        if (ev[i]) cudaEventDestroy(ev[i]);      // released once their work completes
    return st;
}

constexpr size_t kStatusBlockBytes = 16;

int new_graph(diffuser_graph** out, diffuser_graph** g) {
    if (!out) return fail(DIFFUSER_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    *g = new (std::nothrow) diffuser_graph();
    if (!*g) return fail(DIFFUSER_ERR_ALLOC, "host allocation failed");
    (*g)->replay = new (std::nothrow) ReplayCache();   // without it, forwards launch directly
    (*g)->band_deals = dfs::create_band_deals();        // without it, the band path deals in snake order
    // status block: word, padding, then the device address of the host mirror
    cudaError_t err = cudaGetDevice(&(*g)->device);
    int* mirror_dev = nullptr;
    if (err == cudaSuccess) err = cudaMalloc(&(*g)->d_status, kStatusBlockBytes);
    if (err == cudaSuccess) err = cudaHostAlloc(&(*g)->h_status, sizeof(int), cudaHostAllocMapped);
    if (err == cudaSuccess) {
        *(*g)->h_status = 0;
        err = cudaHostGetDevicePointer(&mirror_dev, (*g)->h_status, 0);
    }
    if (err == cudaSuccess) {
        unsigned char block[kStatusBlockBytes] = {0};
        std::memcpy(block + 8, &mirror_dev, sizeof(mirror_dev));
        err = cudaMemcpy((*g)->d_status, block, kStatusBlockBytes, cudaMemcpyHostToDevice);
    }
    if (err != cudaSuccess) {
        cudaFree((*g)->d_status);
        if ((*g)->h_status) cudaFreeHost((*g)->h_status);
        delete (*g)->replay;
        delete *g;
        *g = nullptr;
        return cuda_fail(err, "graph set-up");
    }
    return DIFFUSER_OK;
}

int finish_graph(int status, diffuser_graph* g, diffuser_graph** out) {
    if (status != DIFFUSER_OK) {
        diffuser_graph_free(g);
        return status;
    }
    *out = g;
    return DIFFUSER_OK;
}

}  // namespace dfs

using namespace dfs;

extern "C" {

const char* diffuser_status_string(int status) {
    switch (status) {
        case DIFFUSER_OK: return "ok";
        case DIFFUSER_ERR_INVALID_ARG: return "invalid argument";
        case DIFFUSER_ERR_UNSUPPORTED: return "unsupported dtype, head width or option";
        case DIFFUSER_ERR_OVERFLOW: return "size overflows its index type";
        case DIFFUSER_ERR_ALLOC: return "allocation failed";
        case DIFFUSER_ERR_CUDA: return "CUDA runtime error";
        case DIFFUSER_ERR_DEVICE: return "a kernel reported an error";
        case DIFFUSER_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        default: return "unknown status";
    }
}

const char* diffuser_last_error(void) { return g_last_error.c_str(); }

int diffuser_version(void) { return 100; }

namespace {

int build_token_graph(int64_t n, int32_t r, int32_t dilation, int32_t n_globals,
                      const int32_t* global_idx, int32_t rand_per_row, uint64_t seed, bool causal,
                      diffuser_graph** out, bool uniform = false) {
    try {
        if (n < 1 || n > INT32_MAX) return fail(DIFFUSER_ERR_INVALID_ARG, "n out of range");
        if (r < 0) return fail(DIFFUSER_ERR_INVALID_ARG, "r must be >= 0");
        if (dilation < 1) return fail(DIFFUSER_ERR_INVALID_ARG, "dilation must be >= 1");
        if (n_globals < 0 || n_globals > n)
            return fail(DIFFUSER_ERR_INVALID_ARG, "n_globals out of range");
        if (rand_per_row < 0 || rand_per_row > kMaxRandPerRow)
            return fail(DIFFUSER_ERR_INVALID_ARG, "rand_per_row must lie in [0, 1024]");
        std::vector<int32_t> G(n_globals);
        for (int32_t t = 0; t < n_globals; ++t) {
            G[t] = global_idx ? global_idx[t] : t;
            if (G[t] < 0 || G[t] >= n || (t > 0 && G[t] <= G[t - 1]))
                return fail(DIFFUSER_ERR_INVALID_ARG,
                            "global positions must be strictly increasing in [0, n)");
        }
        // the CSR must stay addressable: a crude upper bound on nnz
        const double bound = (double)n * ((double)n_globals + 2.0 * r + 1 + rand_per_row) +
                             (double)n_globals * n;
        if (bound > (double)kMaxNnz * 4)
            return fail(DIFFUSER_ERR_OVERFLOW, "graph too large");
        diffuser_graph* g = nullptr;
        int st = new_graph(out, &g);
        if (st) return st;
        g->kind = kTokenGraph;
        g->n = n;
        g->r = r;
        g->n_globals = n_globals;
        g->rand_per_row = rand_per_row;
        g->causal = causal;
        g->dilation = dilation;
        g->uniform = uniform ? 1 : 0;
        g->seed = seed;
        g->h_globals = std::move(G);
        st = dilation > 1 ? build_dilated_graph_device(g, nullptr) : build_token_graph_device(g, nullptr);
        return finish_graph(st, g, out);
    } catch (const std::bad_alloc&) {
        return fail(DIFFUSER_ERR_ALLOC, "host allocation failed");
    } catch (...) {
        return fail(DIFFUSER_ERR_INVALID_ARG, "unexpected exception");
    }
}

}  // namespace

int diffuser_build_graph(int64_t n, int32_t r, int32_t n_globals, const int32_t* global_idx,
                         int32_t rand_per_row, uint64_t seed, diffuser_graph** out) {
    return build_token_graph(n, r, 1, n_globals, global_idx, rand_per_row, seed, false, out);
}

int diffuser_build_causal_graph(int64_t n, int32_t r, int32_t n_globals,
                                const int32_t* global_idx, int32_t rand_per_row, uint64_t seed,
                                diffuser_graph** out) {
    return build_token_graph(n, r, 1, n_globals, global_idx, rand_per_row, seed, true, out);
}

int diffuser_build_dilated_graph(int64_t n, int32_t r, int32_t dilation, int32_t n_globals,
                                 const int32_t* global_idx, int32_t rand_per_row, uint64_t seed,
                                 int32_t causal, diffuser_graph** out) {
    return build_token_graph(n, r, dilation, n_globals, global_idx, rand_per_row, seed,
                             causal != 0, out);
}

int diffuser_build_uniform_graph(int64_t n, int32_t r, int32_t n_globals, const int32_t* global_idx,
                                 int32_t positions_per_row, int32_t causal, diffuser_graph** out) {
    return build_token_graph(n, r, 1, n_globals, global_idx, positions_per_row, 0, causal != 0, out,
                             true);
}

int diffuser_build_block_graph(int64_t n, int32_t block, int32_t window_blocks,
                               int32_t rand_blocks, int32_t global_blocks, uint64_t seed,
                               diffuser_graph** out) {
    try {
        if (n < 1 || n > INT32_MAX) return fail(DIFFUSER_ERR_INVALID_ARG, "n out of range");
        if (block < 1) return fail(DIFFUSER_ERR_INVALID_ARG, "block must be >= 1");
        if (window_blocks < 1 || window_blocks > kMaxWindowBlocks || window_blocks % 2 == 0)
            return fail(DIFFUSER_ERR_INVALID_ARG, "window_blocks must be odd, 1..63");
        if (rand_blocks < 0 || rand_blocks > kMaxRandBlocks)
            return fail(DIFFUSER_ERR_INVALID_ARG, "rand_blocks must lie in [0, 64]");
        const int64_t nb = (n + block - 1) / block;
        if (global_blocks < 0 || global_blocks > nb)
            return fail(DIFFUSER_ERR_INVALID_ARG, "global_blocks must lie in [0, ceil(n/block)]");
        diffuser_graph* g = nullptr;
        int st = new_graph(out, &g);
        if (st) return st;
        g->kind = kBlockGraph;
        g->n = n;
        g->block = block;
        g->window_blocks = window_blocks;
        g->rand_blocks = rand_blocks;
        g->global_blocks = global_blocks;
        g->seed = seed;
        st = build_block_graph_device(g, nullptr);
        if (st == DIFFUSER_OK) st = build_block_tiles(g);
        return finish_graph(st, g, out);
    } catch (const std::bad_alloc&) {
        return fail(DIFFUSER_ERR_ALLOC, "host allocation failed");
    } catch (...) {
        return fail(DIFFUSER_ERR_INVALID_ARG, "unexpected exception");
    }
}

int diffuser_graph_info(const diffuser_graph* g, int64_t* n, int64_t* nnz) {
    if (!g) return fail(DIFFUSER_ERR_INVALID_ARG, "graph is NULL");
    if (n) *n = g->n;
    if (nnz) *nnz = g->nnz;
    return DIFFUSER_OK;
}

int diffuser_graph_copy_csr(const diffuser_graph* g, int64_t* row_ptr, int32_t* col_idx) {
    if (!g || !row_ptr || !col_idx) return fail(DIFFUSER_ERR_INVALID_ARG, "NULL argument");
    std::memcpy(row_ptr, g->h_row_ptr.data(), sizeof(int64_t) * (g->n + 1));
    std::memcpy(col_idx, g->h_col.data(), sizeof(int32_t) * g->nnz);
    return DIFFUSER_OK;
}

void diffuser_graph_free(diffuser_graph* g) {
    if (!g) return;
    cudaFree(g->d_row_ptr);
    cudaFree(g->d_col);
    cudaFree(g->d_globals);
    cudaFree(g->d_is_global);
    cudaFree(g->d_gslot);
    cudaFree(g->d_x_ptr);
    cudaFree(g->d_x_col);
    cudaFree(g->d_t_ptr);
    cudaFree(g->d_t_row);
    cudaFree(g->d_t_edge);
    cudaFree(g->d_wp0);
    cudaFree(g->d_tw0);
    cudaFree(g->d_trest);
    cudaFree(g->d_orders);
    cudaFree(g->d_bruns);
    cudaFree(g->d_blk_chunks);
    cudaFree(g->d_blk_tile_ptr);
    cudaFree(g->d_blk_order);
    dfs::destroy_block_deals(g->blk_deals);
    dfs::destroy_band_deals(g->band_deals);
    cudaFree(g->d_status);
    if (g->h_status) cudaFreeHost(g->h_status);
    dfs::destroy_replay_cache(g->replay);
    delete g;
}

int diffuser_workspace_size(const diffuser_graph* g, int64_t B, int64_t H, int32_t d,
                            int32_t dtype, size_t* bytes) {
    int st = check_shape(g, B, H, d, dtype);
    if (st) return st;
    if (!bytes) return fail(DIFFUSER_ERR_INVALID_ARG, "bytes is NULL");
    return workspace_need(g, B, H, dtype, bytes);
}

int diffuser_forward(const void* Q, const void* K, const void* V, int32_t dtype, int64_t B,
                     int64_t H, int32_t d, const diffuser_graph* g, int32_t hops, float alpha,
                     void* out, void* workspace, size_t workspace_bytes, diffuser_stream stream) {
    try {
        return forward_device(Q, K, V, dtype, B, H, d, g, hops, alpha, out, workspace,
                              workspace_bytes, stream);
    } catch (...) {
        return fail(DIFFUSER_ERR_ALLOC, "unexpected exception");
    }
}

int diffuser_backward_workspace_size(const diffuser_graph* g, int64_t B, int64_t H, int32_t d,
                                     int32_t dtype, int32_t hops, size_t* bytes) {
    int st = check_shape(g, B, H, d, dtype);
    if (st) return st;
    if (!bytes) return fail(DIFFUSER_ERR_INVALID_ARG, "bytes is NULL");
    if (hops < 0) return fail(DIFFUSER_ERR_INVALID_ARG, "hops must be >= 0");
    BwdLayout L;
    if ((st = plan_backward_layout(g, B * H, hops, &L))) return st;
    *bytes = L.total;
    return DIFFUSER_OK;
}

int diffuser_backward(const void* Q, const void* K, const void* V, const void* dOut, int32_t dtype,
                      int64_t B, int64_t H, int32_t d, const diffuser_graph* g, int32_t hops,
                      float alpha, void* dQ, void* dK, void* dV, void* workspace,
                      size_t workspace_bytes, diffuser_stream stream) {
    try {
        int st = check_shape(g, B, H, d, dtype);
        if (st) return st;
        if (!Q || !K || !V || !dOut || !dQ || !dK || !dV)
            return fail(DIFFUSER_ERR_INVALID_ARG, "a tensor pointer is NULL");
        if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(dOut) || !aligned16(dQ) ||
            !aligned16(dK) || !aligned16(dV))
            return fail(DIFFUSER_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
        if (hops < 0) return fail(DIFFUSER_ERR_INVALID_ARG, "hops must be >= 0");
        if (!(alpha >= 0.f && alpha <= 1.f))
            return fail(DIFFUSER_ERR_INVALID_ARG, "alpha must lie in [0, 1]");
        const size_t bytes = io_bytes(g, B, H, dtype);
        const void* in[4] = {Q, K, V, dOut};
        void* grads[3] = {dQ, dK, dV};
        for (int x = 0; x < 3; ++x) {
            for (int y = 0; y < 4; ++y)
                if (overlaps(grads[x], bytes, in[y], bytes))
                    return fail(DIFFUSER_ERR_INVALID_ARG, "a gradient overlaps an input");
            for (int y = x + 1; y < 3; ++y)
                if (overlaps(grads[x], bytes, grads[y], bytes))
                    return fail(DIFFUSER_ERR_INVALID_ARG, "the gradients overlap");
        }
        BwdLayout L;
        if ((st = plan_backward_layout(g, B * H, hops, &L))) return st;
        if ((st = check_workspace_bytes(L.total, workspace, workspace_bytes))) return st;
        if ((st = check_device(g))) return st;
        if ((st = check_status_word(g))) return st;
        {
            // the transposed graph, built by the first backward on this graph; the
            // graph stays logically immutable (the lock orders the one-time build)
            static std::mutex mu;
            std::lock_guard<std::mutex> lock(mu);
            if (!g->d_t_ptr && (st = build_transposed_graph(const_cast<diffuser_graph*>(g)))) return st;
        }
        return launch_backward_csr(g, B * H, Q, K, V, dOut, dtype, hops, alpha, dQ, dK, dV,
                                   static_cast<char*>(workspace), L,
                                   g_path.load() != DIFFUSER_PATH_CSR,
                                   static_cast<cudaStream_t>(stream));
    } catch (...) {
        return fail(DIFFUSER_ERR_ALLOC, "unexpected exception");
    }
}

namespace {

// The per-head forward's workspace: device staging for one head's Q, K, V and
// out slices when B > 1 (a head's [B][n][d] slice is strided in BHSD), then the
// largest per-head forward workspace for B units.
int per_head_need(const diffuser_graph* const* graphs, int64_t B, int64_t H, int32_t d,
                  int32_t dtype, size_t* staging, size_t* need) {
    if (!graphs) return fail(DIFFUSER_ERR_INVALID_ARG, "graphs is NULL");
    if (H < 1) return fail(DIFFUSER_ERR_INVALID_ARG, "B and H must be >= 1");   // before graphs[0] is read
    int st = check_shape(graphs[0], B, H, d, dtype);
    if (st) return st;
    size_t fwd = 0;
    for (int64_t h = 0; h < H; ++h) {
        const diffuser_graph* g = graphs[h];
        if (!g) return fail(DIFFUSER_ERR_INVALID_ARG, "a head's graph is NULL");
        if (g->n != graphs[0]->n) return fail(DIFFUSER_ERR_INVALID_ARG, "the heads' graphs differ in n");
        if (g->device != graphs[0]->device)
            return fail(DIFFUSER_ERR_INVALID_ARG, "the heads' graphs live on different devices");
        size_t one = 0;
        if ((st = workspace_need(g, B, 1, dtype, &one))) return st;
        if (one > fwd) fwd = one;
    }
    *staging = B > 1 ? 4 * align_up(io_bytes(graphs[0], B, 1, dtype)) : 0;
    *need = *staging + fwd;
    return DIFFUSER_OK;
}

}  // namespace

int diffuser_per_head_workspace_size(const diffuser_graph* const* graphs, int64_t B, int64_t H,
                                     int32_t d, int32_t dtype, size_t* bytes) {
    try {
        if (!bytes) return fail(DIFFUSER_ERR_INVALID_ARG, "bytes is NULL");
        size_t staging = 0;
        return per_head_need(graphs, B, H, d, dtype, &staging, bytes);
    } catch (...) {
        return fail(DIFFUSER_ERR_ALLOC, "unexpected exception");
    }
}

int diffuser_forward_per_head(const void* Q, const void* K, const void* V, int32_t dtype,
                              int64_t B, int64_t H, int32_t d, const diffuser_graph* const* graphs,
                              int32_t hops, float alpha, void* out, void* workspace,
                              size_t workspace_bytes, diffuser_stream stream) {
    try {
        size_t staging = 0, need = 0;
        int st = per_head_need(graphs, B, H, d, dtype, &staging, &need);
        if (st) return st;
        const diffuser_graph* g0 = graphs[0];
        if (!Q || !K || !V || !out) return fail(DIFFUSER_ERR_INVALID_ARG, "a tensor pointer is NULL");
        if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(out))
            return fail(DIFFUSER_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
        if (hops < 0) return fail(DIFFUSER_ERR_INVALID_ARG, "hops must be >= 0");
        if (!(alpha >= 0.f && alpha <= 1.f))
            return fail(DIFFUSER_ERR_INVALID_ARG, "alpha must lie in [0, 1]");
        const size_t bytes = io_bytes(g0, B, H, dtype);
        if (overlaps(out, bytes, Q, bytes) || overlaps(out, bytes, K, bytes))
            return fail(DIFFUSER_ERR_INVALID_ARG, "out overlaps Q or K");
        if (hops > 0 && overlaps(out, bytes, V, bytes))
            return fail(DIFFUSER_ERR_INVALID_ARG, "out may alias V only when hops == 0");
        if ((st = check_workspace_bytes(need, workspace, workspace_bytes))) return st;
        for (int64_t h = 0; h < H; ++h) {
            if ((st = check_device(graphs[h]))) return st;
            if ((st = check_status_word(graphs[h]))) return st;
        }
        cudaStream_t s = static_cast<cudaStream_t>(stream);
        if (hops == 0) {
            if (out == V) return DIFFUSER_OK;
            cudaError_t err = cudaMemcpyAsync(out, V, bytes, cudaMemcpyDeviceToDevice, s);
            return err == cudaSuccess ? DIFFUSER_OK : cuda_fail(err, "copying V to out (hops = 0)");
        }
        const size_t slice = io_bytes(g0, 1, 1, dtype);         // one [n][d] head slice
        const char* q = static_cast<const char*>(Q);
        const char* k = static_cast<const char*>(K);
        const char* v = static_cast<const char*>(V);
        char* o = static_cast<char*>(out);
        char* ws = static_cast<char*>(workspace);
        for (int64_t h = 0; h < H; ++h) {
            const size_t at = (size_t)h * slice;
            if (B == 1) {
                // head h's slices are contiguous: run it in place
                st = forward_device(q + at, k + at, v + at, dtype, 1, 1, d, graphs[h], hops, alpha,
                                    o + at, ws, workspace_bytes, s);
                if (st) return st;
                continue;
            }
            // gather head h of every batch item (B rows of `slice` bytes, H slices apart),
            // run the B units, scatter the output back
            const size_t seg = staging / 4, pitch = (size_t)H * slice;
            char* sq = ws;
            char* sk = ws + seg;
            char* sv = ws + 2 * seg;
            char* so = ws + 3 * seg;
            cudaError_t err = cudaMemcpy2DAsync(sq, slice, q + at, pitch, slice, B, cudaMemcpyDeviceToDevice, s);
            if (err == cudaSuccess)
                err = cudaMemcpy2DAsync(sk, slice, k + at, pitch, slice, B, cudaMemcpyDeviceToDevice, s);
            if (err == cudaSuccess)
                err = cudaMemcpy2DAsync(sv, slice, v + at, pitch, slice, B, cudaMemcpyDeviceToDevice, s);
            if (err != cudaSuccess) return cuda_fail(err, "gathering a head's slices");
            st = forward_device(sq, sk, sv, dtype, B, 1, d, graphs[h], hops, alpha, so, ws + staging,
                                workspace_bytes - staging, s);
            if (st) return st;
            err = cudaMemcpy2DAsync(o + at, pitch, so, slice, slice, B, cudaMemcpyDeviceToDevice, s);
            if (err != cudaSuccess) return cuda_fail(err, "scattering a head's output");
        }
        return DIFFUSER_OK;
    } catch (...) {
        return fail(DIFFUSER_ERR_ALLOC, "unexpected exception");
    }
}

namespace {

// Status block of the stand-alone projections on each device (the layout of a
// graph's: word, padding, device address of a page-locked host mirror), made
// on the first projection call on that device and kept for the process.
struct ProjStatus {
    int* d = nullptr;
    int* h = nullptr;
};
std::mutex g_proj_mu;
ProjStatus g_proj_status[kMaxReplayDevices];

int projection_status(ProjStatus* out) {
    int dev = -1;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return cuda_fail(err, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxReplayDevices) return fail(DIFFUSER_ERR_UNSUPPORTED, "device index out of range");
    std::lock_guard<std::mutex> lk(g_proj_mu);
    ProjStatus& ps = g_proj_status[dev];
    if (!ps.d) {
        int* d = nullptr;
        int* h = nullptr;
        int* mirror_dev = nullptr;
        err = cudaMalloc(&d, kStatusBlockBytes);
        if (err == cudaSuccess) err = cudaHostAlloc(&h, sizeof(int), cudaHostAllocMapped);
        if (err == cudaSuccess) {
            *h = 0;
            err = cudaHostGetDevicePointer(&mirror_dev, h, 0);
        }
        if (err == cudaSuccess) {
            unsigned char block[kStatusBlockBytes] = {0};
            std::memcpy(block + 8, &mirror_dev, sizeof(mirror_dev));
            err = cudaMemcpy(d, block, kStatusBlockBytes, cudaMemcpyHostToDevice);
        }
        if (err != cudaSuccess) {
            cudaFree(d);
            if (h) cudaFreeHost(h);
            return cuda_fail(err, "projection status block");
        }
        ps.d = d;
        ps.h = h;
    }
    *out = ps;
    return DIFFUSER_OK;
}

int check_projection_pointers(const void* const* in, int nin, void* const* outs, int nout,
                              const size_t* in_bytes, const size_t* out_bytes) {
    for (int x = 0; x < nin; ++x)
        if (!in[x] || !aligned16(in[x])) return fail(DIFFUSER_ERR_INVALID_ARG, "an input is NULL or not 16-byte aligned");
    for (int x = 0; x < nout; ++x) {
        if (!outs[x] || !aligned16(outs[x]))
            return fail(DIFFUSER_ERR_INVALID_ARG, "an output is NULL or not 16-byte aligned");
        for (int y = 0; y < nin; ++y)
            if (overlaps(outs[x], out_bytes[x], in[y], in_bytes[y]))
                return fail(DIFFUSER_ERR_INVALID_ARG, "an output overlaps an input");
        for (int y = x + 1; y < nout; ++y)
            if (overlaps(outs[x], out_bytes[x], outs[y], out_bytes[y]))
                return fail(DIFFUSER_ERR_INVALID_ARG, "the outputs overlap");
    }
    return DIFFUSER_OK;
}

}  // namespace

int diffuser_qkv_projection(const void* X, const void* Wqkv, int64_t B, int64_t n, int32_t D, int32_t H,
                            int32_t d, void* Q, void* K, void* V, diffuser_stream stream) {
    try {
        int st = check_layer_shape(B, n, D, H, d);
        if (st) return st;
        const size_t xb = (size_t)B * n * D * 2, wb = (size_t)3 * H * kHeadDim * D * 2;
        const size_t ob = (size_t)B * H * n * kHeadDim * 2;
        const void* in[2] = {X, Wqkv};
        void* outs[3] = {Q, K, V};
        const size_t inb[2] = {xb, wb}, outb[3] = {ob, ob, ob};
        if ((st = check_projection_pointers(in, 2, outs, 3, inb, outb))) return st;
        ProjStatus ps;
        if ((st = projection_status(&ps))) return st;
        if (*reinterpret_cast<volatile int*>(ps.h) != 0)
            return fail(DIFFUSER_ERR_DEVICE, "a projection kernel reported a failure (see diffuser_projection_status)");
        return launch_qkv_projection(X, Wqkv, B, n, D, H, Q, K, V, ps.d, static_cast<cudaStream_t>(stream));
    } catch (...) {
        return fail(DIFFUSER_ERR_ALLOC, "unexpected exception");
    }
}

int diffuser_output_projection(const void* Z, const void* Wo, int64_t B, int64_t n, int32_t D, int32_t H,
                               int32_t d, void* Y, diffuser_stream stream) {
    try {
        int st = check_layer_shape(B, n, D, H, d);
        if (st) return st;
        const size_t zb = (size_t)B * H * n * kHeadDim * 2, wb = (size_t)D * H * kHeadDim * 2;
        const size_t yb = (size_t)B * n * D * 2;
        const void* in[2] = {Z, Wo};
        void* outs[1] = {Y};
        const size_t inb[2] = {zb, wb}, outb[1] = {yb};
        if ((st = check_projection_pointers(in, 2, outs, 1, inb, outb))) return st;
        ProjStatus ps;
        if ((st = projection_status(&ps))) return st;
        if (*reinterpret_cast<volatile int*>(ps.h) != 0)
            return fail(DIFFUSER_ERR_DEVICE, "a projection kernel reported a failure (see diffuser_projection_status)");
        return launch_output_projection(Z, Wo, B, n, D, H, Y, ps.d, static_cast<cudaStream_t>(stream));
    } catch (...) {
        return fail(DIFFUSER_ERR_ALLOC, "unexpected exception");
    }
}

int diffuser_projection_status(int* status, int reset) {
    if (!status) return fail(DIFFUSER_ERR_INVALID_ARG, "NULL argument");
    ProjStatus ps;
    int st = projection_status(&ps);
    if (st) return st;
    cudaError_t err = cudaMemcpy(status, ps.d, sizeof(int), cudaMemcpyDeviceToHost);
    if (err == cudaSuccess && *status == 0) *status = *reinterpret_cast<volatile int*>(ps.h);
    if (err == cudaSuccess && reset) {
        err = cudaMemset(ps.d, 0, sizeof(int));
        *reinterpret_cast<volatile int*>(ps.h) = 0;
    }
    return err == cudaSuccess ? DIFFUSER_OK : cuda_fail(err, "reading the projection status word");
}

int diffuser_layer_workspace_size(const diffuser_graph* g, int64_t B, int32_t D, int32_t H, int32_t d,
                                  size_t* bytes) {
    try {
        if (!g || !bytes) return fail(DIFFUSER_ERR_INVALID_ARG, "NULL argument");
        int st = check_layer_shape(B, g->n, D, H, d);
        if (st) return st;
        size_t fwd = 0;
        if ((st = workspace_need(g, B, H, DIFFUSER_DTYPE_BF16, &fwd))) return st;
        *bytes = 4 * align_up(io_bytes(g, B, H, DIFFUSER_DTYPE_BF16)) + fwd;
        return DIFFUSER_OK;
    } catch (...) {
        return fail(DIFFUSER_ERR_ALLOC, "unexpected exception");
    }
}

int diffuser_layer_forward(const void* X, const void* Wqkv, const void* Wo, int64_t B, int32_t D, int32_t H,
                           int32_t d, const diffuser_graph* g, int32_t hops, float alpha, void* Y,
                           void* workspace, size_t workspace_bytes, diffuser_stream stream) {
    try {
        if (!g) return fail(DIFFUSER_ERR_INVALID_ARG, "graph is NULL");
        const int64_t n = g->n;
        int st = check_layer_shape(B, n, D, H, d);
        if (st) return st;
        if (hops < 0) return fail(DIFFUSER_ERR_INVALID_ARG, "hops must be >= 0");
        if (!(alpha >= 0.f && alpha <= 1.f)) return fail(DIFFUSER_ERR_INVALID_ARG, "alpha must lie in [0, 1]");
        const size_t xb = (size_t)B * n * D * 2, wqb = (size_t)3 * H * kHeadDim * D * 2;
        const size_t wob = (size_t)D * H * kHeadDim * 2;
        const void* in[3] = {X, Wqkv, Wo};
        void* outs[1] = {Y};
        const size_t inb[3] = {xb, wqb, wob}, outb[1] = {xb};
        if ((st = check_projection_pointers(in, 3, outs, 1, inb, outb))) return st;
        size_t need = 0;
        if ((st = diffuser_layer_workspace_size(g, B, D, H, d, &need))) return st;
        if ((st = check_workspace_bytes(need, workspace, workspace_bytes))) return st;
        if ((st = check_device(g))) return st;
        if ((st = check_status_word(g))) return st;
        const size_t slot = align_up(io_bytes(g, B, H, DIFFUSER_DTYPE_BF16));
        char* ws = static_cast<char*>(workspace);
        char *q = ws, *k = ws + slot, *v = ws + 2 * slot, *z = ws + 3 * slot;
        cudaStream_t s = static_cast<cudaStream_t>(stream);
        if ((st = launch_qkv_projection(X, Wqkv, B, n, D, H, q, k, v, g->d_status, s))) return st;
        if ((st = forward_device(q, k, v, DIFFUSER_DTYPE_BF16, B, H, d, g, hops, alpha, z, ws + 4 * slot,
                                 workspace_bytes - 4 * slot, s)))
            return st;
        return launch_output_projection(z, Wo, B, n, D, H, Y, g->d_status, s);
    } catch (...) {
        return fail(DIFFUSER_ERR_ALLOC, "unexpected exception");
    }
}

int diffuser_host_workspace_size(const diffuser_graph* g, int64_t B, int64_t H, int32_t d,
                                 int32_t dtype, size_t* bytes) {
    if (!bytes) return fail(DIFFUSER_ERR_INVALID_ARG, "bytes is NULL");
    size_t base = 0;
    int st = diffuser_workspace_size(g, B, H, d, dtype, &base);
    if (st) return st;
    *bytes = base + 4 * align_up(io_bytes(g, B, H, dtype));
    return DIFFUSER_OK;
}

int diffuser_forward_host(const void* Q, const void* K, const void* V, int32_t dtype, int64_t B,
                          int64_t H, int32_t d, const diffuser_graph* g, int32_t hops,
                          float alpha, void* out, void* workspace, size_t workspace_bytes,
                          diffuser_stream stream) {
    try {
        int st = check_shape(g, B, H, d, dtype);
        if (st) return st;
        if (!Q || !K || !V || !out) return fail(DIFFUSER_ERR_INVALID_ARG, "a pointer is NULL");
        size_t need = 0;
        if ((st = diffuser_host_workspace_size(g, B, H, d, dtype, &need))) return st;
        if (!workspace || reinterpret_cast<uintptr_t>(workspace) % kAlign)
            return fail(DIFFUSER_ERR_WORKSPACE, "workspace NULL or not 256-byte aligned");
        if (workspace_bytes < need)
            return fail(DIFFUSER_ERR_WORKSPACE, "workspace too small: need " +
                                                    std::to_string(need) + " bytes");
        if ((st = check_device(g))) return st;
        if ((st = check_status_word(g))) return st;
        const size_t bytes = io_bytes(g, B, H, dtype), slot = align_up(bytes);
        char* ws = static_cast<char*>(workspace);
        char* dQ = ws;
        char* dK = ws + slot;
        char* dV = ws + 2 * slot;
        char* dO = ws + 3 * slot;
        BandPlan bp;
        char* fws = ws + 4 * slot;
        const size_t fws_bytes = workspace_bytes - 4 * slot;
        const int64_t units = B * H;
        if (hops > 0 && use_band(g, dtype, &bp)) {
            BandLayout BL;
            if ((st = plan_band_layout(g, bp, units, &BL))) return st;
            return forward_host_overlapped(
                Q, K, V, B, H, g, hops, alpha, out, dQ, dK, dV, dO, fws, fws_bytes, bytes, stream,
                [&](const void* q, const void* k, cudaStream_t s) {
                    return launch_band_scores(g, bp, units, q, k, nullptr, fws, BL, false, s);
                },
                [&](const void* q, const void* k, const void* v, void* o, cudaStream_t s) {
                    return launch_band_hops(g, bp, units, q, k, v, hops, alpha, o, fws, BL, s);
                });
        }
        if (hops > 0 && use_block(g, dtype)) {
            BlockLayout KL;
            if ((st = plan_block_layout(g, units, &KL))) return st;
            return forward_host_overlapped(
                Q, K, V, B, H, g, hops, alpha, out, dQ, dK, dV, dO, fws, fws_bytes, bytes, stream,
                [&](const void* q, const void* k, cudaStream_t s) {
                    return launch_block_scores(g, units, q, k, fws, KL, s);
                },
                [&](const void* q, const void* k, const void* v, void* o, cudaStream_t s) {
                    return launch_block_hops(g, units, q, k, v, hops, alpha, o, fws, KL, s);
                });
        }
        cudaError_t err = cudaMemcpyAsync(dQ, Q, bytes, cudaMemcpyHostToDevice, stream);
        if (err == cudaSuccess) err = cudaMemcpyAsync(dK, K, bytes, cudaMemcpyHostToDevice, stream);
        if (err == cudaSuccess) err = cudaMemcpyAsync(dV, V, bytes, cudaMemcpyHostToDevice, stream);
        if (err != cudaSuccess) return cuda_fail(err, "host-to-device copies");
        st = forward_device(dQ, dK, dV, dtype, B, H, d, g, hops, alpha, dO, ws + 4 * slot,
                            workspace_bytes - 4 * slot, stream);
        if (st) return st;
        err = cudaMemcpyAsync(out, dO, bytes, cudaMemcpyDeviceToHost, stream);
        return err == cudaSuccess ? DIFFUSER_OK : cuda_fail(err, "device-to-host copy");
    } catch (...) {
        return fail(DIFFUSER_ERR_ALLOC, "unexpected exception");
    }
}

int diffuser_attention_weights(const void* Q, const void* K, int32_t dtype, int64_t B, int64_t H,
                               int32_t d, const diffuser_graph* g, float* A_out, void* workspace,
                               size_t workspace_bytes, diffuser_stream stream) {
    try {
        int st = check_shape(g, B, H, d, dtype);
        if (st) return st;
        if (!Q || !K || !A_out) return fail(DIFFUSER_ERR_INVALID_ARG, "a pointer is NULL");
        if (!aligned16(Q) || !aligned16(K) || !aligned16(A_out))
            return fail(DIFFUSER_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
        size_t need = 0;
        if ((st = workspace_need(g, B, H, dtype, &need))) return st;
        if ((st = check_workspace_bytes(need, workspace, workspace_bytes))) return st;
        if ((st = check_device(g))) return st;
        if ((st = check_status_word(g))) return st;
        BandPlan bp;
        if (use_band(g, dtype, &bp)) {
            BandLayout BL;
            char* ws = static_cast<char*>(workspace);
            if ((st = plan_band_layout(g, bp, B * H, &BL))) return st;
            if ((st = launch_band_scores(g, bp, B * H, Q, K, nullptr, ws, BL, true, stream))) return st;
            return launch_band_to_csr(g, bp, B * H, ws, BL, A_out, stream);
        }
        CsrArgs a{g->d_row_ptr, g->d_col, g->n, g->nnz, B * H};
        return launch_score_csr(a, Q, K, dtype, A_out, stream);
    } catch (...) {
        return fail(DIFFUSER_ERR_ALLOC, "unexpected exception");
    }
}

int diffuser_diffuse_csr(const diffuser_graph* g, const float* A, const void* V, int32_t dtype,
                         int64_t B, int64_t H, int32_t d, int32_t hops, float alpha, void* out,
                         void* workspace, size_t workspace_bytes, diffuser_stream stream) {
    try {
        int st = check_shape(g, B, H, d, dtype);
        if (st) return st;
        if (!A || !V || !out) return fail(DIFFUSER_ERR_INVALID_ARG, "a pointer is NULL");
        if (!aligned16(A) || !aligned16(V) || !aligned16(out))
            return fail(DIFFUSER_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
        if (hops < 0) return fail(DIFFUSER_ERR_INVALID_ARG, "hops must be >= 0");
        if (!(alpha >= 0.f && alpha <= 1.f))
            return fail(DIFFUSER_ERR_INVALID_ARG, "alpha must lie in [0, 1]");
        const size_t bytes = io_bytes(g, B, H, dtype);
        if (hops > 0 && overlaps(out, bytes, V, bytes))
            return fail(DIFFUSER_ERR_INVALID_ARG, "out may alias V only when hops == 0");
        Layout L;
        if ((st = plan_layout(g, B, H, &L))) return st;
        if ((st = check_workspace(L, workspace, workspace_bytes))) return st;
        if ((st = check_device(g))) return st;
        if ((st = check_status_word(g))) return st;
        CsrArgs a{g->d_row_ptr, g->d_col, g->n, g->nnz, B * H};
        return run_hops_csr(g, a, A, V, dtype, hops, alpha, out, static_cast<char*>(workspace),
                            L, stream);
    } catch (...) {
        return fail(DIFFUSER_ERR_ALLOC, "unexpected exception");
    }
}

int diffuser_set_path(int path) {
    if (path != DIFFUSER_PATH_AUTO && path != DIFFUSER_PATH_CSR)
        return fail(DIFFUSER_ERR_INVALID_ARG, "unknown path");
    g_path.store(path);
    return DIFFUSER_OK;
}

int diffuser_get_path(void) { return g_path.load(); }

int diffuser_kernels_for(const diffuser_graph* g, int32_t dtype, int* kernels) {
    if (!g || !kernels) return fail(DIFFUSER_ERR_INVALID_ARG, "NULL argument");
    if (dtype != DIFFUSER_DTYPE_FP32 && dtype != DIFFUSER_DTYPE_BF16)
        return fail(DIFFUSER_ERR_UNSUPPORTED, "dtype must be FP32 or BF16");
    BandPlan bp;
    *kernels = use_band(g, dtype, &bp) ? DIFFUSER_KERNELS_BAND
               : use_block(g, dtype)   ? DIFFUSER_KERNELS_BLOCK
                                       : DIFFUSER_KERNELS_CSR;
    return DIFFUSER_OK;
}

int diffuser_graph_status(const diffuser_graph* g, int* status, int reset) {
    if (!g || !status) return fail(DIFFUSER_ERR_INVALID_ARG, "NULL argument");
    int dev = -1;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return cuda_fail(err, "cudaGetDevice");
    if (dev != g->device) return fail(DIFFUSER_ERR_INVALID_ARG, "not the graph's device");
    err = cudaMemcpy(status, g->d_status, sizeof(int), cudaMemcpyDeviceToHost);
    if (err == cudaSuccess && *status == 0 && g->h_status)
        *status = *reinterpret_cast<volatile int*>(g->h_status);
    if (err == cudaSuccess && reset) {
        err = cudaMemset(g->d_status, 0, sizeof(int));
        if (g->h_status) *reinterpret_cast<volatile int*>(g->h_status) = 0;
    }
    if (err != cudaSuccess) return cuda_fail(err, "reading the device status word");
    return DIFFUSER_OK;
}

int diffuser_graph_set_status(const diffuser_graph* g, int status) {
    if (!g) return fail(DIFFUSER_ERR_INVALID_ARG, "NULL argument");
    int dev = -1;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return cuda_fail(err, "cudaGetDevice");
    if (dev != g->device) return fail(DIFFUSER_ERR_INVALID_ARG, "not the graph's device");
    err = cudaMemcpy(g->d_status, &status, sizeof(int), cudaMemcpyHostToDevice);
    if (err != cudaSuccess) return cuda_fail(err, "writing the device status word");
    if (g->h_status) *reinterpret_cast<volatile int*>(g->h_status) = status;
    return DIFFUSER_OK;
}

int64_t diffuser_launch_count(int64_t* per_kind) {
    int64_t total = 0;
    for (int k = 0; k < DIFFUSER_KERNEL_KINDS; ++k) {
        int64_t v = g_launches[k].load(std::memory_order_relaxed);
        if (per_kind) per_kind[k] = v;
        total += v;
    }
    return total;
}

int diffuser_profile_begin(void) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (g_prof_on) return fail(DIFFUSER_ERR_INVALID_ARG, "a profile is already open");
    g_prof_on = true;
    g_prof_records.clear();
    return DIFFUSER_OK;
}

int diffuser_profile_end(double* ms_per_kind, int64_t* launches_per_kind) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (!g_prof_on) return fail(DIFFUSER_ERR_INVALID_ARG, "no profile is open");
    g_prof_on = false;
    double ms[DIFFUSER_KERNEL_KINDS] = {0};
    int64_t cnt[DIFFUSER_KERNEL_KINDS] = {0};
    int status = DIFFUSER_OK;
    for (auto& r : g_prof_records) {
        cudaError_t err = cudaEventSynchronize(r.stop);
        float t = 0.f;
        if (err == cudaSuccess) err = cudaEventElapsedTime(&t, r.start, r.stop);
        if (err != cudaSuccess && status == DIFFUSER_OK) status = cuda_fail(err, "profile events");
        ms[r.kind] += t;
        cnt[r.kind] += 1;
        g_event_pool.push_back(r.start);
        g_event_pool.push_back(r.stop);
    }
    g_prof_records.clear();
    for (int k = 0; k < DIFFUSER_KERNEL_KINDS; ++k) {
        if (ms_per_kind) ms_per_kind[k] = ms[k];
        if (launches_per_kind) launches_per_kind[k] = cnt[k];
    }
    return status;
}

}  // extern "C"
