// kdt_api.cu -- the C ABI (include/kdtree_build.h): argument checks,
// workspace handling, the per-device status word and per-kernel timing.
#include <cstdint>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "kdt_internal.cuh"

namespace kdt {

// Sticky per-device status word (each device that loads the module has its own).
__device__ int g_device_status;

__global__ void status_fold_kernel(const int *s) {
    pdl_enter();
    const int v = *s;
    if (v != 0) atomicCAS(&g_device_status, 0, v);
}

void enqueue_status_fold(int *status, cudaStream_t stream) {
    ProfScope ps(stream, "status_fold", 0.0);
    launch_pdl(status_fold_kernel, 1, 1, 0, stream, status);
}

int *device_status_address() {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    return static_cast<int *>(p);
}

int read_and_clear_device_status(int *out) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int)) != cudaSuccess) return KDT_ECUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess) return KDT_ECUDA;
    *out = v;
    return KDT_OK;
}

// ---- per-kernel timing -------------------------------------------------------

namespace {
struct Pending {
    const char *name;
    cudaEvent_t ev0, ev1;
    double bytes;
    int kernels;
};
struct Total {
    const char *name;
    int64_t launches;
    double ms;
    double bytes;
    int64_t kernels;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<Pending> g_pending;
std::vector<Total> g_totals;
}  // namespace

ProfScope::ProfScope(cudaStream_t s, const char *n, double b)
    : stream(s), name(n), bytes(b), ev0(nullptr), on(false), kernels(1) {
    bool enabled;
    {
        std::lock_guard<std::mutex> g(g_prof_mu);
        enabled = g_prof_on;
    }
    if (!enabled) return;
    if (cudaEventCreate(&ev0) != cudaSuccess) return;
    cudaEventRecord(ev0, stream);
    on = true;
}

ProfScope::~ProfScope() {
    if (!on) return;
    cudaEvent_t ev1;
    if (cudaEventCreate(&ev1) != cudaSuccess) {
        cudaEventDestroy(ev0);
        return;
    }
    cudaEventRecord(ev1, stream);
    std::lock_guard<std::mutex> g(g_prof_mu);
    g_pending.push_back({name, ev0, ev1, bytes, kernels});
}

static void drain_pending_locked() {
    for (auto &p : g_pending) {
        float ms = 0.f;
        cudaEventSynchronize(p.ev1);
        cudaEventElapsedTime(&ms, p.ev0, p.ev1);
        cudaEventDestroy(p.ev0);
        cudaEventDestroy(p.ev1);
        bool found = false;
        for (auto &t : g_totals) {
            if (std::strcmp(t.name, p.name) == 0) {
                t.launches += 1;
                t.ms += ms;
                t.bytes += p.bytes;
                t.kernels += p.kernels;
                found = true;
                break;
            }
        }
        if (!found) g_totals.push_back({p.name, 1, (double)ms, p.bytes, (int64_t)p.kernels});
    }
    g_pending.clear();
}

}  // namespace kdt

using namespace kdt;

static bool aligned256(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

extern "C" {

int kdt_workspace_size(int64_t N, int k, int split_mode, size_t *bytes) {
    if (!bytes) return KDT_EINVAL;
    Plan p;
    const int rc = make_plan(N, k, split_mode, &p);
    if (rc != KDT_OK) return rc;
    *bytes = p.bytes;
    return KDT_OK;
}

int kdt_build_ws(const float *pts, int64_t N, int k, int split_mode, int32_t *perm, void *workspace,
                 size_t workspace_bytes, void *stream) {
    if (!pts || !perm || !workspace) return KDT_EINVAL;
    Plan p;
    const int rc = make_plan(N, k, split_mode, &p);
    if (rc != KDT_OK) return rc;
    if (workspace_bytes < p.bytes) return KDT_ENOMEM;
    if (!aligned256(workspace)) return KDT_EINVAL;
    return enqueue_build(p, carve(p, workspace), pts, perm, static_cast<cudaStream_t>(stream));
}

int kdt_build(const float *pts, int64_t N, int k, int split_mode, int32_t *perm, void *stream) {
    if (!pts || !perm) return KDT_EINVAL;
    Plan p;
    int rc = make_plan(N, k, split_mode, &p);
    if (rc != KDT_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void *ws = nullptr;
    if (cudaMallocAsync(&ws, p.bytes, s) != cudaSuccess) {
        cudaGetLastError();
        return KDT_ENOMEM;
    }
    rc = enqueue_build(p, carve(p, ws), pts, perm, s);
    if (cudaFreeAsync(ws, s) != cudaSuccess && rc == KDT_OK) rc = KDT_ECUDA;
    return rc;
}

int kdt_balanced_slots(int64_t N, int64_t *slots) {
    if (!slots || N < 1 || N > 2147483647LL) return KDT_EINVAL;
    *slots = ((int64_t)1 << make_shape(N).L) - 1;
    return KDT_OK;
}

int kdt_balanced_workspace_size(int64_t N, int k, size_t *bytes) {
    if (!bytes) return KDT_EINVAL;
    Plan p;
    const int rc = make_plan(N, k, KDT_SPLIT_ROUND_ROBIN, &p, kShapeBalanced);
    if (rc != KDT_OK) return rc;
    *bytes = p.bytes;
    return KDT_OK;
}

int kdt_build_balanced(const float *pts, int64_t N, int k, int32_t *slots, void *workspace, size_t workspace_bytes,
                       void *stream) {
    if (!pts || !slots || !workspace) return KDT_EINVAL;
    Plan p;
    const int rc = make_plan(N, k, KDT_SPLIT_ROUND_ROBIN, &p, kShapeBalanced);
    if (rc != KDT_OK) return rc;
    if (workspace_bytes < p.bytes) return KDT_ENOMEM;
    if (!aligned256(workspace)) return KDT_EINVAL;
    return enqueue_build(p, carve(p, workspace), pts, slots, static_cast<cudaStream_t>(stream));
}

int kdt_host_workspace_size(int64_t N, int k, int split_mode, size_t *bytes) {
    if (!bytes) return KDT_EINVAL;
    Plan p;
    const int rc = make_plan(N, k, split_mode, &p);
    if (rc != KDT_OK) return rc;
    const size_t pts_bytes = ((size_t)N * k * 4 + 255) / 256 * 256;
    const size_t perm_bytes = ((size_t)N * 4 + 255) / 256 * 256;
    *bytes = p.bytes + pts_bytes + perm_bytes;
    return KDT_OK;
}

// Device-side address of a page-locked host buffer, or nullptr if the buffer
// is ordinary pageable memory (or the device cannot address it).
static const void *pinned_device_address(const void *host) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, host) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

int kdt_build_host(const float *host_pts, int64_t N, int k, int split_mode, int32_t *host_perm, void *workspace,
                   size_t workspace_bytes, void *stream) {
    if (!host_pts || !host_perm || !workspace) return KDT_EINVAL;
    Plan p;
    int rc = make_plan(N, k, split_mode, &p);
    if (rc != KDT_OK) return rc;
    size_t need = 0;
    kdt_host_workspace_size(N, k, split_mode, &need);
    if (workspace_bytes < need) return KDT_ENOMEM;
    if (!aligned256(workspace)) return KDT_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned char *base = static_cast<unsigned char *>(workspace);
    float *d_pts = reinterpret_cast<float *>(base + p.bytes);
    int32_t *d_perm = reinterpret_cast<int32_t *>(base + p.bytes + ((size_t)N * k * 4 + 255) / 256 * 256);
    const Buffers b = carve(p, workspace);
    // Page-locked host buffers are used in place: the first kernel reads the
    // points across the host link as it converts them, and the kernels that
    // fix nodes write the permutation straight into host memory, so the
    // transfers overlap the build instead of preceding and following it.
    // Pageable buffers are staged through the workspace.
    const float *pts_in = static_cast<const float *>(pinned_device_address(host_pts));
    int32_t *perm_out = static_cast<int32_t *>(const_cast<void *>(pinned_device_address(host_perm)));
    if (!pts_in) {
        if (cudaMemcpyAsync(d_pts, host_pts, (size_t)N * k * 4, cudaMemcpyHostToDevice, s) != cudaSuccess)
            return KDT_ECUDA;
        pts_in = d_pts;
    }
    rc = enqueue_build(p, b, pts_in, perm_out ? perm_out : d_perm, s, pts_in == d_pts);
    if (rc != KDT_OK) return rc;
    if (!perm_out && cudaMemcpyAsync(host_perm, d_perm, (size_t)N * 4, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return KDT_ECUDA;
    int st = 0;
    if (cudaMemcpyAsync(&st, b.status, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return KDT_ECUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KDT_ECUDA;
    return st;
}

int kdt_verify(const float *pts, int64_t N, int k, int split_mode, const int32_t *perm, void *stream) {
    if (!pts || !perm || N < 1 || N > 2147483647LL || k < 1 || k > kMaxK ||
        (split_mode != KDT_SPLIT_ROUND_ROBIN && split_mode != KDT_SPLIT_WIDEST))
        return KDT_EINVAL;
    int result = 0;
    const int rc = enqueue_verify(pts, N, k, split_mode, perm, static_cast<cudaStream_t>(stream), &result);
    if (rc != KDT_OK) return rc;
    return result;
}

int kdt_gather_points(const float *pts, int64_t N, int k, const int32_t *perm, float *out, void *stream) {
    if (!pts || !perm || !out || N < 1 || N > 2147483647LL || k < 1 || k > kMaxK) return KDT_EINVAL;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(pts), a1 = a0 + (uintptr_t)N * k * 4;
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(out), b1 = b0 + (uintptr_t)N * k * 4;
    if (a0 < b1 && b0 < a1) return KDT_EINVAL;  // out overlaps pts
    int *st = device_status_address();
    if (!st) return KDT_ECUDA;
    return enqueue_gather(pts, N, k, perm, out, st, static_cast<cudaStream_t>(stream));
}

int kdt_build_inplace(float *pts, int64_t N, int k, int split_mode, int32_t *perm, void *workspace,
                      size_t workspace_bytes, void *stream) {
    if (!pts || !perm || !workspace) return KDT_EINVAL;
    Plan p;
    const int rc = make_plan(N, k, split_mode, &p);
    if (rc != KDT_OK) return rc;
    if (workspace_bytes < p.bytes) return KDT_ENOMEM;
    if (!aligned256(workspace)) return KDT_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const Buffers b = carve(p, workspace);
    const int rb = enqueue_build(p, b, pts, perm, s);
    if (rb != KDT_OK) return rb;
    return enqueue_inplace_tail(p, b, pts, perm, s);
}

int kdt_node_dims(const float *tree_pts, int64_t N, int k, int split_mode, uint8_t *dims, void *stream) {
    if (!tree_pts || !dims || N < 1 || N > 2147483647LL || k < 1 || k > kMaxK ||
        (split_mode != KDT_SPLIT_ROUND_ROBIN && split_mode != KDT_SPLIT_WIDEST))
        return KDT_EINVAL;
    return enqueue_node_dims(tree_pts, N, k, split_mode, dims, static_cast<cudaStream_t>(stream));
}

int kdt_knn(const float *tree_pts, int64_t N, int k, const uint8_t *dims, const float *queries, int64_t Q, int K,
            int32_t *out_node, float *out_dist2, void *stream) {
    if (!tree_pts || !queries || !out_node || !out_dist2 || N < 1 || N > 2147483647LL || k < 1 || k > kMaxK ||
        Q < 0 || K < 1 || K > KDT_MAX_KNN)
        return KDT_EINVAL;
    int *st = device_status_address();
    if (!st) return KDT_ECUDA;
    return enqueue_knn(tree_pts, N, k, dims, queries, Q, K, out_node, out_dist2, st,
                       static_cast<cudaStream_t>(stream));
}

int kdt_status(void *stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return KDT_ECUDA;
    int v = 0;
    const int rc = read_and_clear_device_status(&v);
    return rc != KDT_OK ? rc : v;
}

const char *kdt_error_string(int code) {
    switch (code) {
        case KDT_OK: return "ok";
        case KDT_EINVAL: return "invalid argument";
        case KDT_ENOMEM: return "out of memory or workspace too small";
        case KDT_ECUDA: return "CUDA runtime error";
        case KDT_ENONFINITE: return "non-finite coordinate";
        case KDT_ETIMEOUT: return "device-side wait timed out";
        case KDT_EINTERNAL: return "internal consistency check failed";
        default: return "unknown error";
    }
}

int kdt_profile_enable(int on) {
    std::lock_guard<std::mutex> g(g_prof_mu);
    g_prof_on = on != 0;
    return KDT_OK;
}

int kdt_profile_reset(void) {
    std::lock_guard<std::mutex> g(g_prof_mu);
    drain_pending_locked();
    g_totals.clear();
    return KDT_OK;
}

int kdt_profile_read(kdt_kernel_stat *out, int cap) {
    std::lock_guard<std::mutex> g(g_prof_mu);
    drain_pending_locked();
    const int n = (int)g_totals.size();
    for (int i = 0; i < n && i < cap && out; ++i) {
        out[i].name = g_totals[i].name;
        out[i].launches = g_totals[i].launches;
        out[i].total_ms = g_totals[i].ms;
        out[i].bytes_alg = g_totals[i].bytes;
        out[i].kernels = g_totals[i].kernels;
    }
    return n;
}

}  // extern "C"
