// kdt_static.cu -- kdt_build_static: the build with a fixed, library-owned
// scratch array instead of an allocation (see include/kdtree_build.h for who
// needs it and its limits).
#include <cstdint>
#include <mutex>

#include "kdt_internal.cuh"

namespace {

// The scratch array.  In host code this name is only a stand-in for the
// device symbol, never a device address: the address comes from
// cudaGetSymbolAddress, looked up once per device.
static __device__ __align__(256) unsigned char g_static_scratch[KDT_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up on
// the first call for that device).  Returns nullptr on failure.
void *scratch_address() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> g(g_mu);
    if (!g_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return nullptr;
        }
        g_addr[dev] = p;
    }
    return g_addr[dev];
}

}  // namespace

extern "C" int kdt_build_static(const float *pts, int64_t N, int k, int split_mode, int32_t *perm, void *stream) {
    if (!pts || !perm) return KDT_EINVAL;
    kdt::Plan p;
    const int rc = kdt::make_plan(N, k, split_mode, &p);
    if (rc != KDT_OK) return rc;
    if (p.bytes > (size_t)KDT_STATIC_SCRATCH_BYTES) return KDT_EINVAL;  // does not fit the array
    void *ws = scratch_address();
    if (!ws) return KDT_ECUDA;
    return kdt::enqueue_build(p, kdt::carve(p, ws), pts, perm, static_cast<cudaStream_t>(stream));
}
