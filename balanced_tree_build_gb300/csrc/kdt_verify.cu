// kdt_verify.cu -- GPU check that a permutation is the left-balanced k-d tree
// of a point set.
//
// The KdTreeGPU page ("An Implementation of a Balanced Kd Tree Builder Using
// GPUs", build section) verifies its trees on the GPU after the build; this is
// that idea for the left-balanced tree.  One thread per node i walks from the
// root to i and checks the k-d condition of "GPU-friendly, Parallel, and
// (Almost-)In-Place Construction of Left-Balanced k-d Trees" (problem
// paragraph) against every ancestor a: i in the left subtree of a requires
// pts[perm[i]] < pts[perm[a]] under a's split order, i in the right subtree
// the reverse.  The split order is the cyclic super key plus input index, so
// the condition is strict and the tree it accepts is unique.  In widest mode
// the walk carries the domain down from the bounding box, clipping it at each
// ancestor's split coordinate, and recomputes each ancestor's dimension.
//
// Independent of the build kernels: comparisons are made on the raw floats,
// not on the build's keys.
#include "kdt_internal.cuh"

namespace kdt {

constexpr int kVerifyThreads = 256;

__device__ __forceinline__ bool pt_less(const float *__restrict__ pts, int k, int p, int64_t a, int64_t b) {
    for (int j = 0; j < k; ++j) {
        int c = p + j;
        if (c >= k) c -= k;
        const float xa = pts[a * k + c], xb = pts[b * k + c];
        if (xa < xb) return true;
        if (xb < xa) return false;
    }
    return a < b;
}

// Finiteness and (widest mode) the bounding box as key min/max.
__global__ void __launch_bounds__(kVerifyThreads) verify_prep_kernel(const float *__restrict__ pts, int64_t N,
                                                                     int k, uint32_t *bbox, int *flags) {
    uint32_t mn[kMaxK], mx[kMaxK];
#pragma unroll
    for (int c = 0; c < kMaxK; ++c) {
        mn[c] = 0xffffffffu;
        mx[c] = 0u;
    }
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int bad = 0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < N; i += stride) {
#pragma unroll
        for (int c = 0; c < kMaxK; ++c) {
            if (c < k) {
                const float f = pts[i * k + c];
                bad |= !isfinite(f);
                const uint32_t key = f2key(f);
                mn[c] = min(mn[c], key);
                mx[c] = max(mx[c], key);
            }
        }
    }
#pragma unroll
    for (int c = 0; c < kMaxK; ++c) {
        if (c < k) {
            const uint32_t a = __reduce_min_sync(0xffffffffu, mn[c]);
            const uint32_t b = __reduce_max_sync(0xffffffffu, mx[c]);
            if ((threadIdx.x & 31) == 0) {
                atomicMin(&bbox[c], a);
                atomicMax(&bbox[k + c], b);
            }
        }
    }
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(&flags[1], 1);
}

__global__ void __launch_bounds__(kVerifyThreads) verify_nodes_kernel(const float *__restrict__ pts, int64_t N,
                                                                      int k, int mode,
                                                                      const int32_t *__restrict__ perm,
                                                                      const uint32_t *__restrict__ bbox,
                                                                      uint32_t *seen, int *flags) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= N) return;
    const int64_t pi = perm[i];
    if (pi < 0 || pi >= N) {
        atomicOr(&flags[0], 1);
        return;
    }
    const uint32_t bit = 1u << (pi & 31);
    if (atomicOr(&seen[pi >> 5], bit) & bit) {
        atomicOr(&flags[0], 1);
        return;
    }
    float lo[kMaxK], hi[kMaxK];
    if (mode == KDT_SPLIT_WIDEST) {
        for (int c = 0; c < k; ++c) {
            lo[c] = key2f(bbox[c]);
            hi[c] = key2f(bbox[k + c]);
        }
    }
    const int depth = level_of(i);
    int64_t a = 0;
    for (int t = depth - 1; t >= 0; --t) {
        const int right = (int)(((uint64_t)(i + 1) >> t) & 1u);
        const int d = mode == KDT_SPLIT_ROUND_ROBIN ? level_of(a) % k : widest_dim(lo, hi, k);
        const int64_t pa = perm[a];
        if (pa < 0 || pa >= N) {
            atomicOr(&flags[0], 1);
            return;
        }
        const bool ok = right ? pt_less(pts, k, d, pa, pi) : pt_less(pts, k, d, pi, pa);
        if (!ok) {
            atomicOr(&flags[0], 1);
            return;
        }
        if (mode == KDT_SPLIT_WIDEST) {
            const float v = pts[pa * k + d];
            if (right) lo[d] = v;
            else hi[d] = v;
        }
        a = 2 * a + 1 + right;
    }
}

int enqueue_verify(const float *pts, int64_t N, int k, int mode, const int32_t *perm, cudaStream_t stream,
                   int *result) {
    const size_t words = (size_t)((N + 31) / 32);
    const size_t bytes = 256 + (size_t)2 * k * 4 + words * 4;
    void *ws = nullptr;
    if (cudaMallocAsync(&ws, bytes, stream) != cudaSuccess) return KDT_ENOMEM;
    int *flags = static_cast<int *>(ws);
    uint32_t *bbox = reinterpret_cast<uint32_t *>(static_cast<unsigned char *>(ws) + 128);
    uint32_t *seen = reinterpret_cast<uint32_t *>(static_cast<unsigned char *>(ws) + 256 + (size_t)2 * k * 4);
    int rc = KDT_OK;
    int h[2] = {0, 0};
    do {
        if (cudaMemsetAsync(flags, 0, 8, stream) != cudaSuccess) { rc = KDT_ECUDA; break; }
        if (cudaMemsetAsync(bbox, 0xff, (size_t)k * 4, stream) != cudaSuccess) { rc = KDT_ECUDA; break; }
        if (cudaMemsetAsync(bbox + k, 0, (size_t)k * 4, stream) != cudaSuccess) { rc = KDT_ECUDA; break; }
        if (cudaMemsetAsync(seen, 0, words * 4, stream) != cudaSuccess) { rc = KDT_ECUDA; break; }
        int64_t blocks = (N + kVerifyThreads - 1) / kVerifyThreads;
        if (blocks > 152 * 16) blocks = 152 * 16;
        verify_prep_kernel<<<(unsigned)blocks, kVerifyThreads, 0, stream>>>(pts, N, k, bbox, flags);
        if (cudaGetLastError() != cudaSuccess) { rc = KDT_ECUDA; break; }
        const int64_t nb = (N + kVerifyThreads - 1) / kVerifyThreads;
        verify_nodes_kernel<<<(unsigned)nb, kVerifyThreads, 0, stream>>>(pts, N, k, mode, perm, bbox, seen, flags);
        if (cudaGetLastError() != cudaSuccess) { rc = KDT_ECUDA; break; }
        if (cudaMemcpyAsync(h, flags, 8, cudaMemcpyDeviceToHost, stream) != cudaSuccess) { rc = KDT_ECUDA; break; }
    } while (0);
    cudaFreeAsync(ws, stream);
    if (cudaStreamSynchronize(stream) != cudaSuccess) return KDT_ECUDA;
    if (rc != KDT_OK) return rc;
    if (h[1]) return KDT_ENONFINITE;
    *result = h[0] ? 1 : 0;
    return KDT_OK;
}

}  // namespace kdt
