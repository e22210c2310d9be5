// kdt_gather.cu -- the points in level order: out[node] = pts[perm[node]],
// and the in-place build that leaves the point array itself in level order.
//
// "GPU-friendly, Parallel, and (Almost-)In-Place Construction of Left-Balanced
// k-d Trees" (introduction and core idea) builds by reordering the data array
// itself into the tree's order, with one tag per point as the only extra
// memory.  This library's build returns the order as a permutation; these
// calls apply it to the points.  Rows are copied as raw 32-bit words, so every
// coordinate (signed zeros included) arrives bit for bit.
#include "kdt_internal.cuh"

namespace kdt {

constexpr int kGatherThreads = 256;

// One thread per node: row perm[u] of `pts` (k consecutive words) to row u of
// `out`; `vec`: rows of 2 or 4 words are 8/16-byte aligned and move as one
// access.  Skips all work when *gate is nonzero (an earlier error); an entry
// of perm outside 0..N-1 is skipped and recorded in *status.
__global__ void __launch_bounds__(kGatherThreads) gather_rows_kernel(const uint32_t *__restrict__ pts, int64_t N,
                                                                     int k, const int32_t *__restrict__ perm,
                                                                     uint32_t *__restrict__ out, const int *gate,
                                                                     int *status, int bad_code, bool vec) {
    if (gate != nullptr && *(volatile const int *)gate != 0) return;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < N; u += stride) {
        const int32_t src = __ldg(perm + u);
        if (src < 0 || (int64_t)src >= N) {
            set_status(status, bad_code);
            continue;
        }
        const uint32_t *row = pts + (int64_t)src * k;
        uint32_t *dst = out + u * k;
        if (vec && k == 4) {
            *reinterpret_cast<uint4 *>(dst) = __ldg(reinterpret_cast<const uint4 *>(row));
        } else if (vec && k == 2) {
            *reinterpret_cast<uint2 *>(dst) = __ldg(reinterpret_cast<const uint2 *>(row));
        } else {
            for (int c = 0; c < k; ++c) dst[c] = __ldg(row + c);
        }
    }
}

// words[0..n) = src[0..n) unless *gate is nonzero.
__global__ void __launch_bounds__(kGatherThreads) copy_words_kernel(const uint32_t *__restrict__ src, int64_t n,
                                                                    uint32_t *__restrict__ dst, const int *gate) {
    if (*(volatile const int *)gate != 0) return;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) dst[i] = __ldg(src + i);
}

static unsigned gather_grid(int64_t n) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 152;
    int64_t blocks = (n + kGatherThreads - 1) / kGatherThreads;
    const int64_t cap = (int64_t)sms * 8;
    return (unsigned)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

static bool rows_vectorisable(const void *a, const void *b) {
    return ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b)) & 15u) == 0;
}

static void launch_gather(const uint32_t *pts, int64_t N, int k, const int32_t *perm, uint32_t *out,
                          const int *gate, int *status, int bad_code, cudaStream_t stream) {
    gather_rows_kernel<<<gather_grid(N), kGatherThreads, 0, stream>>>(pts, N, k, perm, out, gate, status, bad_code,
                                                                    rows_vectorisable(pts, out));
}

int enqueue_gather(const float *pts, int64_t N, int k, const int32_t *perm, float *out, int *status,
                   cudaStream_t stream) {
    ProfScope ps(stream, "gather", (double)N * (4.0 + 8.0 * k));
    launch_gather(reinterpret_cast<const uint32_t *>(pts), N, k, perm, reinterpret_cast<uint32_t *>(out), nullptr,
                  status, KDT_EINVAL, stream);
    return cudaGetLastError() == cudaSuccess ? KDT_OK : KDT_ECUDA;
}

int enqueue_inplace_tail(const Plan &p, const Buffers &b, float *pts, const int32_t *perm, cudaStream_t stream) {
    const int64_t N = p.S.N;
    const int k = p.k;
    // after the build every record buffer is free; buffer 0 (G * 4 * ld >=
    // (k + 1) * N words) holds the reordered rows until they are copied back
    uint32_t *tmp = reinterpret_cast<uint32_t *>(b.rec[0]);
    {
        ProfScope ps(stream, "gather", (double)N * (4.0 + 8.0 * k));
        launch_gather(reinterpret_cast<const uint32_t *>(pts), N, k, perm, tmp, b.status, b.status, KDT_EINTERNAL,
                      stream);
        if (cudaGetLastError() != cudaSuccess) return KDT_ECUDA;
    }
    {
        ProfScope ps(stream, "copyback", (double)N * 8.0 * k);
        copy_words_kernel<<<gather_grid(N * k), kGatherThreads, 0, stream>>>(tmp, N * k,
                                                                            reinterpret_cast<uint32_t *>(pts), b.status);
        if (cudaGetLastError() != cudaSuccess) return KDT_ECUDA;
    }
    enqueue_status_fold(b.status, stream);  // a gather error comes after the build's own fold
    return cudaGetLastError() == cudaSuccess ? KDT_OK : KDT_ECUDA;
}

}  // namespace kdt
