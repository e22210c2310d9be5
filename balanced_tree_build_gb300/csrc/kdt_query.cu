// kdt_query.cu -- queries on a built tree: the split dimension of every node,
// and the K nearest nodes of query points.
//
// The tree is given by its points in level order (tree_pts row u = the point
// stored at node u; kdt_gather_points / kdt_build_inplace produce it).
//
// Nearest neighbours follow "Bigger Buffer k-d Trees on Multi-Many-Core
// Systems" (nearest-neighbour search via k-d trees): go down to the cell that
// holds the query, then back up; on the way up a node's other subtree is
// entered only if the query is closer to the node's splitting plane than the
// current K-th candidate, and the search ends when it comes back to the root.
// On the implicit level-order tree (children 2u+1, 2u+2, parent (u-1)/2) this
// needs no stack: the node it arrived from says whether it came from the
// parent, the near child or the far child.
//
// Result definition (the oracle's): the K smallest (dist2, node) pairs in
// lexicographic order, dist2 = sum over c of (q[c] - p[c])^2 accumulated left
// to right in float32, every operation rounded (no fused multiply-add).  A
// far subtree is skipped only if its plane term exceeds the K-th dist2: every
// point beyond the plane has a coordinate difference at least as large in
// magnitude (rounded subtraction is monotone) and its dist2 is a rounded sum
// of non-negative terms that include that one, so the skip never loses a
// result or a tie.
#include "kdt_internal.cuh"

namespace kdt {

constexpr int kQueryThreads = 128;
constexpr int kDimThreads = 256;

// ---- split dimensions ----------------------------------------------------------

// Bounding box of all points: lo in box[0..k), hi in box[k..2k) as keys.
__global__ void __launch_bounds__(kDimThreads) tree_bbox_kernel(const float *__restrict__ pts, int64_t N, int k,
                                                                uint32_t *box) {
    uint32_t mn[kMaxK], mx[kMaxK];
    for (int c = 0; c < k; ++c) {
        mn[c] = 0xffffffffu;
        mx[c] = 0u;
    }
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < N; i += stride)
        for (int c = 0; c < k; ++c) {
            const uint32_t key = f2key(__ldg(pts + i * k + c));
            mn[c] = min(mn[c], key);
            mx[c] = max(mx[c], key);
        }
    for (int c = 0; c < k; ++c) {
        const uint32_t a = __reduce_min_sync(0xffffffffu, mn[c]);
        const uint32_t b = __reduce_max_sync(0xffffffffu, mx[c]);
        if ((threadIdx.x & 31u) == 0) {
            atomicMin(&box[c], a);
            atomicMax(&box[k + c], b);
        }
    }
}

// dims[u]: round-robin level(u) mod k; widest: the walk from the root, cutting
// the domain at each ancestor's split coordinate, then the widest extent
// ("GPU-friendly, Parallel, and (Almost-)In-Place Construction of
// Left-Balanced k-d Trees", split-widest-dimension paragraphs).
__global__ void __launch_bounds__(kDimThreads) node_dims_kernel(const float *__restrict__ pts, int64_t N, int k,
                                                                int mode, const uint32_t *box, uint8_t *dims) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < N; u += stride) {
        const int depth = level_of(u);
        if (mode == KDT_SPLIT_ROUND_ROBIN) {
            dims[u] = (uint8_t)(depth % k);
            continue;
        }
        float lo[kMaxK], hi[kMaxK];
        for (int c = 0; c < k; ++c) {
            lo[c] = key2f(box[c]);
            hi[c] = key2f(box[k + c]);
        }
        int64_t a = 0;
        for (int t = depth - 1; t >= 0; --t) {
            const int d = widest_dim(lo, hi, k);
            const int right = (int)(((u + 1) >> t) & 1);
            const float s = __ldg(pts + a * k + d);
            if (right) lo[d] = s;
            else hi[d] = s;
            a = 2 * a + 1 + right;
        }
        dims[u] = (uint8_t)widest_dim(lo, hi, k);
    }
}

// ---- K nearest nodes ------------------------------------------------------------

__device__ __forceinline__ float dist2(const float *q, const float *__restrict__ p, int k) {
    float d = 0.f;
    for (int c = 0; c < k; ++c) {
        const float t = __fsub_rn(q[c], __ldg(p + c));
        d = __fadd_rn(d, __fmul_rn(t, t));
    }
    return d;
}

// (dd, node) before (d2, n2) in the result order: dist2, then node id.
__device__ __forceinline__ bool knn_before(float dd, int32_t node, float d2, int32_t n2) {
    return dd < d2 || (dd == d2 && node < n2);
}

// One thread per query.  The K best (dist2, node) pairs are kept sorted
// ascending.  KC > 0: K == KC is known at compile time and the list lives in
// registers (unrolled insertion); KC == 0: any K <= KDT_MAX_KNN, list in
// local memory.
template <int KC>
__global__ void __launch_bounds__(kQueryThreads) knn_kernel(const float *__restrict__ tree, int64_t N, int k,
                                                            const uint8_t *__restrict__ dims,
                                                            const float *__restrict__ queries, int64_t Q, int K,
                                                            int32_t *out_node, float *out_dist2, int *status) {
    constexpr int KA = KC > 0 ? KC : KDT_MAX_KNN;
    const int64_t qi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (qi >= Q) return;
    const int kk = KC > 0 ? KC : K;
    float q[kMaxK];
    for (int c = 0; c < k; ++c) q[c] = __ldg(queries + qi * k + c);
    float bd[KA];
    int32_t bn[KA];
#pragma unroll
    for (int j = 0; j < KA; ++j) {
        if (KC == 0 && j >= kk) break;
        bd[j] = __int_as_float(0x7f800000);  // +infinity
        bn[j] = -1;
    }
    int64_t prev = -1, cur = 0;
    const int64_t cap = 3 * N + 3;  // each node is entered at most three times
    int64_t it = 0;
    for (; it < cap; ++it) {
        const int64_t par = cur == 0 ? -1 : (cur - 1) >> 1;
        int d = dims != nullptr ? (int)dims[cur] : level_of(cur) % k;
        if (d >= k) {  // a caller-supplied dimension out of range
            set_status(status, KDT_EINVAL);
            d = 0;
        }
        const float *p = tree + cur * k;
        const float diff = __fsub_rn(q[d], __ldg(p + d));
        const int64_t near_c = 2 * cur + (diff < 0.f ? 1 : 2);
        const int64_t far_c = 4 * cur + 3 - near_c;
        const float plane = __fmul_rn(diff, diff);
        const float worst = KC > 0 ? bd[KA - 1] : bd[kk - 1];
        int64_t next;
        if (prev == par) {
            // first visit: the node's own point
            const float dd = dist2(q, p, k);
            const int32_t node = (int32_t)cur;
            if (KC > 0) {
                if (knn_before(dd, node, bd[KA - 1], bn[KA - 1])) {
                    // slot j takes the old j-1 if the new pair comes before
                    // it, else the new pair if it comes before the old j
#pragma unroll
                    for (int j = KA - 1; j > 0; --j) {
                        if (knn_before(dd, node, bd[j - 1], bn[j - 1])) {
                            bd[j] = bd[j - 1];
                            bn[j] = bn[j - 1];
                        } else if (knn_before(dd, node, bd[j], bn[j])) {
                            bd[j] = dd;
                            bn[j] = node;
                        }
                    }
                    if (knn_before(dd, node, bd[0], bn[0])) {
                        bd[0] = dd;
                        bn[0] = node;
                    }
                }
            } else if (knn_before(dd, node, bd[kk - 1], bn[kk - 1])) {
                int j = kk - 1;
                while (j > 0 && knn_before(dd, node, bd[j - 1], bn[j - 1])) {
                    bd[j] = bd[j - 1];
                    bn[j] = bn[j - 1];
                    --j;
                }
                bd[j] = dd;
                bn[j] = node;
            }
            const float w2 = KC > 0 ? bd[KA - 1] : bd[kk - 1];
            if (near_c < N) next = near_c;
            else next = (far_c < N && plane <= w2) ? far_c : par;
        } else if (prev == near_c) {
            next = (far_c < N && plane <= worst) ? far_c : par;
        } else {
            next = par;
        }
        if (next < 0) break;
        prev = cur;
        cur = next;
    }
    if (it >= cap) set_status(status, KDT_EINTERNAL);
#pragma unroll
    for (int j = 0; j < KA; ++j) {
        if (KC == 0 && j >= kk) break;
        out_node[qi * kk + j] = bn[j];
        out_dist2[qi * kk + j] = bd[j];
    }
}

static unsigned grid_for(int64_t n, int threads, int per_sm) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 152;
    int64_t blocks = (n + threads - 1) / threads;
    const int64_t cap = (int64_t)sms * per_sm;
    return (unsigned)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

int enqueue_node_dims(const float *tree_pts, int64_t N, int k, int mode, uint8_t *dims, cudaStream_t stream) {
    uint32_t *box = nullptr;
    if (mode == KDT_SPLIT_WIDEST) {
        if (cudaMallocAsync(reinterpret_cast<void **>(&box), (size_t)2 * k * 4, stream) != cudaSuccess) {
            cudaGetLastError();
            return KDT_ENOMEM;
        }
        if (cudaMemsetAsync(box, 0xff, (size_t)k * 4, stream) != cudaSuccess ||
            cudaMemsetAsync(box + k, 0x00, (size_t)k * 4, stream) != cudaSuccess)
            return KDT_ECUDA;
        tree_bbox_kernel<<<grid_for(N, kDimThreads, 4), kDimThreads, 0, stream>>>(tree_pts, N, k, box);
        if (cudaGetLastError() != cudaSuccess) return KDT_ECUDA;
    }
    {
        ProfScope ps(stream, "node_dims", 0.0);
        node_dims_kernel<<<grid_for(N, kDimThreads, 8), kDimThreads, 0, stream>>>(tree_pts, N, k, mode, box, dims);
        if (cudaGetLastError() != cudaSuccess) return KDT_ECUDA;
    }
    if (box && cudaFreeAsync(box, stream) != cudaSuccess) return KDT_ECUDA;
    return KDT_OK;
}

int enqueue_knn(const float *tree_pts, int64_t N, int k, const uint8_t *dims, const float *queries, int64_t Q,
                int K, int32_t *out_node, float *out_dist2, int *status, cudaStream_t stream) {
    if (Q == 0) return KDT_OK;
    ProfScope ps(stream, "knn", 0.0);
    const unsigned blocks = (unsigned)((Q + kQueryThreads - 1) / kQueryThreads);
    switch (K) {
#define KDT_KNN_CASE(KK)                                                                                        \
    case KK:                                                                                                    \
        knn_kernel<KK><<<blocks, kQueryThreads, 0, stream>>>(tree_pts, N, k, dims, queries, Q, K, out_node,   \
                                                             out_dist2, status);                               \
        break;
        KDT_KNN_CASE(1)
        KDT_KNN_CASE(2)
        KDT_KNN_CASE(4)
        KDT_KNN_CASE(8)
        KDT_KNN_CASE(16)
#undef KDT_KNN_CASE
        default:
            knn_kernel<0><<<blocks, kQueryThreads, 0, stream>>>(tree_pts, N, k, dims, queries, Q, K, out_node,
                                                                out_dist2, status);
    }
    return cudaGetLastError() == cudaSuccess ? KDT_OK : KDT_ECUDA;
}

}  // namespace kdt
