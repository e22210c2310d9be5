// kdt_internal.cuh -- private declarations of the GB300 k-d tree builder.
//
// Notation ("GPU-friendly, Parallel, and (Almost-)In-Place Construction of
// Left-Balanced k-d Trees", notation paragraph): nodes are numbered in level
// order, level(i) = floor(log2(i+1)), L = numLevels(N) = level(N-1)+1,
// F(l) = 2^l - 1 nodes above level l.  The paper announces O(1) forms for the
// subtree size ss(s) and the segment begin sb(s,l) but its text does not
// carry them; the forms below are derived from the left-balanced shape
// (levels 0..L-2 full, level L-1 filled from the left with M = N - F(L-1)
// nodes):
//   for s on level l, j = s - F(l), B = 2^(L-1-l), A = B - 1:
//     ss(s)   = A + clamp(M - j*B, 0, B)                (0 if s >= N)
//     sb(s,l) = F(l) + j*A + min(M, j*B)
// sb is the first array position of subtree s's points after level l has been
// split off: the F(l) nodes already fixed occupy positions 0..F(l)-1 and the
// live subtrees follow in node order.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

#include "kdtree_build.h"

namespace kdt {

constexpr int kMaxK = KDT_MAX_K;
constexpr int kMaxWords = kMaxK + 1;  // k coordinate keys + the input index

// ---- integer helpers usable on host and device -----------------------------

__host__ __device__ __forceinline__ int ilog2_u64(uint64_t v) {
#ifdef __CUDA_ARCH__
    return 63 - __clzll((long long)v);
#else
    return 63 - __builtin_clzll(v);
#endif
}

__host__ __device__ __forceinline__ int level_of(int64_t i) { return ilog2_u64((uint64_t)i + 1u); }

__host__ __device__ __forceinline__ int64_t full_nodes(int l) { return ((int64_t)1 << l) - 1; }

// Tree shapes.  KDT_SHAPE_LEFT_BALANCED: the left-balanced complete tree of
// the left-balanced paper (levels full but the last, which fills from the
// left).  KDT_SHAPE_BALANCED: the median-split tree of Brown's builder ("An
// Implementation of a Balanced Kd Tree Builder Using GPUs", overview list):
// a node of n points keeps the point of rank floor((n-1)/2), so its lower
// side has floor((n-1)/2) points and its upper side the rest; nodes are
// numbered in heap order with empty slots where a subtree is empty.
constexpr int kShapeLeftBalanced = 0, kShapeBalanced = 1;

struct Shape {
    int64_t N;  // number of points
    int L;      // numLevels(N): levels of either shape
    int64_t M;  // left-balanced: nodes on the last level
    int kind;   // kShapeLeftBalanced or kShapeBalanced
};

__host__ __device__ __forceinline__ Shape make_shape(int64_t N, int kind = kShapeLeftBalanced) {
    Shape S;
    S.N = N;
    S.L = level_of(N - 1) + 1;
    S.M = N - full_nodes(S.L - 1);
    S.kind = kind;
    return S;
}

// Balanced shape of n points: node i of level l (heap order) covers the gaps
// [g0, g0 + m) among the n + 1 gaps around its in-order positions -- its
// points are the in-order positions [g0, g0 + m - 1) (none if m <= 1) and its
// split point sits at g0 + floor(m/2) - 1.  The lower child gets floor(m/2)
// of the gaps, the upper child the rest: a walk from the root, O(l).
__host__ __device__ __forceinline__ void bal_node(int64_t n, int l, int64_t i, int64_t *g0, int64_t *m) {
    int64_t a = 0, c = n + 1;
    for (int t = l - 1; t >= 0; --t) {
        const int64_t h = c >> 1;
        if ((i >> t) & 1) {
            a += h;
            c -= h;
        } else {
            c = h;
        }
    }
    *g0 = a;
    *m = c;
}

// Largest subtree on level l (the splits of both shapes put at least as many
// points on the side that the largest subtree descends into).
__host__ __device__ __forceinline__ int64_t largest_subtree(const Shape &S, int l);

// ss(s) for node s on level l (0 if the node does not exist).
__host__ __device__ __forceinline__ int64_t seg_size(const Shape &S, int l, int64_t s) {
    if (S.kind == kShapeBalanced) {
        if (l >= S.L) return 0;
        int64_t g0, m;
        bal_node(S.N, l, s - full_nodes(l), &g0, &m);
        return m > 1 ? m - 1 : 0;
    }
    if (l >= S.L || s >= S.N) return 0;
    const int64_t B = (int64_t)1 << (S.L - 1 - l);
    const int64_t A = B - 1;
    const int64_t j = s - full_nodes(l);
    int64_t r = S.M - j * B;
    r = r < 0 ? 0 : (r > B ? B : r);
    return A + r;
}

// sb(s, l) for node s on level l: the first array position of subtree s when
// the F(l) nodes above level l own positions 0..F(l)-1 and the live subtrees
// follow in node order (balanced shape: on levels whose nodes all hold points,
// where the i subtrees before node i are separated by i fixed positions in
// the in-order numbering).
__host__ __device__ __forceinline__ int64_t seg_begin(const Shape &S, int l, int64_t s) {
    if (S.kind == kShapeBalanced) {
        int64_t g0, m;
        const int64_t i = s - full_nodes(l);
        bal_node(S.N, l, i, &g0, &m);
        return full_nodes(l) + g0 - i;
    }
    const int64_t B = (int64_t)1 << (S.L - 1 - l);
    const int64_t A = B - 1;
    const int64_t j = s - full_nodes(l);
    const int64_t t = j * B;
    return full_nodes(l) + j * A + (t < S.M ? t : S.M);
}

__host__ __device__ __forceinline__ int64_t largest_subtree(const Shape &S, int l) {
    if (l >= S.L) return 0;
    if (S.kind == kShapeBalanced) return S.N >> l;  // the upper child of n points has floor(n/2)
    return seg_size(S, l, full_nodes(l));           // the first subtree of a level is the largest
}

// 32-bit forms of ss and sb for device code (left-balanced shape): with
// N < 2^31 every node id, size and position fits; requires l < L and s on
// level l.
__device__ __forceinline__ int32_t seg_size32(const Shape &S, int l, int32_t s) {
    if (s >= (int32_t)S.N) return 0;
    const int32_t B = 1 << (S.L - 1 - l);
    const int32_t j = s - ((1 << l) - 1);
    int32_t r = (int32_t)S.M - j * B;
    r = r < 0 ? 0 : (r > B ? B : r);
    return B - 1 + r;
}

__device__ __forceinline__ int32_t seg_begin32(const Shape &S, int l, int32_t s) {
    const int32_t B = 1 << (S.L - 1 - l);
    const int32_t j = s - ((1 << l) - 1);
    const int32_t t = j * B;
    return ((1 << l) - 1) + j * (B - 1) + (t < (int32_t)S.M ? t : (int32_t)S.M);
}

// Number of node slots of level l that the build visits (left-balanced: the
// nodes that exist; balanced: every slot of the level).
__host__ __device__ __forceinline__ int64_t nodes_on_level(const Shape &S, int l) {
    const int64_t w = (int64_t)1 << l;
    if (S.kind == kShapeBalanced) return w;
    const int64_t left = S.N - full_nodes(l);
    return left < w ? left : w;
}

// ---- programmatic dependent launch ----------------------------------------------
// The build's kernels are launched so that each may be scheduled while the
// one before it drains (its launch and setup overlap that tail).  Every such
// kernel calls pdl_enter() first: it waits until the kernel before it has
// completed and its writes are visible (so, transitively, everything before
// that), then lets the kernel after it be scheduled.

__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <class... KArgs, class... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---- order-preserving float keys -------------------------------------------
// Unsigned comparison of the keys equals IEEE '<' on finite floats, with -0
// folded onto +0 so that the two zeros compare equal (as '<' does).

__device__ __forceinline__ uint32_t f2key(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key2f(uint32_t k) {
    const uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
    return __uint_as_float(u);
}

// Widest extent of a domain: argmax of hi - lo (float32, round to nearest),
// lowest dimension on ties.
__device__ __forceinline__ int widest_dim(const float *lo, const float *hi, int k) {
    int best = 0;
    float ext = __fsub_rn(hi[0], lo[0]);
    for (int d = 1; d < k; ++d) {
        const float e = __fsub_rn(hi[d], lo[d]);
        if (e > ext) {
            ext = e;
            best = d;
        }
    }
    return best;
}

// ---- point records -----------------------------------------------------------
// On the global levels a point travels as a record of words: its k order-
// preserving keys (words 0..k-1) and its input index (word k), grouped four
// to a 16-byte uint4.  A record buffer holds G = ceil((k+1)/4) group columns
// of ld uint4 each -- group g of record q at g * ld + q -- so for k <= 3 a
// whole record is one 128-bit load or store (padding words are unused).

__host__ __device__ __forceinline__ int rec_groups(int k) { return (k + 4) / 4; }

__device__ __forceinline__ uint32_t u4_word(const uint4 &v, int i) {
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

__device__ __forceinline__ void u4_set(uint4 &v, int i, uint32_t x) {
    if (i == 0) v.x = x;
    else if (i == 1) v.y = x;
    else if (i == 2) v.z = x;
    else v.w = x;
}

// Word w of record q.
__device__ __forceinline__ uint32_t rec_word(const uint4 *r, int64_t ld, int w, int64_t q) {
    return reinterpret_cast<const uint32_t *>(r + (int64_t)(w >> 2) * ld + q)[w & 3];
}

// ---- device status ----------------------------------------------------------

__device__ __forceinline__ void set_status(int *status, int code) { atomicCAS(status, 0, code); }

// ---- workspace --------------------------------------------------------------

// Finisher tile limits: a subtree whose point count is at most `tile` is
// finished inside one CTA's shared memory.
struct TilePlan {
    int tile;           // T: max points per finisher CTA
    int nb;             // value buckets of the sorted finisher's counting sort
    size_t smem;        // dynamic shared memory per sorted-finisher CTA
    size_t smem_select; // dynamic shared memory per select-finisher CTA
};

constexpr size_t kSelectSmemMax = 200 * 1024;  // select finisher: at least one CTA per SM

// Per live subtree of a global level: the value bucket that holds the split
// rank, the point counts below it and in it, and the partition cursors.
struct SegSel {
    uint32_t bstar, below, cnt;
    uint32_t curL, curC, curR;
    uint32_t klo, khi;  // keys of the split bucket: [klo, khi)
};

constexpr int kBuckets = 2048;         // value buckets per subtree on global levels
constexpr int kBuckets0 = 16384;       // value buckets of level 0 (one subtree, its own histogram pass)
constexpr int64_t kBuckets0Min = 1 << 24;  // ... from this many points on (below, kBuckets: the pass is latency-bound)
constexpr int kMultiMaxSegs = 1024;    // multi-CTA levels: at most this many subtrees

struct Plan {
    Shape S;
    int k;
    int mode;
    int finish_level;    // first level whose largest subtree fits a finisher tile
    int multi_levels;    // levels [0, multi_levels) use the multi-CTA pipeline
    TilePlan tp;
    int64_t table_cap;   // node-table entries per level
    int64_t hist_rows;   // histogram rows per buffer (multi-CTA levels)
    int64_t sel_cap;     // SegSel entries per table (two tables, by level parity)
    int64_t ld;          // records per group column (N rounded up to 8)
    // byte offsets inside the workspace
    size_t off_status, off_bbox, off_rec[3], off_dom[2], off_dim[2], off_hist[2], off_sel[2], off_fb;
    size_t bytes;
};

// shape: kShapeLeftBalanced (either split rule) or kShapeBalanced (the
// round-robin rule only).
int make_plan(int64_t N, int k, int mode, Plan *p, int shape = kShapeLeftBalanced);

struct Buffers {
    int *status;
    uint32_t *bbox;  // [2k]: min keys then max keys
    uint4 *rec[3];   // record buffers: [0], [1] ping-pong, [2] bucket candidates
    const uint32_t *col0;  // dense keys of coordinate 0 for the first level's histogram, or null
    const float *pts3;     // k = 3 input points that the first level reads in place of records, or null
    float *dom[2];   // node tables: entry e holds lo[k] then hi[k]
    int *dim[2];
    uint32_t *hist[2];  // [rows][kBuckets]
    SegSel *sel[2];     // per live subtree of a global level, by level parity
    uint8_t *fallback;  // [tiles]: 1 = tile left to the select finisher
};

Buffers carve(const Plan &p, void *base);

// Finisher tile choice and launch (kdt_finisher_sorted.cu): the sorted
// finisher runs every tile; tiles it leaves (flag set in Buffers::fallback)
// go to the select finisher (kdt_finisher.cu).
int pick_tile(int k, int mode, TilePlan *tp);
int enqueue_finisher(const Plan &p, const Buffers &b, int src, int32_t *perm, cudaStream_t stream);
size_t select_finisher_smem(int k, int T, int mode);
// Select finisher over the tiles whose flag in `only` is nonzero.
int launch_select_finisher(const Plan &p, const Buffers &b, int src, int32_t *perm, const uint8_t *only,
                           cudaStream_t stream);

// Enqueues one global level l (records move from buffer src to src^1).
int enqueue_level(const Plan &p, const Buffers &b, int l, int src, int32_t *perm, cudaStream_t stream);

// Enqueues the whole build on `stream`.  Returns a KDT_* code for launch errors.
// `pts_in_hbm`: pts is device memory (not host memory mapped into the
// device's address space), so reading it twice costs HBM bandwidth only.
int enqueue_build(const Plan &p, const Buffers &b, const float *pts, int32_t *perm,
                  cudaStream_t stream, bool pts_in_hbm = true);

// Per-kernel timing (profiling switch in kdt_api.cu).  `kernels`: kernel
// launches inside the scope (1 unless the code between the events says so).
struct ProfScope {
    cudaStream_t stream;
    const char *name;
    double bytes;
    cudaEvent_t ev0;
    bool on;
    int kernels;
    ProfScope(cudaStream_t s, const char *n, double b);
    ~ProfScope();
};

// Folds a build's status word into the per-device status word.
void enqueue_status_fold(int *status, cudaStream_t stream);
int read_and_clear_device_status(int *out);

int enqueue_verify(const float *pts, int64_t N, int k, int mode, const int32_t *perm,
                   cudaStream_t stream, int *result);

// Level-order points (kdt_gather.cu): out[u] = pts[perm[u]] (rows of k
// words); bad perm entries are recorded in *status.
int enqueue_gather(const float *pts, int64_t N, int k, const int32_t *perm, float *out, int *status,
                   cudaStream_t stream);
// After enqueue_build: rewrites pts in level order through the workspace
// (skipped if the build recorded an error).
int enqueue_inplace_tail(const Plan &p, const Buffers &b, float *pts, const int32_t *perm, cudaStream_t stream);
// Device address of the calling thread's current device's status word.
int *device_status_address();

// Queries on a built tree (kdt_query.cu).
int enqueue_node_dims(const float *tree_pts, int64_t N, int k, int mode, uint8_t *dims, cudaStream_t stream);
int enqueue_knn(const float *tree_pts, int64_t N, int k, const uint8_t *dims, const float *queries, int64_t Q,
                int K, int32_t *out_node, float *out_dist2, int *status, cudaStream_t stream);

}  // namespace kdt
