// kdt_build.cu -- the build path: init, per-level segment split, shared-memory
// finisher.
//
// Method ("GPU-friendly, Parallel, and (Almost-)In-Place Construction of
// Left-Balanced k-d Trees", core-idea and tag-update passages): all points
// start in the root's subtree; level by level every live subtree s is split
// at the point of rank ss(lChild(s)) under s's split order, that point becomes
// node s, the lower points form subtree lChild(s) and the higher ones
// rChild(s).  After numLevels(N) levels every point sits at its node.
//
// In the paper every step sorts all points by (subtree tag, split key) and
// then reads each point's new tag off its sorted position.  Only one fact of
// that sort is used -- which side of rank ss(lChild(s)) a point falls on --
// so this builder replaces the sort by an exact rank select plus a partition,
// which gives the same subtree sets and therefore the same tree.  The array
// layout is the paper's: after level l the F(l+1) fixed nodes own positions
// 0..F(l+1)-1 (their points go straight to the output), and live subtree s
// of level l+1 occupies [sb(s, l+1), sb(s, l+1) + ss(s)).
//
// Points are carried as 16-byte records: k order-preserving coordinate keys
// plus the input index, four words per group, G = ceil((k+1)/4) group
// columns, double-buffered.  With k = 3 points in device memory the first
// level builds the records itself from the input, so init only reduces the
// bounding box and writes the first coordinate's keys.  Every build kernel
// is launched as a programmatic dependent of the one before it
// (launch_pdl / pdl_enter).
#include <cstdio>

#include "kdt_internal.cuh"
#include "kdt_select.cuh"

namespace kdt {

constexpr int kInitThreads = 256;

// ---------------------------------------------------------------------------
// init: AoS float points -> SoA keys + index; finiteness; bounding box

constexpr int kInitPPT = 4;  // points per thread per iteration

// Folds every thread's per-coordinate key minima and maxima (k <= KM) into
// the CTA's, then into bbox: one global atomic per coordinate and CTA (the
// bounding box's 2k words would otherwise take one per warp each).
template <int KM>
__device__ __forceinline__ void bbox_fold(const uint32_t (&mn)[KM], const uint32_t (&mx)[KM], int k,
                                          uint32_t *bbox) {
    __shared__ uint32_t smn[KM], smx[KM];
    const uint32_t t = threadIdx.x;
    if (t < (uint32_t)KM) {
        smn[t] = 0xffffffffu;
        smx[t] = 0u;
    }
    __syncthreads();
#pragma unroll
    for (int c = 0; c < KM; ++c) {
        if (c < k) {
            const uint32_t a = __reduce_min_sync(0xffffffffu, mn[c]);
            const uint32_t b = __reduce_max_sync(0xffffffffu, mx[c]);
            if ((t & 31u) == 0u) {
                atomicMin(&smn[c], a);
                atomicMax(&smx[c], b);
            }
        }
    }
    __syncthreads();
    if (t < (uint32_t)k) {
        atomicMin(&bbox[t], smn[t]);
        atomicMax(&bbox[k + t], smx[t]);
    }
}

// KM: compile-time bound on k (4, 8, 16 or 32), so that the per-dimension
// minima and maxima stay in registers without reserving 2 * KDT_MAX_K of them
// for small k.  Each point's record (keys, then its input index) is written
// whole: for k <= 3 one 16-byte store, otherwise four words at a time.
template <int KM>
__global__ void __launch_bounds__(kInitThreads) init_kernel(const float *__restrict__ pts, int64_t N,
                                                            int k, int64_t ld, uint4 *__restrict__ rec,
                                                            uint32_t *__restrict__ bbox,
                                                            int *__restrict__ status) {
    pdl_enter();
    uint32_t mn[KM], mx[KM];
#pragma unroll
    for (int c = 0; c < KM; ++c) {
        mn[c] = 0xffffffffu;
        mx[c] = 0u;
    }
    int bad = 0;
    const int64_t nt = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i0 < N; i0 += nt * kInitPPT) {
        if (KM == 4) {
            // the kInitPPT points' loads go out before the stores, one
            // dimension at a time (coalesced across the warp)
            uint4 r[kInitPPT];
#pragma unroll
            for (int u = 0; u < kInitPPT; ++u) r[u] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (c < k) {
                    float f[kInitPPT];
#pragma unroll
                    for (int u = 0; u < kInitPPT; ++u) {
                        const int64_t i = i0 + u * nt;
                        f[u] = i < N ? __ldg(pts + i * k + c) : 0.f;
                    }
#pragma unroll
                    for (int u = 0; u < kInitPPT; ++u) {
                        if (i0 + u * nt < N) {
                            bad |= !isfinite(f[u]);
                            const uint32_t key = f2key(f[u]);
                            u4_set(r[u], c, key);
                            mn[c] = min(mn[c], key);
                            mx[c] = max(mx[c], key);
                        }
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kInitPPT; ++u) {
                const int64_t i = i0 + u * nt;
                if (i < N) {
                    u4_set(r[u], k, (uint32_t)i);
                    rec[i] = r[u];
                }
            }
        } else if ((k & 3) == 0 && (reinterpret_cast<uintptr_t>(pts) & 15u) == 0) {
            // k a multiple of 4, points 16-byte aligned: each group of four
            // keys is one 128-bit load, all of them issued before the stores
            constexpr int GM = KM / 4;
            const int gk = k >> 2;
            const uint4 *p4 = reinterpret_cast<const uint4 *>(pts);
            uint4 v[kInitPPT][GM];
#pragma unroll
            for (int u = 0; u < kInitPPT; ++u) {
                const int64_t i = i0 + u * nt;
#pragma unroll
                for (int g = 0; g < GM; ++g) v[u][g] = g < gk && i < N ? __ldg(p4 + i * gk + g) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < kInitPPT; ++u) {
                const int64_t i = i0 + u * nt;
                if (i >= N) continue;
#pragma unroll
                for (int g = 0; g < GM; ++g) {
                    if (g >= gk) break;
                    uint4 r;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float f = __uint_as_float(u4_word(v[u][g], j));
                        bad |= !isfinite(f);
                        const uint32_t key = f2key(f);
                        mn[4 * g + j] = min(mn[4 * g + j], key);
                        mx[4 * g + j] = max(mx[4 * g + j], key);
                        u4_set(r, j, key);
                    }
                    rec[(int64_t)g * ld + i] = r;
                }
                rec[(int64_t)gk * ld + i] = make_uint4((uint32_t)i, 0u, 0u, 0u);  // word k: the index
            }
        } else {
            // words 0..k of each record: keys, then the index; a group is
            // stored once its four words (or the last, word k) are set
#pragma unroll
            for (int u = 0; u < kInitPPT; ++u) {
                const int64_t i = i0 + u * nt;
                if (i >= N) continue;
                uint4 r = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int wd = 0; wd <= KM; ++wd) {
                    if (wd > k) break;
                    if (wd < k) {
                        const float f = __ldg(pts + i * k + wd);
                        bad |= !isfinite(f);
                        const uint32_t key = f2key(f);
                        if (wd < KM) {
                            mn[wd] = min(mn[wd], key);
                            mx[wd] = max(mx[wd], key);
                        }
                        u4_set(r, wd & 3, key);
                    } else {
                        u4_set(r, wd & 3, (uint32_t)i);
                    }
                    if ((wd & 3) == 3 || wd == k) {
                        rec[(int64_t)(wd >> 2) * ld + i] = r;
                        r = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            }
        }
    }
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) set_status(status, KDT_ENONFINITE);
    bbox_fold<KM>(mn, mx, k, bbox);
}

// k = 3, points 16-byte aligned: four points are three 128-bit loads, and two
// such groups per thread are in flight at once.  Besides the records (`rec`,
// null when the first level reads the points itself), the first
// coordinate's keys go to a dense column (`col0`, may be null) that the
// first level's histogram reads instead of the 16-byte records.
constexpr int kInit3Threads = 256;

__device__ __forceinline__ void init3_point(float x, float y, float z, uint32_t i, uint4 &r, uint32_t *mn,
                                            uint32_t *mx, int &bad) {
    bad |= !isfinite(x) | !isfinite(y) | !isfinite(z);
    r.x = f2key(x);
    r.y = f2key(y);
    r.z = f2key(z);
    r.w = i;
    mn[0] = min(mn[0], r.x);
    mx[0] = max(mx[0], r.x);
    mn[1] = min(mn[1], r.y);
    mx[1] = max(mx[1], r.y);
    mn[2] = min(mn[2], r.z);
    mx[2] = max(mx[2], r.z);
}

__global__ void __launch_bounds__(kInit3Threads, 4) init3_kernel(const float *__restrict__ pts, int64_t N,
                                                                 uint4 *__restrict__ rec, uint32_t *__restrict__ col0,
                                                                 uint32_t *__restrict__ bbox,
                                                                 int *__restrict__ status) {
    pdl_enter();
    uint32_t mn[3] = {0xffffffffu, 0xffffffffu, 0xffffffffu}, mx[3] = {0u, 0u, 0u};
    int bad = 0;
    const int64_t groups = N >> 2;  // groups of four points
    const int64_t nt = (int64_t)gridDim.x * blockDim.x;
    const uint4 *p4 = reinterpret_cast<const uint4 *>(pts);
    for (int64_t g0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g0 < groups; g0 += 2 * nt) {
        uint4 v[2][3];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int64_t g = g0 + u * nt;
#pragma unroll
            for (int j = 0; j < 3; ++j) v[u][j] = g < groups ? __ldg(p4 + 3 * g + j) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int64_t g = g0 + u * nt;
            if (g >= groups) continue;
            float f[12];
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                f[4 * j + 0] = __uint_as_float(v[u][j].x);
                f[4 * j + 1] = __uint_as_float(v[u][j].y);
                f[4 * j + 2] = __uint_as_float(v[u][j].z);
                f[4 * j + 3] = __uint_as_float(v[u][j].w);
            }
            uint4 r[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                init3_point(f[3 * i], f[3 * i + 1], f[3 * i + 2], (uint32_t)(4 * g + i), r[i], mn, mx, bad);
            if (rec)
#pragma unroll
                for (int i = 0; i < 4; ++i) rec[4 * g + i] = r[i];
            if (col0) reinterpret_cast<uint4 *>(col0)[g] = make_uint4(r[0].x, r[1].x, r[2].x, r[3].x);
        }
    }
    // the last N mod 4 points
    const int64_t tail = (int64_t)blockIdx.x * blockDim.x + threadIdx.x + (groups << 2);
    if (tail < N) {
        uint4 r;
        init3_point(pts[3 * tail], pts[3 * tail + 1], pts[3 * tail + 2], (uint32_t)tail, r, mn, mx, bad);
        if (rec) rec[tail] = r;
        if (col0) col0[tail] = r.x;
    }
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) set_status(status, KDT_ENONFINITE);
    bbox_fold<3>(mn, mx, 3, bbox);
}

// Root node table entry: domain = bounding box of all points, dim = widest.
__global__ void root_table_kernel(const uint32_t *bbox, int k, float *dom, int *dim) {
    pdl_enter();
    float lo[kMaxK], hi[kMaxK];
    for (int c = 0; c < k; ++c) {
        lo[c] = key2f(bbox[c]);
        hi[c] = key2f(bbox[k + c]);
        dom[c] = lo[c];
        dom[k + c] = hi[c];
    }
    dim[0] = widest_dim(lo, hi, k);
}

// ---------------------------------------------------------------------------
// plan, workspace and enqueue

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int make_plan(int64_t N, int k, int mode, Plan *p, int shape) {
    if (N < 1 || N > 2147483647LL || k < 1 || k > kMaxK || (mode != 0 && mode != 1)) return KDT_EINVAL;
    if (shape != kShapeLeftBalanced && (shape != kShapeBalanced || mode != KDT_SPLIT_ROUND_ROBIN)) return KDT_EINVAL;
    Plan q{};
    q.S = make_shape(N, shape);
    q.k = k;
    q.mode = mode;
    if (pick_tile(k, mode, &q.tp) != 0) return KDT_EINVAL;
    int lf = 0;
    while (lf < q.S.L && largest_subtree(q.S, lf) > q.tp.tile) ++lf;
    q.finish_level = lf;
    int lm = 0;
    // every level with few subtrees runs on the whole GPU (multi-CTA); the
    // one-CTA-per-subtree kernel needs enough subtrees to fill the SMs
    while (lm < lf && ((int64_t)1 << lm) <= kMultiMaxSegs) ++lm;
    q.multi_levels = lm;
    q.table_cap = (int64_t)1 << lf;
    // every global level but the first gets its histograms from the level
    // above (round-robin rule, k >= 2): one row per subtree of the deepest
    q.hist_rows = lf > 0 ? ((int64_t)1 << (lf - 1)) : 0;
    q.sel_cap = lf > 0 ? ((int64_t)1 << (lf - 1)) : 0;
    size_t off = 0;
    q.off_status = off;
    off = align_up(off + 64, 256);
    q.off_bbox = off;
    off = align_up(off + (size_t)2 * k * 4, 256);
    q.ld = (N + 7) & ~(int64_t)7;
    for (int b = 0; b < 3; ++b) {
        const int64_t rows = (b < 2 || lf > 0) ? q.ld : 0;
        q.off_rec[b] = off;
        off = align_up(off + (size_t)rec_groups(k) * rows * 16, 256);
    }
    for (int b = 0; b < 2; ++b) {
        q.off_dom[b] = off;
        off = align_up(off + (size_t)q.table_cap * 2 * k * 4, 256);
        q.off_dim[b] = off;
        off = align_up(off + (size_t)q.table_cap * 4, 256);
        q.off_hist[b] = off;
        const int64_t words = q.hist_rows * kBuckets;
        off = align_up(off + (size_t)(b == 0 && words < kBuckets0 ? kBuckets0 : words) * 4, 256);  // level 0: kBuckets0
    }
    for (int t = 0; t < 2; ++t) {
        q.off_sel[t] = off;
        off = align_up(off + (size_t)q.sel_cap * sizeof(SegSel), 256);
    }
    q.off_fb = off;
    off = align_up(off + (size_t)q.table_cap, 256);
    q.bytes = off;
    *p = q;
    return KDT_OK;
}

Buffers carve(const Plan &p, void *base) {
    unsigned char *b = static_cast<unsigned char *>(base);
    Buffers r;
    r.status = reinterpret_cast<int *>(b + p.off_status);
    r.bbox = reinterpret_cast<uint32_t *>(b + p.off_bbox);
    for (int i = 0; i < 3; ++i) r.rec[i] = reinterpret_cast<uint4 *>(b + p.off_rec[i]);
    r.col0 = nullptr;
    r.pts3 = nullptr;
    for (int i = 0; i < 2; ++i) {
        r.dom[i] = reinterpret_cast<float *>(b + p.off_dom[i]);
        r.dim[i] = reinterpret_cast<int *>(b + p.off_dim[i]);
        r.hist[i] = reinterpret_cast<uint32_t *>(b + p.off_hist[i]);
    }
    r.sel[0] = reinterpret_cast<SegSel *>(b + p.off_sel[0]);
    r.sel[1] = reinterpret_cast<SegSel *>(b + p.off_sel[1]);
    r.fallback = b + p.off_fb;
    return r;
}

#define KDT_LAUNCH_CHECK()                                      \
    do {                                                        \
        cudaError_t e_ = cudaGetLastError();                    \
        if (e_ != cudaSuccess) return KDT_ECUDA;                \
    } while (0)

int enqueue_build(const Plan &p, const Buffers &b_in, const float *pts, int32_t *perm, cudaStream_t stream,
                  bool pts_in_hbm) {
    Buffers b = b_in;
    const Shape &S = p.S;
    const int k = p.k;
    const double Nd = (double)S.N;
    if (cudaMemsetAsync(b.status, 0, 2 * sizeof(int), stream) != cudaSuccess) return KDT_ECUDA;  // status, level-0 done count
    if (S.kind == kShapeBalanced) {  // heap slots of empty subtrees read -1
        const size_t slots = (((size_t)1) << S.L) - 1;
        if (cudaMemsetAsync(perm, 0xff, slots * sizeof(int32_t), stream) != cudaSuccess) return KDT_ECUDA;
    }
    if (cudaMemsetAsync(b.bbox, 0xff, (size_t)k * 4, stream) != cudaSuccess) return KDT_ECUDA;
    if (cudaMemsetAsync(b.bbox + k, 0x00, (size_t)k * 4, stream) != cudaSuccess) return KDT_ECUDA;
    {
        int dev = 0, sms = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        int64_t blocks = (S.N + kInitThreads * kInitPPT - 1) / (kInitThreads * kInitPPT);
        const int64_t cap = (int64_t)(sms > 0 ? sms : 152) * 16;
        if (blocks > cap) blocks = cap;
        ProfScope ps(stream, "init", 0.0);
        if (k == 3 && (reinterpret_cast<uintptr_t>(pts) & 15u) == 0) {
            // the first level's histogram reads a dense copy of the first
            // coordinate's keys, kept in the candidate buffer until that level
            uint32_t *col0 = p.finish_level > 0 && p.mode == KDT_SPLIT_ROUND_ROBIN
                                 ? reinterpret_cast<uint32_t *>(b.rec[2]) : nullptr;
            b.col0 = col0;
            // with the points in HBM, the first (multi-CTA, round-robin)
            // level reads them directly and builds the records in registers:
            // the 16-byte records are neither written here nor read there
            if (pts_in_hbm && col0 && p.multi_levels > 0) b.pts3 = pts;
            int64_t g3 = (S.N / 4 + 2 * kInit3Threads - 1) / (2 * kInit3Threads);
            const int64_t cap3 = (int64_t)(sms > 0 ? sms : 152) * 16;
            if (g3 > cap3) g3 = cap3;
            if (g3 < 1) g3 = 1;
            launch_pdl(init3_kernel, (unsigned)g3, kInit3Threads, 0, stream, pts, S.N, b.pts3 ? nullptr : b.rec[0], col0,
                                                                    b.bbox, b.status);
        } else if (k <= 3)
            launch_pdl(init_kernel<4>, (unsigned)blocks, kInitThreads, 0, stream, pts, S.N, k, p.ld, b.rec[0], b.bbox,
                                                                          b.status);
        else if (k <= 8)
            launch_pdl(init_kernel<8>, (unsigned)blocks, kInitThreads, 0, stream, pts, S.N, k, p.ld, b.rec[0], b.bbox,
                                                                          b.status);
        else if (k <= 16)
            launch_pdl(init_kernel<16>, (unsigned)blocks, kInitThreads, 0, stream, pts, S.N, k, p.ld, b.rec[0], b.bbox,
                                                                           b.status);
        else
            launch_pdl(init_kernel<32>, (unsigned)blocks, kInitThreads, 0, stream, pts, S.N, k, p.ld, b.rec[0], b.bbox,
                                                                           b.status);
        KDT_LAUNCH_CHECK();
    }
    {
        ProfScope ps(stream, "root_table", 0.0);
        launch_pdl(root_table_kernel, 1, 1, 0, stream, b.bbox, k, b.dom[0], b.dim[0]);
        KDT_LAUNCH_CHECK();
    }
    int src = 0;
    for (int l = 0; l < p.finish_level; ++l) {
        const int rc = enqueue_level(p, b, l, src, perm, stream);
        if (rc != KDT_OK) return rc;
        src ^= 1;
    }
    {
        const int rc = enqueue_finisher(p, b, src, perm, stream);
        if (rc != KDT_OK) return rc;
    }
    enqueue_status_fold(b.status, stream);
    KDT_LAUNCH_CHECK();
    return KDT_OK;
}

}  // namespace kdt
