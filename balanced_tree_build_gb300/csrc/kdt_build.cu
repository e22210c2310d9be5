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
// so this build replaces the sort by an exact rank select plus a partition,
// which gives the same subtree sets and therefore the same tree.  The array
// layout is the paper's: after level l the F(l+1) fixed nodes own positions
// 0..F(l+1)-1 (their points go straight to the output), and live subtree s
// of level l+1 occupies [sb(s, l+1), sb(s, l+1) + ss(s)).
//
// Points are carried as records in structure-of-arrays form: k order-
// preserving coordinate keys plus the input index, double-buffered.
#include <cstdio>

#include "kdt_internal.cuh"
#include "kdt_select.cuh"

namespace kdt {

constexpr int kInitThreads = 256;
constexpr int kFinThreads = 512;
constexpr int kFinWarps = kFinThreads / 32;
constexpr int kWarpMax = 256;          // finisher: subtrees this small go to one warp
constexpr size_t kFinSmemBudget = 200 * 1024;

// ---------------------------------------------------------------------------
// init: AoS float points -> SoA keys + index; finiteness; bounding box

__global__ void __launch_bounds__(kInitThreads) init_kernel(const float *__restrict__ pts, int64_t N,
                                                            int k, uint32_t *__restrict__ keys,
                                                            uint32_t *__restrict__ idx,
                                                            uint32_t *__restrict__ bbox,
                                                            int *__restrict__ status) {
    uint32_t mn[kMaxK], mx[kMaxK];
#pragma unroll
    for (int c = 0; c < kMaxK; ++c) {
        mn[c] = 0xffffffffu;
        mx[c] = 0u;
    }
    int bad = 0;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < N; i += stride) {
#pragma unroll
        for (int c = 0; c < kMaxK; ++c) {
            if (c < k) {
                const float f = pts[i * k + c];
                bad |= !isfinite(f);
                const uint32_t key = f2key(f);
                keys[(int64_t)c * N + i] = key;
                mn[c] = min(mn[c], key);
                mx[c] = max(mx[c], key);
            }
        }
        idx[i] = (uint32_t)i;
    }
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) set_status(status, KDT_ENONFINITE);
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
}

// Root node table entry: domain = bounding box of all points, dim = widest.
__global__ void root_table_kernel(const uint32_t *bbox, int k, float *dom, int *dim) {
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
// finisher: one CTA owns a subtree of at most T points and fixes all of its
// remaining levels in shared memory.

struct FinArgs {
    Shape S;
    int k, mode, l0, T;
    const uint32_t *src_keys, *src_idx;
    int32_t *perm;
    const float *dom;  // node table of level l0 (widest mode)
    int *status;
};

struct FinSmem {
    uint32_t *keys;   // [k][T]
    uint32_t *idx;    // [T]
    uint16_t *ids[2]; // [T] each: local point ids in current order
    uint32_t *hist;   // [kFinWarps * kWarpRadixBins]
    float *sval;      // [T] split coordinate of tile-local node (widest mode)
    uint8_t *sdim;    // [T] split dimension of tile-local node (widest mode)
};

__host__ __device__ inline size_t fin_smem_bytes(int k, int T, int mode) {
    size_t b = (size_t)k * T * 4 + (size_t)T * 4 + (size_t)T * 4 + (size_t)kFinWarps * kWarpRadixBins * 4;
    if (mode == KDT_SPLIT_WIDEST) b += (size_t)T * 5;
    return (b + 15) & ~(size_t)15;
}

__device__ inline FinSmem fin_carve(unsigned char *p, int k, int T, int mode) {
    FinSmem f;
    f.keys = reinterpret_cast<uint32_t *>(p);
    p += (size_t)k * T * 4;
    f.idx = reinterpret_cast<uint32_t *>(p);
    p += (size_t)T * 4;
    f.hist = reinterpret_cast<uint32_t *>(p);
    p += (size_t)kFinWarps * kWarpRadixBins * 4;
    f.ids[0] = reinterpret_cast<uint16_t *>(p);
    p += (size_t)T * 2;
    f.ids[1] = reinterpret_cast<uint16_t *>(p);
    p += (size_t)T * 2;
    f.sval = reinterpret_cast<float *>(p);
    p += mode == KDT_SPLIT_WIDEST ? (size_t)T * 4 : 0;
    f.sdim = p;
    return f;
}

// Word i of the point at offset q of a sub-subtree whose ordered local ids
// start at `ids`.
struct SmemSeg {
    const uint32_t *keys, *idx;
    const uint16_t *ids;
    int T, k, d;
    __device__ __forceinline__ uint32_t operator()(int i, uint32_t q) const {
        const int id = ids[q];
        if (i == k) return idx[id];
        int c = d + i;
        if (c >= k) c -= k;
        return keys[c * T + id];
    }
};

// Split dimension of tile node u (level j) under the widest rule: walk from
// the tile root down to u, clipping the tile root's domain by each ancestor's
// split (the walk of the split-widest-dimension passage, top-down).
__device__ int fin_widest_dim_of(const FinArgs &a, const FinSmem &sm, int64_t s0, int j, int64_t u) {
    float lo[kMaxK], hi[kMaxK];
    const int k = a.k;
    const float *dom = a.dom + (s0 - full_nodes(a.l0)) * 2 * k;
    for (int c = 0; c < k; ++c) {
        lo[c] = dom[c];
        hi[c] = dom[k + c];
    }
    const int depth = j - a.l0;
    const int64_t first = ((s0 + 1) << depth) - 1;
    const int64_t lu = (((int64_t)1 << depth) - 1) + (u - first);
    int64_t cur = 0;
    for (int t = depth - 1; t >= 0; --t) {
        const int bit = (int)(((lu + 1) >> t) & 1);
        const int dd = sm.sdim[cur];
        const float v = sm.sval[cur];
        if (bit) lo[dd] = v;
        else hi[dd] = v;
        cur = 2 * cur + 1 + bit;
    }
    return widest_dim(lo, hi, k);
}

__device__ __forceinline__ int64_t tile_local_index(int64_t s0, int depth, int64_t u) {
    const int64_t first = ((s0 + 1) << depth) - 1;
    return (((int64_t)1 << depth) - 1) + (u - first);
}

__device__ __forceinline__ int fin_dim(const FinArgs &a, const FinSmem &sm, int64_t s0, int j, int64_t u) {
    return a.mode == KDT_SPLIT_ROUND_ROBIN ? j % a.k : fin_widest_dim_of(a, sm, s0, j, u);
}

// Fixes node u (level j) inside one warp: selects its split point among the
// n_u points at ids[cur][off_u..], writes perm[u], and moves the other local
// ids to the children's ranges of ids[cur^1].
//
// The warp owns the subtree of node t (level jt) whose points occupied
// [off_t, off_t + n_t) when the warp took it over.  Offsets below are laid out
// relative to that range, which therefore never moves: the descendants of t
// on each level are packed from off_t.  (Laid out relative to the whole tile
// instead, the ranges would shift left as medians leave, into a range that a
// neighbouring, unsynchronised warp may still be reading.)
__device__ void warp_split_node(const FinArgs &a, const FinSmem &sm, int64_t s0, int64_t t, int jt,
                                uint32_t off_t, int j, int64_t u, int cur, uint32_t *wf, uint32_t *hist) {
    const uint32_t lane = threadIdx.x & 31u;
    const Shape &S = a.S;
    const int depth = j - a.l0;
    const int64_t sub_base_j = seg_begin(S, j, ((t + 1) << (j - jt)) - 1);
    const uint32_t n_u = (uint32_t)seg_size(S, j, u);
    const uint32_t off_u = off_t + (uint32_t)(seg_begin(S, j, u) - sub_base_j);
    const bool has_children = j + 1 < S.L;
    const uint32_t m_u = has_children ? (uint32_t)seg_size(S, j + 1, 2 * u + 1) : 0u;
    uint32_t left_off = 0;
    if (has_children) {
        const int64_t sub_base_j1 = seg_begin(S, j + 1, ((t + 1) << (j + 1 - jt)) - 1);
        left_off = off_t + (uint32_t)(seg_begin(S, j + 1, 2 * u + 1) - sub_base_j1);
    }
    const uint32_t right_off = left_off + m_u;
    const int d = fin_dim(a, sm, s0, j, u);
    const int k = a.k;
    const uint16_t *src = sm.ids[cur] + off_u;
    uint16_t *dst = sm.ids[cur ^ 1];
    const int64_t lu = tile_local_index(s0, depth, u);

    if (n_u <= 32u) {
        // all-pairs rank: each lane holds one point
        const bool valid = lane < n_u;
        const uint32_t my_id = valid ? src[lane] : 0u;
        const uint32_t my_w0 = valid ? sm.keys[d * a.T + my_id] : 0u;
        uint32_t rank = 0;
        for (uint32_t t = 0; t < n_u; ++t) {
            const uint32_t oid = __shfl_sync(0xffffffffu, my_id, t);
            const uint32_t ow0 = __shfl_sync(0xffffffffu, my_w0, t);
            if (valid) {
                bool lt;
                if (ow0 != my_w0) {
                    lt = ow0 < my_w0;
                } else {
                    lt = false;
                    if (oid != my_id) {
                        int i = 1;
                        for (; i < k; ++i) {
                            int c = d + i;
                            if (c >= k) c -= k;
                            const uint32_t x = sm.keys[c * a.T + oid], y = sm.keys[c * a.T + my_id];
                            if (x != y) {
                                lt = x < y;
                                break;
                            }
                        }
                        if (i == k) lt = sm.idx[oid] < sm.idx[my_id];
                    }
                }
                rank += lt ? 1u : 0u;
            }
        }
        if (valid) {
            if (rank == m_u) {
                a.perm[u] = (int32_t)sm.idx[my_id];
                if (a.mode == KDT_SPLIT_WIDEST && lu < a.T) {
                    sm.sval[lu] = key2f(my_w0);
                    sm.sdim[lu] = (uint8_t)d;
                }
            } else if (rank < m_u) {
                dst[left_off + rank] = (uint16_t)my_id;
            } else {
                dst[right_off + rank - m_u - 1u] = (uint16_t)my_id;
            }
        }
        return;
    }

    const SmemSeg acc{sm.keys, sm.idx, src, a.T, k, d};
    const uint32_t med = warp_select(acc, n_u, m_u, k + 1, wf, hist);
    if (med == 0xffffffffu) {
        if (lane == 0) set_status(a.status, KDT_EINTERNAL);
        return;
    }
    // median words into wf (reuse)
    __syncwarp();
    if (lane <= (uint32_t)k) wf[lane] = acc((int)lane, med);
    __syncwarp();
    const uint32_t lt_mask = (1u << lane) - 1u;
    uint32_t lc = 0, rc = 0;
    for (uint32_t q0 = 0; q0 < n_u; q0 += 32) {
        const uint32_t q = q0 + lane;
        int side = -1;
        if (q < n_u) {
            const int c = cmp_words(acc, q, wf, k + 1);
            side = c < 0 ? 0 : (c > 0 ? 1 : -1);
        }
        const uint32_t lm = __ballot_sync(0xffffffffu, side == 0);
        const uint32_t rm = __ballot_sync(0xffffffffu, side == 1);
        if (side == 0) {
            const uint32_t o = lc + __popc(lm & lt_mask);
            if (o < m_u) dst[left_off + o] = src[q];
            else set_status(a.status, KDT_EINTERNAL);
        } else if (side == 1) {
            const uint32_t o = rc + __popc(rm & lt_mask);
            if (o < n_u - m_u - 1u) dst[right_off + o] = src[q];
            else set_status(a.status, KDT_EINTERNAL);
        }
        lc += __popc(lm);
        rc += __popc(rm);
    }
    if (lane == 0) {
        const uint32_t id = src[med];
        a.perm[u] = (int32_t)sm.idx[id];
        if (a.mode == KDT_SPLIT_WIDEST && lu < a.T) {
            sm.sval[lu] = key2f(wf[0]);
            sm.sdim[lu] = (uint8_t)d;
        }
    }
    __syncwarp();
}

__global__ void __launch_bounds__(kFinThreads) finisher_kernel(FinArgs a) {
    extern __shared__ __align__(16) unsigned char fin_smem[];
    __shared__ SelState st;
    __shared__ uint32_t red[64];
    __shared__ uint32_t medw[kMaxWords];
    __shared__ uint32_t wfs[kFinWarps][kMaxWords];
    __shared__ uint32_t cursor[2];
    __shared__ int stop;
    const uint32_t tid = threadIdx.x;
    if (tid == 0) stop = *(volatile int *)a.status;
    __syncthreads();
    if (stop) return;

    const Shape &S = a.S;
    const int k = a.k;
    const FinSmem sm = fin_carve(fin_smem, k, a.T, a.mode);
    const int64_t s0 = full_nodes(a.l0) + blockIdx.x;
    const uint32_t n = (uint32_t)seg_size(S, a.l0, s0);
    const int64_t base = seg_begin(S, a.l0, s0);
    const int64_t N = S.N;
    if (n > (uint32_t)a.T) {
        if (tid == 0) set_status(a.status, KDT_EINTERNAL);
        return;
    }
    for (uint32_t q = tid; q < n; q += blockDim.x) {
        for (int c = 0; c < k; ++c) sm.keys[c * a.T + q] = a.src_keys[(int64_t)c * N + base + q];
        sm.idx[q] = a.src_idx[base + q];
        sm.ids[0][q] = (uint16_t)q;
    }
    __syncthreads();

    // Phase A: the whole CTA splits each large node in turn.
    int j = a.l0, cur = 0;
    while (j < S.L) {
        const int depth = j - a.l0;
        const int64_t first = ((s0 + 1) << depth) - 1;
        if (seg_size(S, j, first) <= (int64_t)kWarpMax) break;
        const int64_t tile_base_j = seg_begin(S, j, first);
        const int64_t tile_base_j1 = seg_begin(S, j + 1, ((s0 + 1) << (depth + 1)) - 1);
        const int64_t count = (int64_t)1 << depth;
        for (int64_t o = 0; o < count; ++o) {
            const int64_t u = first + o;
            if (u >= N) break;
            const uint32_t n_u = (uint32_t)seg_size(S, j, u);
            const uint32_t off_u = (uint32_t)(seg_begin(S, j, u) - tile_base_j);
            const uint32_t m_u = (uint32_t)seg_size(S, j + 1, 2 * u + 1);
            const uint32_t left_off = (uint32_t)(seg_begin(S, j + 1, 2 * u + 1) - tile_base_j1);
            const uint32_t right_off = left_off + m_u;
            const uint32_t nr = n_u - m_u - 1u;
            const int d = fin_dim(a, sm, s0, j, u);
            const uint16_t *src = sm.ids[cur] + off_u;
            uint16_t *dst = sm.ids[cur ^ 1];
            const SmemSeg acc{sm.keys, sm.idx, src, a.T, k, d};
            cta_select(acc, n_u, m_u, k + 1, st, sm.hist, red);
            if (st.err) {
                if (tid == 0) set_status(a.status, KDT_EINTERNAL);
                return;
            }
            if (tid <= (uint32_t)k) medw[tid] = acc((int)tid, st.med_q);
            if (tid < 2) cursor[tid] = 0u;
            __syncthreads();
            const uint32_t lane = tid & 31u, lt_mask = (1u << lane) - 1u;
            for (uint32_t q0 = 0; q0 < n_u; q0 += blockDim.x) {
                const uint32_t q = q0 + tid;
                int side = -1;
                if (q < n_u) {
                    const int c = cmp_words(acc, q, medw, k + 1);
                    side = c < 0 ? 0 : (c > 0 ? 1 : -1);
                }
                const uint32_t lm = __ballot_sync(0xffffffffu, side == 0);
                const uint32_t rm = __ballot_sync(0xffffffffu, side == 1);
                uint32_t lb = 0, rb = 0;
                if (lane == 0) {
                    if (lm) lb = atomicAdd(&cursor[0], __popc(lm));
                    if (rm) rb = atomicAdd(&cursor[1], __popc(rm));
                }
                lb = __shfl_sync(0xffffffffu, lb, 0);
                rb = __shfl_sync(0xffffffffu, rb, 0);
                if (side == 0) {
                    const uint32_t oo = lb + __popc(lm & lt_mask);
                    if (oo < m_u) dst[left_off + oo] = src[q];
                    else set_status(a.status, KDT_EINTERNAL);
                } else if (side == 1) {
                    const uint32_t oo = rb + __popc(rm & lt_mask);
                    if (oo < nr) dst[right_off + oo] = src[q];
                    else set_status(a.status, KDT_EINTERNAL);
                }
            }
            if (tid == 0) {
                a.perm[u] = (int32_t)sm.idx[src[st.med_q]];
                const int64_t lu = tile_local_index(s0, depth, u);
                if (a.mode == KDT_SPLIT_WIDEST && lu < a.T) {
                    sm.sval[lu] = key2f(medw[0]);
                    sm.sdim[lu] = (uint8_t)d;
                }
            }
            __syncthreads();
        }
        cur ^= 1;
        ++j;
    }

    // Phase B: each warp finishes whole subtrees of at most kWarpMax points.
    if (j < S.L) {
        const int w = (int)(tid >> 5);
        const int depth0 = j - a.l0;
        const int64_t first0 = ((s0 + 1) << depth0) - 1;
        const int64_t count0 = (int64_t)1 << depth0;
        uint32_t *hist = sm.hist + w * kWarpRadixBins;
        uint32_t *wf = wfs[w];
        const int64_t tile_base = seg_begin(S, j, first0);
        for (int64_t o = w; o < count0; o += kFinWarps) {
            const int64_t t = first0 + o;
            if (t >= N) break;
            const uint32_t off_t = (uint32_t)(seg_begin(S, j, t) - tile_base);
            int c = cur;
            for (int jj = j; jj < S.L; ++jj, c ^= 1) {
                const int dd = jj - j;
                const int64_t f = ((t + 1) << dd) - 1;
                const int64_t cnt = (int64_t)1 << dd;
                for (int64_t oo = 0; oo < cnt; ++oo) {
                    const int64_t u = f + oo;
                    if (u >= N) break;
                    warp_split_node(a, sm, s0, t, j, off_t, jj, u, c, wf, hist);
                }
                __syncwarp();
            }
        }
    }
}

// ---------------------------------------------------------------------------
// plan, workspace and enqueue

static int pick_tile(int k, int mode, int *T, size_t *smem) {
    static const int cands[] = {8192, 6144, 4096, 3072, 2048, 1024, 512};
    for (int c : cands) {
        const size_t b = fin_smem_bytes(k, c, mode);
        if (b <= kFinSmemBudget) {
            *T = c;
            *smem = b;
            return 0;
        }
    }
    return -1;
}

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int make_plan(int64_t N, int k, int mode, Plan *p) {
    if (N < 1 || N > 2147483647LL || k < 1 || k > kMaxK || (mode != 0 && mode != 1)) return KDT_EINVAL;
    Plan q{};
    q.S = make_shape(N);
    q.k = k;
    q.mode = mode;
    if (pick_tile(k, mode, &q.tp.tile, &q.tp.smem) != 0) return KDT_EINVAL;
    int lf = 0;
    while (lf < q.S.L && seg_size(q.S, lf, full_nodes(lf)) > q.tp.tile) ++lf;
    q.finish_level = lf;
    int lm = 0;
    while (lm < lf && ((int64_t)1 << lm) <= kMultiMaxSegs && seg_size(q.S, lm, full_nodes(lm)) > kMultiMinSize) ++lm;
    q.multi_levels = lm;
    q.table_cap = (int64_t)1 << lf;
    q.hist_rows = lm > 0 ? ((int64_t)1 << (lm - 1)) : 0;
    q.sel_cap = lf > 0 ? ((int64_t)1 << (lf - 1)) : 0;
    size_t off = 0;
    q.off_status = off;
    off = align_up(off + 64, 256);
    q.off_bbox = off;
    off = align_up(off + (size_t)2 * k * 4, 256);
    for (int b = 0; b < 3; ++b) {
        const int64_t rows = (b < 2 || lf > 0) ? N : 0;
        q.off_keys[b] = off;
        off = align_up(off + (size_t)k * rows * 4, 256);
        q.off_idx[b] = off;
        off = align_up(off + (size_t)rows * 4, 256);
    }
    for (int b = 0; b < 2; ++b) {
        q.off_dom[b] = off;
        off = align_up(off + (size_t)q.table_cap * 2 * k * 4, 256);
        q.off_dim[b] = off;
        off = align_up(off + (size_t)q.table_cap * 4, 256);
        q.off_hist[b] = off;
        off = align_up(off + (size_t)q.hist_rows * kBuckets * 4, 256);
    }
    q.off_sel = off;
    off = align_up(off + (size_t)q.sel_cap * sizeof(SegSel), 256);
    q.bytes = off;
    *p = q;
    return KDT_OK;
}

Buffers carve(const Plan &p, void *base) {
    unsigned char *b = static_cast<unsigned char *>(base);
    Buffers r;
    r.status = reinterpret_cast<int *>(b + p.off_status);
    r.bbox = reinterpret_cast<uint32_t *>(b + p.off_bbox);
    for (int i = 0; i < 3; ++i) {
        r.keys[i] = reinterpret_cast<uint32_t *>(b + p.off_keys[i]);
        r.idx[i] = reinterpret_cast<uint32_t *>(b + p.off_idx[i]);
    }
    for (int i = 0; i < 2; ++i) {
        r.dom[i] = reinterpret_cast<float *>(b + p.off_dom[i]);
        r.dim[i] = reinterpret_cast<int *>(b + p.off_dim[i]);
        r.hist[i] = reinterpret_cast<uint32_t *>(b + p.off_hist[i]);
    }
    r.sel = reinterpret_cast<SegSel *>(b + p.off_sel);
    return r;
}

#define KDT_LAUNCH_CHECK()                                      \
    do {                                                        \
        cudaError_t e_ = cudaGetLastError();                    \
        if (e_ != cudaSuccess) return KDT_ECUDA;                \
    } while (0)

int enqueue_build(const Plan &p, const Buffers &b, const float *pts, int32_t *perm, cudaStream_t stream) {
    const Shape &S = p.S;
    const int k = p.k;
    const double Nd = (double)S.N;
    if (cudaMemsetAsync(b.status, 0, sizeof(int), stream) != cudaSuccess) return KDT_ECUDA;
    if (cudaMemsetAsync(b.bbox, 0xff, (size_t)k * 4, stream) != cudaSuccess) return KDT_ECUDA;
    if (cudaMemsetAsync(b.bbox + k, 0x00, (size_t)k * 4, stream) != cudaSuccess) return KDT_ECUDA;
    {
        int dev = 0, sms = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        int64_t blocks = (S.N + kInitThreads - 1) / kInitThreads;
        const int64_t cap = (int64_t)(sms > 0 ? sms : 152) * 8;
        if (blocks > cap) blocks = cap;
        ProfScope ps(stream, "init", 0.0);
        init_kernel<<<(unsigned)blocks, kInitThreads, 0, stream>>>(pts, S.N, k, b.keys[0], b.idx[0], b.bbox,
                                                                   b.status);
        KDT_LAUNCH_CHECK();
    }
    root_table_kernel<<<1, 1, 0, stream>>>(b.bbox, k, b.dom[0], b.dim[0]);
    KDT_LAUNCH_CHECK();
    int src = 0;
    for (int l = 0; l < p.finish_level; ++l) {
        const int rc = enqueue_level(p, b, l, src, perm, stream);
        if (rc != KDT_OK) return rc;
        src ^= 1;
    }
    {
        FinArgs a;
        a.S = S;
        a.k = k;
        a.mode = p.mode;
        a.l0 = p.finish_level;
        a.T = p.tp.tile;
        a.src_keys = b.keys[src];
        a.src_idx = b.idx[src];
        a.perm = perm;
        a.dom = b.dom[p.finish_level & 1];
        a.status = b.status;
        if (cudaFuncSetAttribute(finisher_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.tp.smem) !=
            cudaSuccess)
            return KDT_ECUDA;
        const int64_t ntiles = nodes_on_level(S, p.finish_level);
        const double sort_levels = (double)(S.L - 1 - p.finish_level);
        ProfScope ps(stream, "finisher", 20.0 * Nd * sort_levels + 12.0 * Nd);
        finisher_kernel<<<(unsigned)ntiles, kFinThreads, p.tp.smem, stream>>>(a);
        KDT_LAUNCH_CHECK();
    }
    enqueue_status_fold(b.status, stream);
    KDT_LAUNCH_CHECK();
    return KDT_OK;
}

}  // namespace kdt
