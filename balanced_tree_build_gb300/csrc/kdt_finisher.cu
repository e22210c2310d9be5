// kdt_finisher.cu -- the select finisher: one CTA owns a subtree of at most T
// points and fixes all of its remaining levels on chip by exact rank selects.
// It runs the tiles that the sorted finisher (kdt_finisher_sorted.cu) leaves:
// those whose coordinates fall into too few value buckets (heavy ties,
// tightly clustered values), which its selects handle at any distribution.
//
// The paper's method runs every level over the whole array ("GPU-friendly,
// Parallel, and (Almost-)In-Place Construction of Left-Balanced k-d Trees",
// introduction: every kernel and sort operates on the entire set).  Once a
// subtree fits one CTA's shared memory, the remaining ~half of the levels
// cost one read of its records and one write of its output nodes here.
//
// Inside the CTA the records stay put; a list of 16-bit local ids is
// partitioned level by level (ping-pong).  The work is split by node size:
//   * phase A (nodes > 256 points): the nodes of a level are spread over
//     warp groups (16 / nodes warps each, named barriers); each group splits
//     its node by value buckets (min/max, one histogram, one partition pass)
//     and ranks the few points of the split bucket exactly;
//   * phase B (nodes <= 256): each warp owns whole subtrees; nodes > 32 are
//     split the same way by one warp, nodes <= 32 rank their points with one
//     lane per point, subtrees of <= 7 points are finished by one lane each.
// Phase-B subtrees are laid out relative to the range the warp took over, so
// warps never touch each other's ranges.
#include "kdt_internal.cuh"
#include "kdt_select.cuh"

namespace kdt {

constexpr int kFinThreads = 512;
constexpr int kFinWarps = kFinThreads / 32;
constexpr int kWarpMax = 256;  // phase B: subtrees this small go to one warp
constexpr int kLaneMax = 7;    // subtrees this small go to one lane
constexpr int kCandPerWarp = 64;  // bucket-split candidates per warp
constexpr int kFinHistWords = kFinWarps * kWarpRadixBins;  // 4096

struct FinArgs {
    Shape S;
    int k, mode, l0, T;
    int64_t ld;
    const uint4 *src;  // records of level l0 (group columns of ld records)
    int32_t *perm;
    const float *dom;  // node table of level l0
    const uint8_t *only;  // per tile: nonzero = finish it here
    int *status;
};

size_t select_finisher_smem(int k, int T, int mode) {
    size_t b = (size_t)k * T * 4 + (size_t)T * 4 + (size_t)T * 4 + (size_t)kFinHistWords * 4;
    if (mode == KDT_SPLIT_WIDEST) b += (size_t)T * 5;
    return (b + 15) & ~(size_t)15;
}

struct FinSmem {
    uint32_t *keys;    // [k][T]
    uint32_t *idx;     // [T]
    uint16_t *ids[2];  // [T] each: local point ids in current order
    uint32_t *hist;    // [kFinHistWords]
    float *sval;       // [T] split coordinate of tile-local node (widest mode)
    uint8_t *sdim;     // [T] split dimension of tile-local node (widest mode)
};

__device__ inline FinSmem fin_carve(unsigned char *p, int k, int T, int mode) {
    FinSmem f;
    f.keys = reinterpret_cast<uint32_t *>(p);
    p += (size_t)k * T * 4;
    f.idx = reinterpret_cast<uint32_t *>(p);
    p += (size_t)T * 4;
    f.hist = reinterpret_cast<uint32_t *>(p);
    p += (size_t)kFinHistWords * 4;
    f.ids[0] = reinterpret_cast<uint16_t *>(p);
    p += (size_t)T * 2;
    f.ids[1] = reinterpret_cast<uint16_t *>(p);
    p += (size_t)T * 2;
    f.sval = reinterpret_cast<float *>(p);
    p += mode == KDT_SPLIT_WIDEST ? (size_t)T * 4 : 0;
    f.sdim = p;
    return f;
}

// Word i of the point at offset q of a node whose ordered local ids start at
// `ids`.
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

// Strict split order of dimension d between local points a and b.
__device__ __forceinline__ bool local_less(const FinSmem &sm, int T, int k, int d, uint32_t a, uint32_t b) {
    for (int i = 0; i < k; ++i) {
        int c = d + i;
        if (c >= k) c -= k;
        const uint32_t x = sm.keys[c * T + a], y = sm.keys[c * T + b];
        if (x != y) return x < y;
    }
    return sm.idx[a] < sm.idx[b];
}

__device__ __forceinline__ int64_t tile_local_index(int64_t s0, int depth, int64_t u) {
    const int64_t first = ((s0 + 1) << depth) - 1;
    return (((int64_t)1 << depth) - 1) + (u - first);
}

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
    const int64_t lu = tile_local_index(s0, depth, u);
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

__device__ __forceinline__ int fin_dim(const FinArgs &a, const FinSmem &sm, int64_t s0, int j, int64_t u) {
    return a.mode == KDT_SPLIT_ROUND_ROBIN ? j % a.k : fin_widest_dim_of(a, sm, s0, j, u);
}

__device__ __forceinline__ void record_split(const FinArgs &a, const FinSmem &sm, int64_t s0, int j, int64_t u,
                                             uint32_t id, int d) {
    if (a.mode != KDT_SPLIT_WIDEST) return;
    const int64_t lu = tile_local_index(s0, j - a.l0, u);
    if (lu < a.T) {
        sm.sval[lu] = key2f(sm.keys[d * a.T + id]);
        sm.sdim[lu] = (uint8_t)d;
    }
}

// Geometry of node u (level j) inside a range that starts at `off_root` and
// holds, on level jr, the subtree of node `root` (levels below are packed
// from the same start).
struct NodeGeom {
    uint32_t n, off, m, left_off, right_off;
    bool children;
};

__device__ __forceinline__ NodeGeom node_geom(const Shape &S, int64_t root, int jr, uint32_t off_root, int j,
                                              int64_t u) {
    NodeGeom g;
    const int32_t u32 = (int32_t)u;
    const int32_t first_j = (int32_t)(((root + 1) << (j - jr)) - 1);
    g.n = (uint32_t)seg_size32(S, j, u32);
    g.off = off_root + (uint32_t)(seg_begin32(S, j, u32) - seg_begin32(S, j, first_j));
    g.children = j + 1 < S.L;
    g.m = 0u;
    g.left_off = 0u;
    if (g.children && g.n > 1u) {
        const int32_t first_j1 = 2 * first_j + 1;
        g.m = (uint32_t)seg_size32(S, j + 1, 2 * u32 + 1);
        g.left_off = off_root + (uint32_t)(seg_begin32(S, j + 1, 2 * u32 + 1) - seg_begin32(S, j + 1, first_j1));
    }
    g.right_off = g.left_off + g.m;
    return g;
}

// Group-wide split of node u: select, then partition the other local ids into
// the children's ranges of `dst` (ballot compaction, cursors in `cur2`).
template <class G>
__device__ void group_split_node(const G &grp, const FinArgs &a, const FinSmem &sm, int64_t s0, int j, int64_t u,
                                 const NodeGeom &ng, const uint16_t *src_all, uint16_t *dst, SelState &st,
                                 uint32_t *hist, int bits, uint32_t *red, uint32_t *medw, uint32_t *cur2) {
    const int k = a.k;
    const int d = fin_dim(a, sm, s0, j, u);
    const uint16_t *src = src_all + ng.off;
    const SmemSeg acc{sm.keys, sm.idx, src, a.T, k, d};
    group_select(grp, acc, ng.n, ng.m, k + 1, st, hist, bits, red);
    if (st.err) {
        if (grp.tid() == 0) set_status(a.status, KDT_EINTERNAL);
        return;
    }
    const uint32_t tid = grp.tid(), nt = grp.size();
    for (uint32_t i = tid; i <= (uint32_t)k; i += nt) medw[i] = acc((int)i, st.med_q);  // k + 1 words, k <= 32
    if (tid < 2) cur2[tid] = 0u;
    grp.sync();
    const uint32_t lane = lane_id(), lt = (1u << lane) - 1u;
    const uint32_t nr = ng.n - ng.m - 1u;
    for (uint32_t q0 = 0; q0 < ng.n; q0 += nt) {
        const uint32_t q = q0 + tid;
        int side = -1;
        if (q < ng.n) {
            const int c = cmp_words(acc, q, medw, k + 1);
            side = c < 0 ? 0 : (c > 0 ? 1 : -1);
        }
        const uint32_t lm = __ballot_sync(0xffffffffu, side == 0);
        const uint32_t rm = __ballot_sync(0xffffffffu, side == 1);
        uint32_t lb = 0, rb = 0;
        if (lane == 0) {
            if (lm) lb = atomicAdd(&cur2[0], __popc(lm));
            if (rm) rb = atomicAdd(&cur2[1], __popc(rm));
        }
        lb = __shfl_sync(0xffffffffu, lb, 0);
        rb = __shfl_sync(0xffffffffu, rb, 0);
        if (side == 0) {
            const uint32_t o = lb + __popc(lm & lt);
            if (o < ng.m) dst[ng.left_off + o] = src[q];
            else set_status(a.status, KDT_EINTERNAL);
        } else if (side == 1) {
            const uint32_t o = rb + __popc(rm & lt);
            if (o < nr) dst[ng.right_off + o] = src[q];
            else set_status(a.status, KDT_EINTERNAL);
        }
    }
    if (tid == 0) {
        const uint32_t id = src[st.med_q];
        a.perm[u] = (int32_t)sm.idx[id];
        record_split(a, sm, s0, j, u, id, d);
    }
    grp.sync();
}

// Group-wide split of node u by value buckets: min and max of the split
// coordinate, one histogram of 2^bits buckets over that range, one partition
// pass (points below the split bucket go left, above it right); the few
// points in the split bucket ("candidates", at most `cap`, listed in `cand`)
// are then ranked exactly by pairwise comparison under the full split order.
// Falls back to the exact select when the split coordinate is constant or
// the candidates do not fit.  `pk` holds 8 words of shared scratch.
template <class G>
__device__ void group_bucket_split(const G &grp, const FinArgs &a, const FinSmem &sm, int64_t s0, int j, int64_t u,
                                   const NodeGeom &ng, const uint16_t *src_all, uint16_t *dst, SelState &st,
                                   uint32_t *hist, int bits, uint32_t *red, uint32_t *medw, uint32_t *pk,
                                   uint16_t *cand, uint32_t cap) {
    const int k = a.k, T = a.T;
    const int d = fin_dim(a, sm, s0, j, u);
    const uint16_t *src = src_all + ng.off;
    const uint32_t tid = grp.tid(), nt = grp.size();
    const uint32_t nb = 1u << bits;
    const uint32_t *kd = sm.keys + d * T;
    uint32_t mn = 0xffffffffu, mx = 0u;
    for (uint32_t q = tid; q < ng.n; q += nt) {
        const uint32_t v = kd[src[q]];
        mn = min(mn, v);
        mx = max(mx, v);
    }
    group_minmax(grp, mn, mx, red);
    const float lo = key2f(mn);
    const float rg = __fsub_rn(key2f(mx), lo);
    float scale = 0.f;
    if (rg > 0.f && rg <= 3.0e38f) scale = __fdiv_rn((float)nb, rg);
    if (mn == mx || !(scale > 0.f && scale <= 3.0e38f)) {
        grp.sync();
        group_split_node(grp, a, sm, s0, j, u, ng, src_all, dst, st, hist, bits, red, medw, pk);
        return;
    }
    for (uint32_t b = tid; b < nb; b += nt) hist[b] = 0u;
    grp.sync();
    for (uint32_t q = tid; q < ng.n; q += nt) atomicAdd(&hist[value_bucket(kd[src[q]], lo, scale, nb)], 1u);
    grp.sync();
    {
        const uint32_t per = nb / nt;
        uint32_t sum = 0;
        for (uint32_t i = 0; i < per; ++i) sum += hist[tid * per + i];
        uint32_t total;
        const uint32_t excl = group_exclusive_scan(grp, sum, red, total);
        if (ng.m >= excl && ng.m < excl + sum) {
            uint32_t c = excl;
            for (uint32_t i = 0; i < per; ++i) {
                const uint32_t h = hist[tid * per + i];
                if (ng.m < c + h) {
                    pk[0] = tid * per + i;
                    pk[1] = c;
                    pk[2] = h;
                    break;
                }
                c += h;
            }
        }
        if (tid < 3) pk[4 + tid] = 0u;
    }
    grp.sync();
    const uint32_t bstar = pk[0], below = pk[1], cnt = pk[2];
    if (cnt > cap) {
        grp.sync();
        group_split_node(grp, a, sm, s0, j, u, ng, src_all, dst, st, hist, bits, red, medw, pk);
        return;
    }
    const uint32_t above = ng.n - below - cnt;
    const uint32_t nr = ng.n - ng.m - 1u;
    const uint32_t right_tail = ng.right_off + (nr - above);
    const uint32_t lane = lane_id(), lt = (1u << lane) - 1u;
    for (uint32_t q0 = 0; q0 < ng.n; q0 += nt) {
        const uint32_t q = q0 + tid;
        int side = 3;
        uint32_t id = 0;
        if (q < ng.n) {
            id = src[q];
            const uint32_t b = value_bucket(kd[id], lo, scale, nb);
            side = b < bstar ? 0 : (b > bstar ? 2 : 1);
        }
        const uint32_t lm = __ballot_sync(0xffffffffu, side == 0);
        const uint32_t cm = __ballot_sync(0xffffffffu, side == 1);
        const uint32_t rm = __ballot_sync(0xffffffffu, side == 2);
        uint32_t lb = 0, cb = 0, rb = 0;
        if (lane == 0) {
            if (lm) lb = atomicAdd(&pk[4], __popc(lm));
            if (cm) cb = atomicAdd(&pk[5], __popc(cm));
            if (rm) rb = atomicAdd(&pk[6], __popc(rm));
        }
        lb = __shfl_sync(0xffffffffu, lb, 0);
        cb = __shfl_sync(0xffffffffu, cb, 0);
        rb = __shfl_sync(0xffffffffu, rb, 0);
        if (side == 0) {
            const uint32_t o = lb + __popc(lm & lt);
            if (o < below) dst[ng.left_off + o] = (uint16_t)id;
            else set_status(a.status, KDT_EINTERNAL);
        } else if (side == 2) {
            const uint32_t o = rb + __popc(rm & lt);
            if (o < above) dst[right_tail + o] = (uint16_t)id;
            else set_status(a.status, KDT_EINTERNAL);
        } else if (side == 1) {
            const uint32_t o = cb + __popc(cm & lt);
            if (o < cnt) cand[o] = (uint16_t)id;
            else set_status(a.status, KDT_EINTERNAL);
        }
    }
    grp.sync();
    // exact ranks of the candidates; rank r = m - below is the split point
    const uint32_t r = ng.m - below;
    for (uint32_t q = tid; q < cnt; q += nt) {
        const uint32_t id = cand[q];
        uint32_t rank = 0;
        for (uint32_t t = 0; t < cnt; ++t) {
            const uint32_t o = cand[t];
            if (o != id && local_less(sm, T, k, d, o, id)) ++rank;
        }
        if (rank == r) {
            a.perm[u] = (int32_t)sm.idx[id];
            record_split(a, sm, s0, j, u, id, d);
        } else if (rank < r) {
            dst[ng.left_off + below + rank] = (uint16_t)id;
        } else {
            dst[ng.right_off + rank - r - 1u] = (uint16_t)id;
        }
    }
    grp.sync();
}

// Warp: split node u of at most 32 points, one lane per point.  The rank of
// each point comes from a 32-bucket value ranking (five ballots); if two
// points share a bucket, from all-pairs comparisons.
__device__ void warp_split_small(const FinArgs &a, const FinSmem &sm, int64_t s0, int j, int64_t u,
                                 const NodeGeom &ng, const uint16_t *src_all, uint16_t *dst) {
    const uint32_t lane = lane_id();
    const int k = a.k, T = a.T;
    const int d = fin_dim(a, sm, s0, j, u);
    const uint16_t *src = src_all + ng.off;
    const bool valid = lane < ng.n;
    const uint32_t my_id = valid ? src[lane] : 0u;
    const uint32_t my_w0 = valid ? sm.keys[d * T + my_id] : 0u;
    const uint32_t mn = __reduce_min_sync(0xffffffffu, valid ? my_w0 : 0xffffffffu);
    const uint32_t mx = __reduce_max_sync(0xffffffffu, valid ? my_w0 : 0u);
    const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
    uint32_t rank = 0;
    bool ranked = false;
    if (mn != mx) {
        const int bits = ng.n > 16u ? 10 : 8;
        const uint32_t nb = 1u << bits;
        const float lo = key2f(mn);
        const float r = __fsub_rn(key2f(mx), lo);
        if (r > 0.f && r <= 3.0e38f) {
            const float scale = __fdiv_rn((float)nb, r);
            if (scale <= 3.0e38f) {
                const uint32_t b = value_bucket(my_w0, lo, scale, nb);
                // radix ranking by ballots: `less` = points in lower buckets,
                // `eq` = points in the same bucket (including this one)
                uint32_t eq = vmask, less = 0;
                for (int bit = bits - 1; bit >= 0; --bit) {
                    const uint32_t bl = __ballot_sync(0xffffffffu, valid && ((b >> bit) & 1u));
                    if ((b >> bit) & 1u) {
                        less += __popc(eq & ~bl);
                        eq &= bl;
                    } else {
                        eq &= ~bl;
                    }
                }
                // points sharing a bucket: compare with the few lanes involved
                uint32_t ties = __ballot_sync(0xffffffffu, valid && __popc(eq) > 1);
                while (ties) {
                    const int t = __ffs(ties) - 1;
                    ties &= ties - 1u;
                    const uint32_t oid = __shfl_sync(0xffffffffu, my_id, t);
                    const uint32_t ow0 = __shfl_sync(0xffffffffu, my_w0, t);
                    if (valid && (uint32_t)t != lane && ((eq >> t) & 1u)) {
                        const bool lt = ow0 != my_w0 ? ow0 < my_w0 : local_less(sm, T, k, d, oid, my_id);
                        less += lt ? 1u : 0u;
                    }
                }
                rank = less;
                ranked = true;
            }
        }
    }
    if (!ranked) {
        rank = 0;
        for (uint32_t t = 0; t < ng.n; ++t) {
            const uint32_t oid = __shfl_sync(0xffffffffu, my_id, t);
            const uint32_t ow0 = __shfl_sync(0xffffffffu, my_w0, t);
            if (valid && t != lane) {
                const bool lt = ow0 != my_w0 ? ow0 < my_w0 : local_less(sm, T, k, d, oid, my_id);
                rank += lt ? 1u : 0u;
            }
        }
    }
    if (valid) {
        if (rank == ng.m) {
            a.perm[u] = (int32_t)sm.idx[my_id];
            record_split(a, sm, s0, j, u, my_id, d);
        } else if (rank < ng.m) {
            dst[ng.left_off + rank] = (uint16_t)my_id;
        } else {
            dst[ng.right_off + rank - ng.m - 1u] = (uint16_t)my_id;
        }
    }
}

// One lane finishes the whole subtree of node u (level j, at most kLaneMax
// points at ids[0..n)): sort them in place by the split order, take the split
// rank, recurse on the two sides (explicit stack).
__device__ void lane_finish(const FinArgs &a, const FinSmem &sm, int64_t s0, int j, int64_t u, uint16_t *e,
                            uint32_t n) {
    const int k = a.k, T = a.T;
    struct Item {
        int32_t u;
        int8_t j, lo, n;
    };
    Item stack[8];
    int sp = 0;
    stack[sp++] = Item{(int32_t)u, (int8_t)(j - a.l0), 0, (int8_t)n};
    while (sp > 0) {
        const Item it = stack[--sp];
        if (it.n == 0) continue;
        const int jj = a.l0 + it.j;
        const int d = fin_dim(a, sm, s0, jj, it.u);
        for (int x = it.lo + 1; x < it.lo + it.n; ++x) {
            const uint32_t v = e[x];
            int y = x - 1;
            while (y >= it.lo && local_less(sm, T, k, d, v, e[y])) {
                e[y + 1] = e[y];
                --y;
            }
            e[y + 1] = (uint16_t)v;
        }
        const uint32_t m = (jj + 1 < a.S.L && it.n > 1) ? (uint32_t)seg_size32(a.S, jj + 1, 2 * it.u + 1) : 0u;
        const uint32_t med = e[it.lo + m];
        a.perm[it.u] = (int32_t)sm.idx[med];
        record_split(a, sm, s0, jj, it.u, med, d);
        if (it.n > 1) {
            stack[sp++] = Item{2 * it.u + 2, (int8_t)(it.j + 1), (int8_t)(it.lo + m + 1), (int8_t)(it.n - m - 1)};
            stack[sp++] = Item{2 * it.u + 1, (int8_t)(it.j + 1), it.lo, (int8_t)m};
        }
    }
}

__global__ void __launch_bounds__(kFinThreads, 2) finisher_kernel(FinArgs a) {
    pdl_enter();
    extern __shared__ __align__(16) unsigned char fin_smem[];
    __shared__ SelState st[kFinWarps];
    __shared__ uint32_t red[kFinWarps][64];
    __shared__ uint32_t medw[kFinWarps][kMaxWords];
    __shared__ uint32_t pk[kFinWarps][8];
    __shared__ uint16_t cand[kFinWarps * kCandPerWarp];
    __shared__ int stop;
    const uint32_t tid = threadIdx.x;
    if (a.only != nullptr && a.only[blockIdx.x] == 0) return;
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
    const uint32_t nt = blockDim.x;
    // load the tile's records: words 0..k-1 to the key arrays, word k to
    //    the input indices (G uint4 per record; a batch's loads go out first)
    for (int gi = 0; gi < rec_groups(k); ++gi) {
        const uint4 *col = a.src + (int64_t)gi * a.ld + base;
        for (uint32_t q = tid; q < n; q += 4 * nt) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = q + u * nt < n ? __ldg(col + q + u * nt) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (q + u * nt >= n) continue;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int wd = 4 * gi + j;
                    if (wd < k) sm.keys[wd * a.T + q + u * nt] = u4_word(v[u], j);
                    else if (wd == k) sm.idx[q + u * nt] = u4_word(v[u], j);
                }
            }
        }
    }
    for (uint32_t q = tid; q < n; q += blockDim.x) sm.ids[0][q] = (uint16_t)q;
    __syncthreads();

    const uint32_t w = tid >> 5;
    // Phase A: the nodes of a level are spread over warp groups.
    int j = a.l0, cur = 0;
    while (j < S.L) {
        const int depth = j - a.l0;
        const int64_t first = ((s0 + 1) << depth) - 1;
        if (seg_size(S, j, first) <= (int64_t)kWarpMax) break;
        const int64_t count = min(((int64_t)1 << depth), N - first);
        const int groups = (int)(count < (int64_t)kFinWarps ? count : (int64_t)kFinWarps);
        int gsh = 0;  // groups = 2^gsh for count a power of two; otherwise round down
        while ((2 << gsh) <= groups) ++gsh;
        const int ng = 1 << gsh;
        const uint32_t wpg = kFinWarps / ng;
        const uint32_t g = w / wpg;
        const WarpsGroup grp{g * wpg * 32u, wpg * 32u, (int)g + 1};
        const int bits = min(kCtaRadixBits, 12 - gsh);
        uint32_t *hist = sm.hist + g * (kFinHistWords >> gsh);
        for (int64_t o = g; o < count; o += ng) {
            const int64_t u = first + o;
            const NodeGeom geom = node_geom(S, s0, a.l0, 0u, j, u);
            group_bucket_split(grp, a, sm, s0, j, u, geom, sm.ids[cur], sm.ids[cur ^ 1], st[g], hist, bits, red[g],
                               medw[g], pk[g], cand + g * wpg * kCandPerWarp, wpg * kCandPerWarp);
        }
        __syncthreads();
        cur ^= 1;
        ++j;
    }

    // Phase B: each warp finishes whole subtrees of at most kWarpMax points.
    if (j < S.L) {
        const int depth0 = j - a.l0;
        const int64_t first0 = ((s0 + 1) << depth0) - 1;
        const int64_t count0 = (int64_t)1 << depth0;
        const int64_t tile_base = seg_begin(S, j, first0);
        const WarpsGroup wg{w * 32u, 32u, 0};
        uint32_t *hist = sm.hist + w * kWarpRadixBins;
        for (int64_t o = w; o < count0; o += kFinWarps) {
            const int64_t t = first0 + o;
            if (t >= N) break;
            const uint32_t off_t = (uint32_t)(seg_begin(S, j, t) - tile_base);
            int c = cur;
            for (int jj = j; jj < S.L; ++jj, c ^= 1) {
                const int dd = jj - j;
                const int64_t f = ((t + 1) << dd) - 1;
                if (f >= N) break;
                const int64_t cnt = min(((int64_t)1 << dd), N - f);
                if (seg_size(S, jj, f) <= (int64_t)kLaneMax) {
                    // one lane per remaining subtree
                    for (int64_t o2 = lane_id(); o2 < cnt; o2 += 32) {
                        const int64_t u = f + o2;
                        const NodeGeom geom = node_geom(S, t, j, off_t, jj, u);
                        lane_finish(a, sm, s0, jj, u, sm.ids[c] + geom.off, geom.n);
                    }
                    break;
                }
                for (int64_t oo = 0; oo < cnt; ++oo) {
                    const int64_t u = f + oo;
                    const NodeGeom geom = node_geom(S, t, j, off_t, jj, u);
                    if (geom.n > 32u)
                        group_bucket_split(wg, a, sm, s0, jj, u, geom, sm.ids[c], sm.ids[c ^ 1], st[w], hist,
                                           kWarpRadixBits, red[w], medw[w], pk[w], cand + w * kCandPerWarp,
                                           (uint32_t)kCandPerWarp);
                    else
                        warp_split_small(a, sm, s0, jj, u, geom, sm.ids[c], sm.ids[c ^ 1]);
                }
                __syncwarp();
            }
            __syncwarp();
        }
    }
}

int launch_select_finisher(const Plan &p, const Buffers &b, int src, int32_t *perm, const uint8_t *only,
                           cudaStream_t stream) {
    const Shape &S = p.S;
    FinArgs a;
    a.S = S;
    a.k = p.k;
    a.mode = p.mode;
    a.l0 = p.finish_level;
    a.T = p.tp.tile;
    a.ld = p.ld;
    a.src = b.rec[src];
    a.perm = perm;
    a.dom = b.dom[p.finish_level & 1];
    a.only = only;
    a.status = b.status;
    if (cudaFuncSetAttribute(finisher_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)p.tp.smem_select) != cudaSuccess)
        return KDT_ECUDA;
    const int64_t ntiles = nodes_on_level(S, p.finish_level);
    launch_pdl(finisher_kernel, (unsigned)ntiles, kFinThreads, p.tp.smem_select, stream, a);
    if (cudaGetLastError() != cudaSuccess) return KDT_ECUDA;
    return KDT_OK;
}

}  // namespace kdt
