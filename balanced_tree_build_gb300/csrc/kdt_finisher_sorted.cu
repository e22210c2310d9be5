// kdt_finisher_sorted.cu -- the presorted shared-memory finisher: one CTA
// owns a subtree of at most T points and fixes all of its remaining levels on
// chip, with one sort per dimension and then stable partitions.
//
// Method.  "An Implementation of a Balanced Kd Tree Builder Using GPUs"
// (overview list, after Brown's O(kn log n) builder): sort one reference
// array per coordinate by the super key of that coordinate; the split point of
// a node is then read off the array of its split coordinate at a known
// position, and the other arrays are partitioned around it, which keeps them
// sorted inside each child.  Here the split point of node u is the point of
// rank ss(lChild(u)) ("GPU-friendly, Parallel, and (Almost-)In-Place
// Construction of Left-Balanced k-d Trees", problem paragraph), so the tree is
// the same one the level-by-level method builds.
//
// Per tile (subtree s0 of level l0, n <= T points):
//   1. load the k coordinate keys and the input index of its points;
//   2. for each coordinate c, order the local ids by the super key of c: a
//      counting sort into value buckets of x[c] (a monotone map of the key),
//      then each point's rank inside its bucket by comparison under the full
//      super key.  A bucket of more than kSfMaxBucket points (heavy ties or
//      clustered values) leaves the whole tile to the select finisher, which
//      handles any input;
//   3. levels with fewer nodes than warps: a group of warps per node.  The
//      node's points are marked left / median / right from their offsets in
//      the array of its split coordinate, then every array is partitioned
//      stably into the children's segments (ballot compaction; a count pass
//      gives each warp its start);
//   4. lower levels: each warp owns whole subtrees (at most 8 nodes per
//      level) and splits each array in one pass over its range, without CTA
//      barriers: a byte per position names its node, whose constants come by
//      shuffle from the lane that holds them;
//   5. subtrees of at most 15 points (levels >= L-4): one lane each; every
//      node of the subtree scans the subtree's points in the order of its
//      split coordinate, keeps those carrying its code and ranks them.
//
// Segments of a level are laid out as in the select finisher: node i of the
// level (counted from the tile's first node on it) starts at the sum of the
// sizes of nodes 0..i-1, children follow their parents' order, so the left
// child of node i starts at off(i) - i.
#include "kdt_internal.cuh"
#include "kdt_select.cuh"

namespace kdt {

constexpr int kSfThreads = 512;
constexpr int kSfWarps = kSfThreads / 32;
constexpr int kSfPPT = 8;          // points per thread in the sort (T <= kSfPPT * kSfThreads)
constexpr int kSfMaxBucket = 16;   // larger buckets leave the tile to the select finisher
constexpr size_t kSfSmemBudget = 110 * 1024;  // two CTAs per SM
constexpr int kMaxLevels = 32;

// Constants of level j of the whole tree (B = 2^(L-1-j), notation of the
// closed forms for ss and sb): with level index jv = s - F(j),
//   ss(s) = B-1 + clamp(M - jv*B, 0, B), so the first q = M / B subtrees of
//   the level hold 2B-1 points, subtree q holds B-1+rem (rem = M - q*B) and
//   the rest B-1.
struct SfLevel {
    int32_t B, q, rem;
};

struct SfArgs {
    Shape S;
    int k, mode, l0, T, nb;
    int64_t ld;
    const uint32_t *src_keys, *src_idx;
    int32_t *perm;
    const float *dom;    // node table of level l0 (widest mode)
    uint8_t *fallback;   // per tile: 1 = left to the select finisher
    int *status;
    SfLevel lv[kMaxLevels];
};

static size_t align16(size_t x) { return (x + 15) & ~(size_t)15; }

// Dynamic shared memory of one CTA: reference arrays [k][T] u16, keys [k][T]
// u32 (after the sort: the second reference array set and the side flags),
// input indices [T], nb 16-bit bucket counters, a [T] u16 bucket staging array, and
// in widest mode the split value and dimension of every tile node.
size_t sorted_finisher_smem(int k, int T, int mode, int nb) {
    size_t b = (size_t)2 * k * T + (size_t)4 * k * T + (size_t)4 * T + (size_t)2 * nb + (size_t)2 * T;
    if (mode == KDT_SPLIT_WIDEST) b += (size_t)5 * T;
    return align16(b);
}

struct SfSmem {
    uint16_t *ids0;   // [k][T]
    uint32_t *keys;   // [k][T], live during the sort
    uint16_t *ids1;   // [k][T], aliases keys after the sort
    uint8_t *side;    // [T], aliases keys + 2kT bytes after the sort
    uint32_t *idx;    // [T]
    uint32_t *hist;   // [nb / 2]: two 16-bit bucket counters per word
    uint16_t *stage;  // [T] points grouped by bucket, before ranking
    float *sval;      // [T] split value of tile node (widest mode)
    uint8_t *sdim;    // [T] split dimension of tile node (widest mode)
};

__device__ __forceinline__ SfSmem sf_carve(unsigned char *p, int k, int T, int nb) {
    SfSmem f;
    f.ids0 = reinterpret_cast<uint16_t *>(p);
    p += (size_t)2 * k * T;
    f.keys = reinterpret_cast<uint32_t *>(p);
    f.ids1 = reinterpret_cast<uint16_t *>(p);
    f.side = p + (size_t)2 * k * T;
    p += (size_t)4 * k * T;
    f.idx = reinterpret_cast<uint32_t *>(p);
    p += (size_t)4 * T;
    f.hist = reinterpret_cast<uint32_t *>(p);
    p += (size_t)2 * nb;
    f.stage = reinterpret_cast<uint16_t *>(p);
    p += (size_t)2 * T;
    f.sval = reinterpret_cast<float *>(p);
    p += (size_t)4 * T;
    f.sdim = p;
    return f;
}

// Super-key order of coordinate c between local points a and b whose x[c]
// keys are equal: x[c+1 mod k], ..., x[c-1 mod k], then the input index.
__device__ __forceinline__ bool sk_less_tail(const uint32_t *keys, const uint32_t *idx, int T, int k, int c,
                                             uint32_t a, uint32_t b) {
    for (int i = 1; i < k; ++i) {
        int cc = c + i;
        if (cc >= k) cc -= k;
        const uint32_t x = keys[cc * T + a], y = keys[cc * T + b];
        if (x != y) return x < y;
    }
    return idx[a] < idx[b];
}

// Level j of the tile whose first node on level j has level index jv0:
// sizes, left-child sizes and offsets of its nodes i = 0..cnt-1.
struct TileLevel {
    int32_t B, q, rem, half, M, jv0, S0;

    __device__ __forceinline__ int32_t Sf(int32_t J) const { return B * min(J, q) + (J > q ? rem : 0); }
    __device__ __forceinline__ int32_t size(int32_t i) const {
        int32_t r = M - (jv0 + i) * B;
        r = r < 0 ? 0 : (r > B ? B : r);
        return B - 1 + r;
    }
    // ss(lChild(u)) for node i
    __device__ __forceinline__ int32_t msize(int32_t i) const {
        int32_t r = M - (jv0 + i) * B;
        r = r < 0 ? 0 : (r > half ? half : r);
        return half - 1 + r;
    }
    __device__ __forceinline__ int32_t off(int32_t i) const { return i * (B - 1) + Sf(jv0 + i) - S0; }
};

__device__ __forceinline__ TileLevel make_tile_level(const Shape &S, const SfLevel &c, int j, int64_t first) {
    TileLevel t;
    t.B = c.B;
    t.q = c.q;
    t.rem = c.rem;
    t.half = c.B >> 1;
    t.M = (int32_t)S.M;
    t.jv0 = (int32_t)(first - full_nodes(j));
    t.S0 = t.Sf(t.jv0);
    return t;
}

// Split dimension of tile node i on relative depth `depth` under the widest
// rule: clip the tile root's domain by the splits of the node's ancestors
// (recorded in sval / sdim), top-down.
__device__ int sf_widest_dim(const SfArgs &a, const SfSmem &sm, int64_t s0, int depth, int32_t i) {
    float lo[kMaxK], hi[kMaxK];
    const int k = a.k;
    const float *dom = a.dom + (s0 - full_nodes(a.l0)) * 2 * k;
    for (int c = 0; c < k; ++c) {
        lo[c] = dom[c];
        hi[c] = dom[k + c];
    }
    const int64_t lu = (((int64_t)1 << depth) - 1) + i;
    int64_t cur = 0;
    for (int t = depth - 1; t >= 0; --t) {
        const int bit = (int)(((lu + 1) >> t) & 1);
        const int dd = sm.sdim[cur];
        const float v = sm.sval[cur];
        if (dd < k) {
            if (bit) lo[dd] = v;
            else hi[dd] = v;
        }
        cur = 2 * cur + 1 + bit;
    }
    return widest_dim(lo, hi, k);
}

__device__ __forceinline__ int sf_dim(const SfArgs &a, const SfSmem &sm, int64_t s0, int j, int32_t i) {
    return a.mode == KDT_SPLIT_ROUND_ROBIN ? j % a.k : sf_widest_dim(a, sm, s0, j - a.l0, i);
}

// Node i (level-order id u, relative depth `depth`) takes local point `id`,
// split on dimension d, as its split point.
__device__ __forceinline__ void sf_emit(const SfArgs &a, const SfSmem &sm, int64_t base, int depth, int64_t u,
                                        int32_t i, uint32_t id, int d) {
    a.perm[u] = (int32_t)sm.idx[id];
    if (a.mode == KDT_SPLIT_WIDEST) {
        const int32_t lu = ((1 << depth) - 1) + i;  // < n: tile nodes exist left to right
        if (lu < a.T) {
            sm.sval[lu] = key2f(__ldg(a.src_keys + (int64_t)d * a.ld + base + id));
            sm.sdim[lu] = (uint8_t)d;
        }
    }
}

// CTA-wide min and max (every thread gets both); `red` holds 2 * kSfWarps words.
__device__ __forceinline__ void sf_block_minmax(uint32_t &mn, uint32_t &mx, uint32_t *red) {
    mn = __reduce_min_sync(0xffffffffu, mn);
    mx = __reduce_max_sync(0xffffffffu, mx);
    const uint32_t w = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    if (lane == 0) {
        red[w] = mn;
        red[kSfWarps + w] = mx;
    }
    __syncthreads();
    mn = __reduce_min_sync(0xffffffffu, lane < (uint32_t)kSfWarps ? red[lane] : 0xffffffffu);
    mx = __reduce_max_sync(0xffffffffu, lane < (uint32_t)kSfWarps ? red[kSfWarps + lane] : 0u);
    __syncthreads();
}

// Warp: the split of a node on the array of its split coordinate, whose
// segment `seg` lists the node's points in that order.  The points at
// offsets [qb, qe) go to their child in the same order (offset < m: left
// child, dl[offset]; offset > m: right child, dr[offset - m - 1]), their side
// flags are set (0 left, 1 right, 2 split point) and the split point is
// emitted.  Local ids are masked to the tile (T a power of two), so corrupt
// data cannot address outside it; the per-node counts of the other arrays
// catch it.
__device__ __forceinline__ void sf_split_sorted(const SfArgs &a, const SfSmem &sm, const uint16_t *seg, uint32_t qb,
                                                uint32_t qe, uint32_t m, uint16_t *dl, uint16_t *dr, int64_t base,
                                                int depth, int64_t u, int32_t i, int d) {
    const uint32_t tmask = (uint32_t)a.T - 1u;
    for (uint32_t q = qb + lane_id(); q < qe; q += 32) {
        const uint32_t id = seg[q] & tmask;
        sm.side[id] = (uint8_t)(q < m ? 0u : (q == m ? 2u : 1u));
        if (q < m) dl[q] = (uint16_t)id;
        else if (q > m) dr[(q - m - 1u) & tmask] = (uint16_t)id;
        else sf_emit(a, sm, base, depth, u, i, id, d);
    }
}

// Warp: numbers of left and right points at offsets [qb, qe) of `seg` (qb a
// multiple of 32), packed as left | right << 16.
__device__ __forceinline__ uint32_t sf_count_other(const uint16_t *seg, uint32_t qb, uint32_t qe,
                                                   const uint8_t *side, uint32_t tmask) {
    uint32_t l = 0u, r = 0u;
    for (uint32_t q0 = qb; q0 < qe; q0 += 32) {
        const uint32_t q = q0 + lane_id();
        const uint32_t s = q < qe ? side[seg[q] & tmask] : 2u;
        l += __popc(__ballot_sync(0xffffffffu, s == 0u));
        r += __popc(__ballot_sync(0xffffffffu, s == 1u));
    }
    return l | (r << 16);
}

// Warp: stable partition of the points at offsets [qb, qe) of `seg` by
// their side flags: left points to dl[lp...], right points to dr[rp...] in
// their order (lp, rp: points of the node placed by earlier offsets).
// Returns the final lp | rp << 16.  Destinations are masked to the tile.
__device__ __forceinline__ uint32_t sf_split_other(const uint16_t *seg, uint32_t qb, uint32_t qe,
                                                   const uint8_t *side, uint16_t *dl, uint16_t *dr, uint32_t lp,
                                                   uint32_t rp, uint32_t tmask) {
    const uint32_t lane = lane_id(), lt = (1u << lane) - 1u;
    for (uint32_t q0 = qb; q0 < qe; q0 += 32) {
        const uint32_t q = q0 + lane;
        uint32_t id = 0u, s = 2u;
        if (q < qe) {
            id = seg[q] & tmask;
            s = side[id];
        }
        const uint32_t lb = __ballot_sync(0xffffffffu, s == 0u);
        const uint32_t rb = __ballot_sync(0xffffffffu, s == 1u);
        if (s < 2u) {
            uint16_t *dst = s == 0u ? dl + ((lp + __popc(lb & lt)) & tmask) : dr + ((rp + __popc(rb & lt)) & tmask);
            *dst = (uint16_t)id;
        }
        lp += __popc(lb);
        rp += __popc(rb);
    }
    return lp | (rp << 16);
}

// One lane: the whole subtree of node u (level j, index irel on its tile
// level, nn <= 15 points at offset o of every array).  code[id] (the side
// array) is the local level-order index (root 0) of the subtree node that
// holds point id.  Each local node scans the subtree's points in the order of
// its split coordinate, keeps those with its code and ranks them: rank
// ss(lChild) is its split point, lower ranks take the left child's code,
// higher ones the right child's.  A node of at most 3 points emits its
// children (single points) directly.
__device__ void sf_finish_small(const SfArgs &a, const SfSmem &sm, int64_t s0, int64_t base, int j, int64_t u,
                                int32_t irel, int32_t o, int32_t nn, const uint16_t *A) {
    const Shape &S = a.S;
    const int T = a.T, k = a.k;
    const uint32_t tmask = (uint32_t)T - 1u;
    uint8_t *code = sm.side;
    if (nn < 1 || nn > 15 || o < 0 || o + nn > T) {
        set_status(a.status, KDT_EINTERNAL);
        return;
    }
    for (int32_t q = 0; q < nn; ++q) code[A[o + q] & tmask] = 0;
    uint32_t done = 0u;  // local nodes already emitted by their parent
    const int32_t M = (int32_t)S.M;
    const int d0 = j % k;
    for (int v = 0; v < 15; ++v) {
        if ((done >> v) & 1u) continue;
        const int lev = 31 - __clz(v + 1);
        const int jj = j + lev;
        if (jj >= S.L) break;
        const int32_t vl = v + 1 - (1 << lev);
        const int64_t uv = ((u + 1) << lev) - 1 + vl;
        if (uv >= S.N) continue;
        // ss(uv) and ss(lChild(uv)) from the level's constants (32-bit: uv < 2^31)
        const int32_t B = a.lv[jj].B, half = B >> 1;
        const int32_t rm = M - ((int32_t)uv - ((1 << jj) - 1)) * B;
        const int32_t nv = B - 1 + (rm < 0 ? 0 : (rm > B ? B : rm));
        const int32_t mv = jj + 1 < S.L ? half - 1 + (rm < 0 ? 0 : (rm > half ? half : rm)) : 0;
        const int32_t iv = (irel << lev) + vl;
        int d;
        if (a.mode == KDT_SPLIT_ROUND_ROBIN) {
            d = d0 + lev;
            while (d >= k) d -= k;
        } else {
            d = sf_widest_dim(a, sm, s0, jj - a.l0, iv);
        }
        const bool leaves = nv <= 3;
        if (leaves && v < 7) done |= 3u << (2 * v + 1);
        const uint16_t *seg = A + d * T + o;
        int32_t r = 0;
        for (int32_t q = 0; q < nn; ++q) {
            const uint32_t id = seg[q] & tmask;
            if (code[id] != (uint8_t)v) continue;
            if (r == mv) {
                sf_emit(a, sm, base, jj - a.l0, uv, iv, id, d);
                code[id] = 0xff;
            } else if (leaves) {
                const int64_t c = r < mv ? 2 * uv + 1 : 2 * uv + 2;
                if (c < S.N) a.perm[c] = (int32_t)sm.idx[id];
                else set_status(a.status, KDT_EINTERNAL);
                code[id] = 0xff;
            } else {
                code[id] = (uint8_t)(r < mv ? 2 * v + 1 : 2 * v + 2);
            }
            ++r;
        }
        if (r != nv) set_status(a.status, KDT_EINTERNAL);
    }
}

__global__ void __launch_bounds__(kSfThreads, 2) sorted_finisher_kernel(const __grid_constant__ SfArgs a) {
    extern __shared__ __align__(16) unsigned char sf_smem[];
    __shared__ uint32_t red[2 * kSfWarps];
    __shared__ uint32_t wcnt[kSfWarps][kMaxK];
    __shared__ int stop;
    const uint32_t tid = threadIdx.x, NT = kSfThreads;
    const uint32_t w = tid >> 5, lane = tid & 31u;
    if (tid == 0) stop = *(volatile int *)a.status;
    __syncthreads();
    if (stop) {
        if (tid == 0) a.fallback[blockIdx.x] = 0;
        return;
    }
    const Shape &S = a.S;
    const int k = a.k, T = a.T, nb = a.nb;
    const SfSmem sm = sf_carve(sf_smem, k, T, nb);
    const int64_t s0 = full_nodes(a.l0) + blockIdx.x;
    const uint32_t n = (uint32_t)seg_size(S, a.l0, s0);
    const int64_t base = seg_begin(S, a.l0, s0);
    if (n > (uint32_t)T || (uint32_t)T > kSfPPT * NT || (uint32_t)nb % (2u * NT) != 0u || nb > 65536) {
        if (tid == 0) {
            set_status(a.status, KDT_EINTERNAL);
            a.fallback[blockIdx.x] = 0;
        }
        return;
    }

    // 1. load the tile: all loads of a batch are issued before its stores
    for (int c = 0; c <= k; ++c) {
        const uint32_t *col = (c < k ? a.src_keys + (int64_t)c * a.ld : a.src_idx) + base;
        uint32_t *dstc = c < k ? sm.keys + c * T : sm.idx;
        for (uint32_t q = tid; q < n; q += 4 * NT) {
            uint32_t v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = q + u * NT < n ? __ldg(col + q + u * NT) : 0u;
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (q + u * NT < n) dstc[q + u * NT] = v[u];
        }
    }
    __syncthreads();

    // 2. one reference array per coordinate, sorted by its super key
    bool fail = false;
    for (int c = 0; c < k; ++c) {
        const uint32_t *kc = sm.keys + c * T;
        uint32_t mn = 0xffffffffu, mx = 0u;
        for (uint32_t q = tid; q < n; q += NT) {
            const uint32_t v = kc[q];
            mn = min(mn, v);
            mx = max(mx, v);
        }
        sf_block_minmax(mn, mx, red);
        const float lo = key2f(mn);
        const float rg = __fsub_rn(key2f(mx), lo);
        float scale = 0.f;
        bool spread = false;
        if (mn != mx && rg > 0.f && rg <= 3.0e38f) {
            scale = __fdiv_rn((float)nb, rg);
            spread = scale > 0.f && scale <= 3.0e38f;
        }
        if (!spread && n > (uint32_t)kSfMaxBucket) {  // same decision in every thread
            fail = true;
            break;
        }
        for (uint32_t b = tid; b < (uint32_t)nb / 2u; b += NT) sm.hist[b] = 0u;
        __syncthreads();
        uint32_t pk[kSfPPT];
#pragma unroll
        for (int i = 0; i < kSfPPT; ++i) {
            const uint32_t q = tid + (uint32_t)i * NT;
            pk[i] = 0u;
            if (q < n) {
                const uint32_t b = spread ? value_bucket(kc[q], lo, scale, (uint32_t)nb) : 0u;
                const uint32_t sh = (b & 1u) << 4;
                pk[i] = (b << 16) | ((atomicAdd(&sm.hist[b >> 1], 1u << sh) >> sh) & 0xffffu);
            }
        }
        __syncthreads();
        const uint32_t per = (uint32_t)nb / NT;
        uint16_t *h16 = reinterpret_cast<uint16_t *>(sm.hist);  // counters, then bucket starts
        uint32_t sum = 0u;
        int big = 0;
        for (uint32_t i = 0; i < per; ++i) {
            const uint32_t h = h16[tid * per + i];
            sum += h;
            big |= h > (uint32_t)kSfMaxBucket;
        }
        if (__syncthreads_or(big)) {
            fail = true;
            break;
        }
        uint32_t run = block_exclusive_scan(sum, red);
        for (uint32_t i = 0; i < per; ++i) {
            const uint32_t h = h16[tid * per + i];
            h16[tid * per + i] = (uint16_t)run;
            run += h;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kSfPPT; ++i) {
            const uint32_t q = tid + (uint32_t)i * NT;
            if (q < n) sm.stage[h16[pk[i] >> 16] + (pk[i] & 0xffffu)] = (uint16_t)q;
        }
        __syncthreads();
        // rank inside the bucket under the super key of c
        uint16_t *arr = sm.ids0 + c * T;
#pragma unroll
        for (int i = 0; i < kSfPPT; ++i) {
            const uint32_t q = tid + (uint32_t)i * NT;
            if (q < n) {
                const uint32_t b = pk[i] >> 16;
                const uint32_t beg = h16[b], end = b + 1 < (uint32_t)nb ? h16[b + 1] : n;
                uint32_t rank = 0u;
                if (end - beg > 1u) {
                    const uint32_t kq = kc[q];
                    for (uint32_t x = beg; x < end; ++x) {
                        const uint32_t o = sm.stage[x];
                        const uint32_t ko = kc[o];
                        rank += (ko < kq || (ko == kq && o != q && sk_less_tail(sm.keys, sm.idx, T, k, c, o, q)))
                                    ? 1u
                                    : 0u;
                    }
                }
                arr[beg + rank] = (uint16_t)q;
            }
        }
        __syncthreads();
    }
    if (tid == 0) a.fallback[blockIdx.x] = fail ? 1 : 0;
    if (fail) return;

    // 3. levels with fewer nodes than warps: a group of warps per node
    const uint32_t tmask = (uint32_t)T - 1u;
    uint16_t *A = sm.ids0, *Bq = sm.ids1;
    int j = a.l0;
    for (; j + 4 < S.L; ++j) {
        const int depth = j - a.l0;
        const int32_t cnt = 1 << depth;  // levels <= L-2 are full
        if (cnt >= kSfWarps) break;
        const int64_t first = ((s0 + 1) << depth) - 1;
        const TileLevel tl = make_tile_level(S, a.lv[j], j, first);
        const uint32_t wpg = (uint32_t)(kSfWarps / cnt);
        const int32_t i = (int32_t)(w / wpg);
        const uint32_t r = w % wpg, g0 = w - r;
        const int32_t off = tl.off(i), nn = tl.size(i), m = tl.msize(i);
        const int d = sf_dim(a, sm, s0, j, i);
        const uint32_t nch = ((uint32_t)nn + 31u) / 32u;
        const uint32_t qb = min(32u * (r * nch / wpg), (uint32_t)nn);
        const uint32_t qe = min(32u * ((r + 1u) * nch / wpg), (uint32_t)nn);
        const int32_t lo_l = off - i;
        sf_split_sorted(a, sm, A + d * T + off, qb, qe, (uint32_t)m, Bq + d * T + lo_l, Bq + d * T + lo_l + m, base,
                        depth, first + i, i, d);
        __syncthreads();
        for (int c = 0; c < k; ++c) {
            if (c == d) continue;
            const uint32_t v = sf_count_other(A + c * T + off, qb, qe, sm.side, tmask);
            if (lane == 0) wcnt[w][c] = v;
        }
        __syncthreads();
        for (int c = 0; c < k; ++c) {
            if (c == d) continue;
            const uint32_t pre = __reduce_add_sync(0xffffffffu, lane < r ? wcnt[g0 + lane][c] : 0u);
            const uint32_t fin = sf_split_other(A + c * T + off, qb, qe, sm.side, Bq + c * T + lo_l,
                                                Bq + c * T + lo_l + m, pre & 0xffffu, pre >> 16, tmask);
            if (r == wpg - 1u && fin != ((uint32_t)m | ((uint32_t)(nn - 1 - m) << 16)) && lane == 0)
                set_status(a.status, KDT_EINTERNAL);
        }
        __syncthreads();
        uint16_t *t2 = A;
        A = Bq;
        Bq = t2;
    }

    // 4. lower levels: warp w owns nodes [w*cnt/W, (w+1)*cnt/W) of every
    //    level.  Its subtrees stay packed from the offset `wbase` where it
    //    took them over: in the tile-wide layout a warp's range moves left
    //    level by level (split points leave) and would reach ranges that a
    //    slower neighbour still reads.  A warp owns at most 8 nodes per level
    //    here (this phase starts with one node per warp and ends at level L-5
    //    of tiles of at most 4096 points), so lane l holds the constants of
    //    its l-th node -- start of its segment, ss(lChild), left points of the
    //    nodes before it, split dimension -- and every position finds them by
    //    one shuffle from the byte that names its node (written when the
    //    point moved to its child on the level above).  Each array is then
    //    split in one pass over the warp's range, with no per-node loops: the
    //    array of a node's split dimension by offset, the others by side flag
    //    and running left/right counts (left point: Lpre + right points of
    //    the earlier nodes; right point: Rpre + their left points + m).
    bool warp_owned = false;
    int32_t wbase = 0;
    if (j + 4 < S.L) {
        warp_owned = true;
        uint8_t *pcur = reinterpret_cast<uint8_t *>(sm.stage), *pnxt = pcur + T;  // warp-local node of each position
        {
            const int depth = j - a.l0;
            const int64_t first = ((s0 + 1) << depth) - 1;
            const TileLevel tl = make_tile_level(S, a.lv[j], j, first);
            const int32_t per = (1 << depth) / kSfWarps;
            wbase = tl.off((int32_t)w * per);
            int32_t o = wbase;
            for (int32_t l = 0; l < per; ++l) {
                const int32_t nn = tl.size((int32_t)w * per + l);
                for (int32_t q = (int32_t)lane; q < nn; q += 32) pcur[(o + q) & (int32_t)tmask] = (uint8_t)l;
                o += nn;
            }
            __syncwarp();
        }
        for (; j + 4 < S.L; ++j) {
            const int depth = j - a.l0;
            const int32_t cnt = 1 << depth;
            const int64_t first = ((s0 + 1) << depth) - 1;
            const TileLevel tl = make_tile_level(S, a.lv[j], j, first);
            const int32_t per = cnt / kSfWarps;
            const int32_t ib = (int32_t)w * per;
            if (per > 32) {  // cannot happen for T <= 4096; keeps the shuffles in range
                if (lane == 0) set_status(a.status, KDT_EINTERNAL);
                break;
            }
            // lane l: constants of the warp's node l
            int32_t nn_l = 0, m_l = 0, d_l = 0;
            if ((int32_t)lane < per) {
                nn_l = tl.size(ib + (int32_t)lane);
                m_l = tl.msize(ib + (int32_t)lane);
                d_l = a.mode == KDT_SPLIT_ROUND_ROBIN ? j % k : sf_widest_dim(a, sm, s0, depth, ib + (int32_t)lane);
            }
            int32_t st_l = nn_l, lb_l = m_l;  // inclusive scans, then exclusive
#pragma unroll
            for (int o2 = 1; o2 < 32; o2 <<= 1) {
                const int32_t x = __shfl_up_sync(0xffffffffu, st_l, o2), y = __shfl_up_sync(0xffffffffu, lb_l, o2);
                if ((int32_t)lane >= o2) {
                    st_l += x;
                    lb_l += y;
                }
            }
            const int32_t live_w = __shfl_sync(0xffffffffu, st_l, 31), lefts = __shfl_sync(0xffffffffu, lb_l, 31);
            st_l -= nn_l;
            lb_l -= m_l;
            const uint32_t pk1 = (uint32_t)st_l | ((uint32_t)m_l << 16);
            const uint32_t pk2 = (uint32_t)lb_l | ((uint32_t)d_l << 16);
            // the array of each node's split dimension: sides by offset
            for (int32_t q0 = 0; q0 < live_w; q0 += 32) {
                const int32_t q = q0 + (int32_t)lane;
                const bool v = q < live_w;
                const uint32_t nd = v ? pcur[(wbase + q) & (int32_t)tmask] & 31u : 0u;
                const uint32_t a1 = __shfl_sync(0xffffffffu, pk1, nd), a2 = __shfl_sync(0xffffffffu, pk2, nd);
                if (v) {
                    const int32_t st = (int32_t)(a1 & 0xffffu), m = (int32_t)(a1 >> 16), d = (int32_t)(a2 >> 16);
                    const int32_t r = q - st;  // rank in the node's order on d
                    const uint32_t id = A[d * T + ((wbase + q) & (int32_t)tmask)] & tmask;
                    const int32_t cb = st - (int32_t)nd;  // the children's segments start here
                    if (r == m) {
                        sm.side[id] = 2u;
                        sf_emit(a, sm, base, depth, first + ib + (int32_t)nd, ib + (int32_t)nd, id, d);
                    } else {
                        const bool right = r > m;
                        sm.side[id] = right ? 1u : 0u;
                        const int32_t dst = (wbase + cb + (right ? r - 1 : r)) & (int32_t)tmask;
                        Bq[d * T + dst] = (uint16_t)id;
                        pnxt[dst] = (uint8_t)(2u * nd + (right ? 1u : 0u));
                    }
                }
            }
            __syncwarp();
            // the other arrays: stable partition by side flags
            for (int c = 0; c < k; ++c) {
                if (a.mode == KDT_SPLIT_ROUND_ROBIN && c == j % k) continue;
                uint32_t lp = 0u, rp = 0u;
                const uint32_t lt = (1u << lane) - 1u;
                for (int32_t q0 = 0; q0 < live_w; q0 += 32) {
                    const int32_t q = q0 + (int32_t)lane;
                    const bool v = q < live_w;
                    const uint32_t nd = v ? pcur[(wbase + q) & (int32_t)tmask] & 31u : 0u;
                    const uint32_t a1 = __shfl_sync(0xffffffffu, pk1, nd), a2 = __shfl_sync(0xffffffffu, pk2, nd);
                    uint32_t id = 0u, s = 3u;
                    if (v) {
                        id = A[c * T + ((wbase + q) & (int32_t)tmask)] & tmask;
                        s = sm.side[id];
                    }
                    const uint32_t lb = __ballot_sync(0xffffffffu, s == 0u), rb = __ballot_sync(0xffffffffu, s == 1u);
                    // a node split on c itself was moved by the pass above: counted, not stored
                    if (s < 2u && (int32_t)(a2 >> 16) != c) {
                        const int32_t st = (int32_t)(a1 & 0xffffu), m = (int32_t)(a1 >> 16), lbn = (int32_t)(a2 & 0xffffu);
                        const int32_t dst = s == 0u ? (int32_t)(lp + __popc(lb & lt)) + (st - (int32_t)nd - lbn)
                                                    : (int32_t)(rp + __popc(rb & lt)) + lbn + m;
                        Bq[c * T + ((wbase + dst) & (int32_t)tmask)] = (uint16_t)id;
                    }
                    lp += __popc(lb);
                    rp += __popc(rb);
                }
                if (lane == 0 && (lp != (uint32_t)lefts || rp != (uint32_t)(live_w - per - lefts)))
                    set_status(a.status, KDT_EINTERNAL);
            }
            __syncwarp();
            uint16_t *t2 = A;
            A = Bq;
            Bq = t2;
            uint8_t *t3 = pcur;
            pcur = pnxt;
            pnxt = t3;
        }
    }

    // 5. subtrees of at most 15 points (levels >= L-4): one lane each
    {
        const int depth = j - a.l0;
        const int32_t cnt = 1 << depth;
        const int64_t first = ((s0 + 1) << depth) - 1;
        const int64_t count = min((int64_t)cnt, S.N - first);  // nodes that exist
        const TileLevel tl = make_tile_level(S, a.lv[j], j, first);
        // CTA-wide: tile-wide layout; warp-owned: this warp's own nodes,
        // packed from wbase, and no CTA barrier needed
        int32_t ie = (int32_t)count, step = (int32_t)NT, i0 = (int32_t)tid, shift = 0;
        if (warp_owned) {
            const int32_t ib = (int32_t)w * (cnt / kSfWarps);
            ie = ib + cnt / kSfWarps;
            step = 32;
            i0 = ib + (int32_t)lane;
            shift = wbase - tl.off(ib);
        }
        for (int32_t i = i0; i < ie; i += step) {
            const int64_t u = first + i;
            sf_finish_small(a, sm, s0, base, j, u, i, tl.off(i) + shift, (int32_t)seg_size(S, j, u), A);
        }
    }
}

// Tile size T: the largest candidate whose sorted-finisher CTA fits two per
// SM and whose select-finisher CTA (the fallback for the same tiles) fits one.
int pick_tile(int k, int mode, TilePlan *tp) {
    static const int cands[] = {4096, 2048, 1024, 512};
    for (int T : cands) {
        if (T > kSfPPT * kSfThreads) continue;
        const int nb = T > 2 * kSfThreads ? T : 2 * kSfThreads;  // about one point per bucket
        const size_t a = sorted_finisher_smem(k, T, mode, nb);
        const size_t b = select_finisher_smem(k, T, mode);
        if (a <= kSfSmemBudget && b <= kSelectSmemMax) {
            tp->tile = T;
            tp->nb = nb;
            tp->smem = a;
            tp->smem_select = b;
            return 0;
        }
    }
    return -1;
}

int enqueue_finisher(const Plan &p, const Buffers &b, int src, int32_t *perm, cudaStream_t stream) {
    const Shape &S = p.S;
    if (S.L > kMaxLevels) return KDT_EINVAL;
    SfArgs a;
    a.S = S;
    a.k = p.k;
    a.mode = p.mode;
    a.l0 = p.finish_level;
    a.T = p.tp.tile;
    a.nb = p.tp.nb;
    a.ld = p.ld;
    a.src_keys = b.keys[src];
    a.src_idx = b.idx[src];
    a.perm = perm;
    a.dom = b.dom[p.finish_level & 1];
    a.fallback = b.fallback;
    a.status = b.status;
    for (int j = 0; j < kMaxLevels; ++j) {
        SfLevel &c = a.lv[j];
        c = SfLevel{};
        if (j >= S.L) continue;
        const int lgB = S.L - 1 - j;
        const int64_t B = (int64_t)1 << lgB, q = S.M >> lgB;
        c.B = (int32_t)B;
        c.q = (int32_t)q;
        c.rem = (int32_t)(S.M - q * B);
    }
    if (cudaFuncSetAttribute(sorted_finisher_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)p.tp.smem) != cudaSuccess)
        return KDT_ECUDA;
    const int64_t ntiles = nodes_on_level(S, p.finish_level);
    const double Nd = (double)S.N;
    const double sort_levels = (double)(S.L - 1 - p.finish_level);
    {
        ProfScope ps(stream, "finisher", 20.0 * (Nd - (double)full_nodes(p.finish_level)) * sort_levels + 12.0 * Nd);
        sorted_finisher_kernel<<<(unsigned)ntiles, kSfThreads, p.tp.smem, stream>>>(a);
        if (cudaGetLastError() != cudaSuccess) return KDT_ECUDA;
    }
    ProfScope ps(stream, "finisher_select", 0.0);
    return launch_select_finisher(p, b, src, perm, b.fallback, stream);
}

}  // namespace kdt
