// kdt_finisher_sorted.cu -- the presorted shared-memory finisher: one CTA
// owns a subtree of at most T points and fixes all of its remaining levels on
// chip, with one sort per dimension and then in-place partitions.
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
// Layout: in-order.  The tile's subtree is itself a left-balanced complete
// tree of n nodes (height h, Mt nodes on its last level), and every array
// keeps the points of a live node u in the range of in-order positions that
// u's subtree will occupy: [lo(u), lo(u) + ss(u)).  Sorted by its split
// coordinate, that range already reads [left subtree | u | right subtree], so
// u's split point sits at its final in-order position pos(u) = lo(u) +
// ss(lChild(u)) in the array of its own split coordinate, which therefore
// never moves on u's level.  Only the other arrays are partitioned: left
// points to [lo(u), pos(u)), the split point to pos(u), right points after
// it.  Fixed points are never touched again, so after the last level
// position p holds the point of the node whose in-order position is p in
// every array that was partitioned down to that node's level (the output
// reads such an array).  The in-order position <-> node maps of a
// left-balanced tree have closed forms (below); the only node table is the
// current level's node ranges, built from them.
//
// Per tile (subtree s0 of level l0, n <= T points):
//   1. load the k coordinate keys and the input index of its points;
//   2. for each coordinate c, order the local ids by the super key of c: a
//      counting sort into value buckets of x[c] (a monotone map of the key),
//      then each point's rank inside its bucket by comparison under the full
//      super key.  A bucket of more than kSfMaxBucket points (heavy ties or
//      clustered values) leaves the whole tile to the select finisher, which
//      handles any input.  (Round-robin, k = 3, left-balanced tiles: only the
//      tile root's split coordinate here; the other two are sorted on levels
//      0 and 1 per subtree, see the k = 3 schedule in step 3);
//   3. level by level (8 consecutive positions per thread): the side of
//      every live point (left / split / right, stored as its count
//      increment) from the array of its node's split coordinate; then each
//      array that a later level still needs is partitioned in place: each
//      thread holds its 8 ids in registers, a segmented count over the CTA
//      (segments = node ranges, left and right counts packed in one word)
//      gives every point its destination;
//   4. output: node u reads its point at pos(u) of an array that is final
//      there, and writes perm[u] (coalesced: threads walk level order).
#include "kdt_internal.cuh"
#include "kdt_select.cuh"

namespace kdt {

constexpr int kSfPPT = 8;          // positions (sort points) per thread: T = kSfPPT * threads
constexpr int kSfMaxBucket = 16;   // larger buckets leave the tile to the select finisher
constexpr size_t kSfSmemBudget = 110 * 1024;   // two CTAs of up to 512 threads per SM
constexpr size_t kSfSmemBudget1 = 224 * 1024;  // one 1024-thread CTA per SM (T = 8192)
constexpr int kMaxLevels = 32;
constexpr int kSelectOnlyMinK = 5;  // split-widest tiles with this many dimensions go to the select finisher
constexpr uint32_t kSegHead = 0x80000000u;  // scan word: a node range starts inside the scanned span

struct SfArgs {
    Shape S;
    int k, mode, l0, T, nb;
    int64_t tile0;       // this launch's first tile (subtree of level l0, counted from the level's first)
    int64_t ld;
    const uint4 *src;    // records of level l0 (group columns of ld records)
    int32_t *perm;
    const float *dom;    // node table of level l0 (widest mode)
    uint8_t *fallback;   // per tile: 1 = left to the select finisher
    int *status;
};

static size_t align16(size_t x) { return (x + 15) & ~(size_t)15; }

// Dynamic shared memory of one CTA: reference arrays [k][T] u16, keys [k][T]
// u32 (after the sort: the partition increment of each point), input indices
// [T], nb = 2T 8-bit bucket counters plus a 16-bit first position per four
// buckets (after the sort: the node tables of a level), a [T] u16 bucket
// staging array (after the sort, in widest mode: the split dimension of each
// node of a level), and in widest mode the split value and dimension of
// every tile node, in round-robin mode with k = 3 a segment code per point.
size_t sorted_finisher_smem(int k, int T, int mode, int nb) {
    size_t b = (size_t)2 * k * T + (size_t)4 * k * T + (size_t)4 * T + (size_t)nb + (size_t)nb / 2 + (size_t)2 * T;
    if (mode == KDT_SPLIT_WIDEST) b += (size_t)5 * T;
    else if (k == 3) b += (size_t)T;  // segment code per point (k = 3 schedule)
    return align16(b);
}

struct SfSmem {
    uint16_t *ids;    // [k][T]
    uint32_t *keys;   // [k][T], live during the sort
    uint32_t *side;   // [T] partition increment per point, aliases keys after the sort
    uint32_t *idx;    // [T]
    uint32_t *hist;   // [nb / 4]: four 8-bit bucket counters per word
    uint16_t *base16; // [nb / 4]: first sorted position of each word's four buckets
    uint32_t *ntab;   // [T/2] node ranges of a level (lo | pos << 16), aliases hist after the sort
    uint16_t *stage;  // [T] points grouped by bucket, before ranking
    uint8_t *ldim;    // [T/2] split dimension per node of a level, aliases stage (widest mode)
    float *sval;      // [T] split value of tile node (widest mode)
    uint8_t *sdim;    // [T] split dimension of tile node (widest mode)
    uint8_t *segtab;  // [T] segment code per point on the first two levels (k = 3 round-robin), aliases sval
};

__device__ __forceinline__ SfSmem sf_carve(unsigned char *p, int k, int T, int nb) {
    SfSmem f;
    f.ids = reinterpret_cast<uint16_t *>(p);
    p += (size_t)2 * k * T;
    f.keys = reinterpret_cast<uint32_t *>(p);
    f.side = reinterpret_cast<uint32_t *>(p);
    p += (size_t)4 * k * T;
    f.idx = reinterpret_cast<uint32_t *>(p);
    p += (size_t)4 * T;
    f.hist = reinterpret_cast<uint32_t *>(p);
    f.ntab = f.hist;
    f.base16 = reinterpret_cast<uint16_t *>(p + nb);
    p += (size_t)nb + (size_t)nb / 2;
    f.stage = reinterpret_cast<uint16_t *>(p);
    f.ldim = p;
    p += (size_t)2 * T;
    f.sval = reinterpret_cast<float *>(p);
    f.segtab = p;
    p += (size_t)4 * T;
    f.sdim = p;
    return f;
}

// Super-key order of coordinate c between local points a and b whose x[c]
// keys are equal: x[c+1 mod k], ..., x[c-1 mod k], then the input index.
__device__ __noinline__ bool sk_less_tail(const uint32_t *keys, const uint32_t *idx, int T, int k, int c,
                                          uint32_t a, uint32_t b) {
    for (int i = 1; i < k; ++i) {
        int cc = c + i;
        if (cc >= k) cc -= k;
        const uint32_t x = keys[cc * T + a], y = keys[cc * T + b];
        if (x != y) return x < y;
    }
    return idx[a] < idx[b];
}

// ---- in-order closed forms of the tile's left-balanced shape -------------------
// The tile holds n nodes: levels 0..h-2 full, level h-1 holding the first Mt
// of its 2^(h-1) slots.  In the perfect tree of height h the in-order position
// P of the node at level l, index i is (2i+1)*2^(h-1-l) - 1 and its subtree
// starts at i*2^(h-l); the last-level slots that are empty are the even
// positions P >= 2*Mt, so an actual position p maps to P = p below 2*Mt and
// to P = 2p - 2Mt + 1 above it.

// 1-based level-order index (root 1) of the node at in-order position p < n.
__device__ __forceinline__ uint32_t io_node1(uint32_t p, int h, uint32_t Mt) {
    const uint32_t P = p < 2u * Mt ? p : 2u * p - 2u * Mt + 1u;
    const int b = __ffs((int)(P + 1u)) - 1;
    return (1u << (h - 1 - b)) + ((P + 1u) >> (b + 1));
}

// In-order position of node i of level l.
__device__ __forceinline__ uint32_t io_pos(uint32_t i, int l, int h, uint32_t Mt) {
    const uint32_t P = ((2u * i + 1u) << (h - 1 - l)) - 1u;
    return P < 2u * Mt ? P : (P + 2u * Mt - 1u) >> 1;
}

// First in-order position of the subtree of node i of level l.
__device__ __forceinline__ uint32_t io_lo(uint32_t i, int l, int h, uint32_t Mt) {
    const uint32_t P = i << (h - l);
    return P < 2u * Mt ? P : (P >> 1) + Mt;
}

// The same maps for a tile of the balanced shape (n points): walks over the
// gap ranges of its nodes (see bal_node).  An empty node's "position" is its
// gap start; no point is ever assigned to it.
__device__ __forceinline__ uint32_t tile_node1(bool bal, uint32_t p, int h, uint32_t Mt, uint32_t n) {
    if (!bal) return io_node1(p, h, Mt);
    uint32_t u = 1u, a = 0u, c = n + 1u;
    for (int t = 0; t < 32; ++t) {
        const uint32_t hh = c >> 1;
        if (hh == 0u) return 0u;  // not inside any node: cannot happen for p < n
        const uint32_t pos = a + hh - 1u;
        if (p == pos) return u;
        if (p < pos) {
            c = hh;
            u = 2u * u;
        } else {
            a += hh;
            c -= hh;
            u = 2u * u + 1u;
        }
    }
    return 0u;
}

__device__ __forceinline__ uint32_t tile_pos(bool bal, uint32_t i, int l, int h, uint32_t Mt, uint32_t n) {
    if (!bal) return io_pos(i, l, h, Mt);
    int64_t g0, m;
    bal_node(n, l, i, &g0, &m);
    return (uint32_t)(m >= 2 ? g0 + (m >> 1) - 1 : g0);
}

__device__ __forceinline__ uint32_t tile_lo(bool bal, uint32_t i, int l, int h, uint32_t Mt, uint32_t n) {
    if (!bal) return io_lo(i, l, h, Mt);
    int64_t g0, m;
    bal_node(n, l, i, &g0, &m);
    return (uint32_t)g0;
}

// Orders arr[0, T) = the local ids 0..n-1 (padding ids >= n last) by the
// super key of coordinate c: an in-place bitonic sort in shared memory, used
// for a crowded coordinate of a balanced-shape tile (a value bucket with more
// points than the counting sort ranks).  T is a power of two.
template <int NT>
__device__ void bitonic_sort_ids(uint16_t *arr, const uint32_t *kc, const uint32_t *keys, const uint32_t *idx, int T,
                                 int k, int c, uint32_t n) {
    for (uint32_t q = threadIdx.x; q < (uint32_t)T; q += NT) arr[q] = (uint16_t)q;
    __syncthreads();
    for (uint32_t size = 2; size <= (uint32_t)T; size <<= 1) {
        for (uint32_t stride = size >> 1; stride > 0; stride >>= 1) {
            for (uint32_t t = threadIdx.x; t < (uint32_t)T / 2u; t += NT) {
                const uint32_t i = 2u * t - (t & (stride - 1u)), j = i + stride;
                const uint32_t x = arr[i], y = arr[j];
                // y before x under the order (ids >= n after everything)?
                bool y_first;
                if (x >= n || y >= n) y_first = x >= n && (y < n || y < x);
                else y_first = kc[y] < kc[x] || (kc[y] == kc[x] && sk_less_tail(keys, idx, T, k, c, y, x));
                const bool up = (i & size) == 0u;
                if (y_first == up) {
                    arr[i] = (uint16_t)y;
                    arr[j] = (uint16_t)x;
                }
            }
            __syncthreads();
        }
    }
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

// CTA-wide min and max (every thread gets both); `red` holds 2 * NW words.
template <int NW>
__device__ __forceinline__ void sf_block_minmax(uint32_t &mn, uint32_t &mx, uint32_t *red) {
    mn = __reduce_min_sync(0xffffffffu, mn);
    mx = __reduce_max_sync(0xffffffffu, mx);
    const uint32_t w = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    if (lane == 0) {
        red[w] = mn;
        red[NW + w] = mx;
    }
    __syncthreads();
    mn = __reduce_min_sync(0xffffffffu, lane < (uint32_t)NW ? red[lane] : 0xffffffffu);
    mx = __reduce_max_sync(0xffffffffu, lane < (uint32_t)NW ? red[NW + lane] : 0u);
    __syncthreads();
}

// Orders the local ids 0..n-1 into arr = ids[c] by the super key of
// coordinate c: a counting sort into value buckets of x[c] (a monotone map of
// its key), then each point's rank inside its bucket by comparison under the
// full super key.  With nseg > 1 the points are split into segments first:
// code[q] < nseg is point q's segment, code[q] = 4 + j marks a point that
// already has its position fxp[j]; the buckets are taken per segment (nb /
// nseg each), and a point of segment g that is r-th among the other points
// in (segment, bucket, rank) order goes to position r + g -- the segments are
// the subtrees of consecutive in-order ranges, one fixed point between each
// two.  Returns false (in every thread) if a bucket holds more than
// kSfMaxBucket points: the tile is then left to the select finisher (or, for
// a balanced tile, which has none, the coordinate is sorted outright).
template <int NT, int nseg>
__device__ bool sort_coord(const SfSmem &sm, uint32_t *red, int T, int k, int nb, uint32_t n, int c,
                           const uint8_t *code, const uint32_t *fxp, bool bal) {
    constexpr int NW = NT / 32, E = kSfPPT;
    const uint32_t tid = threadIdx.x;
    const uint32_t tmask0 = (uint32_t)T - 1u;  // positions stay inside the tile's arrays
    const uint32_t *kc = sm.keys + c * T;
    uint16_t *arr = sm.ids + c * T;
    uint32_t mn = 0xffffffffu, mx = 0u;
    for (uint32_t q = tid; q < n; q += NT) {
        const uint32_t v = kc[q];
        mn = min(mn, v);
        mx = max(mx, v);
    }
    sf_block_minmax<NW>(mn, mx, red);
    const uint32_t nbs = (uint32_t)nb / (uint32_t)nseg;  // buckets per segment (powers of two)
    const int lgs = 31 - __clz((int)nbs);
    const float lo = key2f(mn);
    const float rg = __fsub_rn(key2f(mx), lo);
    float scale = 0.f;
    bool spread = false;
    if (mn != mx && rg > 0.f && rg <= 3.0e38f) {
        scale = __fdiv_rn((float)nbs, rg);
        spread = scale > 0.f && scale <= 3.0e38f;
    }
    if (!spread && n > (uint32_t)kSfMaxBucket) {  // same decision in every thread
        if (bal && nseg == 1) {  // balanced tiles have no select fallback: sort this coordinate outright
            bitonic_sort_ids<NT>(arr, kc, sm.keys, sm.idx, T, k, c, n);
            return true;
        }
        return false;
    }
    for (uint32_t b = tid; b < (uint32_t)nb / 4u; b += NT) sm.hist[b] = 0u;
    __syncthreads();
    // bucket and arrival slot of each held point (8-bit counters: a slot of
    // kSfMaxBucket or more gives up before any counter can carry into its
    // neighbour); a point with its position already fixed is not counted
    uint32_t pk[E];
    int big = 0;
#pragma unroll
    for (int i = 0; i < E; ++i) {
        const uint32_t q = tid + (uint32_t)i * NT;
        pk[i] = 0xffffffffu;
        if (q < n) {
            uint32_t g = 0u;
            if (nseg > 1) {
                g = code[q];
                if (g >= 4u) continue;
            }
            const uint32_t b = (g << lgs) + (spread ? value_bucket(kc[q], lo, scale, nbs) : 0u);
            const uint32_t sh = (b & 3u) << 3;
            const uint32_t r = (atomicAdd(&sm.hist[b >> 2], 1u << sh) >> sh) & 0xffu;
            big |= r >= (uint32_t)kSfMaxBucket;
            pk[i] = (b << 16) | r;
        }
    }
    if (__syncthreads_or(big)) {
        if (bal && nseg == 1) {
            bitonic_sort_ids<NT>(arr, kc, sm.keys, sm.idx, T, k, c, n);
            return true;
        }
        return false;
    }
    // exclusive scan of the counts: four counter words (16 buckets) per
    // thread; the first position of each word's buckets goes to base16
    constexpr uint32_t WPT = 4;  // nb / 4 / NT with nb = 2T = 16 NT
    uint32_t hw[WPT], sum = 0u;
#pragma unroll
    for (uint32_t i = 0; i < WPT; ++i) {
        hw[i] = sm.hist[tid * WPT + i];
        sum += (hw[i] * 0x01010101u) >> 24;  // byte sum (each count <= kSfMaxBucket)
    }
    uint32_t run = block_exclusive_scan(sum, red);
#pragma unroll
    for (uint32_t i = 0; i < WPT; ++i) {
        sm.base16[tid * WPT + i] = (uint16_t)run;
        run += (hw[i] * 0x01010101u) >> 24;
    }
    __syncthreads();
    // group the points by bucket; st = first position | size << 16
    uint32_t st[E];
#pragma unroll
    for (int i = 0; i < E; ++i) {
        const uint32_t q = tid + (uint32_t)i * NT;
        st[i] = 0u;
        if (pk[i] != 0xffffffffu) {
            const uint32_t b = pk[i] >> 16, j8 = (b & 3u) << 3;
            const uint32_t wv = sm.hist[b >> 2];
            const uint32_t beg = sm.base16[b >> 2] + (((wv * 0x01010100u) >> j8) & 0xffu);  // bytes below b
            sm.stage[(beg + (pk[i] & 0xffffu)) & tmask0] = (uint16_t)q;
            st[i] = beg | (((wv >> j8) & 0xffu) << 16);
        }
    }
    __syncthreads();
    // rank inside the bucket under the super key of c: compared with the
    // bucket's other points (every slot but the point's own arrival slot);
    // the held points step through their buckets together, so their loads
    // overlap
    uint32_t kq[E], rank[E], smax = 0u;
#pragma unroll
    for (int i = 0; i < E; ++i) {
        const uint32_t q = tid + (uint32_t)i * NT;
        const uint32_t sz = st[i] >> 16;
        rank[i] = 0u;
        kq[i] = sz > 1u ? kc[q] : 0u;
        if (sz > 1u) smax = max(smax, sz - 1u);
    }
    for (uint32_t j = 0; j < smax; ++j) {
#pragma unroll
        for (int i = 0; i < E; ++i) {
            const uint32_t sz = st[i] >> 16;
            if (j + 1u < sz) {
                const uint32_t q = tid + (uint32_t)i * NT;
                const uint32_t jj = j < (pk[i] & 0xffu) ? j : j + 1u;  // skip the own slot
                const uint32_t o = sm.stage[((st[i] & 0xffffu) + jj) & tmask0];
                const uint32_t ko = kc[o];
                rank[i] += (ko < kq[i] || (ko == kq[i] && sk_less_tail(sm.keys, sm.idx, T, k, c, o, q))) ? 1u : 0u;
            }
        }
    }
#pragma unroll
    for (int i = 0; i < E; ++i) {
        const uint32_t q = tid + (uint32_t)i * NT;
        if (q >= n) continue;
        if (pk[i] != 0xffffffffu) arr[((st[i] & 0xffffu) + rank[i] + ((pk[i] >> 16) >> lgs)) & tmask0] = (uint16_t)q;
        else arr[fxp[min(code[q] - 4u, 2u)] & tmask0] = (uint16_t)q;  // nseg > 1: a fixed point
    }
    __syncthreads();
    return true;
}

// Segmented sum: `cur` continues the range of `prev` unless a range starts in
// it (kSegHead); the flag of either side survives in bit 31 (values < 2^29).
__device__ __forceinline__ uint32_t seg_combine(uint32_t prev, uint32_t cur) {
    return (cur & kSegHead) ? cur : prev + cur;
}

// Local id number e of the 8 packed in v.
__device__ __forceinline__ uint32_t ids_at(const uint4 &v, int e) {
    const uint32_t wv = e < 2 ? v.x : (e < 4 ? v.y : (e < 6 ? v.z : v.w));
    return (e & 1) ? (wv >> 16) : (wv & 0xffffu);
}

// RR: round-robin split rule; K3: round-robin with k = 3 (the levels move
// each coordinate array once every three levels).
template <int NT, bool RR, bool K3>
__global__ void __launch_bounds__(NT, 1024 / NT) sorted_finisher_kernel(const __grid_constant__ SfArgs a) {
    pdl_enter();
    constexpr int NW = NT / 32, E = kSfPPT;
    static_assert(!K3 || RR, "the k = 3 schedule is a round-robin one");
    extern __shared__ __align__(16) unsigned char sf_smem[];
    __shared__ uint32_t red[64];
    __shared__ uint32_t wagg[2][NW];  // [round parity][warp]: segmented warp sums
    __shared__ uint64_t wagg64[NW];   // k = 3 schedule: segmented warp sums of the 4-field scan
    __shared__ uint32_t fxp[3];      // k = 3 schedule: in-order positions of the tile root and its children
    __shared__ int stop;
    const uint32_t tid = threadIdx.x;
    const uint32_t w = tid >> 5, lane = tid & 31u;
    if (tid == 0) stop = *(volatile int *)a.status;
    __syncthreads();
    const int64_t tile = a.tile0 + blockIdx.x;
    if (stop) {
        if (tid == 0) a.fallback[tile] = 0;
        return;
    }
    const Shape &S = a.S;
    const int k = a.k, T = a.T, nb = a.nb;
    const SfSmem sm = sf_carve(sf_smem, k, T, nb);
    const int64_t s0 = full_nodes(a.l0) + tile;
    const uint32_t n = (uint32_t)seg_size(S, a.l0, s0);
    const int64_t base = seg_begin(S, a.l0, s0);
    const bool bal = S.kind == kShapeBalanced;  // the tile's own shape: left-balanced or balanced
    if (n < 1u || n > (uint32_t)T || T != E * NT || nb != 2 * T) {
        if (tid == 0) {
            set_status(a.status, KDT_EINTERNAL);
            a.fallback[tile] = 0;
        }
        return;
    }

    // 1. load the tile's records: words 0..k-1 to the key arrays, word k to
    //    the input indices (G uint4 per record; a batch's loads go out first)
    for (int gi = 0; gi < rec_groups(k); ++gi) {
        const uint4 *col = a.src + (int64_t)gi * a.ld + base;
        for (uint32_t q = tid; q < n; q += 4 * NT) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = q + u * NT < n ? __ldg(col + q + u * NT) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (q + u * NT >= n) continue;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int wd = 4 * gi + j;
                    if (wd < k) sm.keys[wd * T + q + u * NT] = u4_word(v[u], j);
                    else if (wd == k) sm.idx[q + u * NT] = u4_word(v[u], j);
                }
            }
        }
    }
    __syncthreads();

    // 2. one reference array per coordinate, sorted by its super key (the
    //    k = 3 schedule of a left-balanced tile: only the tile root's split
    //    coordinate here; the next two are sorted per subtree on levels 0
    //    and 1, when the splits above them are known)
    const bool segs = K3 && !bal;
    bool fail = false;
    for (int c = 0; c < k; ++c) {
        if (segs && c != a.l0 % 3) continue;
        if (!sort_coord<NT, 1>(sm, red, T, k, nb, n, c, nullptr, nullptr, bal)) {
            fail = true;
            break;
        }
    }
    if (tid == 0) a.fallback[tile] = fail ? 1 : 0;
    if (fail) return;

    // 3. levels.  Thread tid owns in-order positions p0 .. p0+7; g[e] is the
    //    1-based level-order index (tile-local) of the node whose final
    //    position is p0+e, followed by a terminating one bit and shifted left
    //    until its leading one is bit 31 (0 past the tile): bit 30 - j is then
    //    the side taken below level j.  On level l, t = g << (l + 1) is 0 if
    //    the position is fixed (the node's level is < l), exactly bit 31 for
    //    the node of level l itself (its split point), and otherwise has the
    //    side in bit 31; the node on level l has index g >> (31 - l).
    //    side[id] holds the point's count increment for the partition: 1
    //    (left), 1 << 16 (right) or 0 (split point).
    const uint32_t tmask = (uint32_t)T - 1u;
    constexpr bool rr = RR;
    const int h = 32 - __clz((int)n);
    const uint32_t Mt = n - ((1u << (h - 1)) - 1u);
    const uint32_t p0 = tid * (uint32_t)E;
    const bool wact = w * 32u * (uint32_t)E < n;  // the warp holds a position of the tile
    // the left-aligned code of the node at in-order position p (0 past the tile)
    auto gcode = [&](uint32_t p) -> uint32_t {
        const uint32_t u1 = p < n ? tile_node1(bal, p, h, Mt, n) : 0u;
        return u1 ? ((u1 << 1) | 1u) << (__clz((int)u1) - 1) : 0u;
    };
    uint32_t g[E];
    const int last = h - 2;  // deepest level that moves an array
    if (!rr) {
        if (tid == 0) sm.ldim[0] = (uint8_t)sf_widest_dim(a, sm, s0, 0, 0);
        __syncthreads();
    }
    if constexpr (K3) {
        // Round-robin, k = 3: each coordinate array is moved once every three
        // levels instead of twice.  On level l the split array d_l is in order
        // for the nodes of level l.  Array d_{l+1} was last in order for the
        // nodes of level l-1 (it was the split array of level l-2); here it
        // absorbs the splits of levels l-1 and l in one pass: each point of a
        // level-(l-1) node w goes to one of w's four grandchildren, or is the
        // split point of w or of one of w's children (fixed at its position).
        // Level 0 moves d_1 by the root's split alone.  The scan carries the
        // four grandchildren's first positions (16-bit fields of a 64-bit
        // word, set at the first position of w's range), so a point's
        // destination is one field of its running value.
        constexpr uint64_t kHead64 = 1ull << 63;
        uint32_t *side32 = sm.side;                                 // [T]: two 16-bit sides, by level parity
        uint16_t *side16 = reinterpret_cast<uint16_t *>(sm.side);
        uint16_t *ptab0 = reinterpret_cast<uint16_t *>(sm.ntab);   // [T/2] in-order position + 1 of each node of a level
        uint16_t *ptab1 = ptab0 + T / 2;
        // Left-balanced tiles sort d_1 and d_2 per subtree instead (levels 0
        // and 1 below): the segment code of each point (its side of the
        // splits above, or which split point it is) goes to segtab, and the
        // sort puts every point at its position for the next level directly.
        int l_first = 0;
        if (segs) {
            if (tid < 3u)
                fxp[tid] = tid == 0u ? tile_pos(bal, 0u, 0, h, Mt, n) : (h >= 2 ? tile_pos(bal, tid - 1u, 1, h, Mt, n) : 0u);
#pragma unroll
            for (int l = 0; l < 2; ++l) {
                if (l >= last) break;
                const int dl = (a.l0 + l) % 3, c = (a.l0 + l + 1) % 3;  // d_l, d_{l+1}
                // A': segment codes from d_l -- level 0: 0 left, 1 right, 4
                //     the root; level 1: 2 * (level-0 side) + side, 5 / 6 the
                //     split points of the root's children
                if (wact) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(sm.ids + dl * T + p0);
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const uint32_t ge = gcode(p0 + (uint32_t)e);
                        const uint32_t t = ge << (l + 1);
                        if (t == 0u) continue;
                        const uint32_t id = ids_at(v, e) & tmask;
                        if (l == 0) sm.segtab[id] = (uint8_t)(t == 0x80000000u ? 4u : (t >> 31));
                        else
                            sm.segtab[id] = (uint8_t)(t == 0x80000000u ? 5u + ((ge >> 30) & 1u)
                                                                        : 2u * sm.segtab[id] + (t >> 31));
                    }
                }
                __syncthreads();
                const bool ok = l == 0 ? sort_coord<NT, 2>(sm, red, T, k, nb, n, c, sm.segtab, fxp, bal)
                                       : sort_coord<NT, 4>(sm, red, T, k, nb, n, c, sm.segtab, fxp, bal);
                if (!ok) {
                    if (tid == 0) a.fallback[tile] = 1;  // crowded: the select finisher takes the tile
                    return;
                }
                if (l == 1) {
                    // the keys are no longer read: level 1's sides go to the
                    // side words for level 2's moves (the root is not looked up)
                    for (uint32_t id = tid; id < n; id += NT) {
                        const uint32_t cd = sm.segtab[id];
                        if (cd == 4u) continue;
                        side16[2u * id + 1u] = (uint16_t)(cd >= 5u ? (0x8000u | fxp[min(cd - 4u, 2u)]) : (cd & 1u));
                    }
                    __syncthreads();
                }
                l_first = l + 1;
            }
        }
#pragma unroll
        for (int e = 0; e < E; ++e) g[e] = gcode(p0 + (uint32_t)e);
        const uint32_t gprev = p0 > 0u ? gcode(p0 - 1u) : 0u;
        int dl = (a.l0 + l_first) % 3;
        for (int l = l_first; l < last; ++l, dl = dl == 2 ? 0 : dl + 1) {
            const uint32_t q = (uint32_t)l & 1u;
            uint16_t *pt_l = q ? ptab1 : ptab0;
            const uint16_t *pt_p = q ? ptab0 : ptab1;  // level l - 1
            const int c = dl == 2 ? 0 : dl + 1;  // d_{l+1}
            for (uint32_t i = tid; i < (1u << l); i += NT) pt_l[i] = (uint16_t)(tile_pos(bal, i, l, h, Mt, n) + 1u);
            if (segs && l == 2) {  // level 1's table was overwritten by the sort's counters
                for (uint32_t i = tid; i < 2u; i += NT) ptab1[i] = (uint16_t)(fxp[1u + i] + 1u);
            }
            // A: side of every point of a level-l node, from d_l: 0 left,
            //    1 right, 0x8000 | position for the node's split point
            if (wact) {
                const uint4 v = *reinterpret_cast<const uint4 *>(sm.ids + dl * T + p0);
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const uint32_t t = g[e] << (l + 1);
                    if (t == 0u) continue;
                    const uint32_t id = ids_at(v, e) & tmask;
                    side16[2u * id + q] = (uint16_t)(t == 0x80000000u ? (0x8000u | (p0 + (uint32_t)e)) : (t >> 31));
                }
            }
            __syncthreads();
            // B: live positions of level l-1 (level 0: the whole tile), running
            //    value before each held point, warp scan
            uint4 iv = make_uint4(0u, 0u, 0u, 0u);
            uint64_t X[E];
            uint32_t mask = 0u;
            uint64_t exw = 0ull;
            if (wact) {
                iv = *reinterpret_cast<const uint4 *>(sm.ids + c * T + p0);
                bool pl = (gprev << l) != 0u;
                uint64_t run = 0ull;
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const bool lv = (g[e] << l) != 0u;
                    if (lv && !pl) {  // first position of a level-(l-1) node w
                        uint64_t base = (uint64_t)(p0 + (uint32_t)e);
                        if (l == 0) {
                            base |= (uint64_t)pt_l[0] << 16;
                        } else {
                            const uint32_t wi = (g[e] >> (32 - l)) ^ (1u << (l - 1));
                            base |= ((uint64_t)pt_l[2u * wi] << 16) | ((uint64_t)pt_p[wi] << 32) |
                                    ((uint64_t)pt_l[2u * wi + 1u] << 48);
                        }
                        run = kHead64 | base;
                    }
                    pl = lv;
                    X[e] = run;
                    if (lv) {
                        mask |= 1u << e;
                        const uint32_t sw = side32[ids_at(iv, e) & tmask];
                        const uint32_t s1 = l == 0 ? 0u : (sw >> (16u * (q ^ 1u))) & 0xffffu;
                        const uint32_t s2 = (sw >> (16u * q)) & 0xffffu;
                        if (!((s1 | s2) & 0x8000u)) run += 1ull << (16u * (2u * s1 + s2));
                    }
                }
                uint64_t x = run;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint64_t y = __shfl_up_sync(0xffffffffu, x, o);
                    if (lane >= (uint32_t)o) x = (x & kHead64) ? x : y + x;
                }
                if (lane == 31u) wagg64[w] = x;
                const uint64_t ex = __shfl_up_sync(0xffffffffu, x, 1);
                exw = lane == 0u ? 0ull : ex;
            }
            __syncthreads();
            // D: carry from the warps before, destinations, in-place stores
            if (wact) {
                uint64_t v = lane < (uint32_t)NW ? wagg64[lane] : 0ull;
#pragma unroll
                for (int o = 1; o < NW; o <<= 1) {
                    const uint64_t y = __shfl_up_sync(0xffffffffu, v, o);
                    if (lane >= (uint32_t)o) v = (v & kHead64) ? v : y + v;
                }
                const uint64_t cw = __shfl_sync(0xffffffffu, v, (w + 31u) & 31u);
                const uint64_t lb =
                    (exw & kHead64) ? (exw & ~kHead64) : (w > 0u ? (cw & ~kHead64) : 0ull) + exw;
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    if (!((mask >> e) & 1u)) continue;
                    const uint32_t id = ids_at(iv, e);
                    const uint32_t sw = side32[id & tmask];
                    const uint32_t s1 = l == 0 ? 0u : (sw >> (16u * (q ^ 1u))) & 0xffffu;
                    const uint32_t s2 = (sw >> (16u * q)) & 0xffffu;
                    uint32_t dst;
                    if (s1 & 0x8000u) {
                        dst = s1 & 0x1fffu;
                    } else if (s2 & 0x8000u) {
                        dst = s2 & 0x1fffu;
                    } else {
                        const uint64_t val = (X[e] & kHead64) ? (X[e] & ~kHead64) : lb + X[e];
                        dst = (uint32_t)(val >> (16u * (2u * s1 + s2))) & 0x1fffu;
                    }
                    if (dst < n) sm.ids[c * T + dst] = (uint16_t)id;
                    else set_status(a.status, KDT_EINTERNAL);
                }
            }
            __syncthreads();
        }
    } else {
#pragma unroll
        for (int e = 0; e < E; ++e) g[e] = gcode(p0 + (uint32_t)e);
        const uint32_t gprev = p0 > 0u ? gcode(p0 - 1u) : 0u;
        const uint32_t allk = k >= 32 ? 0xffffffffu : (1u << k) - 1u;  // k <= KDT_MAX_K = 32
        int dl0 = rr ? a.l0 % k : 0;           // round-robin split coordinate of level l
        int par = 0;
        for (int l = 0; l <= last; ++l, dl0 = dl0 + 1 == k ? 0 : dl0 + 1) {
            // arrays to partition on this level: round-robin -- those that some
            // level in (l, last] splits on (the last - l coordinates after dl0,
            // cyclically), except this level's own; widest -- all (a node's own
            // split array is skipped per point)
            uint32_t mv = allk;
            if (rr) {
                const int m = last - l;
                if (m < k - 1) {
                    // bits dl0+1 .. dl0+m, unwrapped (at most bit 62 for k = 32), then folded mod k
                    const uint64_t run = ((1ull << m) - 1ull) << (dl0 + 1);
                    mv = (uint32_t)((run | (run >> k)) & allk);
                }
                mv &= ~(1u << dl0);
                if (mv == 0u) break;  // k >= 2: only for l >= h-2; k == 1: never moves
            }
            // this level's node ranges: lo | pos << 16 per node
            for (uint32_t i = tid; i < (1u << l); i += NT)
                sm.ntab[i] = tile_lo(bal, i, l, h, Mt, n) | (tile_pos(bal, i, l, h, Mt, n) << 16);
            // live / head masks: a node range starts at p if p is live and p-1
            // is not (p-1 holds a fixed ancestor, or p == 0)
            uint32_t live = 0u, head = 0u;
            if (wact) {
                bool pl = (gprev << (l + 1)) != 0u;
    #pragma unroll
                for (int e = 0; e < E; ++e) {
                    const bool lv = (g[e] << (l + 1)) != 0u;
                    live |= (uint32_t)lv << e;
                    head |= (uint32_t)(lv && !pl) << e;
                    pl = lv;
                }
                if (p0 == 0u) head |= live & 1u;
                // phase A: side increments from the split arrays
                if (rr) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(sm.ids + dl0 * T + p0);
    #pragma unroll
                    for (int e = 0; e < E; ++e) {
                        if (!((live >> e) & 1u)) continue;
                        const uint32_t t = g[e] << (l + 1);
                        sm.side[ids_at(v, e) & tmask] = t == 0x80000000u ? 0u : ((t >> 31) ? 0x10000u : 1u);
                    }
                } else {
    #pragma unroll
                    for (int e = 0; e < E; ++e) {
                        if (!((live >> e) & 1u)) continue;
                        const uint32_t t = g[e] << (l + 1);
                        const uint32_t ga = g[e] >> (31 - l);
                        int d = sm.ldim[ga ^ (1u << l)];
                        if (d >= k) {  // corrupt table: record it, keep every access in range
                            set_status(a.status, KDT_EINTERNAL);
                            d = 0;
                        }
                        const uint32_t id = sm.ids[d * T + p0 + e] & tmask;
                        sm.side[id] = t == 0x80000000u ? 0u : ((t >> 31) ? 0x10000u : 1u);
                        if (t == 0x80000000u) {
                            const uint32_t ib = id < n ? id : 0u;  // a permutation of [0, n) unless corrupt
                            sm.sval[ga - 1u] = key2f(rec_word(a.src, a.ld, d, base + ib));
                            sm.sdim[ga - 1u] = (uint8_t)d;
                        }
                    }
                }
            }
            __syncthreads();
            // phases B and D, one array at a time (B of the next array may run
            // while slower warps finish D of this one: different arrays, and the
            // warp sums alternate between two buffers)
            uint32_t rest = mv;
            while (rest != 0u) {
                const int c = __ffs((int)rest) - 1;
                rest &= rest - 1u;
                uint4 iv = make_uint4(0u, 0u, 0u, 0u);
                uint32_t X[E], mask = 0u, exw = 0u;
                // B: running left | right << 16 counts before each held point,
                // from its range start (kSegHead set) or from p0; warp scan
                if (wact) {
                    iv = *reinterpret_cast<const uint4 *>(sm.ids + c * T + p0);
                    mask = live;
                    if (!rr) {
    #pragma unroll
                        for (int e = 0; e < E; ++e) {
                            if (!((live >> e) & 1u)) continue;
                            if (sm.ldim[(g[e] >> (31 - l)) ^ (1u << l)] == c) mask &= ~(1u << e);  // own split array
                        }
                    }
                    uint32_t run = 0u;
    #pragma unroll
                    for (int e = 0; e < E; ++e) {
                        if ((head >> e) & 1u) run = kSegHead;
                        X[e] = run;
                        if ((mask >> e) & 1u) run += sm.side[ids_at(iv, e) & tmask];
                    }
                    uint32_t x = run;
    #pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
                        if (lane >= (uint32_t)o) x = seg_combine(y, x);
                    }
                    if (lane == 31u) wagg[par][w] = x;
                    const uint32_t ex = __shfl_up_sync(0xffffffffu, x, 1);
                    exw = lane == 0u ? 0u : ex;
                }
                __syncthreads();
                // D: carry from the warps before, destinations, in-place stores
                if (wact) {
                    uint32_t v = lane < (uint32_t)NW ? wagg[par][lane] : 0u;
    #pragma unroll
                    for (int o = 1; o < NW; o <<= 1) {
                        const uint32_t y = __shfl_up_sync(0xffffffffu, v, o);
                        if (lane >= (uint32_t)o) v = seg_combine(y, v);
                    }
                    const uint32_t cw = __shfl_sync(0xffffffffu, v, (w + 31u) & 31u);
                    const uint32_t lb = (exw & kSegHead) ? (exw & ~kSegHead) : (w > 0u ? (cw & ~kSegHead) : 0u) + exw;
    #pragma unroll
                    for (int e = 0; e < E; ++e) {
                        if (!((mask >> e) & 1u)) continue;
                        const uint32_t id = ids_at(iv, e);
                        const uint32_t inc = sm.side[id & tmask];
                        const uint32_t val = (X[e] & kSegHead) ? (X[e] & ~kSegHead) : lb + X[e];
                        const uint32_t nt = sm.ntab[(g[e] >> (31 - l)) ^ (1u << l)];
                        const uint32_t pos = nt >> 16;
                        const uint32_t dst = inc == 1u ? (nt & 0xffffu) + (val & 0xffffu)
                                                       : (inc == 0u ? pos : pos + 1u + (val >> 16));
                        if (dst < n) sm.ids[c * T + dst] = (uint16_t)id;
                        else set_status(a.status, KDT_EINTERNAL);
                    }
                }
                par ^= 1;
            }
            // widest: split dimensions of the next level's nodes (their
            // ancestors' split values were recorded in phase A)
            if (!rr && l + 1 <= last) {
                for (uint32_t i = tid; i < (1u << (l + 1)); i += NT) sm.ldim[i] = (uint8_t)sf_widest_dim(a, sm, s0, l + 1, (int32_t)i);
            }
            __syncthreads();
        }
    }

    // 4. output: node u of the tile (level lv, index i) reads its point at
    //    pos(u) from an array that is final there -- in round-robin mode the
    //    array of its own level's split coordinate (leaves: the one of level
    //    h-2), in widest mode any (all arrays move on every level)
    const uint32_t nodes = bal ? (1u << h) - 1u : n;  // balanced: empty slots keep the -1 written up front
    for (uint32_t u = tid; u < nodes; u += NT) {
        const uint32_t g1 = u + 1u;
        const int lv = 31 - __clz((int)g1);
        const uint32_t i = g1 - (1u << lv);
        if (bal) {
            int64_t g0, m;
            bal_node(n, lv, i, &g0, &m);
            if (m < 2) continue;  // an empty subtree
        }
        const uint32_t p = tile_pos(bal, i, lv, h, Mt, n);
        if (p >= n) {
            set_status(a.status, KDT_EINTERNAL);
            continue;
        }
        const int c = rr ? (a.l0 + min(lv, max(last, 0))) % k : 0;
        const uint32_t id = sm.ids[c * T + p] & tmask;
        a.perm[((s0 + 1) << lv) - 1 + i] = (int32_t)sm.idx[id];
    }
}

// Tile size T: 8192 if its sorted-finisher CTA (1024 threads) fits one per
// SM, else the largest candidate whose CTA (T / 8 threads) fits two per SM;
// the select-finisher CTA (the fallback for the same tiles) must fit one.
// Every global level a larger tile absorbs is a whole-array pass saved.
int pick_tile(int k, int mode, TilePlan *tp) {
    static const int cands[] = {8192, 4096, 2048, 1024, 512};
    for (int T : cands) {
        const int nb = 2 * T;  // about one point per two buckets
        // (split-widest with k >= kSelectOnlyMinK never runs the sorted finisher)
        const size_t a = mode == KDT_SPLIT_WIDEST && k >= kSelectOnlyMinK ? 0 : sorted_finisher_smem(k, T, mode, nb);
        const size_t b = select_finisher_smem(k, T, mode);
        if (a <= (T == 8192 ? kSfSmemBudget1 : kSfSmemBudget) && b <= kSelectSmemMax) {
            tp->tile = T;
            tp->nb = nb;
            tp->smem = a;
            tp->smem_select = b;
            return 0;
        }
    }
    return -1;
}

template <int NT, bool RR, bool K3>
static int launch_sorted_mode(const SfArgs &a, int64_t ntiles, size_t smem, cudaStream_t stream) {
    if (cudaFuncSetAttribute(sorted_finisher_kernel<NT, RR, K3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return KDT_ECUDA;
    launch_pdl(sorted_finisher_kernel<NT, RR, K3>, (unsigned)ntiles, NT, smem, stream, a);
    return cudaGetLastError() == cudaSuccess ? KDT_OK : KDT_ECUDA;
}

template <int NT>
static int launch_sorted(const SfArgs &a, int64_t ntiles, size_t smem, cudaStream_t stream) {
    if (a.mode != KDT_SPLIT_ROUND_ROBIN) return launch_sorted_mode<NT, false, false>(a, ntiles, smem, stream);
    return a.k == 3 ? launch_sorted_mode<NT, true, true>(a, ntiles, smem, stream)
                    : launch_sorted_mode<NT, true, false>(a, ntiles, smem, stream);
}

int enqueue_finisher(const Plan &p, const Buffers &b, int src, int32_t *perm, cudaStream_t stream) {
    const Shape &S = p.S;
    if (S.L > kMaxLevels) return KDT_EINVAL;
    // Split-widest with k >= 5: a presorted tile would move its k - 1 other
    // arrays on every level; one rank select per node is cheaper there
    // (measured, 4M uniform points: k = 5 1.02 vs 1.14 ms, k = 8 1.52 vs
    // 1.85 ms; k = 3: 0.94 vs 0.61 ms the other way).
    if (p.mode == KDT_SPLIT_WIDEST && p.k >= kSelectOnlyMinK && S.kind == kShapeLeftBalanced) {
        ProfScope ps(stream, "finisher_select", 0.0);
        return launch_select_finisher(p, b, src, perm, nullptr, stream);
    }
    SfArgs a;
    a.S = S;
    a.k = p.k;
    a.mode = p.mode;
    a.l0 = p.finish_level;
    a.T = p.tp.tile;
    a.nb = p.tp.nb;
    a.ld = p.ld;
    a.src = b.rec[src];
    a.perm = perm;
    a.dom = b.dom[p.finish_level & 1];
    a.fallback = b.fallback;
    a.status = b.status;
    const int64_t ntiles = nodes_on_level(S, p.finish_level);
    const double Nd = (double)S.N;
    const double sort_levels = (double)(S.L - 1 - p.finish_level);
    // Tiles of at most T/2 points run in half-size CTAs (twice as many per
    // SM).  Subtree sizes on the level do not increase with the index: q
    // subtrees of 2B-1 points, one of B-1+rem, the rest B-1.
    const int Ts = a.T / 2;
    int64_t nbig = ntiles;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 152;
    // (with no more tiles than SMs, one launch runs them all side by side)
    if (Ts >= 512 && S.kind != kShapeBalanced && ntiles > sms) {
        const int lgB = S.L - 1 - p.finish_level;
        const int64_t B = (int64_t)1 << lgB, q = S.M >> lgB, rem = S.M - (q << lgB);
        if (B - 1 <= Ts) {
            nbig = 2 * B - 1 > Ts ? q : 0;
            if (nbig < ntiles && B - 1 + rem > Ts) ++nbig;
            if (nbig > ntiles) nbig = ntiles;
        }
    }
    {
        ProfScope ps(stream, "finisher", 20.0 * (Nd - (double)full_nodes(p.finish_level)) * sort_levels + 12.0 * Nd);
        auto launch = [&](const SfArgs &x, int64_t n_tiles, size_t smem) -> int {
            if (n_tiles <= 0) return KDT_OK;
            switch (x.T / kSfPPT) {
                case 1024: return launch_sorted<1024>(x, n_tiles, smem, stream);
                case 512: return launch_sorted<512>(x, n_tiles, smem, stream);
                case 256: return launch_sorted<256>(x, n_tiles, smem, stream);
                case 128: return launch_sorted<128>(x, n_tiles, smem, stream);
                case 64: return launch_sorted<64>(x, n_tiles, smem, stream);
                default: return KDT_EINVAL;
            }
        };
        a.tile0 = 0;
        ps.kernels = (nbig > 0 ? 1 : 0) + (nbig < ntiles ? 1 : 0);
        int rc = launch(a, nbig, p.tp.smem);
        if (rc != KDT_OK) return rc;
        if (nbig < ntiles) {
            SfArgs b2 = a;
            b2.T = Ts;
            b2.nb = 2 * Ts;
            b2.tile0 = nbig;
            rc = launch(b2, ntiles - nbig, sorted_finisher_smem(a.k, Ts, a.mode, 2 * Ts));
            if (rc != KDT_OK) return rc;
        }
    }
    if (S.kind == kShapeBalanced) return KDT_OK;  // balanced tiles never fall back (crowded coordinates are sorted)
    ProfScope ps(stream, "finisher_select", 0.0);
    return launch_select_finisher(p, b, src, perm, b.fallback, stream);
}

}  // namespace kdt
