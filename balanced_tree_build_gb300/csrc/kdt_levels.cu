// kdt_levels.cu -- the global levels of the build: one record pass per level.
//
// For every live subtree s of level l the method needs the point of rank
// m = ss(lChild(s)) under s's split order, and the split of the other points
// into lChild(s) and rChild(s) ("GPU-friendly, Parallel, and (Almost-)In-Place
// Construction of Left-Balanced k-d Trees", core-idea and tag-update
// passages).  Here that is done in three steps:
//
//  1. histogram: each point's split coordinate falls into one of kBuckets
//     value buckets spread evenly over s's domain [lo, hi] in the split
//     dimension (the bucket index is a monotone function of the coordinate);
//  2. pick: the bucket b* that holds rank m, and the counts below it;
//  3. partition: points in buckets below b* certainly go left, above b*
//     certainly right; they are written straight to the children's ranges.
//     Points in b* ("candidates", typically a few per thousand) go to a side
//     buffer; an exact most-significant-digit select over the full split
//     order (cyclic super key, then input index) among them fixes the split
//     point and places the rest.
//
// Step 1 for level l+1 is fused into step 3 of level l when the next split
// dimension differs from the current one (round-robin rule, k >= 2): the
// child's domain in that dimension is the parent's, so the child's buckets
// are known while the parent is partitioned.  Step 2 for level l+1 then runs
// in the CTA that resolves subtree s on level l (its children's histograms
// are final once its candidates are added; each half of the CTA picks one
// child).  Level 0 has a histogram pass of its own, whose last CTA picks.
// With k = 3 points in device memory, level 0 reads the input points and
// builds the records in registers.
//
// Levels with at most 1024 subtrees are spread over all SMs ("multi-CTA"
// pipeline: separate histogram / pick / partition / resolve kernels with
// per-subtree cursors); once there are more subtrees than that each CTA owns
// one subtree and runs all steps itself ("seg" kernel).
#include "kdt_internal.cuh"
#include "kdt_select.cuh"

namespace kdt {

constexpr int kLvlThreads = 512;
constexpr int kResThreadsMax = 1024;  // resolve CTAs of subtrees with many candidates
constexpr uint32_t kSelList = 2048;   // listed candidates of a resolve CTA's select
constexpr int64_t kHistPoints = 16384;  // histogram pass: points per CTA at least
constexpr int kPickThreads = 256;
constexpr int kEPT = 4;                          // consecutive points per thread per tile (divides 8: rows up to
                                                 // the next multiple of 8 exist in every record buffer)
constexpr int kPartCtas = 8;                     // partition CTAs per SM
constexpr int kPartThreads = 128;                // partition CTAs (multi-CTA and per-subtree)
constexpr int kTile = kPartThreads * kEPT;

// ---- value buckets ----------------------------------------------------------

struct Bucketer {
    float lo, scale;
    int nb;  // number of buckets
    // Monotone non-decreasing in the coordinate: fsub and fmul round to
    // nearest (monotone), truncation and clamping are monotone.
    __device__ __forceinline__ int operator()(uint32_t key) const {
        const float x = key2f(key);
        const float t = __fmul_rn(__fsub_rn(x, lo), scale);
        int b = __float2int_rz(t);
        b = b < 0 ? 0 : b;
        return b < nb ? b : nb - 1;
    }
};

__device__ __forceinline__ Bucketer make_bucketer(float lo, float hi, int nb = kBuckets) {
    const float r = __fsub_rn(hi, lo);
    float scale = 0.f;  // empty or non-finite range: every point in bucket 0
    if (r > 0.f && r <= 3.0e38f) {
        scale = __fdiv_rn((float)nb, r);
        if (!(scale <= 3.0e38f)) scale = 0.f;
    }
    Bucketer b;
    b.lo = lo;
    b.scale = scale;
    b.nb = nb;
    return b;
}

// Finite keys: f2key(-FLT_MAX) .. f2key(FLT_MAX).  Every point's key lies
// there (non-finite input is rejected), and the bucket function is monotone
// on that range.
constexpr uint32_t kKeyMin = 0x00800000u, kKeyMax = 0xff7fffffu;

// Smallest finite key whose bucket is >= b, or kKeyMax + 1 if none: the
// points of buckets < b are exactly the keys below it (binary search on the
// monotone bucket function).
__device__ uint32_t first_key_at_least(const Bucketer &bk, uint32_t b) {
    if (b >= (uint32_t)bk.nb) return kKeyMax + 1u;
    uint32_t lo = kKeyMin, hi = kKeyMax + 1u;
    while (lo < hi) {
        const uint32_t mid = lo + (hi - lo) / 2u;
        if ((uint32_t)bk(mid) >= b) hi = mid;
        else lo = mid + 1u;
    }
    return lo;
}

// Subtree of level l that holds array position p (inverse of sb).
__device__ __forceinline__ int64_t seg_of_pos(const Shape &S, int l, int64_t p) {
    if (S.kind == kShapeBalanced) {  // sb increases along the level: binary search, O(l^2)
        int64_t lo = 0, hi = ((int64_t)1 << l) - 1;
        while (lo < hi) {
            const int64_t mid = (lo + hi + 1) >> 1;
            if (seg_begin(S, l, full_nodes(l) + mid) <= p) lo = mid;
            else hi = mid - 1;
        }
        return full_nodes(l) + lo;
    }
    const int64_t B = (int64_t)1 << (S.L - 1 - l), A = B - 1;
    const int64_t q = p - full_nodes(l);
    const int64_t nf = S.M / B;          // subtrees with a full last-level part
    const int64_t r = S.M - nf * B;      // last-level part of subtree nf
    const int64_t full_end = nf * (A + B);
    int64_t j;
    if (q < full_end) {
        j = q / (A + B);
    } else {
        const int64_t q2 = q - full_end;
        if (r > 0) j = q2 < A + r ? nf : nf + 1 + (q2 - (A + r)) / A;
        else j = nf + q2 / A;
    }
    return full_nodes(l) + j;
}

// ---- per-level arguments -----------------------------------------------------

struct LevelArgs {
    Shape S;
    int k, mode, l;
    const uint4 *src;    // records of this level (G group columns of ld records)
    uint4 *dst, *cand;   // records of the next level; candidates of the split buckets
    int G;               // record groups: ceil((k + 1) / 4)
    int32_t *perm;
    const float *dom_cur;
    const int *dim_cur;
    float *dom_nxt;
    int *dim_nxt;
    uint32_t *hist_cur;  // [subtrees][nbk] (multi-CTA levels)
    int nbk;             // buckets of this level's histogram (kBuckets0 on level 0 of a large build, else kBuckets)
    uint32_t *hist_nxt;  // children's histograms (fused next level) or null
    SegSel *sel;
    int hist_in;         // per-subtree levels: this level's histograms were built by the level above
    int warp_res;        // partition: each warp reserves its own output ranges (no CTA barriers)
    const uint32_t *col0;  // level 0, round-robin: dense keys of the split coordinate (else null)
    // level 0, k = 3: the input points (16-byte aligned float triples, point q
    // at position q), read in place of the records, which are built in
    // registers (else null)
    const float *pts3;
    // resolve: pick the next level's split buckets for this subtree's two
    // children (their histograms are final once its candidates are added)
    int pick_next;
    SegSel *sel_next;      // the next level's selections
    uint32_t *hist_nn;     // histograms of the level after next (cleared for the grandchildren), or null
    int *status;
    int *done;           // histogram pass of a one-subtree level: CTAs finished (the last one picks), or null
    int64_t per_cta;     // positions per CTA (persistent multi-CTA kernels)
    int64_t ld;          // records per group column
};

struct SegInfo {
    int64_t s, j, base, left_begin;
    uint32_t n, m, nr;
    int d;
};

__device__ __forceinline__ SegInfo seg_info(const LevelArgs &a, int64_t s) {
    SegInfo g;
    g.s = s;
    g.j = s - full_nodes(a.l);
    g.base = seg_begin(a.S, a.l, s);
    g.n = (uint32_t)seg_size(a.S, a.l, s);
    g.m = (uint32_t)seg_size(a.S, a.l + 1, 2 * s + 1);
    g.nr = g.n - g.m - 1u;
    g.left_begin = seg_begin(a.S, a.l + 1, 2 * s + 1);
    g.d = a.mode == KDT_SPLIT_ROUND_ROBIN ? a.l % a.k : a.dim_cur[g.j];
    return g;
}

__device__ __forceinline__ Bucketer seg_bucketer(const LevelArgs &a, int64_t j, int d, int nb = kBuckets) {
    const float *dom = a.dom_cur + j * 2 * a.k;
    return make_bucketer(dom[d], dom[a.k + d], nb);
}

__device__ __forceinline__ bool stop_requested(const int *status, int *flag) {
    if (threadIdx.x == 0) *flag = *(volatile const int *)status;
    __syncthreads();
    return *flag != 0;
}

// Child domains: the parent's domain with the split coordinate as the left
// child's upper and the right child's lower bound (the clip by the split
// plane of the split-widest-dimension passage), plus their widest dimension.
__device__ void write_child_domains(const float *dom_p, int k, int d, float split, float *dom_l, int *dim_l,
                                    float *dom_r, int *dim_r) {
    float lo[kMaxK], hi[kMaxK];
    for (int c = 0; c < k; ++c) {
        lo[c] = dom_p[c];
        hi[c] = dom_p[k + c];
    }
    const float h = hi[d];
    hi[d] = split;
    for (int c = 0; c < k; ++c) {
        dom_l[c] = lo[c];
        dom_l[k + c] = hi[c];
    }
    *dim_l = widest_dim(lo, hi, k);
    hi[d] = h;
    lo[d] = split;
    for (int c = 0; c < k; ++c) {
        dom_r[c] = lo[c];
        dom_r[k + c] = hi[c];
    }
    *dim_r = widest_dim(lo, hi, k);
}

// ---- partition of one tile ----------------------------------------------------

// Side of a point relative to the split bucket: 0 left, 1 candidate, 2 right.
// Certain-left points fill lChild's range from its start, certain-right ones
// fill rChild's range from its end, candidates take slots 0..cnt-1 of the
// candidate buffer (slot cnt-1 is position s, the node's own, unused, array
// position; the others are the gap between the two certain groups).
struct PartPlan {
    uint32_t bstar, below, cnt, above;
    uint32_t klo, khi;   // keys of the split bucket b*: [klo, khi)
    int64_t right_tail;  // first position of the certain-right group
};

// Prefetches the record lines of the tile starting at t0 (clipped to ve)
// into L2, so that the tile's loads, issued two tiles later, wait on L2
// rather than DRAM: one 128-byte line (8 records) per thread and group.
__device__ __forceinline__ void prefetch_tile(const LevelArgs &a, int64_t t0, int64_t ve, bool pts3 = false) {
    if (pts3) {  // the tile's float triples: 12 bytes per point
        const char *p = reinterpret_cast<const char *>(a.pts3);
        const int64_t b0 = 12 * t0, b1 = 12 * min(ve, t0 + (int64_t)kTile);
        for (int64_t o = b0 + 128 * (int64_t)threadIdx.x; o < b1; o += 128 * (int64_t)blockDim.x)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(p + o));
        return;
    }
    const uint32_t lines = kTile / 8;  // 128-byte lines per group column
    for (uint32_t t = threadIdx.x; t < (uint32_t)a.G * lines; t += blockDim.x) {
        const uint32_t gi = t / lines;
        const int64_t q = t0 + (int64_t)(t - gi * lines) * 8;
        if (q >= ve) continue;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(a.src + (int64_t)gi * a.ld + q));
    }
}

// Partitions the points of [vb, ve) that fall in the tile starting at t0 (a
// multiple of 4): thread t handles positions t0 + 4t .. t0 + 4t + 3.
// `cursors` points at three counters (left, candidate, right) in shared or
// global memory; `wtot` and `wbase` are 3 words per warp of shared scratch;
// `fh` is the fused children's histogram in shared memory, or null.
//
// Every word of the thread's records that fits the register budget is
// loaded first (128-bit loads), so a thread waits for about one memory
// latency per tile.  Output order is slot-major per warp: for each of the 4
// slots the warp's lanes going to one side write consecutive positions
// (ballot + popcount), so every warp store covers one contiguous run.
template <bool kPts3 = false>
__device__ void part_tile(const LevelArgs &a, const SegInfo &g, const Bucketer &bk, const PartPlan &pp, int64_t t0,
                          int64_t vb, int64_t ve, uint32_t *cursors, uint32_t *wtot, uint32_t *wbase, uint32_t *fh,
                          const Bucketer &bkc, int dn) {
    // positions are below 2^31 (N < 2^31): 32-bit arithmetic from here on
    const int64_t ld = a.ld;
    const int d = g.d;
    const uint32_t tid = threadIdx.x, nt = blockDim.x;
    const uint32_t lane = tid & 31u, w = tid >> 5, nw = nt >> 5;
    const uint32_t lt = (1u << lane) - 1u;
    const uint32_t q0 = (uint32_t)t0 + (uint32_t)kEPT * tid;
    const uint32_t vb32 = (uint32_t)vb, ve32 = (uint32_t)ve;
    const bool any = q0 + (uint32_t)kEPT > vb32 && q0 < ve32;
    // group 0 of the thread's four records (for k <= 3 the whole record);
    // rows up to q0 + 3 < ld exist in every buffer
    uint4 r[kEPT];
    if constexpr (kPts3) {  // level 0, k = 3: four points are three 128-bit words of the input
        if (any && q0 + (uint32_t)kEPT <= (uint32_t)a.S.N) {
            const uint4 *p4 = reinterpret_cast<const uint4 *>(a.pts3) + 3u * (q0 >> 2);
            const uint4 v0 = __ldg(p4), v1 = __ldg(p4 + 1), v2 = __ldg(p4 + 2);
            const uint32_t f[12] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w, v2.x, v2.y, v2.z, v2.w};
#pragma unroll
            for (int i = 0; i < kEPT; ++i)
                r[i] = make_uint4(f2key(__uint_as_float(f[3 * i])), f2key(__uint_as_float(f[3 * i + 1])),
                                  f2key(__uint_as_float(f[3 * i + 2])), q0 + (uint32_t)i);
        } else {
#pragma unroll
            for (int i = 0; i < kEPT; ++i) {
                const uint32_t q = q0 + (uint32_t)i;
                r[i] = any && q < (uint32_t)a.S.N
                           ? make_uint4(f2key(__ldg(a.pts3 + 3u * q)), f2key(__ldg(a.pts3 + 3u * q + 1u)),
                                        f2key(__ldg(a.pts3 + 3u * q + 2u)), q)
                           : make_uint4(0u, 0u, 0u, 0u);
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < kEPT; ++i) r[i] = any ? __ldcs(a.src + q0 + i) : make_uint4(0u, 0u, 0u, 0u);
    }
    uint32_t kx[kEPT];
#pragma unroll
    for (int i = 0; i < kEPT; ++i)
        kx[i] = d < 4 ? u4_word(r[i], d) : (any ? rec_word(a.src, ld, d, q0 + i) : 0u);
    // certain points: two ballots per point (certain, right); the
    // candidates of the split bucket (a few per thousand) are reserved per
    // warp straight from the candidate cursor
    uint32_t mV[kEPT], mR[kEPT];
    uint32_t tL = 0, tR = 0;
    int side[kEPT];
#pragma unroll
    for (int i = 0; i < kEPT; ++i) {
        const uint32_t q = q0 + (uint32_t)i;
        side[i] = 3;
        if (q >= vb32 && q < ve32) side[i] = kx[i] < pp.klo ? 0 : (kx[i] >= pp.khi ? 2 : 1);  // bucket vs b*
        mV[i] = __ballot_sync(0xffffffffu, side[i] == 0 || side[i] == 2);
        mR[i] = __ballot_sync(0xffffffffu, side[i] == 2);
        tL += __popc(mV[i] & ~mR[i]);
        tR += __popc(mR[i]);
    }
    uint32_t oL, oR;
    if (a.warp_res) {  // one reservation per warp and side (cursors spread over many subtrees, or in shared memory)
        uint32_t bL = 0u, bR = 0u;
        if (lane == 0) {
            if (tL) bL = atomicAdd(&cursors[0], tL);
            if (tR) bR = atomicAdd(&cursors[2], tR);
        }
        oL = __shfl_sync(0xffffffffu, bL, 0);
        oR = __shfl_sync(0xffffffffu, bR, 0);
    } else {  // one reservation per CTA and side, then the warps' offsets
        if (lane == 0) {
            wtot[2 * w + 0] = tL;
            wtot[2 * w + 1] = tR;
        }
        __syncthreads();
        if (tid < 2u) {
            uint32_t sum = 0u;
            for (uint32_t v = 0; v < nw; ++v) sum += wtot[2 * v + tid];
            uint32_t base = sum ? atomicAdd(&cursors[tid ? 2 : 0], sum) : 0u;
            for (uint32_t v = 0; v < nw; ++v) {
                wbase[2 * v + tid] = base;
                base += wtot[2 * v + tid];
            }
        }
        __syncthreads();
        oL = wbase[2 * w + 0];
        oR = wbase[2 * w + 1];
    }
    const uint32_t lbeg = (uint32_t)g.left_begin, rtail = (uint32_t)pp.right_tail;
    const uint32_t cgap = lbeg + pp.below, s32 = (uint32_t)g.s;
    // pos: destination position of each point (32 bit); side 3 = not stored
    uint32_t pos[kEPT];
#pragma unroll
    for (int i = 0; i < kEPT; ++i) {
        pos[i] = 0u;
        const uint32_t mL = mV[i] & ~mR[i];
        bool ok = true;
        if (side[i] == 0) {
            const uint32_t o = oL + __popc(mL & lt);
            ok = o < pp.below;
            pos[i] = lbeg + o;
        } else if (side[i] == 2) {
            const uint32_t o = oR + __popc(mR[i] & lt);
            ok = o < pp.above;
            pos[i] = rtail + o;
        }
        oL += __popc(mL);
        oR += __popc(mR[i]);
        const uint32_t cm = __ballot_sync(0xffffffffu, side[i] == 1);
        if (cm) {
            const int leader = __ffs((int)cm) - 1;
            uint32_t cb = 0u;
            if ((int)lane == leader) cb = atomicAdd(&cursors[1], (uint32_t)__popc(cm));
            cb = __shfl_sync(0xffffffffu, cb, leader);
            if (side[i] == 1) {
                const uint32_t o = cb + __popc(cm & lt);
                ok = o < pp.cnt;
                pos[i] = o + 1u < pp.cnt ? cgap + o : s32;  // candidate slot o: the gap, the last one position s
            }
        }
        if (!ok) {
            set_status(a.status, KDT_EINTERNAL);
            side[i] = 3;
        }
    }
    // stores: group 0 from registers, then the other groups (k >= 4)
#pragma unroll
    for (int i = 0; i < kEPT; ++i) {
        if (side[i] == 0 || side[i] == 2) {
            __stcs(a.dst + pos[i], r[i]);  // not read again before the next level's pass: evict first
            if (fh != nullptr && dn < 4) atomicAdd(&fh[(side[i] == 0 ? 0 : kBuckets) + bkc(u4_word(r[i], dn))], 1u);
        } else if (side[i] == 1) {
            a.cand[pos[i]] = r[i];
        }
    }
    for (int gi = 1; gi < a.G; ++gi) {
        uint4 v[kEPT];
#pragma unroll
        for (int i = 0; i < kEPT; ++i) v[i] = any ? __ldg(a.src + (int64_t)gi * ld + q0 + i) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int i = 0; i < kEPT; ++i) {
            if (side[i] == 3) continue;
            (side[i] == 1 ? a.cand : a.dst)[(int64_t)gi * ld + pos[i]] = v[i];
            if (fh != nullptr && (dn >> 2) == gi && side[i] != 1)
                atomicAdd(&fh[(side[i] == 0 ? 0 : kBuckets) + bkc(u4_word(v[i], dn & 3))], 1u);
        }
    }
}

// ---- exact resolve of the candidates -----------------------------------------

// Word i of candidate slot q (split order of dimension d).
struct CandAcc {
    const uint4 *rec;
    int64_t ld, gap_begin, s;  // ld: records per group column
    uint32_t cnt;
    int k, d;
    __device__ __forceinline__ int64_t pos(uint32_t q) const { return q + 1u < cnt ? gap_begin + q : s; }
    __device__ __forceinline__ uint32_t operator()(int i, uint32_t q) const {
        int c = d + i;
        if (i == k) c = k;  // the input index
        else if (c >= k) c -= k;
        return rec_word(rec, ld, c, pos(q));
    }
};

// CTA-wide: selects the split point among the candidates, writes perm[s] and
// the children's node-table entries, and moves the other candidates into the
// gap between the certain groups.  `fuse`: add the candidates to the
// children's histograms of the next level.
__device__ void resolve_segment(const LevelArgs &a, const SegInfo &g, const PartPlan &pp, SelState &st,
                                uint32_t *hist, uint32_t *red, uint32_t *medw, uint32_t *cur2, bool fuse, int dn,
                                uint32_t *qbuf, uint32_t qcap) {
    const uint32_t tid = threadIdx.x, nt = blockDim.x;
    const int k = a.k;
    const int64_t ld = a.ld;
    const uint32_t r = g.m - pp.below;  // rank of the split point among the candidates
    const CandAcc acc{a.cand, ld, g.left_begin + pp.below, g.s, pp.cnt, k, g.d};
    if (pp.cnt <= 32u) {  // a few candidates (deep levels): one warp selects, no CTA barriers per round
        if (tid < 32u) group_select(WarpsGroup{0u, 32u, 1}, acc, pp.cnt, r, k + 1, st, hist, kWarpRadixBits, red);
        __syncthreads();
    } else {
        cta_select(acc, pp.cnt, r, k + 1, st, hist, red, qbuf, qcap);
    }
    if (st.err) {
        if (tid == 0) set_status(a.status, KDT_EINTERNAL);
        return;
    }
    for (uint32_t i = tid; i <= (uint32_t)k; i += nt) medw[i] = acc((int)i, st.med_q);  // k + 1 words, k <= 32
    if (tid < 2) cur2[tid] = 0u;
    __syncthreads();
    Bucketer bkc;
    bkc.lo = 0.f;
    bkc.scale = 0.f;
    if (fuse) bkc = seg_bucketer(a, g.j, dn);
    const uint32_t lane = tid & 31u, lt = (1u << lane) - 1u;
    const uint32_t nright = pp.cnt - 1u - r;
    const int64_t right_begin = g.left_begin + g.m;
    // up to four candidates per thread and round (one if every thread has at
    // most one): their first words, and then each column of the moved
    // records, are loaded before they are used
    constexpr int kRB = 4;
    const int rb = pp.cnt > nt ? kRB : 1;
    for (uint32_t q0 = 0; q0 < pp.cnt; q0 += (uint32_t)rb * nt) {
        uint32_t w0[kRB];
#pragma unroll
        for (int u = 0; u < kRB; ++u) {
            const uint32_t q = q0 + (uint32_t)u * nt + tid;
            w0[u] = u < rb && q < pp.cnt ? acc(0, q) : 0u;
        }
        int side[kRB];
        int64_t pos[kRB], sp[kRB];
#pragma unroll
        for (int u = 0; u < kRB; ++u) {
            const uint32_t q = q0 + (uint32_t)u * nt + tid;
            side[u] = -1;
            pos[u] = 0;
            sp[u] = 0;
            if (u >= rb) continue;  // uniform: rb is the same in every thread
            if (q < pp.cnt) {
                const int c = w0[u] != medw[0] ? (w0[u] < medw[0] ? -1 : 1) : cmp_words(acc, q, medw, k + 1);
                side[u] = c < 0 ? 0 : (c > 0 ? 1 : -1);
            }
            const uint32_t lm = __ballot_sync(0xffffffffu, side[u] == 0);
            const uint32_t rm = __ballot_sync(0xffffffffu, side[u] == 1);
            uint32_t lb = 0, rb2 = 0;
            if (lane == 0) {
                if (lm) lb = atomicAdd(&cur2[0], __popc(lm));
                if (rm) rb2 = atomicAdd(&cur2[1], __popc(rm));
            }
            lb = __shfl_sync(0xffffffffu, lb, 0);
            rb2 = __shfl_sync(0xffffffffu, rb2, 0);
            if (side[u] >= 0) {
                bool ok;
                if (side[u] == 0) {
                    const uint32_t o = lb + __popc(lm & lt);
                    ok = o < r;
                    pos[u] = g.left_begin + pp.below + o;
                } else {
                    const uint32_t o = rb2 + __popc(rm & lt);
                    ok = o < nright;
                    pos[u] = right_begin + o;
                }
                if (ok) {
                    sp[u] = acc.pos(q);
                } else {
                    set_status(a.status, KDT_EINTERNAL);
                    side[u] = -1;
                }
            }
        }
        for (int gi = 0; gi < a.G; ++gi) {
            uint4 v[kRB];
#pragma unroll
            for (int u = 0; u < kRB; ++u) v[u] = side[u] >= 0 ? a.cand[(int64_t)gi * ld + sp[u]] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int u = 0; u < kRB; ++u) {
                if (side[u] < 0) continue;
                a.dst[(int64_t)gi * ld + pos[u]] = v[u];
                if (fuse && (dn >> 2) == gi)
                    atomicAdd(&a.hist_nxt[(2 * g.j + side[u]) * kBuckets + bkc(u4_word(v[u], dn & 3))], 1u);
            }
        }
    }
    __syncthreads();
    if (tid == 0) {
        if (cur2[0] != r || cur2[1] != nright) set_status(a.status, KDT_EINTERNAL);
        a.perm[g.s] = (int32_t)medw[k];
        write_child_domains(a.dom_cur + g.j * 2 * k, k, g.d, key2f(medw[0]), a.dom_nxt + (2 * g.j) * 2 * k,
                            a.dim_nxt + 2 * g.j, a.dom_nxt + (2 * g.j + 1) * 2 * k, a.dim_nxt + 2 * g.j + 1);
    }
}

// Picks the bucket holding rank m from a histogram of nb counts (CTA-wide;
// nb a multiple of the CTA size).  Returns false if the counts do not add up
// to n.
template <class G>
__device__ bool pick_bucket_g(const G &grp, const uint32_t *H, uint32_t n, uint32_t m, uint32_t *red, PartPlan *out,
                              int nb) {
    const uint32_t tid = grp.tid(), nt = grp.size();
    const uint32_t per = (uint32_t)nb / nt;
    uint32_t sum = 0;
    for (uint32_t i = 0; i < per; ++i) sum += H[tid * per + i];
    uint32_t total;
    const uint32_t excl = group_exclusive_scan(grp, sum, red, total);
    if (m >= excl && m < excl + sum) {
        uint32_t c = excl;
        for (uint32_t i = 0; i < per; ++i) {
            const uint32_t h = H[tid * per + i];
            if (m < c + h) {
                out->bstar = tid * per + i;
                out->below = c;
                out->cnt = h;
                out->above = n - c - h;
                break;
            }
            c += h;
        }
    }
    grp.sync();
    return total == n;
}

__device__ bool pick_bucket(const uint32_t *H, uint32_t n, uint32_t m, uint32_t *red, PartPlan *out,
                            int nb = kBuckets) {
    return pick_bucket_g(CtaGroup{}, H, n, m, red, out, nb);
}

// Histogram of the bucket function over word d of records [b, e) into shared
// `hist`; each thread issues eight loads before its atomics (the records are
// in global memory; col points at word d of record 0, stride 4 words).
__device__ __forceinline__ void hist_range(const uint32_t *col, int64_t b, int64_t e, const Bucketer &bk,
                                           uint32_t *hist, int stride = 4) {
    constexpr int kH = 8;
    const uint32_t nt = blockDim.x;
    for (int64_t q0 = b + threadIdx.x; q0 < e; q0 += (int64_t)kH * nt) {
        uint32_t v[kH];
#pragma unroll
        for (int u = 0; u < kH; ++u) {
            const int64_t q = q0 + (int64_t)u * nt;
            v[u] = q < e ? __ldg(col + stride * q) : 0u;
        }
#pragma unroll
        for (int u = 0; u < kH; ++u)
            if (q0 + (int64_t)u * nt < e) atomicAdd(&hist[bk(v[u])], 1u);
    }
}

// ---- multi-CTA pipeline kernels ----------------------------------------------

__device__ void pick_subtree(const LevelArgs &a, int64_t s, PartPlan &pp, uint32_t *red);

// Histogram of each subtree's split coordinate over its value buckets.  With
// a.done set (a level of one subtree) the CTA that finishes last also picks
// the split bucket: the others' counts are in the histogram by then.
__global__ void __launch_bounds__(kLvlThreads) level_hist_kernel(LevelArgs a) {
    pdl_enter();
    extern __shared__ uint32_t hist[];  // [a.nbk]
    __shared__ int stop;
    if (stop_requested(a.status, &stop)) return;
    const int64_t begin = full_nodes(a.l) + (int64_t)blockIdx.x * a.per_cta;
    const int64_t end = min(a.S.N, begin + a.per_cta);
    const int64_t ld = a.ld;
    for (int64_t p = begin; p < end;) {
        const int64_t s = seg_of_pos(a.S, a.l, p);
        const SegInfo g = seg_info(a, s);
        const int64_t pe = min(end, g.base + (int64_t)g.n);
        const Bucketer bk = seg_bucketer(a, g.j, g.d, a.nbk);
        for (uint32_t b = threadIdx.x; b < (uint32_t)a.nbk; b += blockDim.x) hist[b] = 0u;
        __syncthreads();
        if (a.col0 != nullptr) {  // level 0: the dense column of the split coordinate
            hist_range(a.col0, p, pe, bk, hist, 1);
        } else {
            const uint32_t *col = reinterpret_cast<const uint32_t *>(a.src + (int64_t)(g.d >> 2) * ld) + (g.d & 3);
            hist_range(col, p, pe, bk, hist);
        }
        __syncthreads();
        uint32_t *H = a.hist_cur + g.j * a.nbk;
        for (uint32_t b = threadIdx.x; b < (uint32_t)a.nbk; b += blockDim.x)
            if (hist[b]) atomicAdd(&H[b], hist[b]);
        __syncthreads();
        p = pe;
    }
    if (a.done != nullptr) {
        __shared__ int last;
        __shared__ uint32_t red[64];
        __shared__ PartPlan pp;
        __threadfence();  // this CTA's counts are in the histogram before it counts itself done
        __syncthreads();
        if (threadIdx.x == 0) last = atomicAdd(a.done, 1) == (int)gridDim.x - 1;
        __syncthreads();
        if (last) {
            __threadfence();
            pick_subtree(a, full_nodes(a.l), pp, red);
        }
    }
}

// CTA-wide: the split bucket of subtree s of level a.l from its histogram
// (a.nbk buckets), written to a.sel[j] with cleared cursors; with a.hist_nxt
// set, the children's histogram rows of the next level are cleared too.
// `pp` and `red` are shared scratch.
template <class G>
__device__ void pick_subtree_g(const G &grp, const LevelArgs &a, int64_t s, PartPlan &pp, uint32_t *red) {
    const uint32_t tid = grp.tid();
    const SegInfo g = seg_info(a, s);
    const bool ok = pick_bucket_g(grp, a.hist_cur + g.j * a.nbk, g.n, g.m, red, &pp, a.nbk);
    // key bounds of the split bucket: two binary searches in two warps
    if (tid == 32) pp.khi = first_key_at_least(seg_bucketer(a, g.j, g.d, a.nbk), pp.bstar + 1u);
    if (tid == 0) pp.klo = first_key_at_least(seg_bucketer(a, g.j, g.d, a.nbk), pp.bstar);
    grp.sync();
    if (tid == 0) {
        if (!ok) set_status(a.status, KDT_EINTERNAL);
        SegSel sl;
        sl.bstar = pp.bstar;
        sl.below = pp.below;
        sl.cnt = pp.cnt;
        sl.curL = sl.curC = sl.curR = 0u;
        sl.klo = pp.klo;
        sl.khi = pp.khi;
        a.sel[g.j] = sl;
    }
    if (a.hist_nxt) {
        uint32_t *H = a.hist_nxt + 2 * g.j * kBuckets;
        for (uint32_t t = tid; t < 2u * kBuckets; t += grp.size()) H[t] = 0u;
    }
    grp.sync();
}

__device__ void pick_subtree(const LevelArgs &a, int64_t s, PartPlan &pp, uint32_t *red) {
    pick_subtree_g(CtaGroup{}, a, s, pp, red);
}

__global__ void __launch_bounds__(kPickThreads) level_pick_kernel(LevelArgs a) {
    pdl_enter();
    __shared__ uint32_t red[64];
    __shared__ PartPlan pp;
    __shared__ int stop;
    if (stop_requested(a.status, &stop)) return;
    pick_subtree(a, full_nodes(a.l) + blockIdx.x, pp, red);
}

__device__ __forceinline__ PartPlan part_plan(const SegInfo &g, uint32_t bstar, uint32_t below, uint32_t cnt,
                                              uint32_t klo, uint32_t khi) {
    PartPlan pp;
    pp.bstar = bstar;
    pp.below = below;
    pp.cnt = cnt;
    pp.klo = klo;
    pp.khi = khi;
    pp.above = g.n - below - cnt;
    pp.right_tail = g.left_begin + g.m + (g.nr - pp.above);
    return pp;
}

// kPts3: level 0 reads the k = 3 input points in place of records (a.pts3).
template <bool kPts3>
__global__ void __launch_bounds__(kPartThreads, kPartCtas) level_part_kernel(LevelArgs a) {
    pdl_enter();
    __shared__ uint32_t wtot[2 * 32], wbase[2 * 32];
    __shared__ uint32_t fh[2 * kBuckets];
    __shared__ int stop;
    if (stop_requested(a.status, &stop)) return;
    const int64_t begin = full_nodes(a.l) + (int64_t)blockIdx.x * a.per_cta;
    const int64_t end = min(a.S.N, begin + a.per_cta);
    const bool fuse = a.hist_nxt != nullptr;
    const int dn = (a.l + 1) % a.k;
    for (int64_t p = begin; p < end;) {
        const int64_t s = seg_of_pos(a.S, a.l, p);
        const SegInfo g = seg_info(a, s);
        const int64_t pe = min(end, g.base + (int64_t)g.n);
        const Bucketer bk = seg_bucketer(a, g.j, g.d);
        const SegSel sl = a.sel[g.j];
        const PartPlan pp = part_plan(g, sl.bstar, sl.below, sl.cnt, sl.klo, sl.khi);
        Bucketer bkc;
        bkc.lo = 0.f;
        bkc.scale = 0.f;
        if (fuse) {
            bkc = seg_bucketer(a, g.j, dn);
            for (uint32_t b = threadIdx.x; b < 2u * kBuckets; b += blockDim.x) fh[b] = 0u;
        }
        __syncthreads();
        for (int64_t t0 = p & ~(int64_t)(kEPT - 1); t0 < pe; t0 += kTile) {
            if (t0 + 2 * kTile < pe) prefetch_tile(a, t0 + 2 * kTile, pe, kPts3);
            part_tile<kPts3>(a, g, bk, pp, t0, p, pe, &a.sel[g.j].curL, wtot, wbase, fuse ? fh : nullptr, bkc, dn);
        }
        __syncthreads();
        if (fuse) {
            uint32_t *H = a.hist_nxt + 2 * g.j * kBuckets;
            for (uint32_t b = threadIdx.x; b < 2u * kBuckets; b += blockDim.x)
                if (fh[b]) atomicAdd(&H[b], fh[b]);
            __syncthreads();
        }
        p = pe;
    }
}

__global__ void __launch_bounds__(kResThreadsMax) level_resolve_kernel(LevelArgs a) {
    pdl_enter();
    __shared__ SelState st;
    __shared__ uint32_t hist[kCtaRadixBins];
    __shared__ uint32_t qbuf[kSelList];
    __shared__ uint32_t red[64];
    __shared__ uint32_t medw[kMaxWords];
    __shared__ uint32_t cur2[2];
    __shared__ int stop;
    if (stop_requested(a.status, &stop)) return;
    const int64_t s = full_nodes(a.l) + blockIdx.x;
    const SegInfo g = seg_info(a, s);
    const SegSel sl = a.sel[g.j];
    const PartPlan pp = part_plan(g, sl.bstar, sl.below, sl.cnt, sl.klo, sl.khi);
    if (sl.curL != pp.below || sl.curC != pp.cnt || sl.curR != pp.above) {
        if (threadIdx.x == 0) set_status(a.status, KDT_EINTERNAL);
        return;
    }
    resolve_segment(a, g, pp, st, hist, red, medw, cur2, a.hist_nxt != nullptr, (a.l + 1) % a.k, qbuf, kSelList);
    if (a.pick_next && !st.err) {
        // the children's histograms are final now (the part pass flushed its
        // counts before this kernel; this CTA added the candidates'), and so
        // are their domains: pick the next level's split buckets here
        __shared__ PartPlan ppn[2];
        __shared__ uint32_t redn[2][64];
        __syncthreads();
        LevelArgs an = a;
        an.l = a.l + 1;
        an.dom_cur = a.dom_nxt;
        an.dim_cur = a.dim_nxt;
        an.hist_cur = a.hist_nxt;
        an.hist_nxt = a.hist_nn;
        an.sel = a.sel_next;
        an.nbk = kBuckets;
        // the two children at once, one half of the CTA each (named barriers 1, 2)
        const uint32_t half = blockDim.x / 2u, hh = threadIdx.x >= half ? 1u : 0u;
        pick_subtree_g(WarpsGroup{hh * half, half, 1 + (int)hh}, an, 2 * s + 1 + hh, ppn[hh], redn[hh]);
        __syncthreads();
    }
}

// ---- one CTA per subtree -------------------------------------------------------

// One CTA per subtree: histogram (built by the level above when it could,
// else from the split words), pick, partition, exact resolve.  With a fused
// next level the children's histograms are built in shared memory during
// the partition and written out whole (this CTA owns both rows); the
// resolve then adds the candidates' contributions.
__global__ void __launch_bounds__(kPartThreads, 8) level_seg_kernel(LevelArgs a) {
    pdl_enter();
    __shared__ SelState st;
    __shared__ uint32_t hist[kBuckets];
    __shared__ uint32_t fh[2 * kBuckets];
    __shared__ uint32_t red[64];
    __shared__ uint32_t wtot[2 * 32], wbase[2 * 32];
    __shared__ uint32_t cursors[3];
    __shared__ uint32_t medw[kMaxWords];
    __shared__ uint32_t cur2[2];
    __shared__ PartPlan pps;
    __shared__ int stop;
    if (stop_requested(a.status, &stop)) return;
    const int64_t s = full_nodes(a.l) + blockIdx.x;
    const SegInfo g = seg_info(a, s);
    const Bucketer bk = seg_bucketer(a, g.j, g.d);
    const int64_t ld = a.ld;
    const bool fuse = a.hist_nxt != nullptr;
    const int dn = (a.l + 1) % a.k;
    if (a.hist_in) {
        const uint32_t *H = a.hist_cur + g.j * kBuckets;
        for (uint32_t b = threadIdx.x; b < (uint32_t)kBuckets; b += blockDim.x) hist[b] = H[b];
    } else {
        for (uint32_t b = threadIdx.x; b < (uint32_t)kBuckets; b += blockDim.x) hist[b] = 0u;
    }
    if (fuse)
        for (uint32_t b = threadIdx.x; b < 2u * kBuckets; b += blockDim.x) fh[b] = 0u;
    if (threadIdx.x < 3) cursors[threadIdx.x] = 0u;
    __syncthreads();
    if (!a.hist_in) {
        const uint32_t *col = reinterpret_cast<const uint32_t *>(a.src + (int64_t)(g.d >> 2) * ld) + (g.d & 3);
        hist_range(col, g.base, g.base + (int64_t)g.n, bk, hist);
        __syncthreads();
    }
    const bool ok = pick_bucket(hist, g.n, g.m, red, &pps);
    if (!ok) {
        if (threadIdx.x == 0) set_status(a.status, KDT_EINTERNAL);
        return;
    }
    if (threadIdx.x == 32) pps.khi = first_key_at_least(bk, pps.bstar + 1u);
    if (threadIdx.x == 0) pps.klo = first_key_at_least(bk, pps.bstar);
    __syncthreads();
    const PartPlan pp = part_plan(g, pps.bstar, pps.below, pps.cnt, pps.klo, pps.khi);
    Bucketer bkc;
    bkc.lo = 0.f;
    bkc.scale = 0.f;
    if (fuse) bkc = seg_bucketer(a, g.j, dn);  // the children's: the parent's domain in dn
    for (int64_t t0 = g.base & ~(int64_t)(kEPT - 1); t0 < g.base + (int64_t)g.n; t0 += kTile) {
        if (t0 + 2 * kTile < g.base + (int64_t)g.n) prefetch_tile(a, t0 + 2 * kTile, g.base + (int64_t)g.n);
        part_tile(a, g, bk, pp, t0, g.base, g.base + (int64_t)g.n, cursors, wtot, wbase, fuse ? fh : nullptr, bkc,
                  dn);
    }
    __syncthreads();
    if (cursors[0] != pp.below || cursors[1] != pp.cnt || cursors[2] != pp.above) {
        if (threadIdx.x == 0) set_status(a.status, KDT_EINTERNAL);
        return;
    }
    if (fuse) {
        uint32_t *H = a.hist_nxt + 2 * g.j * kBuckets;
        for (uint32_t b = threadIdx.x; b < 2u * kBuckets; b += blockDim.x) H[b] = fh[b];
        __syncthreads();  // before the resolve adds the candidates to the same rows
    }
    // fh is free again (written out above, or unused): the select lists its
    // last candidates there
    resolve_segment(a, g, pp, st, hist, red, medw, cur2, fuse, dn, fh, 2u * kBuckets);
}

// ---- host side ------------------------------------------------------------------

int enqueue_level(const Plan &p, const Buffers &b, int l, int src, int32_t *perm, cudaStream_t stream) {
    const Shape &S = p.S;
    const int k = p.k;
    LevelArgs a;
    a.S = S;
    a.k = k;
    a.mode = p.mode;
    a.l = l;
    a.src = b.rec[src];
    a.dst = b.rec[src ^ 1];
    a.cand = b.rec[2];
    a.G = rec_groups(k);
    a.perm = perm;
    a.dom_cur = b.dom[l & 1];
    a.dim_cur = b.dim[l & 1];
    a.dom_nxt = b.dom[(l + 1) & 1];
    a.dim_nxt = b.dim[(l + 1) & 1];
    a.hist_cur = b.hist[l & 1];
    a.hist_nxt = nullptr;
    a.nbk = kBuckets;
    a.hist_in = 0;
    a.warp_res = 0;  // multi-CTA levels: one global reservation per CTA and tile
    a.col0 = l == 0 ? b.col0 : nullptr;
    a.pts3 = l == 0 && l < p.multi_levels ? b.pts3 : nullptr;
    a.pick_next = 0;
    a.sel_next = b.sel[(l + 1) & 1];
    a.hist_nn = nullptr;
    a.sel = b.sel[l & 1];
    a.status = b.status;
    a.done = nullptr;
    a.per_cta = 0;
    a.ld = p.ld;
    const int64_t nseg = nodes_on_level(S, l);
    const int64_t live = S.N - full_nodes(l);
    const double alg = 20.0 * (double)live;
    const bool fusable = p.mode == KDT_SPLIT_ROUND_ROBIN && k >= 2;
    if (l < p.multi_levels) {
        int dev = 0, sms = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 152;
        const int64_t grid = (int64_t)sms * kPartCtas;  // partition CTAs stay resident
        a.per_cta = (live + grid - 1) / grid;
        const int64_t nblk = (live + a.per_cta - 1) / a.per_cta;
        const bool fused_here = l > 0 && fusable;
        if (l + 1 < p.finish_level && fusable) a.hist_nxt = b.hist[(l + 1) & 1];
        if (!fused_here) {
            // level 0 (one subtree) takes a finer histogram: fewer candidates
            // for the one CTA that resolves its split
            a.nbk = l == 0 && live >= kBuckets0Min ? kBuckets0 : kBuckets;
            if (cudaMemsetAsync(a.hist_cur, 0, (size_t)nseg * a.nbk * 4, stream) != cudaSuccess) return KDT_ECUDA;
            const size_t hsm = (size_t)a.nbk * 4;
            if (cudaFuncSetAttribute(level_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)hsm) !=
                cudaSuccess)
                return KDT_ECUDA;
            ProfScope ps(stream, "hist", 0.0);
            // every CTA flushes its whole histogram row with global atomics:
            // at least kHistPoints points per CTA, and no more CTAs than fit
            // the SMs at once
            LevelArgs ah = a;
            if (nseg == 1) ah.done = b.status + 1;  // zeroed with the status word at the start of the build
            const int64_t per_sm = std::min<int64_t>(2048 / kLvlThreads, (int64_t)(227 * 1024) / ((int64_t)hsm + 1024));
            int64_t gh = (live + kHistPoints - 1) / kHistPoints;
            gh = std::max<int64_t>(1, std::min<int64_t>(gh, (int64_t)sms * std::max<int64_t>(1, per_sm)));
            ah.per_cta = (live + gh - 1) / gh;
            gh = (live + ah.per_cta - 1) / ah.per_cta;
            launch_pdl(level_hist_kernel, (unsigned)gh, kLvlThreads, hsm, stream, ah);
            if (cudaGetLastError() != cudaSuccess) return KDT_ECUDA;
        }
        // picks: by the level above's resolve when it could (this level's
        // histograms were fused there), else by their own kernel; likewise
        // this level's resolve picks for the next level
        if (!fused_here && nseg > 1) {  // one subtree: picked by the histogram pass
            ProfScope ps(stream, "pick", 0.0);
            launch_pdl(level_pick_kernel, (unsigned)nseg, kPickThreads, 0, stream, a);
            if (cudaGetLastError() != cudaSuccess) return KDT_ECUDA;
        }
        if (a.hist_nxt != nullptr && l + 1 < p.multi_levels) {
            a.pick_next = 1;
            if (l + 2 < p.finish_level) a.hist_nn = b.hist[l & 1];  // level l+2's rows, cleared for the grandchildren
        }
        {
            ProfScope ps(stream, "part", alg);
            if (a.pts3 != nullptr) launch_pdl(level_part_kernel<true>, (unsigned)nblk, kPartThreads, 0, stream, a);
            else launch_pdl(level_part_kernel<false>, (unsigned)nblk, kPartThreads, 0, stream, a);
            if (cudaGetLastError() != cudaSuccess) return KDT_ECUDA;
        }
        {
            ProfScope ps(stream, "resolve", 0.0);
            // many candidates per subtree (the top levels): a wider CTA
            const double cand = (double)live / (double)nseg / (double)a.nbk;
            const int rt = cand > 4096.0 ? kResThreadsMax : kLvlThreads;
            launch_pdl(level_resolve_kernel, (unsigned)nseg, rt, 0, stream, a);
            if (cudaGetLastError() != cudaSuccess) return KDT_ECUDA;
        }
    } else {
        // the level above built this level's histograms if it could
        a.hist_in = fusable && l > 0 ? 1 : 0;
        a.warp_res = 1;  // cursors in shared memory
        if (l + 1 < p.finish_level && fusable) a.hist_nxt = b.hist[(l + 1) & 1];
        ProfScope ps(stream, "seg", alg);
        launch_pdl(level_seg_kernel, (unsigned)nseg, kPartThreads, 0, stream, a);
        if (cudaGetLastError() != cudaSuccess) return KDT_ECUDA;
    }
    return KDT_OK;
}

}  // namespace kdt
