// kdt_select.cuh -- exact rank selection under the split order, for a CTA, a
// group of warps, or one warp.
//
// The tree needs, for each subtree s, the point of 0-based rank ss(lChild(s))
// among s's points under the strict order of its split dimension d: the
// cyclic super key (x[d], x[d+1 mod k], ..., x[d-1 mod k]) and then the input
// index ("An Implementation of a Balanced Kd Tree Builder Using GPUs", sort
// paragraph, for the super key; "GPU-friendly, Parallel, and (Almost-)In-Place
// Construction of Left-Balanced k-d Trees", problem paragraph, for the rank
// that the balance condition fixes).
//
// A point's order key is the word sequence w_0..w_k with w_i the
// order-preserving key of x[(d+i) mod k] and w_k the input index.  The select
// narrows the set of "matching" points round by round until one remains:
//   * first round: value buckets evenly spread over [min, max] of x[d] among
//     the points (a monotone function of w_0); for spread-out data this alone
//     leaves one or a few points;
//   * then most-significant-digit rounds over the words: min and max of the
//     current word among the matching points; if equal the word is fixed,
//     otherwise a histogram of the digit below the highest differing bit
//     picks the bucket that holds the wanted rank.
// Because w_k is unique the loop ends with exactly one point.
#pragma once

#include "kdt_internal.cuh"

namespace kdt {

constexpr int kCtaRadixBits = 11;
constexpr int kCtaRadixBins = 1 << kCtaRadixBits;
constexpr int kWarpRadixBits = 8;
constexpr int kWarpRadixBins = 1 << kWarpRadixBits;

struct SelState {
    uint32_t f[kMaxWords];  // fixed words of the selected key
    int j;                  // current word
    int has_prefix;         // bits >= sh of word j are fixed to pv
    int sh;
    uint32_t pv;
    uint32_t r;             // wanted rank among the matching points
    uint32_t cnt;           // number of matching points
    int vb_on;              // value-bucket filter on w_0 active
    uint32_t vb;
    float vlo, vscale;
    uint32_t med_q;         // result: position of the selected point
    int err;
    int listed;             // the matching points' positions are listed in the group's buffer
    uint32_t nq;            // entries of that list
};

// ---- thread groups ------------------------------------------------------------

// All threads of the CTA.
struct CtaGroup {
    __device__ __forceinline__ uint32_t tid() const { return threadIdx.x; }
    __device__ __forceinline__ uint32_t size() const { return blockDim.x; }
    __device__ __forceinline__ void sync() const { __syncthreads(); }
};

// `n` consecutive threads (whole warps) starting at thread `base`,
// synchronised by named barrier `bar` (1..15); a single warp uses __syncwarp.
struct WarpsGroup {
    uint32_t base, n;
    int bar;
    __device__ __forceinline__ uint32_t tid() const { return threadIdx.x - base; }
    __device__ __forceinline__ uint32_t size() const { return n; }
    __device__ __forceinline__ void sync() const {
        if (n == 32u) __syncwarp();
        else asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(n) : "memory");
    }
};

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

// min and max over the group (result in every thread); `red` >= 64 words.
template <class G>
__device__ __forceinline__ void group_minmax(const G &g, uint32_t &mn, uint32_t &mx, uint32_t *red) {
    mn = __reduce_min_sync(0xffffffffu, mn);
    mx = __reduce_max_sync(0xffffffffu, mx);
    const uint32_t nw = g.size() >> 5;
    if (nw == 1u) return;
    const uint32_t w = g.tid() >> 5;
    g.sync();
    if (lane_id() == 0) {
        red[w] = mn;
        red[32 + w] = mx;
    }
    g.sync();
    uint32_t a = lane_id() < nw ? red[lane_id()] : 0xffffffffu;
    uint32_t b = lane_id() < nw ? red[32 + lane_id()] : 0u;
    mn = __reduce_min_sync(0xffffffffu, a);
    mx = __reduce_max_sync(0xffffffffu, b);
}

// Exclusive scan of one value per thread over the group; `total` gets the sum.
template <class G>
__device__ __forceinline__ uint32_t group_exclusive_scan(const G &g, uint32_t v, uint32_t *red, uint32_t &total) {
    const uint32_t lane = lane_id();
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= (uint32_t)o) x += y;
    }
    const uint32_t nw = g.size() >> 5;
    if (nw == 1u) {
        total = __shfl_sync(0xffffffffu, x, 31);
        return x - v;
    }
    const uint32_t w = g.tid() >> 5;
    g.sync();
    if (lane == 31) red[w] = x;
    g.sync();
    uint32_t t = lane < nw ? red[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, t, o);
        if (lane >= (uint32_t)o) t += y;
    }
    total = __shfl_sync(0xffffffffu, t, 31);
    const uint32_t before = w > 0 ? __shfl_sync(0xffffffffu, t, (w - 1) & 31) : 0u;
    return before + x - v;
}

// Block-wide exclusive scan (whole CTA).
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t *red) {
    uint32_t total;
    return group_exclusive_scan(CtaGroup{}, v, red, total);
}

// ---- matching ---------------------------------------------------------------------

__device__ __forceinline__ uint32_t value_bucket(uint32_t key, float lo, float scale, uint32_t nb) {
    const float t = __fmul_rn(__fsub_rn(key2f(key), lo), scale);
    int b = __float2int_rz(t);
    b = b < 0 ? 0 : b;
    return (uint32_t)b < nb ? (uint32_t)b : nb - 1u;
}

// Calls f(q, word j of q) for every matching point q of the group's share of
// [0, n), or of the list `qlist` once the matching points were listed there.
// Word 0 of eight points is loaded before any of them is tested, so a thread
// keeps eight loads in flight (the points may sit in global memory); the
// other words are read only for points that still match.
template <class G, class Acc, class F>
__device__ __forceinline__ void for_matching(const G &g, const Acc &acc, const SelState &st, uint32_t n, uint32_t nb,
                                             const uint32_t *qlist, F f) {
    constexpr int kB = 8;
    const uint32_t tid = g.tid(), nt = g.size();
    const int j = st.j;
    auto test = [&](uint32_t q, uint32_t w0) {
        if (st.vb_on && value_bucket(w0, st.vlo, st.vscale, nb) != st.vb) return;
        if (j > 0 && w0 != st.f[0]) return;
        for (int i = 1; i < j; ++i)
            if (acc(i, q) != st.f[i]) return;
        const uint32_t wj = j == 0 ? w0 : acc(j, q);
        if (st.has_prefix && (wj >> st.sh) != st.pv) return;
        f(q, wj);
    };
    if (st.listed) {
        for (uint32_t i = tid; i < st.nq; i += nt) {
            const uint32_t q = qlist[i];
            test(q, acc(0, q));
        }
        return;
    }
    if (n <= nt) {  // at most one point per thread: nothing to batch
        if (tid < n) test(tid, acc(0, tid));
        return;
    }
    for (uint32_t q0 = tid; q0 < n; q0 += kB * nt) {
        uint32_t w0[kB];
#pragma unroll
        for (int u = 0; u < kB; ++u) {
            const uint32_t q = q0 + (uint32_t)u * nt;
            w0[u] = q < n ? acc(0, q) : 0u;
        }
#pragma unroll
        for (int u = 0; u < kB; ++u) {
            const uint32_t q = q0 + (uint32_t)u * nt;
            if (q < n) test(q, w0[u]);
        }
    }
}

// Three-way comparison of point q with the key words w[0..nw).
template <class Acc>
__device__ __forceinline__ int cmp_words(const Acc &acc, uint32_t q, const uint32_t *w, int nw) {
    for (int i = 0; i < nw; ++i) {
        const uint32_t a = acc(i, q);
        if (a != w[i]) return a < w[i] ? -1 : 1;
    }
    return 0;
}

// Group-wide exact select of rank m among n points (positions 0..n-1 through
// `acc`).  `hist` holds 2^bits words (2^bits a multiple of the group size),
// `red` >= 64 words, `st` is the group's state; all in shared memory.  With a
// list buffer (`qbuf`, `qcap` words of shared memory, or null), once at most
// qcap points still match they are listed there, and the later rounds visit
// only those instead of all n.  On return (after a group barrier) st.med_q
// holds the selected position and st.err is nonzero on an internal
// inconsistency.
template <class G, class Acc>
__device__ void group_select(const G &g, const Acc &acc, uint32_t n, uint32_t m, int nwords, SelState &st,
                             uint32_t *hist, int bits, uint32_t *red, uint32_t *qbuf = nullptr, uint32_t qcap = 0u) {
    const uint32_t tid = g.tid(), nt = g.size();
    const uint32_t nbins = 1u << bits;
    if (tid == 0) {
        st.j = 0;
        st.has_prefix = 0;
        st.sh = 0;
        st.pv = 0;
        st.r = m;
        st.cnt = n;
        st.vb_on = 0;
        st.vb = 0;
        st.vlo = 0.f;
        st.vscale = 0.f;
        st.err = 0;
        st.med_q = 0;
        st.listed = 0;
        st.nq = 0;
    }
    g.sync();
    bool value_round = true;
    for (int guard = 0; guard < 8 * kMaxWords + 2; ++guard) {
        if (st.cnt <= 1u || st.j >= nwords) break;
        const int j = st.j;
        uint32_t mn = 0xffffffffu, mx = 0u;
        for_matching(g, acc, st, n, nbins, qbuf, [&](uint32_t, uint32_t w) {
            mn = min(mn, w);
            mx = max(mx, w);
        });
        group_minmax(g, mn, mx, red);
        if (mn == mx) {
            g.sync();
            if (tid == 0) {
                st.f[j] = mn;
                st.j = j + 1;
                st.has_prefix = 0;
            }
            g.sync();
            value_round = false;
            continue;
        }
        // this round's bucket function
        bool vround = false;
        float vlo = 0.f, vscale = 0.f;
        int sh = 0;
        uint32_t lo = 0;
        if (value_round && j == 0) {
            vlo = key2f(mn);
            const float r = __fsub_rn(key2f(mx), vlo);
            if (r > 0.f && r <= 3.0e38f) {
                vscale = __fdiv_rn((float)nbins, r);
                if (vscale <= 3.0e38f) vround = true;
            }
        }
        value_round = false;
        if (!vround) {
            const int hb = 31 - __clz(mn ^ mx);
            sh = hb - (bits - 1) > 0 ? hb - (bits - 1) : 0;
            lo = mn >> sh;
        }
        for (uint32_t b = tid; b < nbins; b += nt) hist[b] = 0u;
        g.sync();
        for_matching(g, acc, st, n, nbins, qbuf, [&](uint32_t, uint32_t w) {
            const uint32_t b = vround ? value_bucket(w, vlo, vscale, nbins) : (w >> sh) - lo;
            atomicAdd(&hist[b], 1u);
        });
        g.sync();
        const uint32_t per = nbins / nt;
        uint32_t sum = 0;
        for (uint32_t i = 0; i < per; ++i) sum += hist[tid * per + i];
        uint32_t total;
        const uint32_t excl = group_exclusive_scan(g, sum, red, total);
        const uint32_t r = st.r;
        g.sync();
        if (r >= excl && r < excl + sum) {
            uint32_t c = excl;
            for (uint32_t i = 0; i < per; ++i) {
                const uint32_t h = hist[tid * per + i];
                if (r < c + h) {
                    const uint32_t b = tid * per + i;
                    st.r = r - c;
                    st.cnt = h;
                    if (vround) {
                        st.vb_on = 1;
                        st.vb = b;
                        st.vlo = vlo;
                        st.vscale = vscale;
                    } else {
                        st.pv = lo + b;
                        st.sh = sh;
                        st.has_prefix = 1;
                        if (sh == 0) {
                            st.f[j] = st.pv;
                            st.j = j + 1;
                            st.has_prefix = 0;
                        }
                    }
                    break;
                }
                c += h;
            }
        }
        g.sync();
        // few points left of many: list them once
        if (qbuf != nullptr && !st.listed && st.cnt > 1u && st.cnt <= qcap && n > 2u * nt) {
            for_matching(g, acc, st, n, nbins, qbuf, [&](uint32_t q, uint32_t) {
                const uint32_t i = atomicAdd(&st.nq, 1u);
                if (i < qcap) qbuf[i] = q;
            });
            g.sync();
            if (tid == 0) {
                if (st.nq != st.cnt) {
                    st.err = 1;
                    st.cnt = 0u;  // ends the loop
                }
                st.listed = 1;
            }
            g.sync();
        }
    }
    if (st.cnt != 1u && tid == 0) st.err = 1;
    g.sync();
    for_matching(g, acc, st, n, nbins, qbuf, [&](uint32_t q, uint32_t) { st.med_q = q; });
    g.sync();
}

// CTA-wide select with 2^11 buckets (global levels).
template <class Acc>
__device__ __forceinline__ void cta_select(const Acc &acc, uint32_t n, uint32_t m, int nwords, SelState &st,
                                           uint32_t *hist, uint32_t *red, uint32_t *qbuf = nullptr,
                                           uint32_t qcap = 0u) {
    group_select(CtaGroup{}, acc, n, m, nwords, st, hist, kCtaRadixBits, red, qbuf, qcap);
}

}  // namespace kdt
