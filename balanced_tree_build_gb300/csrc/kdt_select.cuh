// kdt_select.cuh -- exact rank selection under the split order, for a CTA or
// a warp.
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
// order-preserving key of x[(d+i) mod k] and w_k the input index.  The
// selection is a most-significant-digit radix select over that sequence: each
// round narrows the set of "matching" points (those that share the chosen
// prefix) until one remains.  A round first takes min and max of the current
// word over the matching points; if they agree the word is fixed, otherwise
// the highest differing bit positions the next digit and a histogram of that
// digit picks the bucket holding the wanted rank.  Because w_k is unique the
// loop ends with exactly one point.
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
    uint32_t mn, mx;
    uint32_t med_q;         // result: position of the selected point
    int err;
};

template <class Acc>
__device__ __forceinline__ bool sel_matches(const Acc &acc, const SelState &st, uint32_t q) {
    for (int i = 0; i < st.j; ++i)
        if (acc(i, q) != st.f[i]) return false;
    if (st.has_prefix && (acc(st.j, q) >> st.sh) != st.pv) return false;
    return true;
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

// ---- block-wide helpers (blockDim.x a multiple of 32, at most 1024) -------

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

__device__ __forceinline__ void block_minmax(uint32_t &mn, uint32_t &mx, uint32_t *red) {
    mn = __reduce_min_sync(0xffffffffu, mn);
    mx = __reduce_max_sync(0xffffffffu, mx);
    const int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    __syncthreads();
    if (lane_id() == 0) {
        red[w] = mn;
        red[32 + w] = mx;
    }
    __syncthreads();
    if (w == 0) {
        uint32_t a = lane_id() < (uint32_t)nw ? red[lane_id()] : 0xffffffffu;
        uint32_t b = lane_id() < (uint32_t)nw ? red[32 + lane_id()] : 0u;
        a = __reduce_min_sync(0xffffffffu, a);
        b = __reduce_max_sync(0xffffffffu, b);
        if (lane_id() == 0) {
            red[0] = a;
            red[32] = b;
        }
    }
    __syncthreads();
    mn = red[0];
    mx = red[32];
}

// Exclusive scan of one value per thread; returns the exclusive prefix.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t *red) {
    const uint32_t lane = lane_id();
    const int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= (uint32_t)o) x += y;
    }
    __syncthreads();
    if (lane == 31) red[w] = x;
    __syncthreads();
    if (w == 0) {
        uint32_t t = lane < (uint32_t)nw ? red[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= (uint32_t)o) t += y;
        }
        red[lane] = t;  // inclusive warp totals
    }
    __syncthreads();
    const uint32_t before = w > 0 ? red[w - 1] : 0u;
    return before + x - v;
}

// CTA-wide exact select of rank m among n points (positions 0..n-1 through
// `acc`).  On return (after a barrier) st.med_q holds the selected position.
// `hist` holds kCtaRadixBins words; `red` at least 64 words.
template <class Acc>
__device__ void cta_select(const Acc &acc, uint32_t n, uint32_t m, int nwords, SelState &st,
                           uint32_t *hist, uint32_t *red) {
    const uint32_t tid = threadIdx.x, nt = blockDim.x;
    if (tid == 0) {
        st.j = 0;
        st.has_prefix = 0;
        st.sh = 0;
        st.pv = 0;
        st.r = m;
        st.cnt = n;
        st.err = 0;
        st.med_q = 0;
    }
    __syncthreads();
    for (int guard = 0; guard < 8 * kMaxWords; ++guard) {
        if (st.cnt <= 1u || st.j >= nwords) break;
        const int j = st.j;
        uint32_t mn = 0xffffffffu, mx = 0u;
        for (uint32_t q = tid; q < n; q += nt) {
            if (sel_matches(acc, st, q)) {
                const uint32_t w = acc(j, q);
                mn = min(mn, w);
                mx = max(mx, w);
            }
        }
        block_minmax(mn, mx, red);
        if (mn == mx) {
            if (tid == 0) {
                st.f[j] = mn;
                st.j = j + 1;
                st.has_prefix = 0;
            }
            __syncthreads();
            continue;
        }
        const int hb = 31 - __clz(mn ^ mx);
        const int sh = hb - (kCtaRadixBits - 1) > 0 ? hb - (kCtaRadixBits - 1) : 0;
        const uint32_t lo = mn >> sh;
        for (uint32_t b = tid; b < (uint32_t)kCtaRadixBins; b += nt) hist[b] = 0u;
        __syncthreads();
        for (uint32_t q = tid; q < n; q += nt) {
            if (sel_matches(acc, st, q)) atomicAdd(&hist[(acc(j, q) >> sh) - lo], 1u);
        }
        __syncthreads();
        // find the bucket that holds rank r
        const uint32_t per = kCtaRadixBins / nt;  // bins per thread (nt divides 2048)
        uint32_t sum = 0;
        for (uint32_t i = 0; i < per; ++i) sum += hist[tid * per + i];
        const uint32_t excl = block_exclusive_scan(sum, red);
        const uint32_t r = st.r;
        __syncthreads();
        if (r >= excl && r < excl + sum) {
            uint32_t c = excl;
            for (uint32_t i = 0; i < per; ++i) {
                const uint32_t h = hist[tid * per + i];
                if (r < c + h) {
                    st.r = r - c;
                    st.cnt = h;
                    st.pv = lo + tid * per + i;
                    st.sh = sh;
                    st.has_prefix = 1;
                    if (sh == 0) {
                        st.f[j] = st.pv;
                        st.j = j + 1;
                        st.has_prefix = 0;
                    }
                    break;
                }
                c += h;
            }
        }
        __syncthreads();
    }
    if (st.cnt != 1u && tid == 0) st.err = 1;
    __syncthreads();
    for (uint32_t q = tid; q < n; q += nt)
        if (sel_matches(acc, st, q)) st.med_q = q;
    __syncthreads();
}

// Warp-wide exact select of rank m among n points.  All 32 lanes call it;
// `wf` is per-warp scratch of kMaxWords words, `hist` kWarpRadixBins words.
// Returns the selected position (same value in every lane), or 0xffffffff
// on an internal inconsistency.
template <class Acc>
__device__ uint32_t warp_select(const Acc &acc, uint32_t n, uint32_t m, int nwords, uint32_t *wf,
                                uint32_t *hist) {
    const uint32_t lane = lane_id();
    int j = 0, has_prefix = 0, sh = 0;
    uint32_t pv = 0, r = m, cnt = n;
    auto matches = [&](uint32_t q) -> bool {
        for (int i = 0; i < j; ++i)
            if (acc(i, q) != wf[i]) return false;
        if (has_prefix && (acc(j, q) >> sh) != pv) return false;
        return true;
    };
    for (int guard = 0; guard < 8 * kMaxWords && cnt > 1u && j < nwords; ++guard) {
        uint32_t mn = 0xffffffffu, mx = 0u;
        for (uint32_t q = lane; q < n; q += 32) {
            if (matches(q)) {
                const uint32_t w = acc(j, q);
                mn = min(mn, w);
                mx = max(mx, w);
            }
        }
        mn = __reduce_min_sync(0xffffffffu, mn);
        mx = __reduce_max_sync(0xffffffffu, mx);
        if (mn == mx) {
            __syncwarp();
            if (lane == 0) wf[j] = mn;
            __syncwarp();
            ++j;
            has_prefix = 0;
            continue;
        }
        const int hb = 31 - __clz(mn ^ mx);
        const int nsh = hb - (kWarpRadixBits - 1) > 0 ? hb - (kWarpRadixBits - 1) : 0;
        const uint32_t lo = mn >> nsh;
#pragma unroll
        for (int b = 0; b < kWarpRadixBins / 32; ++b) hist[lane + 32 * b] = 0u;
        __syncwarp();
        for (uint32_t q = lane; q < n; q += 32)
            if (matches(q)) atomicAdd(&hist[(acc(j, q) >> nsh) - lo], 1u);
        __syncwarp();
        constexpr int per = kWarpRadixBins / 32;
        uint32_t h[per];
        uint32_t sum = 0;
#pragma unroll
        for (int i = 0; i < per; ++i) {
            h[i] = hist[lane * per + i];
            sum += h[i];
        }
        uint32_t incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= (uint32_t)o) incl += y;
        }
        const uint32_t excl = incl - sum;
        const bool mine = r >= excl && r < incl;
        uint32_t nr = 0, ncnt = 0, npv = 0;
        if (mine) {
            uint32_t c = excl;
#pragma unroll
            for (int i = 0; i < per; ++i) {
                if (r >= c && r < c + h[i]) {
                    nr = r - c;
                    ncnt = h[i];
                    npv = lo + lane * per + i;
                }
                c += h[i];
            }
        }
        const uint32_t who = __ballot_sync(0xffffffffu, mine);
        if (who == 0u) return 0xffffffffu;
        const int src = __ffs(who) - 1;
        r = __shfl_sync(0xffffffffu, nr, src);
        cnt = __shfl_sync(0xffffffffu, ncnt, src);
        pv = __shfl_sync(0xffffffffu, npv, src);
        sh = nsh;
        has_prefix = 1;
        if (sh == 0) {
            __syncwarp();
            if (lane == 0) wf[j] = pv;
            __syncwarp();
            ++j;
            has_prefix = 0;
        }
        __syncwarp();
    }
    if (cnt != 1u) return 0xffffffffu;
    uint32_t found = 0xffffffffu;
    for (uint32_t q = lane; q < n; q += 32)
        if (matches(q)) found = q;
    found = __reduce_min_sync(0xffffffffu, found);
    return found;
}

}  // namespace kdt
