/*
 * kdt_oracle.c -- CPU oracle for the left-balanced, complete, level-order k-d tree.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously-correct
 * reference that the CUDA build is checked against.  Only the test suite, the
 * package's smoke() check and bench.py's CPU-baseline / reference leg may load
 * it.  It shares no code, header, table or helper with the CUDA library, and
 * the CUDA library never calls it.
 *
 * Sources (cited by page title and passage):
 *   [W]  "GPU-friendly, Parallel, and (Almost-)In-Place Construction of
 *        Left-Balanced k-d Trees" (Wald, arXiv 2211.00120):
 *          - problem paragraph: k-d condition (left subtree <=, right >= in the
 *            node's split dimension) plus the left-balanced shape;
 *          - notation paragraph: level-order ids, parent/lChild/rChild,
 *            level(i), numLevels(N);
 *          - round-robin paragraph: split dimension l mod k for level l;
 *          - split-widest-dimension paragraphs: domain = bounding box of the
 *            whole data set clipped by the ancestors' split planes, split
 *            dimension = widest extent of that domain.
 *   [R]  "An Implementation of a Balanced Kd Tree Builder Using GPUs"
 *        (Robinson, KdTreeGPU wiki), sort paragraph: on equal primary
 *        coordinates compare the next coordinate, then the next, ... (the
 *        "super key").
 *   [B]  "Bigger Buffer k-d Trees on Multi-Many-Core Systems", nearest
 *        neighbour problem statement (K nearest reference points of a query
 *        in Euclidean distance) -- for the query routines at the end.
 *   [R] again, overview list and build section, for the balanced
 *        (median-split, not left-balanced) tree of Brown's presort-and-
 *        partition builder: the kdo_*_balanced routines.
 *
 * Readings taken where the pages are silent:
 *   - the super key is cyclic from the split dimension p: (x[p], x[p+1 mod k],
 *     ..., x[p-1 mod k]) and, when all coordinates are equal, the original
 *     input index breaks the tie; this makes the order strict and total, so
 *     the tree is unique;
 *   - float comparison uses IEEE '<' (so -0 == +0);
 *   - the split point of subtree s is the element of 0-based rank
 *     |S(lChild(s))| of s's point set under that order;
 *   - widest mode: extent = hi - lo in float32 round-to-nearest; the lowest
 *     dimension wins ties (strict '>' to replace); the domain of a child is the
 *     parent's domain with hi[d] (left) or lo[d] (right) set to the split
 *     point's coordinate;
 *   - non-finite coordinates are rejected.
 *
 * Not reentrant: the qsort comparator reads a file-scope context.  The oracle
 * is single-threaded by design.
 *
 * Mutants: compiling with -DKDO_MUTANT=<n> plants one deliberate mistake (see
 * the KDO_MUTANT blocks).  The test suite builds each mutant and checks that
 * at least one pin fails; the product build never defines it.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#ifndef KDO_MUTANT
#define KDO_MUTANT 0
#endif

#define KDO_OK 0
#define KDO_EINVAL (-1)
#define KDO_ENOMEM (-2)
#define KDO_ENONFINITE (-4)
#define KDO_EINTERNAL (-6)
#define KDO_MAXK 32

/* ---- tree notation ([W] notation paragraph) ------------------------------ */

/* level(i) = floor(log2(i+1)), written as a loop. */
int kdo_level(int64_t i)
{
    int l = 0;
    uint64_t v = (uint64_t)i + 1u;
    while (v > 1u) {
        v >>= 1;
        l++;
    }
    return l;
}

/* numLevels(N) = level(N-1) + 1. */
int kdo_num_levels(int64_t N)
{
    return kdo_level(N - 1) + 1;
}

/* |S(t)|: number of nodes of the subtree rooted at t in the level-order tree
 * of N nodes.  Counted level by level: the depth-j descendants of t are the
 * 2^j consecutive ids starting at 2^j (t+1) - 1; count the ones below N.
 * (Deliberately not the closed form that the CUDA library uses.) */
int64_t kdo_subtree_count(int64_t N, int64_t t)
{
    int64_t total = 0;
    if (t < 0 || t >= N)
        return 0;
    for (int j = 0; j < 63; j++) {
        int64_t first = ((t + 1) << j) - 1;
        int64_t width = (int64_t)1 << j;
        if (first >= N)
            break;
        int64_t have = N - first;
        total += have < width ? have : width;
        if ((t + 1) > (INT64_MAX >> (j + 1)))
            break;
    }
    return total;
}

/* ---- the strict total order <_p ([R] super key + index reading) ---------- */

/* Returns 1 if point a precedes point b under <_p, else 0. */
int kdo_less(const float *pts, int k, int p, int64_t a, int64_t b)
{
    for (int j = 0; j < k; j++) {
#if KDO_MUTANT == 2
        int c = j; /* mutant: non-cyclic super key */
#else
        int c = (p + j) % k;
#endif
        float xa = pts[a * k + c];
        float xb = pts[b * k + c];
        if (xa < xb)
            return 1;
        if (xb < xa)
            return 0;
    }
#if KDO_MUTANT == 3
    return a > b; /* mutant: index tiebreak reversed */
#else
    return a < b;
#endif
}

/* Widest extent of a domain ([W] split-widest-dimension paragraphs): argmax of
 * hi[d] - lo[d] in float32, lowest d on ties. */
int kdo_widest_dim(const float *lo, const float *hi, int k)
{
    int best = 0;
    float ext = hi[0] - lo[0];
    for (int d = 1; d < k; d++) {
        float e = hi[d] - lo[d];
#if KDO_MUTANT == 4
        if (e >= ext) { /* mutant: highest dimension wins ties */
#else
        if (e > ext) {
#endif
            ext = e;
            best = d;
        }
    }
    return best;
}

/* ---- recursive median-split builder --------------------------------------- */

static const float *g_pts;
static int g_k;
static int g_p;

static int cmp_idx(const void *va, const void *vb)
{
    int32_t a = *(const int32_t *)va;
    int32_t b = *(const int32_t *)vb;
    if (kdo_less(g_pts, g_k, g_p, a, b))
        return -1;
    if (kdo_less(g_pts, g_k, g_p, b, a))
        return 1;
    return 0;
}

typedef struct {
    const float *pts;
    int64_t N;
    int k;
    int mode;
    int32_t *perm;
    int bad; /* set if a subtree received the wrong number of points */
} build_ctx;

/* rec(s, P, dom): P holds exactly the points of subtree s.  Sort P under the
 * split order of s, place the element of rank |S(lChild(s))| at node s, and
 * recurse on the two sides with the clipped domains. */
static void rec(build_ctx *c, int64_t s, int32_t *P, int64_t n,
                const float *lo, const float *hi)
{
    if (n == 0)
        return;
    if (s >= c->N || n != kdo_subtree_count(c->N, s)) {
        c->bad = 1; /* cannot happen for the real oracle; keeps mutants in bounds */
        return;
    }
    int d;
    if (c->mode == 0) {
#if KDO_MUTANT == 7
        d = (kdo_level(s) + 1) % c->k; /* mutant: wrong round-robin phase */
#else
        d = kdo_level(s) % c->k;
#endif
    } else {
        d = kdo_widest_dim(lo, hi, c->k);
    }
#if KDO_MUTANT == 1
    int64_t m = kdo_subtree_count(c->N, 2 * s + 1);
    if (m + 1 < n)
        m += 1; /* mutant: split rank off by one */
#else
    int64_t m = kdo_subtree_count(c->N, 2 * s + 1);
#endif
    g_pts = c->pts;
    g_k = c->k;
    g_p = d;
    qsort(P, (size_t)n, sizeof(int32_t), cmp_idx);
    c->perm[s] = P[m];
    float split = c->pts[(int64_t)P[m] * c->k + d];

    float clo[KDO_MAXK], chi[KDO_MAXK];
    memcpy(clo, lo, sizeof(float) * c->k);
    memcpy(chi, hi, sizeof(float) * c->k);
#if KDO_MUTANT == 6
    clo[d] = split; /* mutant: left child clipped on the wrong side */
#else
    chi[d] = split;
#endif
#if KDO_MUTANT == 5
    rec(c, 2 * s + 1, P + m + 1, n - m - 1, clo, chi); /* mutant: sides swapped */
#else
    rec(c, 2 * s + 1, P, m, clo, chi);
#endif

    memcpy(clo, lo, sizeof(float) * c->k);
    memcpy(chi, hi, sizeof(float) * c->k);
    clo[d] = split;
#if KDO_MUTANT == 5
    rec(c, 2 * s + 2, P, m, clo, chi);
#else
    rec(c, 2 * s + 2, P + m + 1, n - m - 1, clo, chi);
#endif
}

static int check_args(const float *pts, int64_t N, int k, int mode)
{
    if (!pts || N < 1 || N > INT32_MAX || k < 1 || k > KDO_MAXK ||
        (mode != 0 && mode != 1))
        return KDO_EINVAL;
    for (int64_t i = 0; i < N * (int64_t)k; i++)
        if (!isfinite(pts[i]))
            return KDO_ENONFINITE;
    return KDO_OK;
}

/* Bounding box of all points: the root domain ([W] widest-dimension init). */
static void bbox(const float *pts, int64_t N, int k, float *lo, float *hi)
{
    for (int d = 0; d < k; d++) {
        lo[d] = pts[d];
        hi[d] = pts[d];
    }
    for (int64_t i = 1; i < N; i++)
        for (int d = 0; d < k; d++) {
            float x = pts[i * k + d];
            if (x < lo[d])
                lo[d] = x;
            if (hi[d] < x)
                hi[d] = x;
        }
}

/* perm[node] = input index of the point stored at level-order node `node`. */
int kdo_build(const float *pts, int64_t N, int k, int mode, int32_t *perm)
{
    int rc = check_args(pts, N, k, mode);
    if (rc != KDO_OK)
        return rc;
    if (!perm)
        return KDO_EINVAL;
    int32_t *P = (int32_t *)malloc(sizeof(int32_t) * (size_t)N);
    if (!P)
        return KDO_ENOMEM;
    for (int64_t i = 0; i < N; i++)
        P[i] = (int32_t)i;
    float lo[KDO_MAXK], hi[KDO_MAXK];
    bbox(pts, N, k, lo, hi);
    build_ctx c = {pts, N, k, mode, perm, 0};
    for (int64_t i = 0; i < N; i++)
        perm[i] = -1;
    rec(&c, 0, P, N, lo, hi);
    free(P);
    return c.bad ? KDO_EINTERNAL : KDO_OK;
}

/* ---- verifier: the definition checked node against every ancestor -------- */

/* Checks node i against each of its ancestors a: if i lies in the left
 * subtree of a then perm[i] <_{d(a)} perm[a], else perm[a] <_{d(a)} perm[i].
 * d(a) is recomputed while walking down from the root (round-robin: level mod
 * k; widest: the domain is clipped by each visited ancestor's split point).
 * Returns 1 if the node satisfies all its conditions. */
static int node_ok(const float *pts, int64_t N, int k, int mode,
                   const int32_t *perm, int64_t i, const float *rlo,
                   const float *rhi)
{
    float lo[KDO_MAXK], hi[KDO_MAXK];
    memcpy(lo, rlo, sizeof(float) * k);
    memcpy(hi, rhi, sizeof(float) * k);
    int depth = kdo_level(i);
    int64_t a = 0;
    for (int j = 0; j < depth; j++) {
        int right = (int)(((uint64_t)(i + 1) >> (depth - 1 - j)) & 1u);
        int d = mode == 0 ? kdo_level(a) % k : kdo_widest_dim(lo, hi, k);
        int64_t pa = perm[a], pi = perm[i];
        if (pa < 0 || pa >= N || pi < 0 || pi >= N)
            return 0;
        if (right) {
            if (!kdo_less(pts, k, d, pa, pi))
                return 0;
            lo[d] = pts[pa * k + d];
        } else {
            if (!kdo_less(pts, k, d, pi, pa))
                return 0;
            hi[d] = pts[pa * k + d];
        }
        a = 2 * a + 1 + right;
    }
    return 1;
}

/* Verifies the given nodes (all nodes if nodes == NULL) and, when check_perm is
 * set, that perm is a permutation of 0..N-1.  Returns 0 if valid, 1 if not
 * (first failing node in *bad_node, or -1 for a permutation failure), <0 on
 * error. */
int kdo_verify(const float *pts, int64_t N, int k, int mode,
               const int32_t *perm, const int64_t *nodes, int64_t count,
               int check_perm, int64_t *bad_node)
{
    int rc = check_args(pts, N, k, mode);
    if (rc != KDO_OK)
        return rc;
    if (!perm)
        return KDO_EINVAL;
    if (bad_node)
        *bad_node = -2;
    if (check_perm) {
        unsigned char *seen = (unsigned char *)calloc((size_t)N, 1);
        if (!seen)
            return KDO_ENOMEM;
        for (int64_t i = 0; i < N; i++) {
            int64_t p = perm[i];
            if (p < 0 || p >= N || seen[p]) {
                free(seen);
                if (bad_node)
                    *bad_node = -1;
                return 1;
            }
            seen[p] = 1;
        }
        free(seen);
    }
    float lo[KDO_MAXK], hi[KDO_MAXK];
    bbox(pts, N, k, lo, hi);
    int64_t n = nodes ? count : N;
    for (int64_t t = 0; t < n; t++) {
        int64_t i = nodes ? nodes[t] : t;
        if (i < 0 || i >= N)
            return KDO_EINVAL;
        if (!node_ok(pts, N, k, mode, perm, i, lo, hi)) {
            if (bad_node)
                *bad_node = i;
            return 1;
        }
    }
    return 0;
}

/* ---- exhaustive search over all orderings (tiny N) ------------------------ */

/* Counts the orderings of 0..N-1 that satisfy the tree conditions (every node
 * against every ancestor); copies the first valid one to first_valid.
 * Heap's algorithm enumerates all N! orderings.  N <= 11. */
int64_t kdo_brute_force(const float *pts, int N, int k, int mode,
                        int32_t *first_valid)
{
    if (check_args(pts, N, k, mode) != KDO_OK || N > 11)
        return -1;
    int32_t a[11];
    int c[11];
    for (int i = 0; i < N; i++) {
        a[i] = i;
        c[i] = 0;
    }
    float lo[KDO_MAXK], hi[KDO_MAXK];
    bbox(pts, N, k, lo, hi);
    int64_t valid = 0;
    for (;;) {
        int ok = 1;
        for (int64_t i = 0; i < N && ok; i++)
            ok = node_ok(pts, N, k, mode, a, i, lo, hi);
        if (ok) {
            if (valid == 0 && first_valid)
                memcpy(first_valid, a, sizeof(int32_t) * N);
            valid++;
        }
        /* next permutation (Heap's algorithm, iterative form) */
        int i = 1;
        while (i < N && c[i] >= i) {
            c[i] = 0;
            i++;
        }
        if (i >= N)
            break;
        int j = (i % 2 == 0) ? 0 : c[i];
        int32_t tmp = a[j];
        a[j] = a[i];
        a[i] = tmp;
        c[i]++;
    }
    return valid;
}

/* ---- the balanced tree of [R] (Brown's presort-and-partition builder) ------
 *
 * [R] overview list: sort one reference array per coordinate; take the median
 * of the first coordinate's array as the first node and partition the other
 * arrays into the points below and above it (the median goes to neither
 * side); repeat on both sides with the next coordinate, cycling through the
 * coordinates, until every point is a node.  [R] build section: the medians
 * of level L form a per-level store in which the children of entry j are
 * entries 2j and 2j+1 of level L+1 -- heap order.
 *
 * Readings where the page is silent: the median of n points is the element of
 * 0-based rank floor((n-1)/2) (the lower median); the order is the strict
 * super key + index order above, so duplicates are kept and the tree is
 * unique; the tree is stored in heap order, entry j of level L in slot
 * 2^L - 1 + j of an array of 2^numLevels(N) - 1 slots, -1 where a subtree is
 * empty.  The height is numLevels(N): the larger side of n points has
 * floor(n/2).
 *
 * The builder is the definition written out: sort the subtree's points under
 * its split order (level mod k), place the lower median, recurse. */

/* Slots of the heap-ordered balanced tree of N points: 2^numLevels(N) - 1. */
int64_t kdo_balanced_slots(int64_t N)
{
    if (N < 1 || N > INT32_MAX)
        return -1;
    return ((int64_t)1 << kdo_num_levels(N)) - 1;
}

static void rec_balanced(const float *pts, int k, int64_t slot, int level,
                         int32_t *P, int64_t n, int32_t *slots, int64_t nslots,
                         int *bad)
{
    if (n == 0)
        return;
    if (slot >= nslots) {
        *bad = 1;
        return;
    }
    g_pts = pts;
    g_k = k;
#if KDO_MUTANT == 7
    g_p = (level + 1) % k; /* mutant: wrong round-robin phase */
#else
    g_p = level % k;
#endif
    qsort(P, (size_t)n, sizeof(int32_t), cmp_idx);
#if KDO_MUTANT == 8
    int64_t m = n / 2; /* mutant: upper median */
#else
    int64_t m = (n - 1) / 2;
#endif
    slots[slot] = P[m];
#if KDO_MUTANT == 9
    rec_balanced(pts, k, 2 * slot + 2, level + 1, P, m, slots, nslots, bad); /* mutant: sides swapped */
    rec_balanced(pts, k, 2 * slot + 1, level + 1, P + m + 1, n - 1 - m, slots, nslots, bad);
#else
    rec_balanced(pts, k, 2 * slot + 1, level + 1, P, m, slots, nslots, bad);
    rec_balanced(pts, k, 2 * slot + 2, level + 1, P + m + 1, n - 1 - m, slots, nslots, bad);
#endif
}

/* slots[s] = input index of the point at heap slot s, -1 for an empty slot;
 * nslots must be kdo_balanced_slots(N). */
int kdo_build_balanced(const float *pts, int64_t N, int k, int32_t *slots, int64_t nslots)
{
    int rc = check_args(pts, N, k, 0);
    if (rc != KDO_OK)
        return rc;
    if (!slots || nslots != kdo_balanced_slots(N))
        return KDO_EINVAL;
    int32_t *P = (int32_t *)malloc(sizeof(int32_t) * (size_t)N);
    if (!P)
        return KDO_ENOMEM;
    for (int64_t i = 0; i < N; i++)
        P[i] = (int32_t)i;
    for (int64_t s = 0; s < nslots; s++)
        slots[s] = -1;
    int bad = 0;
    rec_balanced(pts, k, 0, 0, P, N, slots, nslots, &bad);
    free(P);
    return bad ? KDO_EINTERNAL : KDO_OK;
}

/* Shape of the balanced tree: occ[s] = 1 if slot s holds a point.  Sizes
 * follow the split rule (left floor((n-1)/2), right n-1-left), computed by an
 * explicit stack (no sorting involved). */
static int balanced_shape(int64_t N, uint8_t *occ, int64_t nslots)
{
    typedef struct { int64_t slot, n; } item;
    item *st = (item *)malloc(sizeof(item) * 128);
    if (!st)
        return KDO_ENOMEM;
    int sp = 0;
    memset(occ, 0, (size_t)nslots);
    st[sp++] = (item){0, N};
    while (sp > 0) {
        item it = st[--sp];
        if (it.n == 0)
            continue;
        if (it.slot >= nslots || sp + 2 > 128) {
            free(st);
            return KDO_EINTERNAL;
        }
        occ[it.slot] = 1;
        int64_t m = (it.n - 1) / 2;
        st[sp++] = (item){2 * it.slot + 1, m};
        st[sp++] = (item){2 * it.slot + 2, it.n - 1 - m};
    }
    free(st);
    return KDO_OK;
}

/* Node s (occupied) against each of its ancestors a, split dimension
 * level(a) mod k: the strict order puts it below a if it lies in a's left
 * subtree, above a otherwise. */
static int balanced_node_ok(const float *pts, int64_t N, int k, const int32_t *slots, int64_t s)
{
    int depth = kdo_level(s);
    int64_t a = 0;
    for (int j = 0; j < depth; j++) {
        int right = (int)(((uint64_t)(s + 1) >> (depth - 1 - j)) & 1u);
        int d = kdo_level(a) % k;
        int64_t pa = slots[a], ps = slots[s];
        if (pa < 0 || pa >= N || ps < 0 || ps >= N)
            return 0;
        if (right ? !kdo_less(pts, k, d, pa, ps) : !kdo_less(pts, k, d, ps, pa))
            return 0;
        a = 2 * a + 1 + right;
    }
    return 1;
}

/* Checks that slots holds exactly the shape of the balanced tree of N points
 * (occupied slots as the split rule gives them, -1 elsewhere), that the
 * occupied slots hold a permutation of 0..N-1, and the k-d condition of every
 * node against every ancestor.  By uniqueness, valid == equal to
 * kdo_build_balanced.  Returns 0 if valid, 1 if not (first failing slot in
 * *bad_slot, -1 for a shape or permutation failure), <0 on error. */
int kdo_verify_balanced(const float *pts, int64_t N, int k, const int32_t *slots,
                        int64_t nslots, int64_t *bad_slot)
{
    int rc = check_args(pts, N, k, 0);
    if (rc != KDO_OK)
        return rc;
    if (!slots || nslots != kdo_balanced_slots(N))
        return KDO_EINVAL;
    uint8_t *occ = (uint8_t *)malloc((size_t)nslots);
    uint8_t *seen = (uint8_t *)calloc((size_t)N, 1);
    if (!occ || !seen) {
        free(occ);
        free(seen);
        return KDO_ENOMEM;
    }
    rc = balanced_shape(N, occ, nslots);
    int result = 0;
    if (bad_slot)
        *bad_slot = -1;
    for (int64_t s = 0; rc == KDO_OK && s < nslots && result == 0; s++) {
        int32_t v = slots[s];
        if (!occ[s]) {
            if (v != -1)
                result = 1;
            continue;
        }
        if (v < 0 || v >= N || seen[v])
            result = 1;
        else
            seen[v] = 1;
    }
    for (int64_t s = 0; rc == KDO_OK && s < nslots && result == 0; s++) {
        if (occ[s] && !balanced_node_ok(pts, N, k, slots, s)) {
            result = 1;
            if (bad_slot)
                *bad_slot = s;
        }
    }
    free(occ);
    free(seen);
    return rc != KDO_OK ? rc : result;
}

/* Exhaustive search: every assignment of the N points to the occupied slots
 * (Heap's algorithm over the occupied slots in heap order); counts the
 * assignments that satisfy the k-d condition and stores the first one
 * (N <= 11). */
int64_t kdo_brute_force_balanced(const float *pts, int N, int k, int32_t *first_valid)
{
    if (check_args(pts, N, k, 0) != KDO_OK || N > 11)
        return -1;
    int64_t nslots = kdo_balanced_slots(N);
    uint8_t occ[2048];
    int64_t where[11];
    if (nslots > 2048 || balanced_shape(N, occ, nslots) != KDO_OK)
        return -1;
    int cnt = 0;
    for (int64_t s = 0; s < nslots; s++)
        if (occ[s])
            where[cnt++] = s;
    if (cnt != N)
        return -1;
    int32_t slots[2048];
    int32_t a[11];
    int c[11];
    for (int i = 0; i < N; i++) {
        a[i] = i;
        c[i] = 0;
    }
    int64_t valid = 0;
    for (;;) {
        for (int64_t s = 0; s < nslots; s++)
            slots[s] = -1;
        for (int i = 0; i < N; i++)
            slots[where[i]] = a[i];
        int ok = 1;
        for (int i = 0; i < N && ok; i++)
            ok = balanced_node_ok(pts, N, k, slots, where[i]);
        if (ok) {
            if (valid == 0 && first_valid)
                memcpy(first_valid, slots, sizeof(int32_t) * (size_t)nslots);
            valid++;
        }
        int i = 1; /* next permutation (Heap's algorithm, iterative form) */
        while (i < N && c[i] >= i) {
            c[i] = 0;
            i++;
        }
        if (i >= N)
            break;
        int j = (i % 2 == 0) ? 0 : c[i];
        int32_t tmp = a[j];
        a[j] = a[i];
        a[i] = tmp;
        c[i]++;
    }
    return valid;
}

/* ---- split dimensions of a built tree -------------------------------------
 * dims[u] = the split dimension of level-order node u of the tree whose points
 * in level order are tree_pts (row u = the point stored at node u).
 * Round-robin ([W] round-robin paragraph): level(u) mod k.  Widest ([W]
 * split-widest-dimension paragraphs, the walk): start from the bounding box of
 * all points, go down from the root to u, cutting the domain at each
 * ancestor's split coordinate (hi for a left turn, lo for a right turn), and
 * take the widest extent of the final domain. */
int kdo_node_dims(const float *tree_pts, int64_t N, int k, int mode, uint8_t *dims)
{
    int rc = check_args(tree_pts, N, k, mode);
    if (rc != KDO_OK || !dims)
        return rc != KDO_OK ? rc : KDO_EINVAL;
    float root_lo[KDO_MAXK], root_hi[KDO_MAXK];
    bbox(tree_pts, N, k, root_lo, root_hi);
    for (int64_t u = 0; u < N; u++) {
        int depth = kdo_level(u);
        if (mode == 0) {
            dims[u] = (uint8_t)(depth % k);
            continue;
        }
        float lo[KDO_MAXK], hi[KDO_MAXK];
        memcpy(lo, root_lo, sizeof(float) * k);
        memcpy(hi, root_hi, sizeof(float) * k);
        int64_t a = 0; /* current ancestor */
        for (int t = depth - 1; t >= 0; t--) {
            int d = kdo_widest_dim(lo, hi, k);
            int right = (int)(((u + 1) >> t) & 1);
            float s = tree_pts[a * k + d];
            if (right)
                lo[d] = s;
            else
                hi[d] = s;
            a = 2 * a + 1 + right;
        }
        if (a != u)
            return KDO_EINTERNAL;
        dims[u] = (uint8_t)kdo_widest_dim(lo, hi, k);
    }
    return KDO_OK;
}

/* ---- k nearest neighbours, by brute force ----------------------------------
 * "Bigger Buffer k-d Trees on Multi-Many-Core Systems", nearest-neighbour
 * problem statement: the K points of the reference set closest to a query in
 * Euclidean distance.  Readings where the page is silent: the distance is the
 * squared distance sum_{c=0..k-1} (q[c] - p[c])^2, accumulated left to right
 * in float32 with every operation rounded (no fused multiply-add); the
 * reference points are the tree's nodes; the result is the K smallest pairs
 * (distance, node id) in that lexicographic order, listed ascending -- unique
 * because node ids are distinct.  When N < K the remaining slots hold node -1
 * and distance +infinity. */
float kdo_dist2(const float *q, const float *p, int k)
{
    float d = 0.0f;
    for (int c = 0; c < k; c++) {
        float t = q[c] - p[c];
        d = d + t * t;
    }
    return d;
}

int kdo_knn_brute(const float *tree_pts, int64_t N, int k, const float *queries, int64_t Q, int K,
                  int32_t *out_node, float *out_dist2)
{
    if (!tree_pts || !queries || !out_node || !out_dist2 || N < 1 || N > INT32_MAX || k < 1 ||
        k > KDO_MAXK || Q < 0 || K < 1)
        return KDO_EINVAL;
    for (int64_t qi = 0; qi < Q; qi++) {
        const float *q = queries + qi * k;
        int32_t *bn = out_node + qi * K;
        float *bd = out_dist2 + qi * K;
        int have = 0; /* bn/bd[0..have) sorted ascending by (distance, node) */
        for (int64_t u = 0; u < N; u++) {
            float d = kdo_dist2(q, tree_pts + u * k, k);
            if (have == K) {
                /* not better than the worst kept pair: skip */
                if (!(d < bd[K - 1] || (d == bd[K - 1] && u < bn[K - 1])))
                    continue;
                have--;
            }
            int j = have;
            while (j > 0 && (d < bd[j - 1] || (d == bd[j - 1] && u < bn[j - 1]))) {
                bd[j] = bd[j - 1];
                bn[j] = bn[j - 1];
                j--;
            }
            bd[j] = d;
            bn[j] = (int32_t)u;
            have++;
        }
        for (int j = have; j < K; j++) {
            bn[j] = -1;
            bd[j] = INFINITY;
        }
    }
    return KDO_OK;
}
