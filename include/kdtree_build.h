/*
 * kdtree_build.h -- C ABI of the GB300 left-balanced k-d tree builder.
 *
 * Builds the left-balanced, complete k-d tree over N points of k float32
 * coordinates, stored implicitly in level order: node 0 is the root, node i
 * has children 2i+1 and 2i+2 and parent (i-1)/2 ("GPU-friendly, Parallel, and
 * (Almost-)In-Place Construction of Left-Balanced k-d Trees", notation
 * paragraph).  Every node satisfies the k-d condition of that paper's problem
 * paragraph -- its left subtree lies on the low side and its right subtree on
 * the high side of its split plane -- and the tree's shape is the
 * left-balanced complete shape, which fixes every subtree's size.
 *
 * Ordering.  Points are compared in split dimension p by the strict total
 * order (x[p], x[p+1 mod k], ..., x[p-1 mod k], input index): the cyclic
 * "super key" of "An Implementation of a Balanced Kd Tree Builder Using GPUs"
 * (sort paragraph), with the input index as the final tiebreak.  Coordinates
 * compare as IEEE floats (-0 equals +0).  Under this order the tree is
 * unique, so results are reproducible bit for bit.
 *
 * Split rule (split_mode):
 *   KDT_SPLIT_ROUND_ROBIN (0): dimension level(node) mod k (round-robin
 *       paragraph of the left-balanced paper);
 *   KDT_SPLIT_WIDEST (1): the dimension of widest extent of the node's domain,
 *       lowest dimension on ties; the root's domain is the bounding box of all
 *       points and each child's domain is its parent's cut at the parent's
 *       split coordinate (split-widest-dimension paragraphs of the same
 *       paper).  Extents are float32 differences hi - lo.
 *
 * Output.  perm[node] = input index of the point stored at level-order node
 * `node` (so the points of the tree are pts[perm[0]], pts[perm[1]], ...).
 *
 * Layouts.  pts is row-major N x k float32 (k adjacent coordinates per point,
 * the "coordinate array" layout of the KdTreeGPU page); perm is int32[N].
 * Limits: 1 <= N <= 2^31 - 1, 1 <= k <= KDT_MAX_K.
 *
 * Streams.  `stream` is a cudaStream_t passed as void* (NULL = the legacy
 * default stream).  Calls marked "stream-ordered" only enqueue work and return;
 * the caller synchronises before reading results.  Calls marked "synchronous"
 * return after the work is complete.
 *
 * Errors.  Every call returns a KDT_* code.  Argument errors are detected on
 * the host and returned at once, before anything is enqueued.  Errors found on
 * the device (non-finite input, an internal consistency check) are recorded in
 * a per-device status word that kdt_status() returns and clears; the
 * synchronous calls return them directly.  After a device-side error the
 * contents of perm are unspecified.
 *
 * Thread safety.  Calls on different streams may overlap when each uses its
 * own workspace.  The per-device status word is shared by all builds in the
 * process.
 */
#ifndef KDTREE_BUILD_H
#define KDTREE_BUILD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KDT_OK 0
#define KDT_EINVAL (-1)     /* bad argument (null pointer, N, k, mode, size) */
#define KDT_ENOMEM (-2)     /* device allocation failed, or workspace too small */
#define KDT_ECUDA (-3)      /* a CUDA runtime call failed */
#define KDT_ENONFINITE (-4) /* a coordinate is NaN or infinite */
#define KDT_ETIMEOUT (-5)   /* a bounded device-side wait gave up */
#define KDT_EINTERNAL (-6)  /* a device-side consistency check failed */

#define KDT_SPLIT_ROUND_ROBIN 0
#define KDT_SPLIT_WIDEST 1

#define KDT_MAX_K 32

/* Bytes of device scratch that a build of (N, k, split_mode) needs.
 * Host-only; returns KDT_EINVAL for arguments kdt_build would reject. */
int kdt_workspace_size(int64_t N, int k, int split_mode, size_t *bytes);

/* Builds the tree.  pts (read-only) and perm (fully overwritten) are DEVICE
 * pointers owned by the caller.  Scratch memory is allocated and freed
 * stream-ordered on `stream` (cudaMallocAsync / cudaFreeAsync).
 * Stream-ordered. */
int kdt_build(const float *pts, int64_t N, int k, int split_mode,
              int32_t *perm, void *stream);

/* Same as kdt_build with caller-provided device scratch: `workspace` must hold
 * at least kdt_workspace_size() bytes, be 256-byte aligned and must not be in
 * use by another call until this build completes on `stream`.  Allocates
 * nothing.  Stream-ordered. */
int kdt_build_ws(const float *pts, int64_t N, int k, int split_mode,
                 int32_t *perm, void *workspace, size_t workspace_bytes,
                 void *stream);

/* Host-buffer variant: host_pts and host_perm are HOST pointers.  Page-locked
 * (pinned) buffers are used in place: the build's first kernel reads the
 * points across the host link while converting them, and the kernels that fix
 * nodes write the permutation straight into host_perm, so the transfers
 * overlap the build.  Pageable buffers are staged: the points are copied into
 * `workspace` first and the permutation is copied back at the end.  Device
 * scratch is `workspace` (at least kdt_host_workspace_size() bytes).
 * Synchronous; returns device-side errors directly. */
int kdt_host_workspace_size(int64_t N, int k, int split_mode, size_t *bytes);
int kdt_build_host(const float *host_pts, int64_t N, int k, int split_mode,
                   int32_t *host_perm, void *workspace, size_t workspace_bytes,
                   void *stream);

/* Checks that perm (DEVICE pointer) is the tree of pts: perm is a permutation
 * of 0..N-1 and every node satisfies the k-d condition against every one of
 * its ancestors under the order and split rule above (the verifier idea of
 * the KdTreeGPU page).  Because the tree is unique, "valid" is equivalent to
 * "equal to the reference result".  Allocates its scratch stream-ordered.
 * Synchronous: returns 0 if valid, 1 if not, or a negative KDT_* code. */
int kdt_verify(const float *pts, int64_t N, int k, int split_mode,
               const int32_t *perm, void *stream);

/* The points in level order: out[node * k + c] = pts[perm[node] * k + c] for
 * every node and coordinate, copied as raw 32-bit words (bit-exact, signed
 * zeros included).  This applies a build's permutation to the data, the
 * reordered point array that "GPU-friendly, Parallel, and (Almost-)In-Place
 * Construction of Left-Balanced k-d Trees" produces (introduction, core
 * idea).  pts (N x k, read-only), perm (int32[N], read-only) and out (N x k,
 * fully overwritten) are DEVICE pointers owned by the caller; out must not
 * overlap pts (KDT_EINVAL).  An entry of perm outside 0..N-1 is skipped and
 * recorded as KDT_EINVAL in the device status word (kdt_status).
 * Allocates nothing.  Stream-ordered. */
int kdt_gather_points(const float *pts, int64_t N, int k, const int32_t *perm,
                      float *out, void *stream);

/* In-place build: builds the tree of pts exactly as kdt_build_ws (perm
 * receives the permutation), then rewrites pts itself in level order, so that
 * afterwards pts[node * k + c] is coordinate c of the point stored at `node`
 * (bit-exact).  `workspace` (at least kdt_workspace_size() bytes, 256-byte
 * aligned) is the only temporary; nothing is allocated.  pts is read by the
 * build before it is rewritten; if the build records a device-side error, pts
 * is left unchanged.  pts and perm are DEVICE pointers.  Stream-ordered. */
int kdt_build_inplace(float *pts, int64_t N, int k, int split_mode,
                      int32_t *perm, void *workspace, size_t workspace_bytes,
                      void *stream);

/* ---- the balanced tree of Brown's builder ---------------------------------
 * "An Implementation of a Balanced Kd Tree Builder Using GPUs", overview
 * list: sort one reference array per coordinate, take the median of the
 * first coordinate's array as the first node, partition the other arrays into
 * the points below and above it, and repeat on both sides with the next
 * coordinate, cycling through the coordinates; build section: the medians of
 * level L form a per-level store whose entry j has its children at entries 2j
 * and 2j+1 of level L+1.  This tree is balanced but not left-balanced: a node
 * of n points keeps the point of rank floor((n-1)/2) under the split order
 * (dimension level mod k; the same strict super key + input index order as
 * above, so duplicates are kept and the tree is unique), its lower subtree
 * gets floor((n-1)/2) points and its upper subtree the rest.
 *
 * Storage: heap order, the node of entry j of level L in slot 2^L - 1 + j;
 * slots[s] = input index of the point at slot s, -1 where the subtree is
 * empty.  The tree has numLevels(N) levels, so slots has
 * kdt_balanced_slots(N) = 2^numLevels(N) - 1 entries (< 2N). */

/* Number of heap slots of the balanced tree of N points.  Host-only. */
int kdt_balanced_slots(int64_t N, int64_t *slots);

/* Bytes of device scratch for kdt_build_balanced.  Host-only. */
int kdt_balanced_workspace_size(int64_t N, int k, size_t *bytes);

/* Builds the balanced tree.  pts (N x k float32, read-only), slots
 * (int32[kdt_balanced_slots(N)], fully overwritten) and workspace (at least
 * kdt_balanced_workspace_size bytes, 256-byte aligned, not in use by another
 * call until this one completes on `stream`) are DEVICE pointers owned by the
 * caller.  Same limits and errors as kdt_build.  Allocates nothing.
 * Stream-ordered. */
int kdt_build_balanced(const float *pts, int64_t N, int k, int32_t *slots,
                       void *workspace, size_t workspace_bytes, void *stream);

/* ---- queries on a built tree ------------------------------------------------
 * tree_pts is the tree's points in level order (row u = the point stored at
 * node u: the output of kdt_gather_points or kdt_build_inplace), N x k float32,
 * a DEVICE pointer.  Results refer to node ids; perm[node] gives the input
 * index. */

/* Split dimension of every node: dims[u] (uint8[N], DEVICE, fully
 * overwritten).  Round-robin: level(u) mod k.  Widest: the walk of the
 * split-widest-dimension paragraphs of the left-balanced paper -- the root's
 * domain is the bounding box of all points, each step down cuts it at the
 * ancestor's split coordinate, the node's dimension is the widest extent of
 * its domain (float32 hi - lo, lowest dimension on ties) -- which are the
 * dimensions the build used.  Allocates 2k words stream-ordered (widest).
 * Stream-ordered. */
int kdt_node_dims(const float *tree_pts, int64_t N, int k, int split_mode,
                  uint8_t *dims, void *stream);

#define KDT_MAX_KNN 64

/* The K nearest nodes of each query ("Bigger Buffer k-d Trees on
 * Multi-Many-Core Systems", nearest-neighbour search via k-d trees: down to
 * the query's cell, then back up, entering a node's other subtree only when
 * its splitting plane is within the current K-th distance; no stack on the
 * implicit tree).  Result: for query i, out_node[i*K + j] and
 * out_dist2[i*K + j] (j = 0..K-1) are the K smallest pairs (dist2, node) in
 * lexicographic order, ascending, where dist2 = sum over c = 0..k-1 of
 * (q[c] - p[c])^2 accumulated left to right in float32 with every operation
 * rounded (no fused multiply-add).  Slots beyond N hold node -1 and dist2
 * +infinity.  dims: the tree's split dimensions (kdt_node_dims); NULL means
 * round-robin.  queries is Q x k float32; all pointers are DEVICE pointers,
 * out_* fully overwritten.  1 <= K <= KDT_MAX_KNN, Q >= 0.  A dims entry >= k
 * is recorded as KDT_EINVAL in the device status word.  Allocates nothing.
 * Stream-ordered. */
int kdt_knn(const float *tree_pts, int64_t N, int k, const uint8_t *dims,
            const float *queries, int64_t Q, int K, int32_t *out_node,
            float *out_dist2, void *stream);

/* Synchronises `stream`, then returns and clears the calling thread's current
 * device's status word (KDT_OK if no device-side error was recorded). */
int kdt_status(void *stream);

/* Human-readable name of a KDT_* code (static string). */
const char *kdt_error_string(int code);

/* Per-kernel timing.  When enabled, the build records CUDA events around each
 * of its kernel launches, or around a family's group of launches (on the
 * build's stream), and accumulates, per kernel family, the number of timed
 * scopes, their total device time and the kernels launched inside them.
 * kdt_profile_read fills up to `cap` entries (names are static strings) and
 * returns the number of families; it synchronises on the events it reads.
 * kdt_profile_reset clears the totals.  Off by default. */
typedef struct {
    const char *name;
    int64_t launches;  /* timed scopes */
    double total_ms;
    double bytes_alg;  /* algorithmic bytes summed over the scopes */
    int64_t kernels;   /* kernel launches inside those scopes */
} kdt_kernel_stat;

int kdt_profile_enable(int on);
int kdt_profile_reset(void);
int kdt_profile_read(kdt_kernel_stat *out, int cap);

/* Build without any device allocation, for callers that cannot allocate.
 * The paper has no counterpart to this entry point; it is a library convenience.
 *
 * Some callers are not allowed to call cudaMalloc or cudaMallocAsync at the
 * point where they build a tree: a plugin whose host application owns every
 * byte of device memory through its own pool, a latency-critical loop where
 * an allocation could synchronise the device or fail under memory pressure,
 * or a caller that simply has no allocator to hand.  This entry point takes
 * the same inputs and output as kdt_build but uses, as its scratch, one
 * fixed array of KDT_STATIC_SCRATCH_BYTES bytes that the library reserves on
 * every device that loads it (held until the process exits).
 *
 * Limit: the build must fit the array, i.e. kdt_workspace_size(N, k,
 * split_mode) <= KDT_STATIC_SCRATCH_BYTES (about 0.5-1 million points for
 * k = 3); larger builds are rejected with KDT_EINVAL before anything is
 * enqueued.  Other argument errors also return KDT_EINVAL.
 *
 * Set-up: the first call on each device looks up the array's device address
 * (with that device current); make that first call before any stream
 * capture.  Every call clears the parts of the array that must start at
 * zero, so one call's leftovers never affect the next.  All calls share the
 * one array: calls whose work overlaps on the GPU (for example on two
 * streams without ordering between them) race and corrupt each other's
 * results; order them on one stream or with events.
 *
 * pts and perm are DEVICE pointers as for kdt_build.  Stream-ordered. */
#define KDT_STATIC_SCRATCH_BYTES (32u * 1024u * 1024u)
int kdt_build_static(const float *pts, int64_t N, int k, int split_mode,
                     int32_t *perm, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KDTREE_BUILD_H */
