/*
 * mce.h -- C ABI of the GB300 maximal clique enumeration library (libmce_gb300.so).
 *
 * The problem is the one stated in "Parallelizing Maximal Clique Enumeration on GPUs"
 * (arXiv 2212.01473v2), Section 2.1: given a simple undirected graph G = (V, E), find every
 * maximal clique -- every complete subgraph that no further vertex can extend -- exactly, with
 * no sampling or approximation.
 *
 * The search is the Bron-Kerbosch algorithm with pivoting (Section 2.3, Algorithm 2; pivot
 * chosen over P u X, Tomita's rule), split into independent first-level subtrees
 * (Section 2.4, Algorithm 3) taken in degeneracy order (Section 2.4, "Degeneracy Ordering"),
 * each solved on a binary-encoded induced subgraph over P u X (Sections 2.4 and 3.4, "full"
 * induced subgraph) with the compact X representation of Section 3.5 and the worker list of
 * Section 3.3.  mce_config selects the alternatives of the same pages: partial induced
 * subgraphs (Section 3.4, and the rule of Section 4.5 that picks them) and independent
 * second-level subtrees (Section 3.2, Algorithm 4).  Everything runs on one GPU.
 *
 * Conventions shared by every entry point
 *   - Streams are passed as `void *` holding a cudaStream_t (NULL = the legacy default
 *     stream).  Calls that take a stream only enqueue work on it, in stream order, and return
 *     without waiting, unless their comment says they synchronise.
 *   - "device pointer" means memory the current CUDA device can address (cudaMalloc, a
 *     PyTorch CUDA tensor, managed memory).  "host pointer" means ordinary host memory.
 *   - A handle is bound to the CUDA device that was current when mce_create ran; every later
 *     call must be made with that device current.  Handles are not thread-safe.
 *   - Return codes report argument errors and CUDA launch/allocation failures at call time.
 *     Errors that the GPU detects while running (a wait limit exceeded, an output buffer
 *     overflow) are recorded in a status word on the device and returned by mce_last_error.
 *   - Vertex ids are int32 in [0, n).  Results always name vertices by these original ids.
 */
#ifndef MCE_H
#define MCE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct mce_graph mce_graph;   /* opaque; owned by the library */

typedef enum mce_status {
    MCE_OK = 0,
    MCE_ERR_INVALID_ARG = 1,       /* a NULL pointer, a negative size, offsets not monotone   */
    MCE_ERR_NOT_SIMPLE = 2,        /* a self-loop or a repeated neighbour                      */
    MCE_ERR_NOT_SYMMETRIC = 3,     /* u in N(v) but v not in N(u)                              */
    MCE_ERR_ID_RANGE = 4,          /* a neighbour id or a root id outside [0, n)               */
    MCE_ERR_OUT_OF_MEMORY = 5,     /* a device or host allocation failed                       */
    MCE_ERR_BUFFER_TOO_SMALL = 6,  /* an output buffer cannot hold the result                  */
    MCE_ERR_DEVICE_TIMEOUT = 7,    /* a device-side wait exceeded mce_config.spin_limit_ns     */
    MCE_ERR_LIMIT = 8,             /* the graph exceeds a documented size limit of the library */
    MCE_ERR_CUDA = 9,              /* any other CUDA runtime error                             */
    MCE_ERR_INTERNAL = 10          /* a device-side consistency check failed (a library bug)   */
} mce_status;

/*
 * Tuning knobs.  Fill with mce_config_default() and change fields; pass NULL for defaults.
 *   worker_list      1: warps that run out of first-level subtrees receive branches donated by
 *                    busy warps (Section 3.3); 0: static first-level distribution only.
 *   donate_min_p     a branch is donated only if |P| at its root is at least this (Section 3.3
 *                    uses 10) and at least a quarter of |P| of its first-level subtree (copying
 *                    a branch into another warp's workspace is not free).
 *   warps_per_block  warps per CTA of the search kernel (0 = library default).
 *   blocks_per_sm    CTAs per SM of the search kernel (0 = as many as can be resident).
 *   profile          1: record CUDA events around the ordering and around every search launch,
 *                    so that mce_get_info reports per-stage device times; 0 (default): none.
 *   donate_rule      0 (default): donate only when unexplored branches remain both at the
 *                    donor's level and at an earlier level (Section 3.3); 1: when either holds.
 *   spin_limit_ns    upper bound on any single device-side wait (grid barrier, idle warp
 *                    waiting for a donation); on expiry the kernel records
 *                    MCE_ERR_DEVICE_TIMEOUT and returns instead of hanging (an idle warp
 *                    that waited this long instead leaves the worker list, which is not an
 *                    error).
 *   induced          induced subgraph of a subtree (Section 3.4): 1 = full (bitset rows for
 *                    every vertex of P u X; pivot from P u X), 2 = partial (rows for P only;
 *                    P-X adjacencies are binary searches in the graph; pivot from P u X_P),
 *                    0 (default) = the rule of Section 4.5: partial iff Delta / d > 200.
 *   subtree_level    1 (default): independent first-level subtrees, one per vertex
 *                    (Algorithm 3); 2: independent second-level subtrees, one per edge
 *                    (Algorithm 4, Section 3.2).  Other values: MCE_ERR_INVALID_ARG.
 *   overlap_builds   1 (default): the subtrees of the roots with rows of 1, 2 and 4 words
 *                    (full induced subgraphs, first-level subtrees) are built ahead of their
 *                    search on a stream of the handle's own, forked from and joined back to
 *                    the caller's stream, so a narrower class's build overlaps the wider
 *                    classes' search; 0: each build runs on the caller's stream just before
 *                    its search (mce_info.ms_build is then the build's own time).  Results
 *                    are the same.  Other values: MCE_ERR_INVALID_ARG.
 */
typedef struct mce_config {
    int32_t worker_list;
    int32_t donate_min_p;
    int32_t warps_per_block;
    int32_t blocks_per_sm;
    int32_t profile;
    int32_t donate_rule;
    int64_t spin_limit_ns;
    int32_t induced;
    int32_t subtree_level;
    int32_t overlap_builds;
} mce_config;

#define MCE_NUM_WIDTHS 6   /* search kernels, one per bitset row width 1, 2, 4, 8, 16, 32 words */

/* Sizes and diagnostics of a handle (filled by mce_get_info). */
typedef struct mce_info {
    int32_t n;                 /* vertices                                                   */
    int32_t degeneracy;        /* d: largest core number (Section 2.4)                        */
    int64_t m;                 /* undirected edges                                            */
    int32_t max_degree;        /* Delta                                                       */
    int32_t hist_len;          /* d + 2: length of the size histogram in mce_count's output   */
    int32_t peel_rounds;       /* rounds of the parallel peel                                 */
    int32_t n_workers;         /* warps of the search kernel (each one a DFS worker)          */
    int64_t workspace_bytes;   /* device workspace held by the handle                         */
    uint64_t tree_nodes;       /* search-tree nodes visited by the last count/enumerate       */
    uint64_t donations;        /* branches donated through the worker list, last call         */
    /* last call, per row-width class k (row width 1 << k words): */
    uint64_t words[MCE_NUM_WIDTHS];    /* bitset words scored or intersected (pivot scans,
                                          child sets, X_X tests): the search's integer work  */
    int32_t roots[MCE_NUM_WIDTHS];     /* first-level roots of the full schedule per class   */
    int32_t workers[MCE_NUM_WIDTHS];   /* warps launched per class (0: class not launched)   */
    float ms_search[MCE_NUM_WIDTHS];   /* device time per class launch (profile = 1 only)    */
    float ms_order;                    /* device time of the last mce_order/mce_create order */
    int32_t launches;                  /* kernels launched by the last order + count calls   */
    int32_t induced;                   /* induced subgraph in use: 1 full, 2 partial         */
    int32_t subtree_level;             /* 1: first-level subtrees, 2: second-level subtrees  */
    float ms_peel;                     /* the peel's part of ms_order (profile = 1 only)     */
    int64_t peel_live;                 /* vertices still in the graph, summed over the peel's
                                          rounds (the live lists its rounds scan)            */
    float ms_build[MCE_NUM_WIDTHS];    /* device time of the launch that builds the subtrees
                                          of the class's roots ahead of its search (rows of
                                          1, 2, 4 words; 0 where the search builds them
                                          itself; profile = 1 only).  ms_search excludes it. */
} mce_info;

/* Writes the default configuration into *cfg.  Returns MCE_ERR_INVALID_ARG if cfg is NULL. */
mce_status mce_config_default(mce_config *cfg);

/*
 * Copies a graph into the library and prepares it (input side of Section 2.1's problem).
 *   offsets  int32[n+1], offsets[0] = 0, non-decreasing; adj int32[offsets[n]]: the neighbours
 *            of v are adj[offsets[v] .. offsets[v+1]), in any order.  Both are host pointers
 *            if is_device_ptr == 0, else device pointers.  The graph must be simple and
 *            undirected: every edge listed in both directions, no self-loops, no repeats.
 *            The library copies both arrays; the caller may free them on return.
 *   n        number of vertices, 0 <= n < 2^30.  offsets[n] must be < 2^31.
 *   cfg      NULL for defaults.
 *   stream   the copy, the input checks and the first degeneracy ordering run on it.
 *   out      receives the handle; *out is NULL on failure.
 * Synchronises `stream` (the input checks and the workspace size are read back to the host).
 * Device memory comes from a memory pool the library keeps per device (stream-ordered, on
 * `stream`); mce_destroy returns it to that pool, which keeps it for later handles until the
 * process ends or mce_trim_memory hands it back to the driver.
 * Errors: MCE_ERR_INVALID_ARG, MCE_ERR_ID_RANGE, MCE_ERR_NOT_SIMPLE, MCE_ERR_NOT_SYMMETRIC,
 * MCE_ERR_OUT_OF_MEMORY, MCE_ERR_LIMIT (n of 2^30 or more, a first-level P larger than 1024
 * vertices, a degree of 2^21 or more, or with second-level subtrees n + m of 2^31 or more),
 * MCE_ERR_CUDA.
 */
mce_status mce_create(const int32_t *offsets, const int32_t *adj, int32_t n, int is_device_ptr,
                      const mce_config *cfg, void *stream, mce_graph **out);

/*
 * Recomputes the degeneracy order (Section 2.4, "Degeneracy Ordering"): a parallel k-core peel
 * on the GPU, then the split of every adjacency into earlier (X) and later (P) neighbours and
 * the heavy-first schedule of the subtrees.  mce_count, mce_count_roots and
 * mce_enumerate use the order computed last; mce_create computes it once.  This entry point
 * exists so that a timing loop can include the preprocessing, as Section 4.1 ("Reporting of
 * Measurements") does.  Asynchronous on `stream`.
 */
mce_status mce_order(mce_graph *g, void *stream);

/*
 * Counts all maximal cliques (Section 2.1) with one launch of the persistent search kernel.
 *   d_out  device pointer to uint64[2 + hist_len] (hist_len from mce_info):
 *          d_out[0] = number of maximal cliques,
 *          d_out[1] = hash = sum over cliques C of mix64(sum_{c in C} key(c)) mod 2^64 with
 *                     key(c) = mix64((c + 1) * 0x9E3779B97F4A7C15) and mix64 the SplitMix64
 *                     output function -- independent of clique order and of vertex order,
 *          d_out[2 + k] = number of maximal cliques with k vertices.
 *          The pages define no summary; this one is the library's own.
 * Asynchronous on `stream`; the caller owns d_out.
 */
mce_status mce_count(mce_graph *g, void *stream, uint64_t *d_out);

/*
 * Same as mce_count, restricted to the first-level subtrees (Algorithm 3) of the given roots:
 * the maximal cliques whose earliest vertex in the current degeneracy order is one of them.
 * With second-level subtrees (mce_config.subtree_level = 2) the same cliques are found through
 * the subtrees of each root's edges to its later neighbours (Algorithm 4).
 * Summing the outputs over a partition of V gives mce_count's output, which makes runs
 * resumable and lets large graphs be processed in pieces.
 *   d_roots  device pointer to int32[n_roots], original vertex ids (duplicates count twice).
 * Root ids are checked on the device: an id outside [0, n) records MCE_ERR_ID_RANGE.
 */
mce_status mce_count_roots(mce_graph *g, void *stream, const int32_t *d_roots, int32_t n_roots,
                           uint64_t *d_out);

/*
 * Writes every maximal clique as its vertex ids sorted ascending:
 *   clique i = d_ids[d_offsets[i] .. d_offsets[i+1]), i < count.  Cliques are grouped by size
 *   (ascending); the order inside a size group is unspecified.
 *   d_ids      device int32[cap_ids]; d_offsets device int64[cap_cliques + 1].
 *   h_sizes    host int64[2]: receives {number of cliques, number of ids}.
 * Runs a counting pass first when the handle has no count of the full graph for its current
 * order (the sizes come from it, as in count-scan-write compaction), then the writing pass.
 * Synchronises `stream` once to read the sizes.  If a capacity is too small, nothing is written
 * and MCE_ERR_BUFFER_TOO_SMALL is returned with the required sizes in h_sizes.
 */
mce_status mce_enumerate(mce_graph *g, void *stream, int32_t *d_ids, int64_t cap_ids,
                         int64_t *d_offsets, int64_t cap_cliques, int64_t *h_sizes);

/*
 * mce_enumerate restricted to the subtrees of the given roots (the cliques mce_count_roots
 * counts for them), so that an enumeration larger than device memory can be written in pieces:
 * the caller takes the roots in batches, and copies each batch's output out (for example to a
 * pinned host buffer, overlapping the next batch) before reusing the buffers.
 *   d_roots    device int32[n_roots], original vertex ids; n_roots = 0 writes nothing.
 *   d_ids, d_offsets, h_sizes  as for mce_enumerate (d_offsets[0 .. count] is written).
 * Runs a counting pass over the roots, then the writing pass.  Synchronises `stream` once.
 * Errors: MCE_ERR_BUFFER_TOO_SMALL with the required sizes in h_sizes (nothing is written),
 * MCE_ERR_ID_RANGE for a root id outside [0, n), and those of mce_count_roots.
 */
mce_status mce_enumerate_roots(mce_graph *g, void *stream, const int32_t *d_roots,
                               int32_t n_roots, int32_t *d_ids, int64_t cap_ids,
                               int64_t *d_offsets, int64_t cap_cliques, int64_t *h_sizes);

/*
 * Copies the current degeneracy order to device buffers (diagnostics and tests):
 *   d_rank[v] = position of v in the order, d_core[v] = core number of v; either may be NULL.
 */
mce_status mce_get_order(mce_graph *g, void *stream, int32_t *d_rank, int32_t *d_core);

/*
 * Activity profile of the last search (diagnostics).  Only a library built with MCE_PROFILE
 * defined collects it (the normal build leaves it zero): SM clock cycles summed over warps, per
 * row-width class k, at out[k * 16 + a] for activity a = 0 subtree build (rows and X_X list),
 * 1 pivot selection, 2 child sets and leaf checks, 3 X_X partition, 4 donation, 5 waiting in the
 * worker list, 6 the slowest single first-level root, 7 number of roots, 8 small subtrees solved
 * whole, 9 split of N(v) into P and X, and inside a = 0: 10 hash and row set-up, 11 the walk of
 * the later-neighbour lists, 12 the X_X list and vertex keys.  Section 4.5 of the pages breaks
 * execution time down the same way from per-block SM clocks.  Then 16 values for the last
 * ordering, as seen by its first CTA, in nanoseconds: out[96 + p] for rounds run by all CTAs and
 * out[104 + p] for rounds run by one CTA, phase p = 0 scan, 1 report exchange, 2 decide and
 * write, 3 edge removal, 4 end-of-round barrier, 5 number of rounds (rounds run from a frontier,
 * without a scan, count as rounds run by one CTA); out[102] is the largest
 * degree of a vertex removed by the first CTA.  Then, per row-width class k, the load of every
 * SM in the last search (Section 4.3 judges the worker list by per-block loads): at
 * out[112 + k * 256 + s] the SM clock cycles that warps on SM s spent holding work (time in the
 * kernel minus time waiting in the worker list), for s < 256.
 *   out  host uint64[16 * MCE_NUM_WIDTHS + 16 + 256 * MCE_NUM_WIDTHS].  Synchronises the device.
 */
mce_status mce_get_profile(mce_graph *g, uint64_t *out);

/*
 * Degeneracy order of a small graph without allocating anything.
 *
 * The paper has no counterpart: this is a packaging of mce_order's peel for callers that are
 * not allowed to allocate device memory -- code that runs inside a framework whose caching
 * allocator owns all of the GPU's memory, plug-ins that are only ever handed buffers, or
 * latency-critical paths that must not pay for cudaMalloc and the synchronisation it implies.
 * It neither creates a handle nor calls cudaMalloc, cudaFree or any allocating library routine;
 * its scratch space is one fixed array of about 6.2 MiB in device memory, which every GPU that
 * loads the library holds until the process exits.
 *   d_offsets, d_adj  device pointers to a simple undirected graph as a CSR (the same layout as
 *                     mce_create).  The input is NOT checked: validate it with mce_create first
 *                     if it may be malformed.
 *   n                 0 <= n <= 262144; larger graphs return MCE_ERR_LIMIT and nothing runs.
 *   d_rank, d_core    device int32[n]: position in the canonical degeneracy order and core
 *                     number, identical to what mce_get_order reports for the same graph.
 *   d_result          device int32[2]: {degeneracy d, device-side status (0 or an mce_status)}.
 *   stream            the work is enqueued on it; the call returns without waiting.
 * The first call on each device looks up the device address of the scratch array
 * (cudaGetSymbolAddress); make that first call before any stream capture starts.  All calls
 * share the one array, so calls that can overlap on the GPU (different streams or host
 * threads) race with each other: keep them in one stream, one at a time.  Each call clears
 * the part of the array that must start at zero.
 */
mce_status mce_order_noalloc(const int32_t *d_offsets, const int32_t *d_adj, int32_t n,
                             int32_t *d_rank, int32_t *d_core, int32_t *d_result, void *stream);

/* Synchronises `stream`, then returns (and clears) the device-side status of the handle. */
mce_status mce_last_error(mce_graph *g, void *stream);

/* Fills *info; the diagnostics refer to the last completed call (synchronises the device). */
mce_status mce_get_info(mce_graph *g, mce_info *info);

/* Frees the handle and returns its device memory to the library's pool (synchronises the
 * device first).  NULL is a no-op. */
void mce_destroy(mce_graph *g);

/*
 * Returns the device memory that the library's pool for the current device keeps cached (the
 * memory of destroyed handles) to the driver; memory of live handles stays.  The library keeps
 * freed memory so that creating a handle after destroying another one needs no cudaMalloc; a
 * caller that shares the GPU with another allocator (for example a framework's caching
 * allocator) calls this once it has destroyed its handles.  Synchronises the device.
 * Errors: MCE_ERR_CUDA.
 */
mce_status mce_trim_memory(void);

/* Static English description of a status code. */
const char *mce_status_str(mce_status s);

#ifdef __cplusplus
}
#endif

#endif /* MCE_H */
