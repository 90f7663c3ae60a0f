// Input checks and adjacency sorting for mce_create.
//
// The problem is stated for simple undirected graphs ("Parallelizing Maximal Clique
// Enumeration on GPUs", Section 2.1).  Reading the graph is excluded from the reported times on
// the pages (Section 4.1, "Reporting of Measurements"); this file is that reading step.  It runs
// once per handle, not in the timed path.
#include <climits>

#include "mce_internal.cuh"

namespace mce {

namespace {

constexpr int kThreads = 256;

// Lists longer than this are validated by many CTAs each (validate_big_kernel).
constexpr int kValidateSplit = 1024;
constexpr int kValidateChunk = 4096;   // entries per CTA of a long list

// Offsets must be non-decreasing and inside [0, nnz]; adjacency ids inside [0, n).  Lists that
// are not sorted ascending are appended to `unsorted_list`; stats[1] counts, and big_list
// receives, the lists longer than kValidateSplit, stats[2] is the largest degree.
__global__ void __launch_bounds__(kThreads) check_kernel(DevGraph g, int *unsorted_list,
                                                         int *stats, int *big_list)
{
    int *unsorted_n = stats;
    const int lane = threadIdx.x & 31;
    const int warps = gridDim.x * (blockDim.x >> 5);
    for (int v = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; v < g.n; v += warps) {
        const int lo = g.offs[v], hi = g.offs[v + 1];
        if (lo < 0 || hi < lo || (long long)hi > g.nnz) {
            if (lane == 0) set_status(g.ctrl, MCE_ERR_INVALID_ARG);
            continue;
        }
        bool bad_id = false, unsorted = false;
        for (int i = lo + lane; i < hi; i += 32) {
            const int u = g.adj[i];
            bad_id |= (u < 0 || u >= g.n);
            if (i > lo && g.adj[i - 1] > u) unsorted = true;
        }
        if (__any_sync(0xffffffffu, bad_id)) {
            if (lane == 0) set_status(g.ctrl, MCE_ERR_ID_RANGE);
        } else if (__any_sync(0xffffffffu, unsorted)) {
            if (lane == 0) unsorted_list[atomicAdd(unsorted_n, 1)] = v;
        }
        if (lane == 0 && hi - lo > kValidateSplit) {
            big_list[atomicAdd(&stats[1], 1)] = v;
            atomicMax(&stats[2], hi - lo);
        }
    }
}

// Bitonic sort of one list per CTA in shared memory (lists of at most 4096 entries).
constexpr int kSmemSortMax = 4096;

__global__ void __launch_bounds__(512) sort_small_kernel(const int *offs, int *adj,
                                                         const int *list, int n_list)
{
    __shared__ int keys[kSmemSortMax];
    for (int li = blockIdx.x; li < n_list; li += gridDim.x) {
        const int v = list[li];
        const int lo = offs[v], len = offs[v + 1] - lo;
        if (len > kSmemSortMax) continue;
        int p2 = 1;
        while (p2 < len) p2 <<= 1;
        for (int i = threadIdx.x; i < p2; i += blockDim.x) keys[i] = i < len ? adj[lo + i] : INT_MAX;
        __syncthreads();
        for (int k = 2; k <= p2; k <<= 1) {
            for (int j = k >> 1; j > 0; j >>= 1) {
                for (int i = threadIdx.x; i < p2; i += blockDim.x) {
                    const int ixj = i ^ j;
                    if (ixj > i) {
                        const bool up = (i & k) == 0;
                        const int a = keys[i], b = keys[ixj];
                        if ((a > b) == up) { keys[i] = b; keys[ixj] = a; }
                    }
                }
                __syncthreads();
            }
        }
        for (int i = threadIdx.x; i < len; i += blockDim.x) adj[lo + i] = keys[i];
        __syncthreads();
    }
}

// Bitonic sort of one long list in global scratch by a single CTA.
__global__ void __launch_bounds__(1024) sort_large_kernel(const int *offs, int *adj, int v,
                                                          int *scratch)
{
    const int lo = offs[v], len = offs[v + 1] - lo;
    int p2 = 1;
    while (p2 < len) p2 <<= 1;
    for (int i = threadIdx.x; i < p2; i += blockDim.x) scratch[i] = i < len ? adj[lo + i] : INT_MAX;
    __syncthreads();
    for (int k = 2; k <= p2; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < p2; i += blockDim.x) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const bool up = (i & k) == 0;
                    const int a = scratch[i], b = scratch[ixj];
                    if ((a > b) == up) { scratch[i] = b; scratch[ixj] = a; }
                }
            }
            __syncthreads();
        }
    }
    for (int i = threadIdx.x; i < len; i += blockDim.x) adj[lo + i] = scratch[i];
}

__device__ __forceinline__ bool sorted_contains(const int *a, int len, int key)
{
    int lo = 0, hi = len;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] < key) lo = mid + 1;
        else hi = mid;
    }
    return lo < len && a[lo] == key;
}

// On sorted lists: no self-loop and no repeated neighbour; and symmetry.  Symmetry is checked on
// the forward entries only (u in N(v) with u > v: is v in N(u)?), and the forward and backward
// entries are counted into fb[0], fb[1].  With no repeats, reversal maps forward entries into
// backward ones injectively, so equal counts make it a bijection: every backward entry has its
// reverse too.  A warp takes a list of at most kValidateSplit entries (longer ones: below).
__device__ __forceinline__ void validate_range(const DevGraph &g, int v, int lo, int hi, int first,
                                               int step, unsigned long long *fb)
{
    const int lane = threadIdx.x & 31;
    bool not_simple = false, asym = false;
    unsigned nf = 0, nbk = 0;
    for (int i = first; i < hi; i += step) {
        const int u = g.adj[i];
        not_simple |= (u == v) || (i > lo && g.adj[i - 1] == u);
        if (u > v) {
            ++nf;
            const int ulo = g.offs[u];
            asym |= !sorted_contains(g.adj + ulo, g.offs[u + 1] - ulo, v);
        } else if (u < v) {
            ++nbk;
        }
    }
    const unsigned wf = __reduce_add_sync(0xffffffffu, nf);
    const unsigned wb = __reduce_add_sync(0xffffffffu, nbk);
    if (lane == 0) {
        if (wf) atomicAdd(&fb[0], (unsigned long long)wf);
        if (wb) atomicAdd(&fb[1], (unsigned long long)wb);
    }
    if (__any_sync(0xffffffffu, not_simple)) {
        if (lane == 0) set_status(g.ctrl, MCE_ERR_NOT_SIMPLE);
    } else if (__any_sync(0xffffffffu, asym)) {
        if (lane == 0) set_status(g.ctrl, MCE_ERR_NOT_SYMMETRIC);
    }
}

__global__ void __launch_bounds__(kThreads) validate_kernel(DevGraph g, unsigned long long *fb)
{
    const int lane = threadIdx.x & 31;
    const int warps = gridDim.x * (blockDim.x >> 5);
    for (int v = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; v < g.n; v += warps) {
        const int lo = g.offs[v], hi = g.offs[v + 1];
        if (hi - lo > kValidateSplit) continue;
        validate_range(g, v, lo, hi, lo + lane, 32, fb);
    }
}

// A long list: CTA (x, y) takes chunks y, y + gridDim.y, ... of kValidateChunk entries of the
// list of big_list[x].
__global__ void __launch_bounds__(kThreads) validate_big_kernel(DevGraph g, const int *big_list,
                                                                unsigned long long *fb)
{
    const int v = big_list[blockIdx.x];
    const int lo = g.offs[v], hi = g.offs[v + 1];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (long long c0 = lo + (long long)blockIdx.y * kValidateChunk; c0 < hi;
         c0 += (long long)gridDim.y * kValidateChunk) {
        const int c1 = (int)(c0 + kValidateChunk < hi ? c0 + kValidateChunk : hi);
        // warps interleave over the chunk; the repeat test reads the entry before, as above
        validate_range(g, v, lo, c1, (int)c0 + warp * 32 + lane, kThreads, fb);
    }
}

int grid_for(long long work_items, int per_block)
{
    long long b = (work_items + per_block - 1) / per_block;
    if (b < 1) b = 1;
    if (b > 65535LL * 32) b = 65535LL * 32;
    return (int)b;
}

}  // namespace

cudaError_t launch_ingest_check(const DevGraph &g, int *d_unsorted_list, int *d_stats,
                                int *d_big_list, cudaStream_t s)
{
    if (g.n == 0) return cudaSuccess;
    check_kernel<<<grid_for(g.n, kThreads / 32), kThreads, 0, s>>>(g, d_unsorted_list, d_stats,
                                                                   d_big_list);
    return cudaGetLastError();
}

cudaError_t launch_ingest_sort(const DevGraph &g, int *adj_mut, const int *d_list, int n_list,
                               int *scratch, long long scratch_len, cudaStream_t s)
{
    if (n_list <= 0) return cudaSuccess;
    sort_small_kernel<<<n_list < 4096 ? n_list : 4096, 512, 0, s>>>(g.offs, adj_mut, d_list,
                                                                    n_list);
    (void)scratch;
    (void)scratch_len;
    return cudaGetLastError();
}

// Sorts one list longer than the shared-memory limit (the caller loops over such lists).
cudaError_t launch_ingest_sort_large(const DevGraph &g, int *adj_mut, int v, int *scratch,
                                     cudaStream_t s)
{
    sort_large_kernel<<<1, 1024, 0, s>>>(g.offs, adj_mut, v, scratch);
    return cudaGetLastError();
}

cudaError_t launch_ingest_validate(const DevGraph &g, const int *d_big_list, int n_big,
                                   int max_degree, unsigned long long *d_fb, cudaStream_t s)
{
    if (g.n == 0) return cudaSuccess;
    validate_kernel<<<grid_for(g.n, kThreads / 32), kThreads, 0, s>>>(g, d_fb);
    if (n_big > 0) {
        int chunks = (max_degree + kValidateChunk - 1) / kValidateChunk;
        if (chunks > 65535) chunks = 65535;
        validate_big_kernel<<<dim3(n_big, chunks), kThreads, 0, s>>>(g, d_big_list, d_fb);
    }
    return cudaGetLastError();
}

}  // namespace mce
