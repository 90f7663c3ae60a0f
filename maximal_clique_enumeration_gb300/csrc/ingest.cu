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

// Offsets must be non-decreasing and inside [0, nnz]; adjacency ids inside [0, n).  Lists that
// are not sorted ascending are appended to `unsorted_list`.
__global__ void __launch_bounds__(kThreads) check_kernel(DevGraph g, int *unsorted_list,
                                                         int *unsorted_n)
{
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

// On sorted lists: no self-loop, no repeated neighbour, and v in N(u) for every u in N(v).
__global__ void __launch_bounds__(kThreads) validate_kernel(DevGraph g)
{
    const int lane = threadIdx.x & 31;
    const int warps = gridDim.x * (blockDim.x >> 5);
    for (int v = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; v < g.n; v += warps) {
        const int lo = g.offs[v], hi = g.offs[v + 1];
        bool not_simple = false, asym = false;
        for (int i = lo + lane; i < hi; i += 32) {
            const int u = g.adj[i];
            not_simple |= (u == v) || (i > lo && g.adj[i - 1] == u);
            const int ulo = g.offs[u];
            asym |= !sorted_contains(g.adj + ulo, g.offs[u + 1] - ulo, v);
        }
        if (__any_sync(0xffffffffu, not_simple)) {
            if (lane == 0) set_status(g.ctrl, MCE_ERR_NOT_SIMPLE);
        } else if (__any_sync(0xffffffffu, asym)) {
            if (lane == 0) set_status(g.ctrl, MCE_ERR_NOT_SYMMETRIC);
        }
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

cudaError_t launch_ingest_check(const DevGraph &g, int *d_unsorted_list, int *d_unsorted_n,
                                cudaStream_t s)
{
    if (g.n == 0) return cudaSuccess;
    check_kernel<<<grid_for(g.n, kThreads / 32), kThreads, 0, s>>>(g, d_unsorted_list,
                                                                   d_unsorted_n);
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

cudaError_t launch_ingest_validate(const DevGraph &g, cudaStream_t s)
{
    if (g.n == 0) return cudaSuccess;
    validate_kernel<<<grid_for(g.n, kThreads / 32), kThreads, 0, s>>>(g);
    return cudaGetLastError();
}

}  // namespace mce
