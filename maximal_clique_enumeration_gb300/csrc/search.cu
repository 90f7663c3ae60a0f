// Host side of the search: launches, and the small kernels around it (worker-list reset,
// result finalisation, enumeration layout).  The search kernels themselves are in
// search_impl.cuh, instantiated by search_full.cu and search_partial.cu.
#include "mce_internal.cuh"

namespace mce {

namespace {

// Before each launch: empty worker list (slot i expects push number i) and fresh counters.
__global__ void search_prep_kernel(unsigned *seq, int n, DevCtrl *ctrl)
{
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    for (int i = t; i < n; i += gridDim.x * blockDim.x) seq[i] = (unsigned)i;
    if (t == 0) {
        ctrl->next_root = 0ULL;
        ctrl->busy = 0;
        ctrl->ring_head = 0;
        ctrl->ring_tail = 0;
    }
}

// Output: d_out = [count, hash, hist[0..hist_len)], adding the isolated vertices when the
// search skipped them (full-graph count).
__global__ void finalize_kernel(DevGraph g, DevOut o, unsigned long long *d_out,
                                int include_isolated)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const unsigned long long iso = include_isolated ? (unsigned long long)g.ctrl->n_iso : 0ULL;
    if (i == 0) {
        d_out[0] = g.ctrl->result[0] + iso;
        d_out[1] = g.ctrl->result[1] + (include_isolated ? g.ctrl->iso_hash : 0ULL);
    }
    if (i < o.hist_len) d_out[2 + i] = o.hist[i] + (i == 1 ? iso : 0ULL);
}

// Enumeration layout from a count: cliques grouped by size, in ascending size.
__global__ void enum_layout_kernel(const unsigned long long *counts, int hist_len,
                                   long long *region_ids, long long *region_cl,
                                   unsigned long long *cursor, long long *totals)
{
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    long long ids = 0, cl = 0;
    for (int k = 0; k < hist_len; ++k) {
        region_ids[k] = ids;
        region_cl[k] = cl;
        cursor[k] = 0ULL;
        const long long c = (long long)counts[2 + k];
        cl += c;
        ids += c * k;
    }
    region_ids[hist_len] = ids;
    region_cl[hist_len] = cl;
    totals[0] = cl;
    totals[1] = ids;
}

// Isolated vertices (skipped by the full-graph search) as cliques of size 1.
__global__ void enum_isolated_kernel(DevGraph g, DevOut o)
{
    for (int v = blockIdx.x * blockDim.x + threadIdx.x; v < g.n; v += gridDim.x * blockDim.x) {
        if (g.offs[v + 1] != g.offs[v]) continue;
        const unsigned long long slot = atomicAdd(&o.cursor[1], 1ULL);
        const long long cl = o.region_cl[1] + (long long)slot;
        if (cl >= o.region_cl[2]) {
            set_status(g.ctrl, MCE_ERR_BUFFER_TOO_SMALL);
            continue;
        }
        const long long base = o.region_ids[1] + (long long)slot;
        o.offsets[cl] = base;
        o.ids[base] = v;
    }
}

__global__ void enum_close_kernel(DevOut o, const long long *totals)
{
    if (threadIdx.x == 0 && blockIdx.x == 0) o.offsets[totals[0]] = totals[1];
}

}  // namespace

// Kernel instances, one translation unit per variant (built in parallel): full or partial
// induced subgraphs, first- or second-level subtrees.
const void *search_kernel_full(int cls, bool big);
const void *search_kernel_partial(int cls, bool big);
const void *search_kernel_full_l2(int cls, bool big);
const void *search_kernel_partial_l2(int cls, bool big);

static const void *search_kernel_ptr(int cls, int ip, int l2, bool big)
{
    if (l2) return ip ? search_kernel_partial_l2(cls, big) : search_kernel_full_l2(cls, big);
    return ip ? search_kernel_partial(cls, big) : search_kernel_full(cls, big);
}

cudaError_t search_configure(int cls, int ip, int l2, size_t smem)
{
    for (int big = 0; big < 2; ++big) {
        const cudaError_t e = cudaFuncSetAttribute(search_kernel_ptr(cls, ip, l2, big != 0),
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)smem);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t search_occupancy(int group, int ip, int l2, int threads, size_t smem,
                             int *blocks_per_sm)
{
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        blocks_per_sm, search_kernel_ptr(group / 2, ip, l2, (group & 1) == 0), threads, smem);
}

cudaError_t launch_search(const SearchArgs &a, int blocks, int threads, size_t smem,
                          cudaStream_t s)
{
    SearchArgs aa = a;
    void *args[] = {&aa};
    return cudaLaunchKernel(search_kernel_ptr(a.cls, a.g.ip, a.g.l2, (a.group & 1) == 0),
                            dim3(blocks), dim3(threads), args, smem, s);
}

cudaError_t launch_search_prep(const SearchArgs &a, cudaStream_t s)
{
    const int n = a.n_workers > 0 ? a.n_workers : 1;
    search_prep_kernel<<<(n + 255) / 256, 256, 0, s>>>(a.ring_seq, n, a.g.ctrl);
    return cudaGetLastError();
}

cudaError_t launch_finalize(const DevGraph &g, const DevOut &o, unsigned long long *d_out,
                            int include_isolated, cudaStream_t s)
{
    const int n = o.hist_len > 1 ? o.hist_len : 1;
    finalize_kernel<<<(n + 255) / 256, 256, 0, s>>>(g, o, d_out, include_isolated);
    return cudaGetLastError();
}

cudaError_t launch_enum_layout(const DevGraph &g, const unsigned long long *d_counts,
                               int hist_len, long long *region_ids, long long *region_cl,
                               unsigned long long *cursor, long long *d_totals, cudaStream_t s)
{
    (void)g;
    enum_layout_kernel<<<1, 32, 0, s>>>(d_counts, hist_len, region_ids, region_cl, cursor,
                                        d_totals);
    return cudaGetLastError();
}

cudaError_t launch_enum_isolated(const DevGraph &g, const DevOut &o, cudaStream_t s)
{
    if (g.n == 0) return cudaSuccess;
    int b = (g.n + 255) / 256;
    if (b > 4096) b = 4096;
    enum_isolated_kernel<<<b, 256, 0, s>>>(g, o);
    return cudaGetLastError();
}

cudaError_t launch_enum_close(const DevOut &o, const long long *d_totals, cudaStream_t s)
{
    enum_close_kernel<<<1, 32, 0, s>>>(o, d_totals);
    return cudaGetLastError();
}

}  // namespace mce
