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

// ---- offsets of the records of subtrees built ahead (a 64-bit exclusive scan of their sizes)

constexpr int kRecThreads = 256;   // 4 places per thread: kScanBlock places per CTA

// Record size (quads) of the root at place i: roots of the launch groups of row width 1, 2
// and 4 words (groups 0 .. 5) have one.
__device__ __forceinline__ long long record_quads(const DevGraph &g, const int *roots,
                                                  const int *range, int i)
{
    for (int gi = 0; gi < 6; ++gi) {
        const int k = gi / 2;
        if (i >= range[2 * gi] && i < range[2 * gi + 1]) {
            const int v = roots[i];
            const int np = g.pcount[v];
            if (np <= 0 || np > kMaxP) return 0;
            return rec_quads(g.offs[v + 1] - g.offs[v], np, 1 << k);
        }
    }
    return 0;
}

__device__ __forceinline__ long long block_excl_scan_ll(long long v, long long *total,
                                                        long long *sh)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    long long inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) sh[w] = inc;
    __syncthreads();
    long long before = 0, t = 0;
    for (int j = 0; j < nw; ++j) {
        const long long c = sh[j];
        if (j < w) before += c;
        t += c;
    }
    __syncthreads();
    *total = t;
    return before + inc - v;
}

__global__ void __launch_bounds__(kRecThreads) rec_partial_kernel(DevGraph g, const int *roots,
                                                                  const int *range, int n,
                                                                  long long *sums)
{
    __shared__ long long sh[32];
    const int base = blockIdx.x * kScanBlock + threadIdx.x * 4;
    long long v = 0;
    for (int j = 0; j < 4; ++j)
        if (base + j < n) v += record_quads(g, roots, range, base + j);
    long long tot;
    block_excl_scan_ll(v, &tot, sh);
    if (threadIdx.x == 0) sums[blockIdx.x] = tot;
}

__global__ void __launch_bounds__(1024) rec_sums_kernel(long long *sums, int nb)
{
    __shared__ long long sh[32];
    long long carry = 0;
    for (int c0 = 0; c0 < nb; c0 += blockDim.x) {
        const int i = c0 + threadIdx.x;
        const long long v = i < nb ? sums[i] : 0;
        long long tot;
        const long long ex = block_excl_scan_ll(v, &tot, sh);
        if (i < nb) sums[i] = carry + ex;
        carry += tot;
    }
}

__global__ void __launch_bounds__(kRecThreads) rec_final_kernel(DevGraph g, const int *roots,
                                                                const int *range, int n,
                                                                const long long *sums,
                                                                long long *out)
{
    __shared__ long long sh[32];
    const int base = blockIdx.x * kScanBlock + threadIdx.x * 4;
    long long x[4], v = 0;
    for (int j = 0; j < 4; ++j) {
        x[j] = base + j < n ? record_quads(g, roots, range, base + j) : 0;
        v += x[j];
    }
    long long tot;
    long long run = sums[blockIdx.x] + block_excl_scan_ll(v, &tot, sh);
    for (int j = 0; j < 4; ++j) {
        if (base + j < n) out[base + j] = run;
        run += x[j];
        if (base + j == n - 1) out[n] = run;
    }
}

}  // namespace

// Kernel instances, one translation unit per variant (built in parallel): full or partial
// induced subgraphs, first- or second-level subtrees.
const void *search_kernel_full(int cls, bool big);
const void *search_kernel_partial(int cls, bool big);
const void *search_kernel_full_l2(int cls, bool big);
const void *search_kernel_partial_l2(int cls, bool big);

const void *search_kernel_full_rec(int cls, bool big);

static const void *search_kernel_ptr(int cls, int ip, int l2, bool big)
{
    if (l2) return ip ? search_kernel_partial_l2(cls, big) : search_kernel_full_l2(cls, big);
    return ip ? search_kernel_partial(cls, big) : search_kernel_full(cls, big);
}

// Does launch group `group` have a variant that searches subtrees built ahead?
static bool has_rec_variant(int group, int ip, int l2)
{
    return !ip && !l2 && group / 2 <= 2;
}

cudaError_t search_configure(int cls, int ip, int l2, size_t smem)
{
    for (int big = 0; big < 2; ++big) {
        const cudaError_t e = cudaFuncSetAttribute(search_kernel_ptr(cls, ip, l2, big != 0),
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)smem);
        if (e != cudaSuccess) return e;
    }
    for (int big = 0; big < 2 && has_rec_variant(2 * cls + 1, ip, l2); ++big) {
        const cudaError_t e = cudaFuncSetAttribute(search_kernel_full_rec(cls, big != 0),
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)smem);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t search_occupancy(int group, int ip, int l2, int threads, size_t smem,
                             int *blocks_per_sm)
{
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        blocks_per_sm, search_kernel_ptr(group / 2, ip, l2, (group & 1) == 0), threads, smem);
    if (e != cudaSuccess || !has_rec_variant(group, ip, l2)) return e;
    // one geometry serves both variants
    int rec = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &rec, search_kernel_full_rec(group / 2, (group & 1) == 0), threads, smem);
    if (rec < *blocks_per_sm) *blocks_per_sm = rec;
    return e;
}

cudaError_t launch_search(const SearchArgs &a, int blocks, int threads, size_t smem, bool rec,
                          cudaStream_t s)
{
    SearchArgs aa = a;
    void *args[] = {&aa};
    const void *k = rec && has_rec_variant(a.group, a.g.ip, a.g.l2)
                        ? search_kernel_full_rec(a.cls, (a.group & 1) == 0)
                        : search_kernel_ptr(a.cls, a.g.ip, a.g.l2, (a.group & 1) == 0);
    return cudaLaunchKernel(k, dim3(blocks), dim3(threads), args, smem, s);
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

cudaError_t launch_record_offsets(const DevGraph &g, const int *roots, const int *range,
                                  int n_slots, long long *scan_tmp, long long *rec_off,
                                  cudaStream_t s)
{
    cudaError_t e = cudaMemsetAsync(rec_off, 0, sizeof(long long), s);
    if (e != cudaSuccess || n_slots == 0) return e;
    const int nb = (n_slots + kScanBlock - 1) / kScanBlock;
    rec_partial_kernel<<<nb, kRecThreads, 0, s>>>(g, roots, range, n_slots, scan_tmp);
    rec_sums_kernel<<<1, 1024, 0, s>>>(scan_tmp, nb);
    rec_final_kernel<<<nb, kRecThreads, 0, s>>>(g, roots, range, n_slots, scan_tmp, rec_off);
    return cudaGetLastError();
}

cudaError_t build_occupancy(int cls, int *blocks_per_sm)
{
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        blocks_per_sm, build_kernel_full(cls), kBuildThreads,
        (size_t)(kBuildThreads / 32) * build_smem_per_warp(cls));
}

cudaError_t launch_build(const SearchArgs &a, int blocks, cudaStream_t s)
{
    SearchArgs aa = a;
    void *args[] = {&aa};
    return cudaLaunchKernel(build_kernel_full(a.cls), dim3(blocks), dim3(kBuildThreads), args,
                            (size_t)(kBuildThreads / 32) * build_smem_per_warp(a.cls), s);
}

}  // namespace mce
