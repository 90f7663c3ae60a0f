// Host side of the C ABI declared in include/mce.h.
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <initializer_list>
#include <mutex>
#include <new>
#include <vector>

#include "mce_internal.cuh"

using namespace mce;

struct mce_graph {
    int device = 0;
    int n = 0;
    long long nnz = 0;
    mce_config cfg{};
    int sm_count = 0;
    int peel_blocks = 0;
    int search_threads = 0, n_workers = 0;
    int build_blocks[3] = {};  // CTAs of the build launches of row width 1, 2, 4 words
    // per launch group g = 2k + b (row width 1 << k; b = 0 big-workspace roots, 1 the rest)
    int grp_blocks[kNumGroups] = {}, grp_workers[kNumGroups] = {}, grp_count[kNumGroups] = {};
    unsigned long long grp_ws[kNumGroups] = {};
    size_t cls_smem[kNumClasses] = {};
    long long uroots_cap = 0;
    int n_uroots = 0;         // length of the caller's root list of the current call
    int small_lo = 1, small_hi = kSmallP;     // |P| range of the nodes solved whole
    bool records = true;      // build the subtrees of narrow roots ahead of the search
    int record_mask = 7;      // of the row widths 1, 2, 4 words (bits 0, 1, 2)
    unsigned *bb = nullptr;   // their records (bb_quads quads) and offsets by schedule place
    long long bb_quads = 0;
    long long *rec_off = nullptr, *rec_scan = nullptr;
    long long *urec_off = nullptr, *urec_scan = nullptr;   // the same for a caller's roots
    // the builds run on a stream of the handle's own, forked from the caller's stream, so that
    // the build of a narrower group overlaps the search of the wider ones
    cudaStream_t side = nullptr;
    cudaEvent_t ev_fork = nullptr, ev_join = nullptr, ev_built[6] = {};   // per launch group
    bool unit_own = false;    // unit_cnt / unit_scan were reallocated for a caller's root list
    int degeneracy = 0, max_degree = 0, hist_len = 2, rounds = 0;
    unsigned long long ws_words = 0;
    std::vector<void *> allocs;
    cudaStream_t alloc_stream = nullptr;   // stream the next allocations are ordered on
    DevGraph g{};
    unsigned long long *hist_acc = nullptr;     // [hist_len]
    unsigned int *ws = nullptr;
    int *ring = nullptr, *flag = nullptr;
    unsigned *ring_seq = nullptr;
    long long *region_ids = nullptr, *region_cl = nullptr, *totals = nullptr;
    unsigned long long *cursor = nullptr;
    unsigned long long *count_cache = nullptr;  // [2 + hist_len], full-graph count
    unsigned long long *roots_count = nullptr;  // [2 + hist_len], count of a root batch
    bool count_cache_valid = false;
    // profiling: events around the order and around each class launch
    cudaEvent_t ev_order[3] = {nullptr, nullptr, nullptr};   // start, end, after the peel
    cudaEvent_t ev_grp[kNumGroups][2] = {};
    bool grp_timed[kNumGroups] = {};
    cudaEvent_t ev_bld[6][2] = {};               // around the build launches (groups 0 .. 5)
    bool bld_timed[6] = {};
    bool order_timed = false;
    int launches_order = 0, launches_count = 0;
};

namespace {

mce_status from_cuda(cudaError_t e)
{
    if (e == cudaSuccess) return MCE_OK;
    if (e == cudaErrorMemoryAllocation) return MCE_ERR_OUT_OF_MEMORY;
    return MCE_ERR_CUDA;
}

#define MCE_TRY(expr)                                        \
    do {                                                     \
        mce_status _st = from_cuda(expr);                    \
        if (_st != MCE_OK) return _st;                       \
    } while (0)

// Device memory comes from one stream-ordered pool per device, owned by the library, that keeps
// freed memory instead of returning it to the driver: a handle created after another one was
// destroyed reuses its memory without a cudaMalloc / cudaFree round trip each time.
constexpr int kMaxDevices = 64;
cudaMemPool_t g_pool[kMaxDevices];
std::mutex g_pool_lock;

cudaMemPool_t device_pool(int device)
{
    if (device < 0 || device >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_pool_lock);
    if (!g_pool[device]) {
        cudaMemPoolProps props{};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = device;
        cudaMemPool_t pool = nullptr;
        if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        uint64_t keep = UINT64_MAX;
        cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
        g_pool[device] = pool;
    }
    return g_pool[device];
}

template <typename T>
mce_status dev_alloc(mce_graph *h, T **p, size_t count)
{
    void *q = nullptr;
    const size_t bytes = count * sizeof(T) > 0 ? count * sizeof(T) : 16;
    cudaMemPool_t pool = device_pool(h->device);
    // ordered on the stream of the call that allocates; that call synchronises it or uses the
    // memory on it before any other stream can
    cudaError_t e = pool ? cudaMallocFromPoolAsync(&q, bytes, pool, h->alloc_stream)
                         : cudaMalloc(&q, bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *p = nullptr;
        return MCE_ERR_OUT_OF_MEMORY;
    }
    h->allocs.push_back(q);
    *p = static_cast<T *>(q);
    return MCE_OK;
}

#define MCE_ALLOC(h, p, count)                               \
    do {                                                     \
        mce_status _st = dev_alloc((h), &(p), (count));      \
        if (_st != MCE_OK) return _st;                       \
    } while (0)

mce_status read_status(mce_graph *h, cudaStream_t s)
{
    int st = 0;
    MCE_TRY(cudaMemcpyAsync(&st, &h->g.ctrl->status, sizeof(int), cudaMemcpyDeviceToHost, s));
    MCE_TRY(cudaStreamSynchronize(s));
    return (mce_status)st;
}

// Makes the handle's device current for the lifetime of this object (and restores the caller's
// device afterwards), so that synchronisation and frees act on the device that owns the memory.
struct OnDevice {
    int saved = -1;
    explicit OnDevice(int device)
    {
        if (cudaGetDevice(&saved) != cudaSuccess) {
            cudaGetLastError();
            saved = -1;
        }
        if (saved != device) cudaSetDevice(device);
    }
    ~OnDevice()
    {
        int cur = -1;
        if (saved >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != saved) cudaSetDevice(saved);
        cudaGetLastError();
    }
};

// Returns one allocation of the handle to the pool (ordered on stream s) and forgets it.
void dev_free(mce_graph *h, void *p, cudaStream_t s)
{
    if (!p) return;
    for (size_t i = 0; i < h->allocs.size(); ++i) {
        if (h->allocs[i] != p) continue;
        h->allocs[i] = h->allocs.back();
        h->allocs.pop_back();
        if (device_pool(h->device)) cudaFreeAsync(p, s);
        else cudaFree(p);
        return;
    }
}

void free_all(mce_graph *h)
{
    OnDevice on(h->device);
    if (!h->allocs.empty()) {
        // no work of this handle may still be running on any stream (as cudaFree would wait)
        cudaDeviceSynchronize();
        cudaGetLastError();
        for (void *p : h->allocs) {
            if (device_pool(h->device)) cudaFreeAsync(p, 0);
            else cudaFree(p);
        }
        cudaStreamSynchronize(0);
        cudaGetLastError();
    }
    h->allocs.clear();
    for (int i = 0; i < 3; ++i)
        if (h->ev_order[i]) cudaEventDestroy(h->ev_order[i]);
    for (int k = 0; k < kNumGroups; ++k)
        for (int i = 0; i < 2; ++i)
            if (h->ev_grp[k][i]) cudaEventDestroy(h->ev_grp[k][i]);
    for (cudaEvent_t e : {h->ev_fork, h->ev_join})
        if (e) cudaEventDestroy(e);
    for (int gi = 0; gi < 6; ++gi)
        for (cudaEvent_t e : {h->ev_built[gi], h->ev_bld[gi][0], h->ev_bld[gi][1]})
            if (e) cudaEventDestroy(e);
    if (h->side) cudaStreamDestroy(h->side);
    h->side = nullptr;
}

// Resets the per-search accumulators of the control block.
mce_status reset_search(mce_graph *h, cudaStream_t s)
{
    DevCtrl *c = h->g.ctrl;
    MCE_TRY(cudaMemsetAsync(&c->tree_nodes, 0, 4 * sizeof(unsigned long long), s));
    MCE_TRY(cudaMemsetAsync(c->words, 0, sizeof(c->words), s));
    MCE_TRY(cudaMemsetAsync(c->prof, 0, sizeof(c->prof), s));
    MCE_TRY(cudaMemsetAsync(h->g.prof_sm, 0, sizeof(unsigned long long) * kNumClasses * kProfSms,
                            s));
    for (int k = 0; k < kNumGroups; ++k) h->grp_timed[k] = false;
    for (int gi = 0; gi < 6; ++gi) h->bld_timed[gi] = false;
    MCE_TRY(cudaMemsetAsync(h->hist_acc, 0, sizeof(unsigned long long) * h->hist_len, s));
    return MCE_OK;
}

// One launch per row-width class, widest first: the prep kernel empties the worker list and
// the counters, then the persistent search kernel of that class runs.
mce_status run_search(mce_graph *h, cudaStream_t s, bool user_roots, const DevOut *enum_out)
{
    mce_status st = reset_search(h, s);
    if (st != MCE_OK) return st;
    SearchArgs a{};
    a.g = h->g;
    a.out.hist = h->hist_acc;
    a.out.hist_len = h->hist_len;
    if (enum_out) {
        a.out = *enum_out;
        a.out.hist = h->hist_acc;
        a.out.hist_len = h->hist_len;
    }
    a.roots = user_roots ? h->g.uroots : h->g.sched;
    a.range = user_roots ? h->g.ctrl->ucls : h->g.ctrl->cls;
    a.uoff = user_roots ? h->g.uroots_uoff : h->g.sched_uoff;
    a.ws = h->ws;
    a.ring = h->ring;
    a.ring_seq = h->ring_seq;
    a.flag = h->flag;
    a.worker_list = h->cfg.worker_list;
    a.donate_min_p = h->cfg.donate_min_p;
    a.donate_rule = h->cfg.donate_rule;
    a.spin_limit_ns = h->cfg.spin_limit_ns;
    a.small_lo = h->small_lo;
    a.small_hi = h->small_hi;
    if (h->bb) {
        a.bb = h->bb;
        a.bb_quads = h->bb_quads;
        a.rec_off = user_roots ? h->urec_off : h->rec_off;
    }
    // roots of row width <= 4 words: subtrees built ahead when the records fit (the
    // schedule's always do; a caller's list is checked on the device, and the plain search
    // launch after the record search does the work when they do not)
    auto launched = [&](int gi) {
        return h->grp_workers[gi] != 0 && (user_roots || h->grp_count[gi] != 0);
    };
    auto with_records = [&](int gi) {
        const int k = gi / 2;
        return a.bb != nullptr && k <= 2 && ((h->record_mask >> k) & 1) &&
               launched(gi);
    };
    const long long *gate = a.bb ? a.rec_off + (user_roots ? h->n_uroots : h->n) : nullptr;
    // launch order: widest rows first, per width the big-workspace group first, except where
    // both groups of a width search records: then the normal group goes first (its build is
    // the long one; the big group's, the covering tests of a few hubs, overlaps its search)
    int order[kNumGroups];
    for (int o = 0; o < kNumGroups; ++o) order[o] = group_at(o);
    for (int o = 0; o + 1 < kNumGroups; o += 2)
        if (with_records(order[o]) && with_records(order[o + 1])) {
            const int t = order[o];
            order[o] = order[o + 1];
            order[o + 1] = t;
        }
    bool forked = false;
    if (h->side) {
        // all builds on the side stream, in the order of the searches
        for (int o = 0; o < kNumGroups; ++o) {
            const int gi = order[o], k = gi / 2;
            if (!with_records(gi)) continue;
            if (!forked) {
                MCE_TRY(cudaEventRecord(h->ev_fork, s));
                MCE_TRY(cudaStreamWaitEvent(h->side, h->ev_fork, 0));
                forked = true;
            }
            SearchArgs b = a;
            b.cls = k;
            b.group = gi;
            b.rec_gate = gate;
            if (h->cfg.profile) MCE_TRY(cudaEventRecord(h->ev_bld[gi][0], h->side));
            MCE_TRY(launch_build(b, h->build_blocks[k], h->side));
            if (h->cfg.profile) {
                MCE_TRY(cudaEventRecord(h->ev_bld[gi][1], h->side));
                h->bld_timed[gi] = true;
            }
            MCE_TRY(cudaEventRecord(h->ev_built[gi], h->side));
        }
        if (forked) MCE_TRY(cudaEventRecord(h->ev_join, h->side));
    }
    for (int o = 0; o < kNumGroups; ++o) {
        const int gi = order[o], k = gi / 2;
        if (!launched(gi)) continue;                      // no root of the call in this group
        a.cls = k;
        a.group = gi;
        a.ws_words = h->grp_ws[gi];
        a.n_workers = h->grp_workers[gi];
        MCE_TRY(cudaMemsetAsync(h->flag, 0, sizeof(int) * (size_t)a.n_workers, s));
        MCE_TRY(launch_search_prep(a, s));
        const bool rec = with_records(gi);
        a.rec_gate = rec ? gate : nullptr;
        if (rec) {
            if (forked) {
                MCE_TRY(cudaStreamWaitEvent(s, h->ev_built[gi], 0));
            } else {
                if (h->cfg.profile) MCE_TRY(cudaEventRecord(h->ev_bld[gi][0], s));
                MCE_TRY(launch_build(a, h->build_blocks[k], s));
                if (h->cfg.profile) {
                    MCE_TRY(cudaEventRecord(h->ev_bld[gi][1], s));
                    h->bld_timed[gi] = true;
                }
            }
        }
        if (h->cfg.profile) MCE_TRY(cudaEventRecord(h->ev_grp[gi][0], s));
        if (rec) {
            MCE_TRY(launch_search(a, h->grp_blocks[gi], h->search_threads, h->cls_smem[k], true,
                                  s));
            h->launches_count += user_roots ? 2 : 1;   // build (+ the plain search launch)
        }
        if (!rec || user_roots)
            MCE_TRY(launch_search(a, h->grp_blocks[gi], h->search_threads, h->cls_smem[k],
                                  false, s));
        if (h->cfg.profile) {
            MCE_TRY(cudaEventRecord(h->ev_grp[gi][1], s));
            h->grp_timed[gi] = true;
        }
        h->launches_count += 2;                           // prep and search
    }
    if (forked) MCE_TRY(cudaStreamWaitEvent(s, h->ev_join, 0));
    return MCE_OK;
}

}  // namespace

extern "C" {

mce_status mce_config_default(mce_config *cfg)
{
    if (!cfg) return MCE_ERR_INVALID_ARG;
    cfg->worker_list = 1;
    cfg->donate_min_p = 10;
    cfg->warps_per_block = kDefaultWarpsPerBlock;
    cfg->blocks_per_sm = 0;
    cfg->profile = 0;
    cfg->donate_rule = 0;
    cfg->spin_limit_ns = 20LL * 1000 * 1000 * 1000;
    cfg->induced = 0;
    cfg->subtree_level = 1;
    cfg->overlap_builds = 1;
    return MCE_OK;
}

const char *mce_status_str(mce_status s)
{
    switch (s) {
    case MCE_OK: return "ok";
    case MCE_ERR_INVALID_ARG: return "invalid argument";
    case MCE_ERR_NOT_SIMPLE: return "graph is not simple (self-loop or repeated neighbour)";
    case MCE_ERR_NOT_SYMMETRIC: return "graph is not symmetric";
    case MCE_ERR_ID_RANGE: return "vertex id out of range";
    case MCE_ERR_OUT_OF_MEMORY: return "out of memory";
    case MCE_ERR_BUFFER_TOO_SMALL: return "output buffer too small";
    case MCE_ERR_DEVICE_TIMEOUT: return "device-side wait exceeded the spin limit";
    case MCE_ERR_LIMIT: return "graph exceeds a size limit of the library";
    case MCE_ERR_CUDA: return "CUDA error";
    case MCE_ERR_INTERNAL: return "internal consistency check failed on the device";
    }
    return "unknown status";
}

static mce_status order_impl(mce_graph *h, cudaStream_t s);

static mce_status create_impl(mce_graph *h, const int32_t *offsets, const int32_t *adj, int32_t n,
                              int is_device_ptr, cudaStream_t s)
{
    MCE_TRY(cudaGetDevice(&h->device));
    MCE_TRY(cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, h->device));
    h->alloc_stream = s;
    h->n = n;
    // offsets[0] and offsets[n] (= number of adjacency entries)
    int first = 0, last = 0;
    const cudaMemcpyKind k = is_device_ptr ? cudaMemcpyDeviceToHost : cudaMemcpyHostToHost;
    MCE_TRY(cudaMemcpy(&first, offsets, sizeof(int), k));
    MCE_TRY(cudaMemcpy(&last, offsets + n, sizeof(int), k));
    if (first != 0 || last < 0 || (last > 0 && !adj)) return MCE_ERR_INVALID_ARG;
    h->nnz = last;

    DevGraph &g = h->g;
    int *offs = nullptr, *adjm = nullptr;
    MCE_ALLOC(h, offs, (size_t)n + 1);
    MCE_ALLOC(h, adjm, (size_t)h->nnz);
    MCE_ALLOC(h, g.ctrl, 1);
    MCE_TRY(cudaMemsetAsync(g.ctrl, 0, sizeof(DevCtrl), s));
    const cudaMemcpyKind kin = is_device_ptr ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice;
    MCE_TRY(cudaMemcpyAsync(offs, offsets, sizeof(int) * ((size_t)n + 1), kin, s));
    if (h->nnz) MCE_TRY(cudaMemcpyAsync(adjm, adj, sizeof(int) * (size_t)h->nnz, kin, s));
    g.n = n;
    g.nnz = h->nnz;
    g.offs = offs;
    g.adj = adjm;

    // input checks: offsets, id range, sortedness
    // (stats: unsorted lists, long lists, largest degree; fb: forward and backward entries)
    int *d_list = nullptr, *d_stats = nullptr, *d_big = nullptr;
    unsigned long long *d_fb = nullptr;
    MCE_ALLOC(h, d_list, (size_t)n + 1);
    MCE_ALLOC(h, d_big, (size_t)n + 1);
    MCE_ALLOC(h, d_stats, 4);
    MCE_ALLOC(h, d_fb, 2);
    MCE_TRY(cudaMemsetAsync(d_stats, 0, 4 * sizeof(int), s));
    MCE_TRY(cudaMemsetAsync(d_fb, 0, 2 * sizeof(unsigned long long), s));
    MCE_TRY(launch_ingest_check(g, d_list, d_stats, d_big, s));
    mce_status st = read_status(h, s);
    if (st != MCE_OK) return st;
    int stats[4] = {0, 0, 0, 0};
    MCE_TRY(cudaMemcpy(stats, d_stats, sizeof(stats), cudaMemcpyDeviceToHost));
    const int n_unsorted = stats[0];
    if (n_unsorted > 0) {
        MCE_TRY(launch_ingest_sort(g, adjm, d_list, n_unsorted, nullptr, 0, s));
        std::vector<int> list(n_unsorted), hoffs((size_t)n + 1);
        MCE_TRY(cudaMemcpy(list.data(), d_list, sizeof(int) * n_unsorted, cudaMemcpyDeviceToHost));
        MCE_TRY(cudaMemcpy(hoffs.data(), offs, sizeof(int) * ((size_t)n + 1),
                           cudaMemcpyDeviceToHost));
        int *scratch = nullptr;
        long long scratch_len = 0;
        for (int v : list) {
            const long long len = hoffs[v + 1] - hoffs[v];
            if (len <= 4096) continue;
            long long p2 = 1;
            while (p2 < len) p2 <<= 1;
            if (p2 > scratch_len) {
                MCE_ALLOC(h, scratch, (size_t)p2);
                scratch_len = p2;
            }
            MCE_TRY(launch_ingest_sort_large(g, adjm, v, scratch, s));
        }
    }
    MCE_TRY(launch_ingest_validate(g, d_big, stats[1], stats[2], d_fb, s));
    st = read_status(h, s);
    if (st != MCE_OK) return st;
    unsigned long long fb[2] = {0ULL, 0ULL};
    MCE_TRY(cudaMemcpy(fb, d_fb, sizeof(fb), cudaMemcpyDeviceToHost));
    if (fb[0] != fb[1]) return MCE_ERR_NOT_SYMMETRIC;

    // degeneracy order buffers
    MCE_ALLOC(h, g.rank, (size_t)n);
    MCE_ALLOC(h, g.core, (size_t)n);
    MCE_ALLOC(h, g.round_of, (size_t)n);
    MCE_ALLOC(h, g.order, (size_t)n);
    MCE_ALLOC(h, g.pcount, (size_t)n);
    MCE_ALLOC(h, g.sched, (size_t)n);
    MCE_ALLOC(h, g.deg, (size_t)n);
    MCE_ALLOC(h, g.alive_a, (size_t)n);
    MCE_ALLOC(h, g.alive_b, (size_t)n);
    MCE_ALLOC(h, g.bucket, (size_t)kNumBuckets);
    MCE_ALLOC(h, g.padj, (size_t)(h->nnz > 0 ? h->nnz : 1));
    int coop = 0;
    MCE_TRY(cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, h->device));
    if (!coop) return MCE_ERR_CUDA;
    h->peel_blocks = h->sm_count;
    MCE_ALLOC(h, g.blk_cnt, (size_t)2 * h->peel_blocks);
    MCE_ALLOC(h, g.blk_min, (size_t)2 * h->peel_blocks);
    MCE_ALLOC(h, g.blk_cm, (size_t)2 * h->peel_blocks);
    MCE_ALLOC(h, g.blk_rd, (size_t)h->peel_blocks);
    MCE_ALLOC(h, g.blk_gone, (size_t)2 * h->peel_blocks);
    MCE_ALLOC(h, g.front, (size_t)3 * kFrontCap);
    MCE_ALLOC(h, g.rstart, (size_t)n + 1);
    if (h->cfg.profile) {
        for (int i = 0; i < 3; ++i) MCE_TRY(cudaEventCreate(&h->ev_order[i]));
        for (int k = 0; k < kNumGroups; ++k) {
            MCE_TRY(cudaEventCreate(&h->ev_grp[k][0]));
            MCE_TRY(cudaEventCreate(&h->ev_grp[k][1]));
        }
        for (int gi = 0; gi < 6; ++gi) {
            MCE_TRY(cudaEventCreate(&h->ev_bld[gi][0]));
            MCE_TRY(cudaEventCreate(&h->ev_bld[gi][1]));
        }
    }
    g.ip = h->cfg.induced == 2 ? 1 : 0;
    g.l2 = h->cfg.subtree_level == 2 ? 1 : 0;
    // second-level subtrees are counted in int32 prefixes: at most one per edge and vertex
    if (g.l2 && (long long)n + h->nnz / 2 >= (1LL << 31)) return MCE_ERR_LIMIT;
    if (g.l2) {
        MCE_ALLOC(h, g.unit_cnt, (size_t)n + 1);
        MCE_ALLOC(h, g.sched_uoff, (size_t)n + 1);
        MCE_ALLOC(h, g.unit_scan, (size_t)n / kScanBlock + 2);
    }
    {
        mce_status so = order_impl(h, s);
        if (so != MCE_OK) return so;
    }
    st = read_status(h, s);
    if (st != MCE_OK) return st;
    DevCtrl c{};
    MCE_TRY(cudaMemcpy(&c, g.ctrl, sizeof(DevCtrl), cudaMemcpyDeviceToHost));
    // induced subgraphs (Section 4.5): partial when Delta / d > 200, full otherwise, unless the
    // configuration fixes one; the schedule and workspace sizes depend on it, so a change of
    // mode orders once more
    const int ip = h->cfg.induced == 2 ||
                   (h->cfg.induced == 0 && (long long)c.max_degree > 200LL * c.degeneracy);
    if (ip != g.ip) {
        g.ip = ip;
        mce_status so = order_impl(h, s);
        if (so != MCE_OK) return so;
        st = read_status(h, s);
        if (st != MCE_OK) return st;
        MCE_TRY(cudaMemcpy(&c, g.ctrl, sizeof(DevCtrl), cudaMemcpyDeviceToHost));
    }
    h->degeneracy = c.degeneracy;
    h->rounds = c.rounds;
    h->max_degree = c.max_degree;
    h->hist_len = c.degeneracy + 2;
    if (c.max_pcount > kMaxP || c.max_degree > kMaxCode) return MCE_ERR_LIMIT;

    // search kernel geometry, per row-width class: as many CTAs as can be resident
    // (Section 3.3); each warp gets a workspace for the largest root of its class
    int wpb = h->cfg.warps_per_block > 0 ? h->cfg.warps_per_block : kDefaultWarpsPerBlock;
    if (wpb > 4) wpb = 4;
    h->search_threads = 32 * wpb;
    size_t ws_total = 32;
    int group_per_sm[kNumGroups] = {};
    for (int k = 0; k < kNumClasses; ++k) {
        h->cls_smem[k] = search_smem_bytes(k, h->hist_len, wpb);
        MCE_TRY(search_configure(k, g.ip, g.l2, h->cls_smem[k]));
        for (int gi = 2 * k; gi < 2 * k + 2; ++gi) {
            MCE_TRY(search_occupancy(gi, g.ip, g.l2, h->search_threads, h->cls_smem[k],
                                     &group_per_sm[gi]));
            if (group_per_sm[gi] < 1) return MCE_ERR_CUDA;
            if (h->cfg.blocks_per_sm > 0 && h->cfg.blocks_per_sm < group_per_sm[gi])
                group_per_sm[gi] = h->cfg.blocks_per_sm;
        }
    }
    for (int k = 0; k < 3; ++k) {
        int per_sm = 0;
        MCE_TRY(build_occupancy(k, &per_sm));
        h->build_blocks[k] = (per_sm > 0 ? per_sm : 1) * h->sm_count;
    }
    for (int gi = 0; gi < kNumGroups; ++gi) {
        const bool big = (gi & 1) == 0;
        h->grp_count[gi] = c.cls[2 * gi + 1] - c.cls[2 * gi];
        // whole 128-byte lines per warp: no two warps share an L1 line of workspace
        unsigned long long need = (c.ws_grp[gi] + 31) & ~31ULL;
        if (gi == 1 && need < 32) need = 32;              // isolated roots use 1 word
        if (need == 0) continue;                          // no vertex of the graph in this group
        int blocks = group_per_sm[gi] * h->sm_count;
        if (big) {
            // as many warps as the big-workspace budget allows, at most one launch's worth
            long long warps = kBigBudgetWords / (long long)need;
            if (warps < wpb) warps = wpb;
            if (warps / wpb < blocks) blocks = (int)(warps / wpb);
        }
        h->grp_blocks[gi] = blocks;
        h->grp_workers[gi] = blocks * wpb;
        h->grp_ws[gi] = need;
        if ((size_t)h->grp_workers[gi] * need > ws_total) ws_total = (size_t)h->grp_workers[gi] * need;
        if (h->grp_workers[gi] > h->n_workers) h->n_workers = h->grp_workers[gi];
    }
    h->ws_words = ws_total;
    MCE_ALLOC(h, h->ws, ws_total);
    // subtrees built ahead of the search (full induced subgraphs of first-level subtrees): one
    // record per root of the schedule's launch groups of row width <= 4 words, when all
    // of them fit in kRecCapQuads
    if (h->records && !g.ip && !g.l2 && n > 0) {
        MCE_ALLOC(h, h->rec_off, (size_t)n + 1);
        MCE_ALLOC(h, h->rec_scan, (size_t)n / kScanBlock + 2);
        MCE_TRY(launch_record_offsets(g, g.sched, g.ctrl->cls, n, h->rec_scan, h->rec_off, s));
        long long total = 0;
        MCE_TRY(cudaMemcpyAsync(&total, h->rec_off + n, sizeof(long long),
                                cudaMemcpyDeviceToHost, s));
        MCE_TRY(cudaStreamSynchronize(s));
        // all or nothing: without room for every record the search builds every subtree
        if (total > 0 && total <= kRecCapQuads &&
            dev_alloc(h, &h->bb, (size_t)total * 4) == MCE_OK)
            h->bb_quads = total;
        else
            h->bb = nullptr;
        if (h->bb && h->cfg.overlap_builds) {
            MCE_TRY(cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking));
            for (cudaEvent_t *e : {&h->ev_fork, &h->ev_join})
                MCE_TRY(cudaEventCreateWithFlags(e, cudaEventDisableTiming));
            for (int gi = 0; gi < 6; ++gi)
                MCE_TRY(cudaEventCreateWithFlags(&h->ev_built[gi], cudaEventDisableTiming));
        }
    }
    MCE_ALLOC(h, h->ring, (size_t)h->n_workers);
    MCE_ALLOC(h, h->flag, (size_t)h->n_workers);
    MCE_ALLOC(h, h->ring_seq, (size_t)h->n_workers);
    MCE_ALLOC(h, g.ubucket, (size_t)kNumBuckets);
    MCE_ALLOC(h, g.prof_sm, (size_t)kNumClasses * kProfSms);
    MCE_ALLOC(h, h->hist_acc, (size_t)h->hist_len + 1);
    MCE_ALLOC(h, h->region_ids, (size_t)h->hist_len + 2);
    MCE_ALLOC(h, h->region_cl, (size_t)h->hist_len + 2);
    MCE_ALLOC(h, h->cursor, (size_t)h->hist_len + 1);
    MCE_ALLOC(h, h->totals, 2);
    MCE_ALLOC(h, h->count_cache, (size_t)h->hist_len + 2);
    MCE_ALLOC(h, h->roots_count, (size_t)h->hist_len + 2);
    // the allocations are ordered on s: complete them before the handle is used on any stream
    MCE_TRY(cudaStreamSynchronize(s));
    return MCE_OK;
}

mce_status mce_create(const int32_t *offsets, const int32_t *adj, int32_t n, int is_device_ptr,
                      const mce_config *cfg, void *stream, mce_graph **out)
{
    if (!out) return MCE_ERR_INVALID_ARG;
    *out = nullptr;
    if (n < 0 || !offsets) return MCE_ERR_INVALID_ARG;
    if (n >= kRoundUnsorted) return MCE_ERR_LIMIT;      // the peel marks places below 2^30
    mce_graph *h = new (std::nothrow) mce_graph();
    if (!h) return MCE_ERR_OUT_OF_MEMORY;
    if (cfg) h->cfg = *cfg;
    else mce_config_default(&h->cfg);
    if (h->cfg.donate_min_p < 1) h->cfg.donate_min_p = 1;
    if (h->cfg.induced < 0 || h->cfg.induced > 2 || h->cfg.subtree_level < 1 ||
        h->cfg.subtree_level > 2 || h->cfg.overlap_builds < 0 || h->cfg.overlap_builds > 1) {
        delete h;
        return MCE_ERR_INVALID_ARG;
    }
    if (h->cfg.spin_limit_ns <= 0) h->cfg.spin_limit_ns = 20LL * 1000 * 1000 * 1000;
#ifdef MCE_AB_ENV
    // measurement builds only: the solver's |P| range from the environment
    if (const char *e = getenv("MCE_AB_SMALL_LO")) h->small_lo = atoi(e);
    if (const char *e = getenv("MCE_AB_SMALL_HI")) h->small_hi = atoi(e);
    if (const char *e = getenv("MCE_AB_RECORDS")) h->records = atoi(e) != 0;
    if (const char *e = getenv("MCE_AB_RECORD_MASK")) h->record_mask = atoi(e);
    if (h->small_hi > kSmallPMax) h->small_hi = kSmallPMax;
#endif
    mce_status st = create_impl(h, offsets, adj, n, is_device_ptr, (cudaStream_t)stream);
    if (st != MCE_OK) {
        cudaStreamSynchronize((cudaStream_t)stream);
        cudaGetLastError();
        free_all(h);
        delete h;
        return st;
    }
    *out = h;
    return MCE_OK;
}

static mce_status order_impl(mce_graph *h, cudaStream_t s)
{
    h->count_cache_valid = false;
    MCE_TRY(cudaMemsetAsync(h->g.ctrl->peel_prof, 0, sizeof(h->g.ctrl->peel_prof), s));
    if (h->cfg.profile) MCE_TRY(cudaEventRecord(h->ev_order[0], s));
    MCE_TRY(launch_order(h->g, h->peel_blocks, h->cfg.spin_limit_ns, s,
                         h->cfg.profile && h->n > 0 ? h->ev_order[2] : nullptr));
    // the schedule places the roots of a bucket in a different order at each call: the
    // records' offsets follow it (their total does not change)
    if (h->bb)
        MCE_TRY(launch_record_offsets(h->g, h->g.sched, h->g.ctrl->cls, h->n, h->rec_scan,
                                      h->rec_off, s));
    if (h->cfg.profile) {
        MCE_TRY(cudaEventRecord(h->ev_order[1], s));
        h->order_timed = true;
    }
    // peel, its rank pass, orient count (with the split) / scan / scatter (+ subtree count and
    // its scan)
    h->launches_order = h->n > 0 ? (h->g.l2 ? 9 : 5) + (h->bb ? 3 : 0) : 0;
    return MCE_OK;
}

mce_status mce_order(mce_graph *h, void *stream)
{
    if (!h) return MCE_ERR_INVALID_ARG;
    return order_impl(h, (cudaStream_t)stream);
}

static mce_status count_impl(mce_graph *h, cudaStream_t s, const int32_t *d_roots,
                             long long n_roots, uint64_t *d_out)
{
    if (h->n == 0) {
        MCE_TRY(cudaMemsetAsync(d_out, 0, sizeof(uint64_t) * (2 + (size_t)h->hist_len), s));
        return MCE_OK;
    }
    h->launches_count = 1;                                  // finalize
    h->alloc_stream = s;
    if (d_roots) {
        h->launches_count += 3;                             // root binning
        if (n_roots > h->uroots_cap) {
            // grow geometrically, and give the replaced buffers back to the pool (in stream
            // order: work already queued on s still reads them)
            long long cap = h->uroots_cap * 2 > n_roots ? h->uroots_cap * 2 : n_roots;
            if (cap > INT32_MAX) cap = INT32_MAX;
            dev_free(h, h->g.uroots, s);
            h->g.uroots = nullptr;
            h->uroots_cap = 0;
            int *buf = nullptr;
            MCE_ALLOC(h, buf, (size_t)cap);
            h->g.uroots = buf;
            if (h->g.l2) {
                // second-level subtrees: their prefix over the caller's roots, and scan scratch
                // (the schedule's own buffers stay: mce_order uses them)
                dev_free(h, h->g.uroots_uoff, s);
                h->g.uroots_uoff = nullptr;
                if (h->unit_own) {
                    dev_free(h, h->g.unit_cnt, s);
                    dev_free(h, h->g.unit_scan, s);
                }
                const size_t len = (size_t)(cap > h->n ? cap : h->n);
                MCE_ALLOC(h, h->g.uroots_uoff, (size_t)cap + 1);
                MCE_ALLOC(h, h->g.unit_cnt, len + 1);
                MCE_ALLOC(h, h->g.unit_scan, len / kScanBlock + 2);
                h->unit_own = true;
            }
            if (h->bb) {
                // offsets of the records of the caller's roots, and their scan scratch
                dev_free(h, h->urec_off, s);
                dev_free(h, h->urec_scan, s);
                h->urec_off = h->urec_scan = nullptr;
                MCE_ALLOC(h, h->urec_off, (size_t)cap + 1);
                MCE_ALLOC(h, h->urec_scan, (size_t)cap / kScanBlock + 2);
            }
            h->uroots_cap = cap;
        }
        h->n_uroots = (int)n_roots;
        MCE_TRY(launch_bin_roots(h->g, d_roots, (int)n_roots, s));
        if (h->bb) {
            MCE_TRY(launch_record_offsets(h->g, h->g.uroots, h->g.ctrl->ucls, (int)n_roots,
                                          h->urec_scan, h->urec_off, s));
            h->launches_count += 3;
        }
        if (h->g.l2) {
            MCE_TRY(launch_unit_offsets(h->g, h->g.uroots, (int)n_roots, h->g.uroots_uoff, s));
            h->launches_count += 4;
        }
    }
    mce_status st = run_search(h, s, d_roots != nullptr, nullptr);
    if (st != MCE_OK) return st;
    DevOut o{};
    o.hist = h->hist_acc;
    o.hist_len = h->hist_len;
    MCE_TRY(launch_finalize(h->g, o, (unsigned long long *)d_out, d_roots ? 0 : 1, s));
    return MCE_OK;
}

mce_status mce_count(mce_graph *h, void *stream, uint64_t *d_out)
{
    if (!h || !d_out) return MCE_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    mce_status st = count_impl(h, s, nullptr, 0, d_out);
    if (st != MCE_OK) return st;
    MCE_TRY(cudaMemcpyAsync(h->count_cache, d_out, sizeof(uint64_t) * (2 + (size_t)h->hist_len),
                            cudaMemcpyDeviceToDevice, s));
    h->count_cache_valid = true;
    return MCE_OK;
}

mce_status mce_count_roots(mce_graph *h, void *stream, const int32_t *d_roots, int32_t n_roots,
                           uint64_t *d_out)
{
    if (!h || !d_out || n_roots < 0 || (n_roots > 0 && !d_roots)) return MCE_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (n_roots == 0) {
        MCE_TRY(cudaMemsetAsync(d_out, 0, sizeof(uint64_t) * (2 + (size_t)h->hist_len), s));
        return MCE_OK;
    }
    return count_impl(h, s, d_roots, n_roots, d_out);
}

mce_status mce_enumerate(mce_graph *h, void *stream, int32_t *d_ids, int64_t cap_ids,
                         int64_t *d_offsets, int64_t cap_cliques, int64_t *h_sizes)
{
    if (!h || !h_sizes || cap_ids < 0 || cap_cliques < 0) return MCE_ERR_INVALID_ARG;
    if ((cap_ids > 0 && !d_ids) || !d_offsets) return MCE_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (!h->count_cache_valid) {
        mce_status st = mce_count(h, stream, (uint64_t *)h->count_cache);
        if (st != MCE_OK) return st;
    }
    MCE_TRY(launch_enum_layout(h->g, h->count_cache, h->hist_len, h->region_ids, h->region_cl,
                               h->cursor, h->totals, s));
    long long tot[2] = {0, 0};
    MCE_TRY(cudaMemcpyAsync(tot, h->totals, sizeof(tot), cudaMemcpyDeviceToHost, s));
    MCE_TRY(cudaStreamSynchronize(s));
    h_sizes[0] = tot[0];
    h_sizes[1] = tot[1];
    if (tot[0] > cap_cliques || tot[1] > cap_ids) return MCE_ERR_BUFFER_TOO_SMALL;
    DevOut o{};
    o.hist = h->hist_acc;
    o.hist_len = h->hist_len;
    o.ids = d_ids;
    o.offsets = (long long *)d_offsets;
    o.region_ids = h->region_ids;
    o.region_cl = h->region_cl;
    o.cursor = h->cursor;
    if (h->n > 0) {
        mce_status st = run_search(h, s, false, &o);
        if (st != MCE_OK) return st;
        MCE_TRY(launch_enum_isolated(h->g, o, s));
    }
    MCE_TRY(launch_enum_close(o, h->totals, s));
    return MCE_OK;
}

mce_status mce_enumerate_roots(mce_graph *h, void *stream, const int32_t *d_roots,
                               int32_t n_roots, int32_t *d_ids, int64_t cap_ids,
                               int64_t *d_offsets, int64_t cap_cliques, int64_t *h_sizes)
{
    if (!h || !h_sizes || n_roots < 0 || (n_roots > 0 && !d_roots) || cap_ids < 0 ||
        cap_cliques < 0)
        return MCE_ERR_INVALID_ARG;
    if ((cap_ids > 0 && !d_ids) || !d_offsets) return MCE_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    const bool search = n_roots > 0 && h->n > 0;
    if (search) {
        mce_status st = count_impl(h, s, d_roots, n_roots, (uint64_t *)h->roots_count);
        if (st != MCE_OK) return st;
    } else {
        MCE_TRY(cudaMemsetAsync(h->roots_count, 0, sizeof(uint64_t) * (2 + (size_t)h->hist_len),
                                s));
    }
    MCE_TRY(launch_enum_layout(h->g, h->roots_count, h->hist_len, h->region_ids, h->region_cl,
                               h->cursor, h->totals, s));
    long long tot[2] = {0, 0};
    MCE_TRY(cudaMemcpyAsync(tot, h->totals, sizeof(tot), cudaMemcpyDeviceToHost, s));
    mce_status st = read_status(h, s);                  // synchronises s
    if (st != MCE_OK) return st;
    h_sizes[0] = tot[0];
    h_sizes[1] = tot[1];
    if (tot[0] > cap_cliques || tot[1] > cap_ids) return MCE_ERR_BUFFER_TOO_SMALL;
    DevOut o{};
    o.hist = h->hist_acc;
    o.hist_len = h->hist_len;
    o.ids = d_ids;
    o.offsets = (long long *)d_offsets;
    o.region_ids = h->region_ids;
    o.region_cl = h->region_cl;
    o.cursor = h->cursor;
    if (search) {
        // the roots are still binned from the counting pass
        st = run_search(h, s, true, &o);
        if (st != MCE_OK) return st;
    }
    MCE_TRY(launch_enum_close(o, h->totals, s));
    return MCE_OK;
}

mce_status mce_get_order(mce_graph *h, void *stream, int32_t *d_rank, int32_t *d_core)
{
    if (!h) return MCE_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (h->n == 0) return MCE_OK;
    if (d_rank)
        MCE_TRY(cudaMemcpyAsync(d_rank, h->g.rank, sizeof(int) * (size_t)h->n,
                                cudaMemcpyDeviceToDevice, s));
    if (d_core)
        MCE_TRY(cudaMemcpyAsync(d_core, h->g.core, sizeof(int) * (size_t)h->n,
                                cudaMemcpyDeviceToDevice, s));
    return MCE_OK;
}

mce_status mce_last_error(mce_graph *h, void *stream)
{
    if (!h) return MCE_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    mce_status st = read_status(h, s);
    if (st == MCE_ERR_CUDA) return st;
    MCE_TRY(cudaMemsetAsync(&h->g.ctrl->status, 0, sizeof(int), s));
    MCE_TRY(cudaStreamSynchronize(s));
    return st;
}

mce_status mce_get_info(mce_graph *h, mce_info *info)
{
    if (!h || !info) return MCE_ERR_INVALID_ARG;
    MCE_TRY(cudaDeviceSynchronize());
    DevCtrl c{};
    MCE_TRY(cudaMemcpy(&c, h->g.ctrl, sizeof(DevCtrl), cudaMemcpyDeviceToHost));
    memset(info, 0, sizeof(*info));
    info->n = h->n;
    info->degeneracy = h->degeneracy;
    info->m = h->nnz / 2;
    info->max_degree = h->max_degree;
    info->hist_len = h->hist_len;
    info->peel_rounds = c.rounds;
    info->n_workers = h->n_workers;
    info->workspace_bytes = (long long)(h->ws_words * 4ULL) + h->bb_quads * 16;
    info->induced = h->g.ip ? 2 : 1;
    info->subtree_level = h->g.l2 ? 2 : 1;
    info->tree_nodes = c.tree_nodes;
    info->donations = c.donations;
    for (int k = 0; k < kNumClasses; ++k) {
        info->words[k] = c.words[k];
        info->roots[k] = h->grp_count[2 * k] + h->grp_count[2 * k + 1];
        info->workers[k] = h->grp_workers[2 * k + 1] > h->grp_workers[2 * k]
                               ? h->grp_workers[2 * k + 1] : h->grp_workers[2 * k];
        info->ms_search[k] = 0.f;
        for (int b = 0; b < 2; ++b) {
            const int gi = 2 * k + b;
            if (!h->grp_timed[gi]) continue;
            float ms = 0.f;
            MCE_TRY(cudaEventElapsedTime(&ms, h->ev_grp[gi][0], h->ev_grp[gi][1]));
            info->ms_search[k] += ms;
        }
        info->ms_build[k] = 0.f;
        for (int b = 0; b < 2 && k < 3; ++b) {
            const int gi = 2 * k + b;
            if (!h->bld_timed[gi]) continue;
            float ms = 0.f;
            MCE_TRY(cudaEventElapsedTime(&ms, h->ev_bld[gi][0], h->ev_bld[gi][1]));
            info->ms_build[k] += ms;
        }
    }
    if (h->order_timed && h->n > 0) {
        MCE_TRY(cudaEventElapsedTime(&info->ms_order, h->ev_order[0], h->ev_order[1]));
        MCE_TRY(cudaEventElapsedTime(&info->ms_peel, h->ev_order[0], h->ev_order[2]));
    }
    info->peel_live = c.peel_live;
    info->launches = h->launches_order + h->launches_count;
    return MCE_OK;
}

mce_status mce_get_profile(mce_graph *h, uint64_t *out)
{
    if (!h || !out) return MCE_ERR_INVALID_ARG;
    MCE_TRY(cudaDeviceSynchronize());
    MCE_TRY(cudaMemcpy(out, h->g.ctrl->prof, sizeof(h->g.ctrl->prof), cudaMemcpyDeviceToHost));
    MCE_TRY(cudaMemcpy(out + kProfSlots * kNumClasses, h->g.ctrl->peel_prof,
                       sizeof(h->g.ctrl->peel_prof), cudaMemcpyDeviceToHost));
    MCE_TRY(cudaMemcpy(out + kProfSlots * kNumClasses + 16, h->g.prof_sm,
                       sizeof(unsigned long long) * kNumClasses * kProfSms,
                       cudaMemcpyDeviceToHost));
    return MCE_OK;
}

void mce_destroy(mce_graph *h)
{
    if (!h) return;
    {
        OnDevice on(h->device);
        cudaDeviceSynchronize();
    }
    free_all(h);
    delete h;
}

mce_status mce_trim_memory(void)
{
    int dev = 0;
    MCE_TRY(cudaGetDevice(&dev));
    cudaMemPool_t pool = device_pool(dev);
    if (!pool) return MCE_OK;
    MCE_TRY(cudaDeviceSynchronize());
    MCE_TRY(cudaMemPoolTrimTo(pool, 0));
    return MCE_OK;
}

}  // extern "C"
