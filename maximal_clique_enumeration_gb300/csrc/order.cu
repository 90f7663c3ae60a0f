// Degeneracy order on the GPU ("Parallelizing Maximal Clique Enumeration on GPUs",
// Section 2.4, "Degeneracy Ordering"; its time is part of the reported time, Section 4.1).
//
// The pages do not say how the order is computed.  This file computes one particular
// degeneracy order, the "canonical peel": level k starts at 0; a round removes, all at once,
// every remaining vertex with at most k remaining neighbours; when a round would be empty, k
// rises to the smallest remaining degree.  A vertex's position is its (round, id) rank, and
// its core number is the level at which it was removed.  Every vertex then has at most d
// later neighbours, d being the degeneracy (largest level).
//
// One cooperative kernel runs all rounds: the remaining vertices stay in an id-ordered list
// that is compacted stably every round, so each round's removals come out already in id
// order and the order needs no sort.  Two grid-wide barriers separate the phases of a round;
// once at most kPeelSoloVertices vertices remain, CTA 0 finishes alone with CTA barriers.
// Every barrier wait is bounded by spin_limit_ns.
//
// Then small kernels count every vertex's later neighbours |P| (Algorithm 3's P), count the
// isolated vertices, bucket the first-level roots by |P|, heaviest first, and store the
// later-neighbour lists N+(v) as a CSR (scan of |P|, then a stable split of each adjacency).
#include <climits>

#include <cuda/atomic>

#include "mce_internal.cuh"

namespace mce {

namespace {

// Grid-wide barrier for a cooperative launch.  Returns false if the wait exceeded the limit
// (MCE_ERR_DEVICE_TIMEOUT recorded) or some CTA recorded an error.
//
// The arrival counter only grows: a CTA adds 1 with release order, and the barrier it joined is
// complete once the counter reaches the next multiple of the grid size (acquire order), so no
// CTA has to reset anything and the last arrival frees every waiter at once.  The status word is
// polled beside the counter, so an error elsewhere ends the wait early.
__device__ bool grid_barrier(DevCtrl *ctrl, long long limit_ns)
{
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        cuda::atomic_ref<unsigned int, cuda::thread_scope_device> count(ctrl->bar_count);
        const unsigned int nb = gridDim.x;
        const unsigned int old = count.fetch_add(1u, cuda::memory_order_release);
        const unsigned int target = (old / nb + 1u) * nb;
        const volatile int *status = &ctrl->status;
        const unsigned long long t0 = globaltimer_ns();
        unsigned int polls = 0;
        while (true) {
            const unsigned int c = count.load(cuda::memory_order_acquire);
            if (*status != 0) {
                ok = 0;
                break;
            }
            if ((int)(c - target) >= 0) break;
            if ((++polls & 63u) == 1) {                  // check the clock now and then
                if ((long long)(globaltimer_ns() - t0) > limit_ns) {
                    set_status(ctrl, MCE_ERR_DEVICE_TIMEOUT);
                    ok = 0;
                    break;
                }
                if (polls > 4096) __nanosleep(128);      // a long wait: stop hammering L2
            }
        }
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

__device__ __forceinline__ int warp_incl_scan(int v, int lane)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

// Exclusive scan of one value per thread over the CTA; *total = CTA sum.
__device__ __forceinline__ int block_excl_scan_int(int v, int *total, int *sh)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int inc = warp_incl_scan(v, lane);
    if (lane == 31) sh[w] = inc;
    __syncthreads();
    int before = 0, t = 0;
    for (int i = 0; i < nw; ++i) {
        const int c = sh[i];
        if (i < w) before += c;
        t += c;
    }
    __syncthreads();
    *total = t;
    return before + inc - v;
}

// Phase timers of the MCE_PROFILE build (CTA 0, thread 0; nanoseconds): slot = phase, +8 when
// the round runs in a single CTA.  Phases: 0 scan, 1 report exchange (barrier), 2 decide and
// write, 3 edge removal, 4 end-of-round barrier, 5 rounds, 6 max edges of one removed vertex.
#ifdef MCE_PROFILE
#define PEEL_MARK(var) unsigned long long var = globaltimer_ns()
#define PEEL_ADD(slot, var)                                                            \
    do {                                                                               \
        if (blockIdx.x == 0 && threadIdx.x == 0) {                                     \
            const unsigned long long now_ = globaltimer_ns();                          \
            g.ctrl->peel_prof[(slot) + (solo ? 8 : 0)] += now_ - (var);                \
            var = now_;                                                                \
        }                                                                              \
    } while (0)
#else
#define PEEL_MARK(var) (void)0
#define PEEL_ADD(slot, var) (void)0
#endif

// Each thread holds up to kPeelItems consecutive entries of its CTA's part of the live list.
constexpr int kPeelItems = 8;
constexpr int kPeelBigDegree = 1024;   // removed vertices this wide are handled by a whole CTA
constexpr int kPeelBigQueue = 256;     // ... up to this many per round and CTA (then by warps)
constexpr long long kPeelSoloEntries = 1 << 20;   // and the single-CTA finish needs few edges left

// One round of the peel, in a CTA that owns live[lo, hi):
//   scan   -- load ids and current degrees once (kept in registers across the exchange) and
//             report (#deg <= k, least degree above k, #vertices at that degree);
//   decide -- from every CTA's report: if some vertex has deg <= k the round removes those,
//             else the level rises to the least degree d' and the round removes deg == d';
//   write  -- stable compaction: removed vertices get their rank (round, id order), round and
//             core number; survivors go to the next live list;
//   remove -- the CTA subtracts one degree from every neighbour of its own removed vertices
//             (degrees of vertices already removed are never read again).
// Grid barriers: after the scan (reports) and after the removal (degrees, next live list).
__global__ void __launch_bounds__(kPeelThreads, 1) peel_kernel(DevGraph g, long long limit_ns)
{
    __shared__ int sh[32];
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int lane = tid & 31, wib = tid >> 5, wpb = nthr >> 5;
    const int n = g.n;
    for (int v = blockIdx.x * nthr + tid; v < n; v += gridDim.x * nthr) {
        g.deg[v] = g.offs[v + 1] - g.offs[v];
        g.round_of[v] = -1;
        g.alive_a[v] = v;
    }
    if (!grid_barrier(g.ctrl, limit_ns)) return;

    int *alive = g.alive_a, *alive_next = g.alive_b;
    int n_alive = n, k = 0, r = 0, pos = 0, phase = 0, dmax = 0;
    // adjacency entries of the remaining vertices, read from the offsets themselves (callers of
    // the allocation-free entry point pass no edge count)
    long long live_entries = n > 0 ? (long long)g.offs[n] - (long long)g.offs[0] : 0;
    long long live_sum = 0;           // live vertices summed over rounds (CTA 0 keeps it)
    bool solo = false;
    int nb = gridDim.x, b = blockIdx.x;
    const int tile = nthr * kPeelItems;
    __shared__ long long s_removed;
    while (n_alive > 0) {
        if (!solo && r > 0) {
            // every CTA learns how many adjacency entries the last round removed
            if (wib == 0) {
                long long t = 0;
                for (int i = lane; i < nb; i += 32) t += g.blk_rd[i];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
                if (lane == 0) s_removed = t;
            }
            __syncthreads();
            live_entries -= s_removed;
        }
        // one CTA finishes once few vertices and few edges remain (a dense core keeps the grid)
        if (!solo && n_alive <= kPeelSoloVertices && live_entries <= kPeelSoloEntries) {
            if (blockIdx.x != 0) return;
            solo = true;
            nb = 1;
            b = 0;
        }
        PEEL_MARK(t_ph);
        const int chunk = (n_alive + nb - 1) / nb;
        const int lo = min(b * chunk, n_alive), hi = min(lo + chunk, n_alive);
        const bool in_regs = chunk <= tile;        // the same in every CTA
        int vid[kPeelItems], vdg[kPeelItems];
        // -- scan
        int cnt_le = 0, mmin = INT_MAX, cnt_m = 0;
        for (int t0 = lo; t0 < hi; t0 += tile) {
#pragma unroll
            for (int j = 0; j < kPeelItems; ++j) {
                const int i = t0 + tid * kPeelItems + j;
                vid[j] = i < hi ? alive[i] : -1;
            }
#pragma unroll
            for (int j = 0; j < kPeelItems; ++j) vdg[j] = vid[j] >= 0 ? g.deg[vid[j]] : INT_MAX;
#pragma unroll
            for (int j = 0; j < kPeelItems; ++j) {
                const int d = vdg[j];
                if (vid[j] < 0) continue;
                if (d <= k) ++cnt_le;
                else if (d < mmin) { mmin = d; cnt_m = 1; }
                else if (d == mmin) ++cnt_m;
            }
        }
        // CTA report in one exchange: (#deg <= k, least degree above k, #at that degree)
        __shared__ int s_rep[3][32];
        __shared__ int s_dec[3];
        {
            const int wle = __reduce_add_sync(0xffffffffu, cnt_le);
            const int wmin = __reduce_min_sync(0xffffffffu, mmin);
            const int wcm = __reduce_add_sync(0xffffffffu, mmin == wmin ? cnt_m : 0);
            if (lane == 0) { s_rep[0][wib] = wle; s_rep[1][wib] = wmin; s_rep[2][wib] = wcm; }
            __syncthreads();
            if (wib == 0) {
                const int a0 = lane < wpb ? s_rep[0][lane] : 0;
                const int a1 = lane < wpb ? s_rep[1][lane] : INT_MAX;
                const int a2 = lane < wpb ? s_rep[2][lane] : 0;
                const int bm = __reduce_min_sync(0xffffffffu, a1);
                const int t_le = __reduce_add_sync(0xffffffffu, a0);
                const int t_cm = __reduce_add_sync(0xffffffffu, a1 == bm ? a2 : 0);
                if (lane == 0) { s_dec[0] = t_le; s_dec[1] = bm; s_dec[2] = t_cm; }
            }
            __syncthreads();
        }
        cnt_le = s_dec[0];
        const int bmin = s_dec[1];
        cnt_m = s_dec[2];
        PEEL_ADD(0, t_ph);
        // -- decide (identically in every CTA)
        int total, prefix, newk;
        if (solo) {
            if (cnt_le > 0) { newk = k; total = cnt_le; }
            else { newk = bmin; total = cnt_m; }
            prefix = 0;
        } else {
            if (tid == 0) {
                g.blk_cnt[phase * nb + b] = cnt_le;
                g.blk_min[phase * nb + b] = bmin;
                g.blk_cm[phase * nb + b] = cnt_m;
            }
            if (!grid_barrier(g.ctrl, limit_ns)) return;
            PEEL_ADD(1, t_ph);
            // warp 0 reads every CTA's report
            __shared__ int s_glob[3];
            if (wib == 0) {
                int tle = 0, ple = 0, gm = INT_MAX;
                for (int i = lane; i < nb; i += 32) {
                    const int c = g.blk_cnt[phase * nb + i];
                    tle += c;
                    if (i < b) ple += c;
                    gm = min(gm, g.blk_min[phase * nb + i]);
                }
                tle = __reduce_add_sync(0xffffffffu, tle);
                ple = __reduce_add_sync(0xffffffffu, ple);
                gm = __reduce_min_sync(0xffffffffu, gm);
                if (tle == 0) {
                    int tm = 0, pm = 0;
                    for (int i = lane; i < nb; i += 32) {
                        const int c = g.blk_min[phase * nb + i] == gm ? g.blk_cm[phase * nb + i] : 0;
                        tm += c;
                        if (i < b) pm += c;
                    }
                    tle = __reduce_add_sync(0xffffffffu, tm);
                    ple = __reduce_add_sync(0xffffffffu, pm);
                } else {
                    gm = k;
                }
                if (lane == 0) { s_glob[0] = tle; s_glob[1] = ple; s_glob[2] = gm; }
            }
            __syncthreads();
            total = s_glob[0];
            prefix = s_glob[1];
            newk = s_glob[2];
            phase ^= 1;
        }
        k = newk;
        dmax = k;
        // -- write: this round's removals in id order, and the stably compacted survivors
        __shared__ int s_front[kPeelThreads * kPeelItems];   // this CTA's removed vertices
        const int my_first = pos + prefix;
        int bf = my_first, bs = lo - prefix;
        for (int t0 = lo; t0 < hi; t0 += tile) {
            if (!in_regs) {
#pragma unroll
                for (int j = 0; j < kPeelItems; ++j) {
                    const int i = t0 + tid * kPeelItems + j;
                    vid[j] = i < hi ? alive[i] : -1;
                    vdg[j] = vid[j] >= 0 ? g.deg[vid[j]] : INT_MAX;
                }
            }
            int nf = 0, nv = 0;
#pragma unroll
            for (int j = 0; j < kPeelItems; ++j) {
                nv += vid[j] >= 0;
                nf += vid[j] >= 0 && vdg[j] <= k;
            }
            int tot;
            const int ex = block_excl_scan_int((nv << 16) | nf, &tot, sh);  // both < 2^16
            const int rf = ex & 0xffff, rv = ex >> 16;
            const int tf = tot & 0xffff, tv = tot >> 16;
            int of = bf + rf, os = bs + (rv - rf);
#pragma unroll
            for (int j = 0; j < kPeelItems; ++j) {
                const int v = vid[j];
                if (v < 0) continue;
                if (vdg[j] <= k) {
                    g.order[of] = v;
                    g.rank[v] = of;
                    g.round_of[v] = r;
                    g.core[v] = k;
                    if (in_regs) s_front[of - my_first] = v;
                    ++of;
                } else {
                    alive_next[os++] = v;
                }
            }
            bf += tf;
            bs += tv - tf;
        }
        // degrees re-read by the write step (slices longer than one tile) must not move before
        // every CTA has written
        if (in_regs || solo) __syncthreads();
        else if (!grid_barrier(g.ctrl, limit_ns)) return;
        PEEL_ADD(2, t_ph);
        // -- remove this CTA's vertices: one warp per vertex, lanes over its neighbours; a vertex
        // with kPeelBigDegree or more neighbours is queued and then handled by the whole CTA
        __shared__ int s_big[kPeelBigQueue];
        __shared__ int s_nbig;
        __shared__ unsigned long long s_rd;       // adjacency entries this CTA removes
        if (tid == 0) {
            s_nbig = 0;
            s_rd = 0ULL;
        }
        __syncthreads();
        for (int e = wib; e < bf - my_first; e += wpb) {
            const int v = in_regs ? s_front[e] : g.order[my_first + e];
            const int elo = g.offs[v], ehi = g.offs[v + 1];
            if (lane == 0) atomicAdd(&s_rd, (unsigned long long)(ehi - elo));
            if (ehi - elo >= kPeelBigDegree) {
                int slot = 0;
                if (lane == 0) slot = atomicAdd(&s_nbig, 1);
                slot = __shfl_sync(0xffffffffu, slot, 0);
                if (slot < kPeelBigQueue) {
                    if (lane == 0) s_big[slot] = v;
                    continue;
                }
            }
            for (int j = elo + lane; j < ehi; j += 32) atomicSub(&g.deg[g.adj[j]], 1);
#ifdef MCE_PROFILE
            if (lane == 0 && blockIdx.x == 0)
                atomicMax(&g.ctrl->peel_prof[6], (unsigned long long)(ehi - elo));
#endif
        }
        __syncthreads();
        const int nbig = min(s_nbig, kPeelBigQueue);
        for (int i = 0; i < nbig; ++i) {
            const int v = s_big[i];
            const int elo = g.offs[v], ehi = g.offs[v + 1];
            for (int j = elo + tid; j < ehi; j += nthr) atomicSub(&g.deg[g.adj[j]], 1);
#ifdef MCE_PROFILE
            if (tid == 0 && blockIdx.x == 0)
                atomicMax(&g.ctrl->peel_prof[6], (unsigned long long)(ehi - elo));
#endif
        }
        if (!solo && tid == 0) g.blk_rd[b] = (long long)s_rd;
        __syncthreads();
        PEEL_ADD(3, t_ph);
        if (solo) __syncthreads();
        else if (!grid_barrier(g.ctrl, limit_ns)) return;
        PEEL_ADD(4, t_ph);
#ifdef MCE_PROFILE
        if (blockIdx.x == 0 && tid == 0) g.ctrl->peel_prof[5 + (solo ? 8 : 0)]++;
#endif
        live_sum += n_alive;
        pos += total;
        n_alive -= total;
        ++r;
        int *t = alive;
        alive = alive_next;
        alive_next = t;
    }
    if (blockIdx.x == 0 && tid == 0) {
        g.ctrl->degeneracy = dmax;
        g.ctrl->rounds = r;
        g.ctrl->peel_live = live_sum;
    }
}

constexpr int kOrientThreads = 256;

// |P(v)| = number of neighbours later in the order, and N+(v) itself: the later neighbours, in
// id order, at the front of v's own slot of padj (padj[offs[v] .. offs[v] + |P(v)|)); isolated
// vertices; |P| histogram; the per-warp workspace bound; Delta.
__global__ void __launch_bounds__(kOrientThreads) orient_count_kernel(DevGraph g)
{
    __shared__ int s_bucket[kNumBuckets];
    for (int i = threadIdx.x; i < kNumBuckets; i += blockDim.x) s_bucket[i] = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int warps = gridDim.x * (blockDim.x >> 5);
    int n_iso = 0, maxp = 0, maxdeg = 0;
    unsigned long long iso_hash = 0, ws = 0;
    unsigned long long ws_grp[kNumGroups] = {};
    for (int v = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; v < g.n; v += warps) {
        const int lo = g.offs[v], hi = g.offs[v + 1];
        const int rv = g.rank[v];
        const unsigned lt = (1u << lane) - 1u;
        int c = 0;
        for (int j0 = lo; j0 < hi; j0 += 32) {
            const int j = j0 + lane;
            const int w = j < hi ? g.adj[j] : 0;
            const bool later = j < hi && g.rank[w] > rv;
            const unsigned m = __ballot_sync(0xffffffffu, later);
            if (later) g.padj[lo + c + __popc(m & lt)] = w;
            c += __popc(m);
        }
        if (lane == 0) {
            g.pcount[v] = c;
            const int deg = hi - lo;
            maxdeg = max(maxdeg, deg);
            if (deg == 0) {
                ++n_iso;
                iso_hash += mix64(vertex_key(v));
            }
            if (c > 0) {
                atomicAdd(&s_bucket[sched_bucket(c, deg, g.ip, g.l2, g.core[v])], 1);
                maxp = max(maxp, c);
                if (c <= kMaxP) {
                    const unsigned long long need = (unsigned long long)ws_layout(deg, c, g.ip, g.l2).total;
                    ws = need > ws ? need : ws;
                    const int gi = 2 * wclass_index(c) + (need > (unsigned long long)kWsCapWords ? 0 : 1);
                    ws_grp[gi] = need > ws_grp[gi] ? need : ws_grp[gi];
                }
            }
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kNumBuckets; i += blockDim.x)
        if (s_bucket[i]) atomicAdd(&g.bucket[i], s_bucket[i]);
    if (lane == 0) {
        if (n_iso) {
            atomicAdd(&g.ctrl->n_iso, n_iso);
            atomicAdd(&g.ctrl->iso_hash, iso_hash);
        }
        atomicMax(&g.ctrl->max_pcount, maxp);
        atomicMax(&g.ctrl->max_degree, maxdeg);
        atomicMax(&g.ctrl->ws_words, ws);
        for (int k = 0; k < kNumGroups; ++k)
            if (ws_grp[k]) atomicMax(&g.ctrl->ws_grp[k], ws_grp[k]);
    }
}

// Turns a schedule-bucket histogram into bucket cursors and records where each launch group
// starts and ends in the resulting order.
__device__ void buckets_to_cursors(int *bucket, int *cls, unsigned long long *total)
{
    int run = 0;
    for (int o = 0; o < kNumGroups; ++o) {
        const int gi = group_at(o);
        cls[2 * gi] = run;
        for (int b = o == 0 ? 0 : 1 + o * kCostBuckets; b < 1 + (o + 1) * kCostBuckets; ++b) {
            const int cnt = bucket[b];
            bucket[b] = run;
            run += cnt;
        }
        cls[2 * gi + 1] = run;
    }
    if (total) *total = (unsigned long long)run;
}

__global__ void orient_scan_kernel(DevGraph g)
{
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    buckets_to_cursors(g.bucket, g.ctrl->cls, &g.ctrl->n_sched);
}

__global__ void __launch_bounds__(kOrientThreads) orient_scatter_kernel(DevGraph g)
{
    for (int v = blockIdx.x * blockDim.x + threadIdx.x; v < g.n; v += gridDim.x * blockDim.x) {
        const int c = g.pcount[v];
        if (c > 0) g.sched[atomicAdd(&g.bucket[sched_bucket(c, g.offs[v + 1] - g.offs[v], g.ip, g.l2, g.core[v])], 1)] = v;
    }
}

// ---- exclusive scan of an int array (three passes: CTA sums, scan of the sums, final)

constexpr int kScanThreads = 256;   // 4 elements per thread

__global__ void __launch_bounds__(kScanThreads) scan_partial_kernel(const int *in, int n, int *sums)
{
    __shared__ int sh[32];
    const int base = blockIdx.x * kScanBlock + threadIdx.x * 4;
    int v = 0;
    for (int i = 0; i < 4; ++i) v += base + i < n ? in[base + i] : 0;
    int tot;
    block_excl_scan_int(v, &tot, sh);
    if (threadIdx.x == 0) sums[blockIdx.x] = tot;
}

__global__ void __launch_bounds__(1024) scan_sums_kernel(int *sums, int nb)
{
    __shared__ int sh[32];
    int carry = 0;
    for (int c0 = 0; c0 < nb; c0 += blockDim.x) {
        const int i = c0 + threadIdx.x;
        const int v = i < nb ? sums[i] : 0;
        int tot;
        const int ex = block_excl_scan_int(v, &tot, sh);
        if (i < nb) sums[i] = carry + ex;
        carry += tot;
    }
}

__global__ void __launch_bounds__(kScanThreads) scan_final_kernel(const int *in, int n,
                                                                  const int *sums, int *out)
{
    __shared__ int sh[32];
    const int base = blockIdx.x * kScanBlock + threadIdx.x * 4;
    int x[4], v = 0;
    for (int i = 0; i < 4; ++i) {
        x[i] = base + i < n ? in[base + i] : 0;
        v += x[i];
    }
    int tot;
    int run = sums[blockIdx.x] + block_excl_scan_int(v, &tot, sh);
    for (int i = 0; i < 4; ++i) {
        if (base + i < n) out[base + i] = run;
        run += x[i];
        if (base + i == n - 1) out[n] = run;
    }
}

// A caller's root list, grouped by row-width class and heaviest first (like the schedule).
__global__ void __launch_bounds__(kOrientThreads) bin_count_kernel(DevGraph g, const int *roots,
                                                                   int n_roots)
{
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_roots; i += gridDim.x * blockDim.x) {
        const int v = roots[i];
        if (v < 0 || v >= g.n) {
            set_status(g.ctrl, MCE_ERR_ID_RANGE);
            continue;
        }
        atomicAdd(&g.ubucket[sched_bucket(g.pcount[v], g.offs[v + 1] - g.offs[v], g.ip, g.l2, g.core[v])], 1);
    }
}

__global__ void bin_scan_kernel(DevGraph g)
{
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    buckets_to_cursors(g.ubucket, g.ctrl->ucls, nullptr);
}

__global__ void __launch_bounds__(kOrientThreads) bin_scatter_kernel(DevGraph g, const int *roots,
                                                                     int n_roots)
{
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_roots; i += gridDim.x * blockDim.x) {
        const int v = roots[i];
        if (v < 0 || v >= g.n) continue;
        g.uroots[atomicAdd(&g.ubucket[sched_bucket(g.pcount[v], g.offs[v + 1] - g.offs[v], g.ip, g.l2, g.core[v])], 1)] = v;
    }
}

}  // namespace

cudaError_t launch_bin_roots(const DevGraph &g, const int *roots, int n_roots, cudaStream_t s)
{
    cudaError_t e = cudaMemsetAsync(g.ubucket, 0, sizeof(int) * kNumBuckets, s);
    if (e != cudaSuccess) return e;
    int b = (n_roots + kOrientThreads - 1) / kOrientThreads;
    if (b < 1) b = 1;
    if (b > 4096) b = 4096;
    bin_count_kernel<<<b, kOrientThreads, 0, s>>>(g, roots, n_roots);
    bin_scan_kernel<<<1, 32, 0, s>>>(g);
    bin_scatter_kernel<<<b, kOrientThreads, 0, s>>>(g, roots, n_roots);
    return cudaGetLastError();
}

// Second-level subtrees of each root (Algorithm 4): one per later neighbour w, i.e. per edge
// {v, w} ordered v before w; an isolated root has one, which reports the clique {v}.
__global__ void __launch_bounds__(kOrientThreads) unit_count_kernel(DevGraph g, const int *roots,
                                                                   int n_roots, int n_slots)
{
    const int len = n_roots >= 0 ? n_roots : (int)g.ctrl->n_sched;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_slots; i += gridDim.x * blockDim.x) {
        int c = 0;
        if (i < len) {
            const int v = roots[i];
            const int p = g.pcount[v];
            c = p > 0 ? p : (g.offs[v + 1] == g.offs[v] ? 1 : 0);
        }
        g.unit_cnt[i] = c;
    }
}

cudaError_t launch_unit_offsets(const DevGraph &g, const int *roots, int n_roots, int *uoff,
                                cudaStream_t s)
{
    const int n_slots = n_roots >= 0 ? n_roots : g.n;
    cudaError_t e = cudaMemsetAsync(uoff, 0, sizeof(int), s);
    if (e != cudaSuccess || n_slots == 0) return e;
    int b = (n_slots + kOrientThreads - 1) / kOrientThreads;
    if (b > 4096) b = 4096;
    unit_count_kernel<<<b, kOrientThreads, 0, s>>>(g, roots, n_roots, n_slots);
    const int nb = (n_slots + kScanBlock - 1) / kScanBlock;
    scan_partial_kernel<<<nb, kScanThreads, 0, s>>>(g.unit_cnt, n_slots, g.unit_scan);
    scan_sums_kernel<<<1, 1024, 0, s>>>(g.unit_scan, nb);
    scan_final_kernel<<<nb, kScanThreads, 0, s>>>(g.unit_cnt, n_slots, g.unit_scan, uoff);
    return cudaGetLastError();
}

// The whole peel: one cooperative launch over peel_blocks CTAs.
cudaError_t launch_peel(const DevGraph &g, int peel_blocks, long long spin_limit_ns,
                        cudaStream_t s)
{
    DevGraph gg = g;
    long long lim = spin_limit_ns;
    void *args[] = {&gg, &lim};
    return cudaLaunchCooperativeKernel((const void *)peel_kernel, dim3(peel_blocks),
                                       dim3(kPeelThreads), args, 0, s);
}

cudaError_t launch_order(const DevGraph &g, int peel_blocks, long long spin_limit_ns,
                         cudaStream_t s, cudaEvent_t ev_peel)
{
    if (g.n == 0) return cudaSuccess;
    // reset the fields the kernels accumulate into
    cudaError_t e = cudaMemsetAsync(&g.ctrl->bar_count, 0, sizeof(unsigned int), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(&g.ctrl->max_pcount, 0, sizeof(int), s);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(&g.ctrl->ws_words, 0, sizeof(unsigned long long) * (1 + kNumGroups), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(&g.ctrl->n_iso, 0, 2 * sizeof(int), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(&g.ctrl->iso_hash, 0, sizeof(unsigned long long), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(g.bucket, 0, sizeof(int) * kNumBuckets, s);
    if (e != cudaSuccess) return e;
    e = launch_peel(g, peel_blocks, spin_limit_ns, s);
    if (e != cudaSuccess) return e;
    if (ev_peel && (e = cudaEventRecord(ev_peel, s)) != cudaSuccess) return e;
    int blocks = (int)((g.n + kOrientThreads / 32 - 1) / (kOrientThreads / 32));
    if (blocks > 8192) blocks = 8192;
    orient_count_kernel<<<blocks, kOrientThreads, 0, s>>>(g);
    orient_scan_kernel<<<1, 32, 0, s>>>(g);
    int sb = (g.n + kOrientThreads - 1) / kOrientThreads;
    if (sb > 8192) sb = 8192;
    orient_scatter_kernel<<<sb, kOrientThreads, 0, s>>>(g);
    if (g.l2) {
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        return launch_unit_offsets(g, g.sched, -1, g.sched_uoff, s);
    }
    return cudaGetLastError();
}

}  // namespace mce

// ------------------------------------------------------------------ allocation-free order
//
// mce_order_noalloc: the degeneracy order of a small graph with no allocation at all, for
// callers that may not call cudaMalloc (see include/mce.h).  The peel kernel above runs
// unchanged; only its scratch (degrees, live lists, the removal order, the barrier counters)
// lives in one fixed array in device memory instead of a handle's buffers.

namespace mce {

namespace {

constexpr int kNoAllocMaxN = 1 << 18;        // vertices
constexpr int kNoAllocMaxBlocks = 1024;      // CTAs of the cooperative peel
constexpr int kNoAllocCtrlWords = (int)((sizeof(DevCtrl) + 255) / 256 * 64);
constexpr int kNoAllocWords = kNoAllocCtrlWords + 8 * kNoAllocMaxBlocks + 5 * kNoAllocMaxN;
constexpr int kNoAllocMaxDevices = 64;

// The whole scratch area: 5 MiB + a few KiB, held by every device that loads the library.
static __device__ __align__(256) int g_noalloc_scratch[kNoAllocWords];

int *g_noalloc_ptr[kNoAllocMaxDevices];      // device address of the array, per device

// Clears what the peel reads before writing: the status word and the barrier counter.
__global__ void noalloc_prep_kernel()
{
    DevCtrl *c = reinterpret_cast<DevCtrl *>(g_noalloc_scratch);
    c->status = 0;
    c->bar_count = 0u;
    c->degeneracy = 0;
    c->rounds = 0;
}

__global__ void noalloc_result_kernel(int *d_result)
{
    const DevCtrl *c = reinterpret_cast<const DevCtrl *>(g_noalloc_scratch);
    d_result[0] = c->degeneracy;
    d_result[1] = c->status;
}

}  // namespace

}  // namespace mce

extern "C" mce_status mce_order_noalloc(const int32_t *d_offsets, const int32_t *d_adj, int32_t n,
                                        int32_t *d_rank, int32_t *d_core, int32_t *d_result,
                                        void *stream)
{
    using namespace mce;
    if (n < 0 || !d_result) return MCE_ERR_INVALID_ARG;
    if (n > kNoAllocMaxN) return MCE_ERR_LIMIT;          // checked first: the size is the news
    if (n > 0 && (!d_offsets || !d_adj || !d_rank || !d_core)) return MCE_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MCE_ERR_CUDA;
    if (dev < 0 || dev >= kNoAllocMaxDevices) return MCE_ERR_LIMIT;
    if (!g_noalloc_ptr[dev]) {                    // set-up, once per device
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return MCE_ERR_CUDA;
        }
        g_noalloc_ptr[dev] = static_cast<int *>(p);
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return MCE_ERR_CUDA;
    const int blocks = sms < kNoAllocMaxBlocks ? sms : kNoAllocMaxBlocks;
    int *base = g_noalloc_ptr[dev];
    cudaStream_t s = (cudaStream_t)stream;
    DevGraph g{};
    g.n = n;
    g.offs = d_offsets;
    g.adj = d_adj;
    g.rank = d_rank;
    g.core = d_core;
    g.ctrl = reinterpret_cast<DevCtrl *>(base);
    g.blk_cnt = base + kNoAllocCtrlWords;
    g.blk_min = g.blk_cnt + 2 * kNoAllocMaxBlocks;
    g.blk_cm = g.blk_min + 2 * kNoAllocMaxBlocks;
    g.blk_rd = reinterpret_cast<long long *>(g.blk_cm + 2 * kNoAllocMaxBlocks);
    g.deg = g.blk_cm + 4 * kNoAllocMaxBlocks;
    g.round_of = g.deg + kNoAllocMaxN;
    g.alive_a = g.round_of + kNoAllocMaxN;
    g.alive_b = g.alive_a + kNoAllocMaxN;
    g.order = g.alive_b + kNoAllocMaxN;
    noalloc_prep_kernel<<<1, 1, 0, s>>>();
    if (cudaGetLastError() != cudaSuccess) return MCE_ERR_CUDA;
    if (n > 0 && launch_peel(g, blocks, 20LL * 1000 * 1000 * 1000, s) != cudaSuccess) {
        cudaGetLastError();
        return MCE_ERR_CUDA;
    }
    noalloc_result_kernel<<<1, 1, 0, s>>>(d_result);
    return cudaGetLastError() == cudaSuccess ? MCE_OK : MCE_ERR_CUDA;
}
