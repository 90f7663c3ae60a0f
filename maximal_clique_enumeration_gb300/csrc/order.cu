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
// One cooperative kernel runs all rounds.  The remaining vertices stay in an id-ordered list
// that is compacted stably in every round that scans it, so those rounds' removals come out in
// id order.  Most rounds need no scan: at level k, a round that keeps the level removes exactly
// the vertices whose degree fell to k in the round before, which that round's edge removal
// collects; such a round takes one grid barrier instead of two and reads no live list.  Once at
// most kPeelSoloVertices vertices remain, CTA 0 finishes alone with CTA barriers.  Every barrier
// wait is bounded by spin_limit_ns.
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

// Phase timers of the MCE_PROFILE build (CTA 0, thread 0; nanoseconds): slot = phase, +8 for
// frontier rounds and rounds run in a single CTA (prof_off).  Phases: 0 scan, 1 report exchange (barrier), 2 decide and
// write, 3 edge removal, 4 end-of-round barrier, 5 rounds, 6 max edges of one removed vertex.
#ifdef MCE_PROFILE
#define PEEL_MARK(var) unsigned long long var = globaltimer_ns()
#define PEEL_ADD(slot, var)                                                            \
    do {                                                                               \
        if (blockIdx.x == 0 && threadIdx.x == 0) {                                     \
            const unsigned long long now_ = globaltimer_ns();                          \
            g.ctrl->peel_prof[(slot) + prof_off] += now_ - (var);                      \
            var = now_;                                                                \
        }                                                                              \
    } while (0)
#else
#define PEEL_MARK(var) (void)0
#define PEEL_ADD(slot, var) (void)0
#endif

// Each thread holds up to kPeelItems consecutive entries of its CTA's part of the live list.
constexpr int kPeelItems = 8;
constexpr int kPeelTile = kPeelThreads * kPeelItems;
constexpr int kPeelBigDegree = 1024;   // removed vertices this wide are handled by a whole CTA
constexpr int kPeelBigQueue = 256;     // ... up to this many per round and CTA (then by warps)
constexpr long long kPeelSoloEntries = 1 << 20;   // and the single-CTA finish needs few edges left
constexpr int kPeelInFlight = 8;       // adjacency entries a thread has in flight in edge removal
// Dynamic shared memory: the CTA's removed vertices of a scan round (kPeelTile), then in
// frontier rounds the frontier's entry offsets (kFrontCap + 1) and adjacency bases (kFrontCap);
// the sort of the rank pass reuses the first part.
constexpr size_t kPeelSmemBytes = (size_t)(kPeelTile + 2 * kFrontCap + 8) * sizeof(int);
static_assert(kFrontCap <= kPeelTile, "a frontier segment sorts in the first part");

// Appends u to the frontier of the next round (warp-aggregated; entries beyond kFrontCap are
// counted, not stored).  All 32 lanes call it, `want` says whether this lane has a vertex.
__device__ __forceinline__ void front_append(bool want, int u, int *front, int *front_cnt)
{
    const unsigned m = __ballot_sync(0xffffffffu, want);
    if (!m) return;
    const int lane = threadIdx.x & 31, leader = __ffs(m) - 1;
    int base = 0;
    if (lane == leader) base = atomicAdd(front_cnt, __popc(m));
    base = __shfl_sync(0xffffffffu, base, leader);
    const int at = base + __popc(m & ((1u << lane) - 1u));
    if (want && at < kFrontCap) front[at] = u;
}

// Subtracts one from the degree of every adjacency entry in [f_begin, f_end) of the flattened
// list of vertices s_vert / their offsets s_off, kPeelInFlight entries in flight, appending to the
// next frontier every vertex whose degree falls from k + 1 to k (at level k those are exactly
// the vertices the next round removes; a vertex removed earlier, or in this round, already has
// degree <= k and is never appended).  Every lane of the warp calls it (appends are ballots).
__device__ void remove_flat(const DevGraph &g, const int *s_off, const int *s_base, int n_vert,
                            int f_begin, int f_end, int k, int *front, int *front_cnt)
{
    int lo = 0, hi = n_vert;                      // owner of f_begin: last i with s_off[i] <= f
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_off[mid] <= f_begin) lo = mid;
        else hi = mid;
    }
    int own = lo;
    // the warp runs until its longest thread is done (ballots need every lane)
    int rounds = (f_end - f_begin + kPeelInFlight - 1) / kPeelInFlight;
    rounds = __reduce_max_sync(0xffffffffu, rounds > 0 ? rounds : 0);
    for (int it = 0; it < rounds; ++it) {
        const int f0 = f_begin + it * kPeelInFlight;
        int u[kPeelInFlight], old[kPeelInFlight];
#pragma unroll
        for (int t = 0; t < kPeelInFlight; ++t) {
            const int f = f0 + t;
            u[t] = -1;
            if (f < f_end) {
                while (s_off[own + 1] <= f) ++own;
                u[t] = __ldg(g.adj + s_base[own] + (f - s_off[own]));
            }
        }
#pragma unroll
        for (int t = 0; t < kPeelInFlight; ++t) old[t] = u[t] >= 0 ? atomicSub(&g.deg[u[t]], 1) : 0;
#pragma unroll
        for (int t = 0; t < kPeelInFlight; ++t)
            front_append(u[t] >= 0 && old[t] == k + 1, u[t], front, front_cnt);
    }
}

// Sorts s[0 .. cnt) ascending, cnt <= kFrontCap (room for the next power of two): bitonic, in
// one warp's registers up to 32 entries, else by the whole CTA in shared memory.
__device__ void block_sort(int *s, int cnt)
{
    const int lane = threadIdx.x & 31;
    if (cnt <= 32) {
        if (threadIdx.x < 32) {
            int x = lane < cnt ? s[lane] : INT_MAX;
#pragma unroll
            for (int kk = 2; kk <= 32; kk <<= 1) {
#pragma unroll
                for (int j = kk >> 1; j > 0; j >>= 1) {
                    const int y = __shfl_xor_sync(0xffffffffu, x, j);
                    const bool take_min = ((lane & j) == 0) == ((lane & kk) == 0);
                    x = take_min ? min(x, y) : max(x, y);
                }
            }
            if (lane < cnt) s[lane] = x;
        }
        __syncthreads();
        return;
    }
    int p2 = 64;
    while (p2 < cnt) p2 <<= 1;
    for (int i = cnt + (int)threadIdx.x; i < p2; i += blockDim.x) s[i] = INT_MAX;
    __syncthreads();
    for (int kk = 2; kk <= p2; kk <<= 1) {
        for (int j = kk >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < p2; i += blockDim.x) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const int a = s[i], b = s[ixj];
                    if ((a > b) == ((i & kk) == 0)) {
                        s[i] = b;
                        s[ixj] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
}

// The canonical peel (see the top of this file) in one cooperative kernel, with two kinds of
// round:
//   scan round (the first round, every round that raises the level, and every round whose
//   vertices did not fit a frontier) -- a CTA owns live[lo, hi):
//     scan   -- load ids, current degrees and removal marks once (kept in registers across the
//               exchange) and report (#deg <= k, least degree above k, #vertices at that degree,
//               #entries removed by frontier rounds since the last compaction);
//     decide -- from every CTA's report: if some vertex has deg <= k the round removes those,
//               else the level rises to the least degree d' and the round removes deg == d';
//     write  -- stable compaction: removed vertices get their rank (round, id order), round and
//               core number; survivors go to the next live list;
//     remove -- the CTA subtracts one degree from every neighbour of its own removed vertices;
//   frontier round -- at level k a round that keeps the level removes exactly the vertices
//   whose degree fell to k during the round before, which that round's edge removal collected
//   (the frontier): no scan and no exchange, every CTA takes a share of the frontier's
//   vertices (round, core number, unsorted place in the order) and of their adjacency entries.
// Every round's edge removal collects the next frontier.  Grid barriers: two per scan round
// (after the reports, and at the end), one per frontier round.  A second kernel then sorts
// each frontier round's vertices by id in place and writes their ranks.  Once few vertices and
// few edges remain, CTA 0 goes on alone (CTA barriers only).
__global__ void __launch_bounds__(kPeelThreads, 1) peel_kernel(DevGraph g, long long limit_ns)
{
    extern __shared__ int s_dyn[];
    int *s_front = s_dyn;                       // scan round: this CTA's removed vertices
    int *s_off = s_dyn + kPeelTile;             // frontier round: entry offsets [cnt + 1]
    int *s_base = s_off + kFrontCap + 8;        // frontier round: adjacency bases [cnt]
    __shared__ int sh[32];
    __shared__ int s_rep[4][32];
    __shared__ int s_dec[4];
    __shared__ int s_glob[5];
    __shared__ int s_big[kPeelBigQueue];
    __shared__ int s_nbig;
    __shared__ unsigned long long s_rd;
    __shared__ long long s_removed;
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int lane = tid & 31, wib = tid >> 5, wpb = nthr >> 5;
    const int n = g.n;
    DevCtrl *c = g.ctrl;
    for (int v = blockIdx.x * nthr + tid; v < n; v += gridDim.x * nthr) {
        g.deg[v] = g.offs[v + 1] - g.offs[v];
        g.round_of[v] = -1;
        g.alive_a[v] = v;
    }
    if (blockIdx.x == 0 && tid < 3) c->front_cnt[tid] = 0;
    if (!grid_barrier(c, limit_ns)) return;

    int *alive = g.alive_a, *alive_next = g.alive_b;
    int n_live = n;     // entries of the live list (frontier rounds remove without compacting)
    int n_alive = n;    // vertices not removed yet
    int k = 0, r = 0, pos = 0, phase = 0, dmax = 0;
    // adjacency entries of the remaining vertices, read from the offsets themselves (callers of
    // the allocation-free entry point pass no edge count)
    long long live_entries = n > 0 ? (long long)g.offs[n] - (long long)g.offs[0] : 0;
    long long live_sum = 0;   // live-list entries scanned plus frontier vertices, over rounds
    bool solo = false;
    int nb = gridDim.x, b = blockIdx.x;
    while (n_alive > 0) {
        // round r reads the frontier round r - 1 collected, collects into the next buffer, and
        // clears the one after (last read in round r - 1); three buffers, so no read races a write
        const int fr_in = r % 3, fr_out = (r + 1) % 3, fr_clear = (r + 2) % 3;
        int *front_in = g.front + (size_t)fr_in * kFrontCap;
        int *front_out = g.front + (size_t)fr_out * kFrontCap;
        const int fc = r > 0 ? *(volatile int *)&c->front_cnt[fr_in] : 0;   // same in every CTA
        if (b == 0 && tid == 0) c->front_cnt[fr_clear] = 0;
        // one CTA finishes once few vertices and few edges remain (a dense core keeps the grid)
        if (!solo && n_live <= kPeelSoloVertices && live_entries <= kPeelSoloEntries) {
            if (blockIdx.x != 0) return;
            solo = true;
            nb = 1;
            b = 0;
        }
        PEEL_MARK(t_ph);
        const bool frontier = fc > 0 && fc <= kFrontCap;
        const int prof_off = solo || frontier ? 8 : 0;
        (void)prof_off;
        if (frontier) {
            // ================================================ frontier round
            // the frontier's adjacency entries, flattened (every CTA the whole prefix)
            {
                int dsum = 0;
                const int per = (fc + nthr - 1) / nthr;       // <= kFrontCap / threads
                const int i0 = min(tid * per, fc), i1 = min(i0 + per, fc);
                for (int i = i0; i < i1; ++i) {
                    const int v = __ldcg(front_in + i);
                    const int lo_v = g.offs[v];
                    s_base[i] = lo_v;
                    s_off[i] = g.offs[v + 1] - lo_v;
                    dsum += s_off[i];
                }
                int tot;
                int run = block_excl_scan_int(dsum, &tot, sh);
                for (int i = i0; i < i1; ++i) {
                    const int d = s_off[i];
                    s_off[i] = run;
                    run += d;
                }
                if (tid == 0) s_off[fc] = tot;
                __syncthreads();
            }
            const int edges = s_off[fc];
            // this CTA's share of the frontier: round, core number, place in the order (the
            // rank pass sorts the round's places by id at the end)
            {
                const int v0 = (int)((long long)fc * b / nb), v1 = (int)((long long)fc * (b + 1) / nb);
                for (int i = v0 + tid; i < v1; i += nthr) {
                    const int v = __ldcg(front_in + i);
                    g.order[pos + i] = v;
                    g.round_of[v] = r;
                    g.core[v] = k;
                }
            }
            if (b == 0 && tid == 0) g.rstart[r] = pos | kRoundUnsorted;
            PEEL_ADD(2, t_ph);
            // this CTA's share of the entries, a contiguous piece per thread
            {
                const long long e0 = (long long)edges * b / nb, e1 = (long long)edges * (b + 1) / nb;
                const int f_begin = (int)(e0 + (e1 - e0) * tid / nthr);
                const int f_end = (int)(e0 + (e1 - e0) * (tid + 1) / nthr);
                remove_flat(g, s_off, s_base, fc, f_begin, f_end, k, front_out,
                            &c->front_cnt[fr_out]);
            }
            __syncthreads();
            PEEL_ADD(3, t_ph);
            if (solo) __syncthreads();
            else if (!grid_barrier(c, limit_ns)) return;
            PEEL_ADD(4, t_ph);
#ifdef MCE_PROFILE
            if (blockIdx.x == 0 && tid == 0) c->peel_prof[5 + prof_off]++;
#endif
            live_entries -= edges;
            live_sum += fc;
            pos += fc;
            n_alive -= fc;
            ++r;
            continue;
        }
        // ==================================================== scan round
        const int chunk = (n_live + nb - 1) / nb;
        const int lo = min(b * chunk, n_live), hi = min(lo + chunk, n_live);
        const bool in_regs = chunk <= kPeelTile;   // the same in every CTA
        int vid[kPeelItems], vdg[kPeelItems];
        // -- scan (an entry removed by a frontier round gets vdg = -1)
        int cnt_le = 0, mmin = INT_MAX, cnt_m = 0, cnt_gone = 0;
        for (int t0 = lo; t0 < hi; t0 += kPeelTile) {
#pragma unroll
            for (int j = 0; j < kPeelItems; ++j) {
                const int i = t0 + tid * kPeelItems + j;
                vid[j] = i < hi ? alive[i] : -1;
            }
#pragma unroll
            for (int j = 0; j < kPeelItems; ++j) {
                if (vid[j] < 0) {
                    vdg[j] = INT_MAX;
                    continue;
                }
                const int d = g.deg[vid[j]], gone = g.round_of[vid[j]];
                vdg[j] = gone >= 0 ? -1 : d;
            }
#pragma unroll
            for (int j = 0; j < kPeelItems; ++j) {
                const int d = vdg[j];
                if (vid[j] < 0) continue;
                if (d < 0) ++cnt_gone;
                else if (d <= k) ++cnt_le;
                else if (d < mmin) { mmin = d; cnt_m = 1; }
                else if (d == mmin) ++cnt_m;
            }
        }
        // CTA report in one exchange: (#deg <= k, least degree above k, #at that degree, #gone)
        {
            const int wle = __reduce_add_sync(0xffffffffu, cnt_le);
            const int wmin = __reduce_min_sync(0xffffffffu, mmin);
            const int wcm = __reduce_add_sync(0xffffffffu, mmin == wmin ? cnt_m : 0);
            const int wgo = __reduce_add_sync(0xffffffffu, cnt_gone);
            if (lane == 0) {
                s_rep[0][wib] = wle;
                s_rep[1][wib] = wmin;
                s_rep[2][wib] = wcm;
                s_rep[3][wib] = wgo;
            }
            __syncthreads();
            if (wib == 0) {
                const int a0 = lane < wpb ? s_rep[0][lane] : 0;
                const int a1 = lane < wpb ? s_rep[1][lane] : INT_MAX;
                const int a2 = lane < wpb ? s_rep[2][lane] : 0;
                const int a3 = lane < wpb ? s_rep[3][lane] : 0;
                const int bm = __reduce_min_sync(0xffffffffu, a1);
                const int t_le = __reduce_add_sync(0xffffffffu, a0);
                const int t_cm = __reduce_add_sync(0xffffffffu, a1 == bm ? a2 : 0);
                const int t_go = __reduce_add_sync(0xffffffffu, a3);
                if (lane == 0) { s_dec[0] = t_le; s_dec[1] = bm; s_dec[2] = t_cm; s_dec[3] = t_go; }
            }
            __syncthreads();
        }
        cnt_le = s_dec[0];
        const int bmin = s_dec[1];
        cnt_m = s_dec[2];
        cnt_gone = s_dec[3];
        PEEL_ADD(0, t_ph);
        // -- decide (identically in every CTA)
        int total, prefix, newk, total_gone, prefix_gone;
        if (solo) {
            if (cnt_le > 0) { newk = k; total = cnt_le; }
            else { newk = bmin; total = cnt_m; }
            prefix = 0;
            total_gone = cnt_gone;
            prefix_gone = 0;
        } else {
            if (tid == 0) {
                g.blk_cnt[phase * nb + b] = cnt_le;
                g.blk_min[phase * nb + b] = bmin;
                g.blk_cm[phase * nb + b] = cnt_m;
                g.blk_gone[phase * nb + b] = cnt_gone;
            }
            if (!grid_barrier(c, limit_ns)) return;
            PEEL_ADD(1, t_ph);
            // warp 0 reads every CTA's report
            if (wib == 0) {
                int tle = 0, ple = 0, gm = INT_MAX, tgo = 0, pgo = 0;
                for (int i = lane; i < nb; i += 32) {
                    const int cl = g.blk_cnt[phase * nb + i];
                    const int cg = g.blk_gone[phase * nb + i];
                    tle += cl;
                    tgo += cg;
                    if (i < b) { ple += cl; pgo += cg; }
                    gm = min(gm, g.blk_min[phase * nb + i]);
                }
                tle = __reduce_add_sync(0xffffffffu, tle);
                ple = __reduce_add_sync(0xffffffffu, ple);
                tgo = __reduce_add_sync(0xffffffffu, tgo);
                pgo = __reduce_add_sync(0xffffffffu, pgo);
                gm = __reduce_min_sync(0xffffffffu, gm);
                if (tle == 0) {
                    int tm = 0, pm = 0;
                    for (int i = lane; i < nb; i += 32) {
                        const int cm = g.blk_min[phase * nb + i] == gm ? g.blk_cm[phase * nb + i] : 0;
                        tm += cm;
                        if (i < b) pm += cm;
                    }
                    tle = __reduce_add_sync(0xffffffffu, tm);
                    ple = __reduce_add_sync(0xffffffffu, pm);
                } else {
                    gm = k;
                }
                if (lane == 0) {
                    s_glob[0] = tle; s_glob[1] = ple; s_glob[2] = gm; s_glob[3] = tgo;
                    s_glob[4] = pgo;
                }
            }
            __syncthreads();
            total = s_glob[0];
            prefix = s_glob[1];
            newk = s_glob[2];
            total_gone = s_glob[3];
            prefix_gone = s_glob[4];
            phase ^= 1;
        }
        k = newk;
        dmax = k;
        if (b == 0 && tid == 0) g.rstart[r] = pos;
        // -- write: this round's removals in id order, and the stably compacted survivors
        const int my_first = pos + prefix;
        int bf = my_first, bs = lo - prefix - prefix_gone;
        for (int t0 = lo; t0 < hi; t0 += kPeelTile) {
            if (!in_regs) {
#pragma unroll
                for (int j = 0; j < kPeelItems; ++j) {
                    const int i = t0 + tid * kPeelItems + j;
                    vid[j] = i < hi ? alive[i] : -1;
                    vdg[j] = vid[j] < 0 ? INT_MAX : (g.round_of[vid[j]] >= 0 ? -1 : g.deg[vid[j]]);
                }
            }
            int nf = 0, ns = 0;
#pragma unroll
            for (int j = 0; j < kPeelItems; ++j) {
                nf += vid[j] >= 0 && vdg[j] >= 0 && vdg[j] <= k;
                ns += vid[j] >= 0 && vdg[j] > k;
            }
            int tot;
            const int ex = block_excl_scan_int((ns << 16) | nf, &tot, sh);  // both < 2^16
            const int rf = ex & 0xffff, rs = ex >> 16;
            const int tf = tot & 0xffff, ts = tot >> 16;
            int of = bf + rf, os = bs + rs;
#pragma unroll
            for (int j = 0; j < kPeelItems; ++j) {
                const int v = vid[j];
                if (v < 0 || vdg[j] < 0) continue;
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
            bs += ts;
        }
        // degrees re-read by the write step (slices longer than one tile) must not move before
        // every CTA has written
        if (in_regs || solo) __syncthreads();
        else if (!grid_barrier(c, limit_ns)) return;
        PEEL_ADD(2, t_ph);
        // -- remove this CTA's vertices: one warp per vertex, lanes over its neighbours
        // (kPeelInFlight at a time); a vertex with kPeelBigDegree or more neighbours is queued
        // and then handled by the whole CTA
        if (tid == 0) {
            s_nbig = 0;
            s_rd = 0ULL;
        }
        __syncthreads();
        int *fcnt = &c->front_cnt[fr_out];
        for (int e = wib; e < bf - my_first; e += wpb) {
            const int v = in_regs ? s_front[e] : g.order[my_first + e];
            const int elo = g.offs[v], ehi = g.offs[v + 1];
            if (ehi - elo >= kPeelBigDegree) {
                int slot = 0;
                if (lane == 0) slot = atomicAdd(&s_nbig, 1);
                slot = __shfl_sync(0xffffffffu, slot, 0);
                if (slot < kPeelBigQueue) {
                    if (lane == 0) s_big[slot] = v;
                    continue;
                }
            }
            if (lane == 0) atomicAdd(&s_rd, (unsigned long long)(ehi - elo));
            for (int j0 = elo; j0 < ehi; j0 += 32 * kPeelInFlight) {
                int u[kPeelInFlight], old[kPeelInFlight];
#pragma unroll
                for (int t = 0; t < kPeelInFlight; ++t) {
                    const int j = j0 + t * 32 + lane;
                    u[t] = j < ehi ? __ldg(g.adj + j) : -1;
                }
#pragma unroll
                for (int t = 0; t < kPeelInFlight; ++t)
                    old[t] = u[t] >= 0 ? atomicSub(&g.deg[u[t]], 1) : 0;
#pragma unroll
                for (int t = 0; t < kPeelInFlight; ++t)
                    front_append(u[t] >= 0 && old[t] == k + 1, u[t], front_out, fcnt);
            }
#ifdef MCE_PROFILE
            if (lane == 0 && blockIdx.x == 0) atomicMax(&c->peel_prof[6], (unsigned long long)(ehi - elo));
#endif
        }
        __syncthreads();
        const int nbig = min(s_nbig, kPeelBigQueue);
        for (int i = 0; i < nbig; ++i) {
            const int v = s_big[i];
            const int elo = g.offs[v], ehi = g.offs[v + 1];
            if (tid == 0) s_rd += (unsigned long long)(ehi - elo);
            for (int j0 = elo + wib * 32 * kPeelInFlight; j0 < ehi; j0 += nthr * kPeelInFlight) {
                int u[kPeelInFlight], old[kPeelInFlight];
#pragma unroll
                for (int t = 0; t < kPeelInFlight; ++t) {
                    const int j = j0 + t * 32 + lane;
                    u[t] = j < ehi ? __ldg(g.adj + j) : -1;
                }
#pragma unroll
                for (int t = 0; t < kPeelInFlight; ++t)
                    old[t] = u[t] >= 0 ? atomicSub(&g.deg[u[t]], 1) : 0;
#pragma unroll
                for (int t = 0; t < kPeelInFlight; ++t)
                    front_append(u[t] >= 0 && old[t] == k + 1, u[t], front_out, fcnt);
            }
#ifdef MCE_PROFILE
            if (tid == 0 && blockIdx.x == 0) atomicMax(&c->peel_prof[6], (unsigned long long)(ehi - elo));
#endif
        }
        if (!solo && tid == 0) g.blk_rd[b] = (long long)s_rd;
        __syncthreads();
        PEEL_ADD(3, t_ph);
        if (solo) __syncthreads();
        else if (!grid_barrier(c, limit_ns)) return;
        PEEL_ADD(4, t_ph);
#ifdef MCE_PROFILE
        if (blockIdx.x == 0 && tid == 0) c->peel_prof[5 + prof_off]++;
#endif
        // every CTA learns how many adjacency entries the round removed
        if (!solo) {
            if (wib == 0) {
                long long t = 0;
                for (int i = lane; i < nb; i += 32) t += g.blk_rd[i];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
                if (lane == 0) s_removed = t;
            }
            __syncthreads();
            live_entries -= s_removed;
        } else {
            live_entries -= (long long)s_rd;
        }
        live_sum += n_live;
        pos += total;
        n_alive -= total;
        n_live -= total + total_gone;
        ++r;
        int *t = alive;
        alive = alive_next;
        alive_next = t;
    }
    if (blockIdx.x == 0 && tid == 0) {
        c->degeneracy = dmax;
        c->rounds = r;
        c->peel_live = live_sum;
        g.rstart[r] = pos;
    }
}

// Rank pass after the peel: each frontier round's places in the order sorted by id (a vertex's
// rank is its (round, id) position), then every vertex of such a round gets its rank.  One
// round per CTA at a time.
__global__ void __launch_bounds__(kPeelThreads) peel_rank_kernel(DevGraph g)
{
    __shared__ int s[kFrontCap];
    if (load_status(g.ctrl) != 0) return;
    const int rounds = g.ctrl->rounds;
    for (int q = blockIdx.x; q < rounds; q += gridDim.x) {
        const int s0 = g.rstart[q];
        if (!(s0 & kRoundUnsorted)) continue;
        const int start = s0 & ~kRoundUnsorted, end = g.rstart[q + 1] & ~kRoundUnsorted;
        const int cnt = end - start;             // <= kFrontCap
        for (int i = threadIdx.x; i < cnt; i += blockDim.x) s[i] = g.order[start + i];
        __syncthreads();
        block_sort(s, cnt);                      // ends with __syncthreads
        for (int i = threadIdx.x; i < cnt; i += blockDim.x) {
            const int v = s[i];
            g.order[start + i] = v;
            g.rank[v] = start + i;
        }
        __syncthreads();
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

// Warp-aggregated s[key] += 1 in shared memory for the active lanes; returns the old value
// plus the lane's rank among the active lanes with the same key.  Every lane of the warp calls
// it (the lanes with one key add once, so a popular bucket costs one atomic per warp).
__device__ __forceinline__ int warp_agg_inc(int *s, int key, bool active)
{
    const unsigned act = __ballot_sync(0xffffffffu, active);
    int r = 0;
    if (active) {
        const int lane = threadIdx.x & 31;
        const unsigned peers = __match_any_sync(act, key);
        const int leader = __ffs(peers) - 1;
        int base = 0;
        if (lane == leader) base = atomicAdd(s + key, __popc(peers));
        base = __shfl_sync(peers, base, leader);
        r = base + __popc(peers & ((1u << lane) - 1u));
    }
    return r;
}

// Places the items of [lo, hi) (one CTA's segment) into out[] at their buckets' cursors:
// the CTA counts its items per bucket in shared memory, reserves each bucket's range with one
// global atomic, then writes every item at its place in that range.  item(i, &b) returns the
// value to place and sets its bucket b, or returns -1 for an item that is not placed.
template <class Item>
__device__ void segment_scatter(int lo, int hi, int *s_cur, int *cursor, int *out, Item item)
{
    for (int i = threadIdx.x; i < kNumBuckets; i += blockDim.x) s_cur[i] = 0;
    __syncthreads();
    for (int b0 = lo; b0 < hi; b0 += blockDim.x) {     // the same trip count for the whole CTA
        const int i = b0 + threadIdx.x;
        int b = 0;
        const int v = i < hi ? item(i, &b) : -1;
        warp_agg_inc(s_cur, b, v >= 0);
    }
    __syncthreads();
    for (int k = threadIdx.x; k < kNumBuckets; k += blockDim.x) {
        const int c = s_cur[k];
        s_cur[k] = c ? atomicAdd(cursor + k, c) : 0;
    }
    __syncthreads();
    for (int b0 = lo; b0 < hi; b0 += blockDim.x) {
        const int i = b0 + threadIdx.x;
        int b = 0;
        const int v = i < hi ? item(i, &b) : -1;
        const int at = warp_agg_inc(s_cur, b, v >= 0);
        if (v >= 0) out[at] = v;
    }
}

// Items per CTA of the segmented scatters.
constexpr int kScatterSegment = 2048;

__global__ void __launch_bounds__(kOrientThreads) orient_scatter_kernel(DevGraph g)
{
    __shared__ int s_cur[kNumBuckets];
    const int lo = blockIdx.x * kScatterSegment;
    const int hi = min(g.n, lo + kScatterSegment);
    segment_scatter(lo, hi, s_cur, g.bucket, g.sched, [&](int v, int *b) {
        const int c = g.pcount[v];
        if (c <= 0) return -1;
        *b = sched_bucket(c, g.offs[v + 1] - g.offs[v], g.ip, g.l2, g.core[v]);
        return v;
    });
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
    __shared__ int s_cnt[kNumBuckets];
    for (int i = threadIdx.x; i < kNumBuckets; i += blockDim.x) s_cnt[i] = 0;
    __syncthreads();
    for (int b0 = blockIdx.x * blockDim.x; b0 < n_roots; b0 += gridDim.x * blockDim.x) {
        const int i = b0 + threadIdx.x;
        const int v = i < n_roots ? roots[i] : 0;
        const bool ok = i < n_roots && v >= 0 && v < g.n;
        if (i < n_roots && !ok) set_status(g.ctrl, MCE_ERR_ID_RANGE);
        const int b = ok ? sched_bucket(g.pcount[v], g.offs[v + 1] - g.offs[v], g.ip, g.l2,
                                        g.core[v])
                         : 0;
        warp_agg_inc(s_cnt, b, ok);
    }
    __syncthreads();
    for (int k = threadIdx.x; k < kNumBuckets; k += blockDim.x)
        if (s_cnt[k]) atomicAdd(&g.ubucket[k], s_cnt[k]);
}

__global__ void bin_scan_kernel(DevGraph g)
{
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    buckets_to_cursors(g.ubucket, g.ctrl->ucls, nullptr);
}

__global__ void __launch_bounds__(kOrientThreads) bin_scatter_kernel(DevGraph g, const int *roots,
                                                                     int n_roots)
{
    __shared__ int s_cur[kNumBuckets];
    const int lo = blockIdx.x * kScatterSegment;
    const int hi = min(n_roots, lo + kScatterSegment);
    segment_scatter(lo, hi, s_cur, g.ubucket, g.uroots, [&](int i, int *b) {
        const int v = roots[i];
        if (v < 0 || v >= g.n) return -1;
        *b = sched_bucket(g.pcount[v], g.offs[v + 1] - g.offs[v], g.ip, g.l2, g.core[v]);
        return v;
    });
}

}  // namespace

cudaError_t launch_bin_roots(const DevGraph &g, const int *roots, int n_roots, cudaStream_t s)
{
    cudaError_t e = cudaMemsetAsync(g.ubucket, 0, sizeof(int) * kNumBuckets, s);
    if (e != cudaSuccess) return e;
    int b = (n_roots + kOrientThreads - 1) / kOrientThreads;
    if (b < 1) b = 1;
    if (b > 1024) b = 1024;
    bin_count_kernel<<<b, kOrientThreads, 0, s>>>(g, roots, n_roots);
    bin_scan_kernel<<<1, 32, 0, s>>>(g);
    const int segs = (n_roots + kScatterSegment - 1) / kScatterSegment;
    bin_scatter_kernel<<<segs > 0 ? segs : 1, kOrientThreads, 0, s>>>(g, roots, n_roots);
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

// The whole peel: one cooperative launch over peel_blocks CTAs (its dynamic shared memory
// exceeds the default 48 KiB: the limit is raised once per device).
cudaError_t launch_peel(const DevGraph &g, int peel_blocks, long long spin_limit_ns,
                        cudaStream_t s)
{
    constexpr int kMaxDev = 64;
    static bool configured[kMaxDev] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev || !configured[dev]) {
        e = cudaFuncSetAttribute((const void *)peel_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPeelSmemBytes);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < kMaxDev) configured[dev] = true;
    }
    DevGraph gg = g;
    long long lim = spin_limit_ns;
    void *args[] = {&gg, &lim};
    e = cudaLaunchCooperativeKernel((const void *)peel_kernel, dim3(peel_blocks),
                                    dim3(kPeelThreads), args, kPeelSmemBytes, s);
    if (e != cudaSuccess) return e;
    peel_rank_kernel<<<peel_blocks, kPeelThreads, 0, s>>>(g);
    return cudaGetLastError();
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
    orient_scatter_kernel<<<(g.n + kScatterSegment - 1) / kScatterSegment, kOrientThreads, 0, s>>>(g);
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
constexpr int kNoAllocWords = kNoAllocCtrlWords + 10 * kNoAllocMaxBlocks + 3 * kFrontCap +
                              6 * kNoAllocMaxN + 64;
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
    g.blk_gone = g.blk_cm + 4 * kNoAllocMaxBlocks;
    g.front = g.blk_gone + 2 * kNoAllocMaxBlocks;
    g.deg = g.front + 3 * kFrontCap;
    g.round_of = g.deg + kNoAllocMaxN;
    g.alive_a = g.round_of + kNoAllocMaxN;
    g.alive_b = g.alive_a + kNoAllocMaxN;
    g.order = g.alive_b + kNoAllocMaxN;
    g.rstart = g.order + kNoAllocMaxN;        // rounds <= n, plus one
    noalloc_prep_kernel<<<1, 1, 0, s>>>();
    if (cudaGetLastError() != cudaSuccess) return MCE_ERR_CUDA;
    if (n > 0 && launch_peel(g, blocks, 20LL * 1000 * 1000 * 1000, s) != cudaSuccess) {
        cudaGetLastError();
        return MCE_ERR_CUDA;
    }
    noalloc_result_kernel<<<1, 1, 0, s>>>(d_result);
    return cudaGetLastError() == cudaSuccess ? MCE_OK : MCE_ERR_CUDA;
}
