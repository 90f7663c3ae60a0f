// Device code of the search (included by search_full.cu and search_partial.cu, which
// instantiate its kernels).
//
// The search: Bron-Kerbosch with Tomita pivoting over independent first-level subtrees, one
// subtree per warp ("Parallelizing Maximal Clique Enumeration on GPUs", Sections 2.3-2.4 and 3).
//
// GB300 mapping (the pages assign a subtree to a thread block; here a warp is the unit of
// work, so that the many small subtrees of sparse graphs do not pay for block-wide barriers):
//   * one persistent kernel, as many CTAs as can be resident (Section 3.3); every warp claims
//     first-level roots from a global counter, heaviest |P| first;
//   * per root v, the warp builds the binary-encoded induced subgraph over P u X
//     (Sections 2.4 "Induced Subgraphs" and 3.4, the full variant): one bitset row per vertex
//     of N(v), with one column per vertex of P = later neighbours;
//   * X is kept compact (Section 3.5): X_P is a per-level bitset over the P columns, X_X a
//     single list of X rows that is partitioned in place as the search descends, with the end
//     of each level's part saved in its stack entry;
//   * the depth-first search is iterative with an explicit stack in the warp's workspace;
//     bitsets are spread over "sub-warps" of G lanes, each lane holding one 16-byte chunk of a
//     row (W <= 4 words: G = 1, every lane holds a whole row), so that row loads are 128-bit
//     and a pivot step scores 32/G rows at once; popcounts are reduced with shuffles.
// Rows, lists and the stack live in global memory (served by L1/L2); each warp has its own
// workspace sized at mce_create for the largest root of the graph.
#pragma once

#include <climits>

#include <cuda/atomic>

#include "mce_internal.cuh"

// Which induced subgraph the including translation unit builds (Section 3.4): 0 = full (rows
// for every vertex of P u X), 1 = partial (rows for P only; P-X adjacencies are looked up in
// the original graph, and the pivot comes from P u X_P).
// And which subtrees it searches: 0 = first-level (one per vertex, Algorithm 3), 1 =
// second-level (one per edge, Algorithm 4).
#if !defined(MCE_SEARCH_IP) || !defined(MCE_SEARCH_L2)
#error "define MCE_SEARCH_IP and MCE_SEARCH_L2 before including search_impl.cuh"
#endif

namespace mce {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr bool kIP = MCE_SEARCH_IP != 0;
constexpr bool kL2 = MCE_SEARCH_L2 != 0;

template <int W>
struct Geo {
    static constexpr int CH = W < 4 ? W : 4;   // words per lane chunk
    static constexpr int G = W / CH;           // lanes per row
    static constexpr int R = 32 / G;           // rows per warp step
};

template <int CH>
struct Ck {
    unsigned w[CH];
};

template <int CH>
__device__ __forceinline__ Ck<CH> ck_zero()
{
    Ck<CH> c;
#pragma unroll
    for (int i = 0; i < CH; ++i) c.w[i] = 0u;
    return c;
}

template <int CH>
__device__ __forceinline__ Ck<CH> ck_load(const unsigned *p)
{
    Ck<CH> c;
    if constexpr (CH == 4) {
        const uint4 t = *reinterpret_cast<const uint4 *>(p);
        c.w[0] = t.x; c.w[1] = t.y; c.w[2] = t.z; c.w[3] = t.w;
    } else if constexpr (CH == 2) {
        const uint2 t = *reinterpret_cast<const uint2 *>(p);
        c.w[0] = t.x; c.w[1] = t.y;
    } else {
        c.w[0] = *p;
    }
    return c;
}

template <int CH>
__device__ __forceinline__ void ck_store(unsigned *p, const Ck<CH> &c)
{
    if constexpr (CH == 4) {
        *reinterpret_cast<uint4 *>(p) = make_uint4(c.w[0], c.w[1], c.w[2], c.w[3]);
    } else if constexpr (CH == 2) {
        *reinterpret_cast<uint2 *>(p) = make_uint2(c.w[0], c.w[1]);
    } else {
        *p = c.w[0];
    }
}

template <int CH>
__device__ __forceinline__ Ck<CH> ck_and(const Ck<CH> &a, const Ck<CH> &b)
{
    Ck<CH> c;
#pragma unroll
    for (int i = 0; i < CH; ++i) c.w[i] = a.w[i] & b.w[i];
    return c;
}

template <int CH>
__device__ __forceinline__ Ck<CH> ck_andnot(const Ck<CH> &a, const Ck<CH> &b)
{
    Ck<CH> c;
#pragma unroll
    for (int i = 0; i < CH; ++i) c.w[i] = a.w[i] & ~b.w[i];
    return c;
}

template <int CH>
__device__ __forceinline__ Ck<CH> ck_or(const Ck<CH> &a, const Ck<CH> &b)
{
    Ck<CH> c;
#pragma unroll
    for (int i = 0; i < CH; ++i) c.w[i] = a.w[i] | b.w[i];
    return c;
}

template <int CH>
__device__ __forceinline__ bool ck_nonzero(const Ck<CH> &a)
{
    unsigned t = 0;
#pragma unroll
    for (int i = 0; i < CH; ++i) t |= a.w[i];
    return t != 0;
}

template <int CH>
__device__ __forceinline__ int ck_popc(const Ck<CH> &a)
{
    int t = 0;
#pragma unroll
    for (int i = 0; i < CH; ++i) t += __popc(a.w[i]);
    return t;
}

// Sum over the G lanes of a sub-warp (all lanes get the sum).
template <int G>
__device__ __forceinline__ int subwarp_sum(int x)
{
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
    return x;
}

template <int G>
__device__ __forceinline__ int subwarp_min(int x)
{
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) x = min(x, __shfl_xor_sync(kFull, x, o));
    return x;
}

// The bitset with bits [0, np) set, in chunk layout (lane chunk q holds words q*CH ..).
template <int W>
__device__ __forceinline__ Ck<Geo<W>::CH> bits_prefix(int np, int q)
{
    constexpr int CH = Geo<W>::CH;
    Ck<CH> c;
#pragma unroll
    for (int i = 0; i < CH; ++i) {
        const int k = q * CH + i;
        const int lo = k * 32;
        c.w[i] = np >= lo + 32 ? kFull : (np > lo ? ((1u << (np - lo)) - 1u) : 0u);
    }
    return c;
}

// Bits of `c` with index < b.
template <int W>
__device__ __forceinline__ Ck<Geo<W>::CH> bits_below(const Ck<Geo<W>::CH> &c, int b, int q)
{
    constexpr int CH = Geo<W>::CH;
    Ck<CH> r;
    const int wb = b >> 5;
    const unsigned m = (1u << (b & 31)) - 1u;
#pragma unroll
    for (int i = 0; i < CH; ++i) {
        const int k = q * CH + i;
        r.w[i] = k < wb ? c.w[i] : (k == wb ? (c.w[i] & m) : 0u);
    }
    return r;
}

// Index of the lowest set bit of `c` above `after` (after = -1: the lowest), or INT_MAX.
template <int W>
__device__ __forceinline__ int lowest_above(const Ck<Geo<W>::CH> &c, int after, int q)
{
    constexpr int CH = Geo<W>::CH;
    int best = INT_MAX;
#pragma unroll
    for (int i = CH - 1; i >= 0; --i) {
        const int k = q * CH + i;
        unsigned w = c.w[i];
        const int lo = k * 32;
        if (after >= lo + 31) w = 0u;
        else if (after >= lo) w &= ~((2u << (after - lo)) - 1u);
        if (w) best = lo + __ffs(w) - 1;
    }
    return subwarp_min<Geo<W>::G>(best);
}

struct Acc {
    unsigned long long count, hash, nodes, donations;
    unsigned long long words;   // bitset words scored / intersected / tested (lane 0 counts)
#ifdef MCE_PROFILE
    unsigned long long prof[kProfSlots];
#endif
};

// Activity timers of the MCE_PROFILE build (no code otherwise).
#ifdef MCE_PROFILE
#define PROF_START(var) const long long var = clock64()
#define PROF_ADD(acc, slot, var) ((acc).prof[slot] += (unsigned long long)(clock64() - (var)))
#else
#define PROF_START(var) (void)0
#define PROF_ADD(acc, slot, var) (void)0
#endif
enum { kProfBuild = 0, kProfPivot, kProfChild, kProfPartition, kProfDonate, kProfIdle,
       kProfMaxRoot, kProfRoots, kProfSmall, kProfSplit, kProfHash, kProfWalk, kProfXList };

struct RootCtx {
    unsigned *rowsP, *rowsX;
    int *pids;
    unsigned long long *pkey;
    int *rids, *xids, *xx, *spill, *plist;
    unsigned *stack;
    int deg, np, nx, LV;
    int rsize;          // |R| at level 0 (1 for a first-level root, 2 for a second-level one)
    int lay_deg, lay_np;   // the workspace layout in use: that of a root of this degree and |P|
};

// Inbox header of a warp workspace (word offsets) and inbox states.
enum { kHdrDeg = 0, kHdrNp = 1, kHdrK = 2, kHdrRsize = 3, kHdrS = 4, kHdrLayDeg = 6,
       kHdrLayNp = 7, kHdrP = 16, kHdrXP = 48 };
enum : int { kInboxIdle = 0, kInboxFull = 1, kInboxRetired = 2, kInboxClaimed = 4 };
constexpr long long kDonateCheckCycles = 2048;   // a donor looks at the worker list this often

using dev_int = cuda::atomic_ref<int, cuda::thread_scope_device>;
using dev_uint = cuda::atomic_ref<unsigned, cuda::thread_scope_device>;
using dev_ull = cuda::atomic_ref<unsigned long long, cuda::thread_scope_device>;

// Regions of a workspace laid out for a root of degree lay_deg with lay_np later neighbours,
// holding a subtree with np vertices in P and nx in X (the same sizes for a first-level root;
// at most those for a second-level subtree of that root).  X rows follow the P rows.
template <int W>
__device__ __forceinline__ RootCtx make_ctx(unsigned *ws, int lay_deg, int lay_np, int np, int nx)
{
    const WsLayout lay = ws_layout(lay_deg, lay_np, kIP, kL2);
    RootCtx r;
    r.rowsP = ws + lay.rowsP;
    r.rowsX = r.rowsP + (long long)np * W;
    r.pids = reinterpret_cast<int *>(ws + lay.pids);
    r.pkey = reinterpret_cast<unsigned long long *>(ws + lay.pkey);
    r.rids = reinterpret_cast<int *>(ws + lay.rids);
    r.xids = reinterpret_cast<int *>(ws + lay.xids);
    r.xx = reinterpret_cast<int *>(ws + lay.xx);
    r.spill = reinterpret_cast<int *>(ws + lay.spill);
    r.plist = reinterpret_cast<int *>(ws + lay.plist);
    r.stack = ws + lay.stack;
    r.deg = np + nx;
    r.np = np;
    r.nx = nx;
    r.LV = lay.LV;
    r.rsize = 1;
    r.lay_deg = lay_deg;
    r.lay_np = lay_np;
    return r;
}

#ifndef MCE_SMEM_STACK
#define MCE_SMEM_STACK 1
#endif
constexpr bool kSmemStack = MCE_SMEM_STACK != 0;
#ifndef MCE_SMEM_STACK_MIN_W
#define MCE_SMEM_STACK_MIN_W 1
#endif

// Stack entry of level L.  The first StackLevels<W> levels live in the warp's shared memory,
// in the space of the P hash and its filter, which no search uses (a subtree's build, when the
// search kernel runs one, ends before its search starts); the others in the workspace.  The
// search carries a pointer to the warp's scratch words (the build's cursor arrays), which
// follow the hash and the filter: the stack starts a fixed distance before it.
template <int W>
struct StackLevels {
    static constexpr int k = W == 1 ? 0 : W == 2 ? 1 : W == 4 ? 2 : W == 8 ? 3 : W == 16 ? 4 : 5;
    static constexpr int LV = (8 + 3 * W + 3) & ~3;               // ws_layout's level size
    static constexpr int value = kSmemStack && W >= MCE_SMEM_STACK_MIN_W ? (64 << k) * 2 + kFilterWords : 0;
    static constexpr int levels = value / LV;
};

template <int W>
__device__ __forceinline__ unsigned *stack_at(unsigned *scratch, const RootCtx &r, int L)
{
    if (L < StackLevels<W>::levels) return scratch - StackLevels<W>::value + L * StackLevels<W>::LV;
    return r.stack + (long long)L * r.LV;
}

// Id of element e of the clique R u {c} at level L: R's level-0 part, then the vertex chosen
// at each level below L, then c.
template <int W>
__device__ __forceinline__ int clique_elem(unsigned *scratch, const RootCtx &r, int L, int c,
                                           int e)
{
    if (e < r.rsize) return r.rids[e];
    const int loc = e < r.rsize + L ? (int)stack_at<W>(scratch, r, e - r.rsize)[3] : c;
    return r.pids[loc];
}

// Reports the maximal clique R u {c}: `size` vertices, hash input `hsum` (sum of keys).
template <int W>
__device__ void report(const SearchArgs &a, const RootCtx &r, int L, int c, int size,
                       unsigned long long hsum, Acc &acc, unsigned long long *s_hist, int lane,
                       unsigned *scratch)
{
    if (size >= a.out.hist_len) {                   // cannot happen: size <= d + 1
        if (lane == 0) set_status(a.g.ctrl, MCE_ERR_INTERNAL);
        return;
    }
    if (a.out.ids == nullptr) {
        if (lane == 0) {
            acc.count++;
            acc.hash += mix64(hsum);
            atomicAdd(&s_hist[size], 1ULL);
        }
        return;
    }
    // enumeration: slot in the group of cliques of this size, then ids in ascending order
    unsigned long long slot = 0;
    if (lane == 0) slot = atomicAdd(&a.out.cursor[size], 1ULL);
    slot = __shfl_sync(kFull, slot, 0);
    const long long cl = a.out.region_cl[size] + (long long)slot;
    if (cl >= a.out.region_cl[size + 1]) {          // more cliques than the counting pass saw
        if (lane == 0) set_status(a.g.ctrl, MCE_ERR_BUFFER_TOO_SMALL);
        return;
    }
    const long long base = a.out.region_ids[size] + (long long)slot * size;
    if (lane == 0) a.out.offsets[cl] = base;
    for (int e = lane; e < size; e += 32) {
        const int id = clique_elem<W>(scratch, r, L, c, e);
        int rk = 0;
        for (int f = 0; f < size; ++f) rk += clique_elem<W>(scratch, r, L, c, f) < id;
        a.out.ids[base + rk] = id;
    }
}

// Writes the indices of the set bits of a chunked bitset to out[], ascending; returns how many.
template <int W>
__device__ __forceinline__ int list_bits(const Ck<Geo<W>::CH> &b, int *out, int lane)
{
    constexpr int CH = Geo<W>::CH;
    int cnt = 0;
#pragma unroll
    for (int k = 0; k < W; ++k) {
        // with whole rows per lane (G = 1) every lane already holds word k
        const unsigned wk = Geo<W>::G == 1 ? b.w[k % CH] : __shfl_sync(kFull, b.w[k % CH], k / CH);
        const bool bit = (wk >> lane) & 1u;
        const unsigned m = __ballot_sync(kFull, bit);
        if (bit) out[cnt + __popc(m & ((1u << lane) - 1u))] = k * 32 + lane;
        cnt += __popc(m);
    }
    __syncwarp();
    return cnt;
}

// Is id in the id-sorted list a[lo .. hi)?
__device__ __forceinline__ bool sorted_has(const int *a, int lo, int hi, int id)
{
    const int end = hi;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(a + mid) < id) lo = mid + 1;
        else hi = mid;
    }
    return lo < end && __ldg(a + lo) == id;
}

// Partial induced subgraphs: is the X vertex x adjacent to the P vertex p?  p comes after x in
// the order, so it is in x's later-neighbour list N+(x), which is sorted by id: a binary search
// of the original graph (Section 3.4).
__device__ __forceinline__ bool x_adjacent(const DevGraph &g, int x, int p)
{
    int lo = __ldg(g.offs + x);
    const int end = lo + __ldg(g.pcount + x);
    int hi = end;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(g.padj + mid) < p) lo = mid + 1;
        else hi = mid;
    }
    return lo < end && __ldg(g.padj + lo) == p;
}

// Tomita pivot over P u X_P (bits of P | XP) and the live X_X rows xx[0..lpX): the row with
// the most neighbours in P, ties to the smaller code.  Returns -1 when some vertex of X is
// adjacent to all of P (no maximal clique below this node: every branch would be cut).  With
// partial induced subgraphs X_X has no rows, and the pivot comes from P u X_P only (Section 3.5,
// last paragraph).
template <int W>
__device__ int choose_pivot(const RootCtx &r, const Ck<Geo<W>::CH> &P, const Ck<Geo<W>::CH> &PX,
                            int npop, int lpX, Acc &acc, int lane)
{
    constexpr int CH = Geo<W>::CH, G = Geo<W>::G, R = Geo<W>::R;
    const int q = lane % G, sub = lane / G;
    // list the members of P u X_P
    const int cntp = list_bits<W>(PX, r.plist, lane);
    const int total = kIP ? cntp : cntp + lpX;
    unsigned best = 0;
    for (int base = 0; base < total; base += R) {
        const int t = base + sub;
        const bool valid = t < total;
        int code = 0;
        const unsigned *row = r.rowsP;
        if (valid) {
            if (t < cntp) {
                code = r.plist[t];
                row = r.rowsP + (long long)code * W;
            } else {
                const int x = r.xx[t - cntp];
                code = r.np + x;
                row = r.rowsX + (long long)x * W;
            }
        }
        const Ck<CH> rc = valid ? ck_load<CH>(row + q * CH) : ck_zero<CH>();
        const int cnt = subwarp_sum<G>(ck_popc<CH>(ck_and<CH>(P, rc)));
        if (valid) {
            const unsigned key = ((unsigned)cnt << kMaxIdxBits) | (unsigned)(kMaxCode - code);
            best = key > best ? key : best;
        }
        if (lane == 0) acc.words += (unsigned long long)W * (unsigned)min(R, total - base);
        if (__any_sync(kFull, valid && cnt == npop)) return -1;
    }
    best = __reduce_max_sync(kFull, best);
    return kMaxCode - (int)(best & (unsigned)kMaxCode);
}

// Does some live X_X row have bit c?  (X_X n N(c) non-empty)
template <int W>
__device__ __forceinline__ bool xx_hits(const DevGraph &g, const RootCtx &r, int lpX, int c,
                                        Acc &acc, int lane)
{
    const int wc = c >> 5;
    const unsigned bit = 1u << (c & 31);
    const int pc = kIP ? r.pids[c] : 0;
    for (int base = 0; base < lpX; base += 32) {
        const int i = base + lane;
        bool hit = false;
        if (i < lpX) {
            if constexpr (kIP) hit = x_adjacent(g, r.xids[r.xx[i]], pc);
            else hit = (r.rowsX[(long long)r.xx[i] * W + wc] & bit) != 0u;
        }
        if (lane == 0) acc.words += (unsigned)min(32, lpX - base);
        if (__any_sync(kFull, hit)) return true;
    }
    return false;
}

// Moves the X_X rows adjacent to c to the front of xx[0..lpX) (order kept) and returns their
// number; the others follow, so the parent's range xx[0..lpX) still holds the same set.
template <int W>
__device__ int xx_partition(const DevGraph &g, const RootCtx &r, int lpX, int c, int lane)
{
    const int wc = c >> 5;
    const unsigned bit = 1u << (c & 31);
    const int pc = kIP ? r.pids[c] : 0;
    const unsigned lt = (1u << lane) - 1u;
    if (lpX <= 32) {
        // one row per lane: every lane has read its row before any lane writes, so the rows go
        // straight to their places (kept first, then the others, each in the old order)
        const bool in = lane < lpX;
        const int x = in ? r.xx[lane] : 0;
        bool keep = false;
        if (in) {
            if constexpr (kIP) keep = x_adjacent(g, r.xids[x], pc);
            else keep = (r.rowsX[(long long)x * W + wc] & bit) != 0u;
        }
        const unsigned mk = __ballot_sync(kFull, keep);
        const unsigned mr = __ballot_sync(kFull, in && !keep);
        __syncwarp();
        if (keep) r.xx[__popc(mk & lt)] = x;
        else if (in) r.xx[__popc(mk) + __popc(mr & lt)] = x;
        __syncwarp();
        return __popc(mk);
    }
    int kept = 0, rem = 0;
    for (int base = 0; base < lpX; base += 32) {
        const int i = base + lane;
        const bool in = i < lpX;
        const int x = in ? r.xx[i] : 0;
        bool keep = false;
        if (in) {
            if constexpr (kIP) keep = x_adjacent(g, r.xids[x], pc);
            else keep = (r.rowsX[(long long)x * W + wc] & bit) != 0u;
        }
        const unsigned mk = __ballot_sync(kFull, keep);
        const unsigned mr = __ballot_sync(kFull, in && !keep);
        if (keep) r.xx[kept + __popc(mk & lt)] = x;
        else if (in) r.spill[rem + __popc(mr & lt)] = x;
        kept += __popc(mk);
        rem += __popc(mr);
        __syncwarp();
    }
    for (int t = lane; t < rem; t += 32) r.xx[kept + t] = r.spill[t];
    __syncwarp();
    return kept;
}

// ------------------------------------------------------------------ small subtrees
//
// Most nodes of a search tree sit near its leaves: on R-MAT, four in five internal nodes have
// |P| <= 8.  Below a node (R, P, X) the search reports exactly the cliques R u C with C a
// nonempty subset of P that is a clique, that no other vertex of P extends, and that no vertex
// of X extends (the invariant of Algorithm 2: every vertex adjacent to all of R is in R, P or
// X).  Which pivots the search would pick below the node changes only the path to these
// cliques, not the set.  So for |P| = k <= kSmallP the warp decides all 2^k subsets at once
// instead of walking the subtree:
//   * P's members p_0 .. p_{k-1} (ascending) renumber the node's columns; N_i is the closed
//     neighbourhood of p_i inside P, as a k-bit mask;
//   * C is a maximal clique of G[P] iff, for every i < k, C is a subset of N_i exactly when i is
//     in C; the 2^k subsets are bit-sliced over the lanes (lane l holds subsets
//     32 l .. 32 l + 31), so each of the k tests is a handful of word operations;
//   * each such C (there are few) is reported unless some vertex of X is adjacent to all of it:
//     for X_P that is one AND of C's own rows (the rows are symmetric on the columns of P), for
//     X_X the lanes test 32 rows at a time, as the pivot scan would.
// Count mode only (enumeration walks the subtree, so that every clique is written as before).


// kSubsets5[m]: bit t set iff the 5-bit value t is a subset of the 5-bit value m.
struct Subsets5 {
    unsigned v[32];
    constexpr Subsets5() : v()
    {
        for (int m = 0; m < 32; ++m) {
            unsigned w = 0;
            for (int t = 0; t < 32; ++t)
                if ((t & ~m) == 0) w |= 1u << t;
            v[m] = w;
        }
    }
};
__constant__ Subsets5 kSubsets5 = Subsets5();

// Subsets C (of up to 10 bits) that lane l's word holds, C = 32 l + t: the bits t with C a
// subset of m.
__device__ __forceinline__ unsigned subsets_of(unsigned m, int lane)
{
    return kSubsets5.v[m & 31u] & ((((unsigned)lane & ~(m >> 5)) & 31u) ? 0u : 0xffffffffu);
}

// The same word's subsets that contain element i.
__device__ __forceinline__ unsigned subsets_with(int i, int lane)
{
    constexpr unsigned kZ[5] = {0xAAAAAAAAu, 0xCCCCCCCCu, 0xF0F0F0F0u, 0xFF00FF00u, 0xFFFF0000u};
    return i < 5 ? kZ[i] : (((unsigned)lane >> (i - 5)) & 1u ? 0xffffffffu : 0u);
}

// The bits of v at the positions of the set bits of m, packed in ascending order (m is the same
// in every lane, so the loop is uniform).
template <int W>
__device__ __forceinline__ unsigned gather_bits(const Ck<W> &v, const Ck<W> &m)
{
    unsigned out = 0;
    int j = 0;
#pragma unroll
    for (int w = 0; w < W; ++w) {
        unsigned pm = m.w[w];
        const unsigned vw = v.w[w];
        while (pm) {
            const int b = __ffs(pm) - 1;
            out |= ((vw >> b) & 1u) << j;
            ++j;
            pm &= pm - 1u;
        }
    }
    return out;
}

// Reports every maximal clique below the node (R, P, X_P u X_X) at level L, |P| = k <= kSmallP
// (rows of whole words per lane, W <= 4).  scratch: 36 words of the warp's shared memory.
template <int W>
__device__ void solve_small(const SearchArgs &a, const RootCtx &r, const Ck<W> &P,
                            const Ck<W> &XP, int lpX, unsigned long long S, int L, int k,
                            Acc &acc, unsigned long long *s_hist, unsigned *scratch, int lane)
{
    int *mem = reinterpret_cast<int *>(scratch);                          // columns of P
    unsigned long long *keys = reinterpret_cast<unsigned long long *>(scratch + 16);
    // lane j < k: the column of p_j (the j-th member of P, ascending)
    int my_p = 0;
    {
        int j = 0;
#pragma unroll
        for (int w = 0; w < W; ++w) {
            unsigned pm = P.w[w];
            while (pm) {
                const int b = __ffs(pm) - 1;
                if (lane == j) my_p = w * 32 + b;
                ++j;
                pm &= pm - 1u;
            }
        }
    }
    unsigned adj = 0;                                         // lane i < k: N(p_i) n P, packed
    if (lane < k) {
        mem[lane] = my_p;
        adj = gather_bits<W>(ck_load<W>(r.rowsP + (long long)my_p * W), P);
        keys[lane] = r.pkey[my_p];
    }
    // maximal cliques of G[P]: subsets of {0..k-1} with [C subset of N_i] == [i in C] for all i
    unsigned V = subsets_of((1u << k) - 1u, lane);
    for (int i = 0; i < k; ++i) {
        const unsigned ni = __shfl_sync(kFull, adj, i) | (1u << i);
        V &= ~(subsets_of(ni, lane) ^ subsets_with(i, lane));
    }
    __syncwarp();                                             // mem[], keys[] written
    const int rsize = r.rsize + L;
    unsigned long long words = (unsigned long long)k * W + (unsigned long long)k * ((1u << k) + 31u) / 32u;
    unsigned cand = __ballot_sync(kFull, V != 0u);
    while (cand) {
        // the next candidate C (the same in every lane), as a set of columns
        const int src = __ffs(cand) - 1;
        const unsigned vs = __shfl_sync(kFull, V, src);
        const unsigned C = (unsigned)src * 32u + (unsigned)(__ffs(vs) - 1);
        if (lane == src) V &= V - 1u;
        cand = __ballot_sync(kFull, V != 0u);
        // C as columns, and the columns adjacent to every member of C (rows are symmetric on
        // the columns of P, so X_P's members adjacent to all of C are XP & AND of C's rows)
        Ck<W> cb = ck_zero<W>(), common;
#pragma unroll
        for (int w = 0; w < W; ++w) common.w[w] = 0xffffffffu;
        unsigned long long sum = S;
        for (unsigned cm = C; cm; cm &= cm - 1u) {
            const int j = __ffs(cm) - 1;
            const int col = mem[j];
#pragma unroll
            for (int w = 0; w < W; ++w) cb.w[w] |= (col >> 5) == w ? 1u << (col & 31) : 0u;
            common = ck_and<W>(common, ck_load<W>(r.rowsP + (long long)col * W));
            sum += keys[j];
        }
        words += (unsigned long long)__popc(C) * W;
        // extended by a vertex of X: a member of X_P adjacent to all of C, or an X_X row
        // containing all of C
        bool dominated = ck_nonzero<W>(ck_and<W>(XP, common));
        for (int base = 0; base < lpX && !dominated; base += 32) {
            const int t = base + lane;
            bool hit = false;
            if (t < lpX) {
                const int x = r.xx[t];
                if constexpr (kIP) {
                    hit = true;
                    const int xid = r.xids[x];
                    for (unsigned cm = C; cm && hit; cm &= cm - 1u)
                        hit = x_adjacent(a.g, xid, r.pids[mem[__ffs(cm) - 1]]);
                } else {
                    const Ck<W> rc = ck_load<W>(r.rowsX + (long long)x * W);
                    hit = !ck_nonzero<W>(ck_andnot<W>(cb, rc));
                }
            }
            dominated = __any_sync(kFull, hit);
            words += (unsigned long long)W * (unsigned)min(32, lpX - base);
        }
        if (dominated) continue;
        const int size = rsize + __popc(C);
        if (lane == 0) {
            if (size >= a.out.hist_len) {                     // cannot happen: size <= d + 1
                set_status(a.g.ctrl, MCE_ERR_INTERNAL);
            } else {
                acc.count++;
                acc.hash += mix64(sum);
                acc.nodes++;
                atomicAdd(&s_hist[size], 1ULL);
            }
        }
    }
    if (lane == 0) acc.words += words;
    __syncwarp();
}

// The same for rows wider than 4 words, whose lanes hold 4-word chunks: lane l holds chunk
// q = l % G of P, X_P and of every row it loads.  P's members are listed from the chunks (a
// prefix of their counts over the G lanes of a row); N_i takes k single bits of p_i's row; an
// X_P member extends C when the chunks of XP & AND of C's rows are nonzero in some lane; an X_X
// row (one per lane) extends C when it holds C's at most kSmallPMax columns.
template <int W>
__device__ void solve_small_wide(const SearchArgs &a, const RootCtx &r, const Ck<Geo<W>::CH> &P,
                                 const Ck<Geo<W>::CH> &XP, int lpX, unsigned long long S, int L,
                                 int k, Acc &acc, unsigned long long *s_hist, unsigned *scratch,
                                 int lane)
{
    constexpr int CH = Geo<W>::CH, G = Geo<W>::G;
    const int q = lane % G;
    int *mem = reinterpret_cast<int *>(scratch);                          // columns of P
    unsigned long long *keys = reinterpret_cast<unsigned long long *>(scratch + 16);
    {
        const int cnt = ck_popc<CH>(P);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < G; o <<= 1) {
            const int y = __shfl_up_sync(kFull, incl, o, G);
            if (q >= o) incl += y;
        }
        if (lane < G) {
            int j = incl - cnt;
#pragma unroll
            for (int w = 0; w < CH; ++w) {
                unsigned pm = P.w[w];
                while (pm) {
                    mem[j++] = (q * CH + w) * 32 + __ffs(pm) - 1;
                    pm &= pm - 1u;
                }
            }
        }
    }
    __syncwarp();
    unsigned adj = 0;                                         // lane i < k: N(p_i) n P, packed
    if (lane < k) {
        const int my_p = mem[lane];
        const unsigned *row = r.rowsP + (long long)my_p * W;
        for (int j = 0; j < k; ++j) {
            const int cj = mem[j];
            adj |= ((row[cj >> 5] >> (cj & 31)) & 1u) << j;
        }
        keys[lane] = r.pkey[my_p];
    }
    unsigned V = subsets_of((1u << k) - 1u, lane);
    for (int i = 0; i < k; ++i) {
        const unsigned ni = __shfl_sync(kFull, adj, i) | (1u << i);
        V &= ~(subsets_of(ni, lane) ^ subsets_with(i, lane));
    }
    __syncwarp();                                             // keys[] written
    const int rsize = r.rsize + L;
    unsigned long long words = (unsigned long long)k * k + (unsigned long long)k * ((1u << k) + 31u) / 32u;
    unsigned cand = __ballot_sync(kFull, V != 0u);
    while (cand) {
        const int src = __ffs(cand) - 1;
        const unsigned vs = __shfl_sync(kFull, V, src);
        const unsigned C = (unsigned)src * 32u + (unsigned)(__ffs(vs) - 1);
        if (lane == src) V &= V - 1u;
        cand = __ballot_sync(kFull, V != 0u);
        Ck<CH> common;
#pragma unroll
        for (int w = 0; w < CH; ++w) common.w[w] = 0xffffffffu;
        unsigned long long sum = S;
        for (unsigned cm = C; cm; cm &= cm - 1u) {
            const int j = __ffs(cm) - 1;
            common = ck_and<CH>(common, ck_load<CH>(r.rowsP + (long long)mem[j] * W + q * CH));
            sum += keys[j];
        }
        const int c = __popc(C);
        words += (unsigned long long)c * W;
        bool dominated = __any_sync(kFull, ck_nonzero<CH>(ck_and<CH>(XP, common)));
        for (int base = 0; base < lpX && !dominated; base += 32) {
            const int t = base + lane;
            bool hit = false;
            if (t < lpX) {
                const int x = r.xx[t];
                hit = true;
                if constexpr (kIP) {
                    const int xid = r.xids[x];
                    for (unsigned cm = C; cm && hit; cm &= cm - 1u)
                        hit = x_adjacent(a.g, xid, r.pids[mem[__ffs(cm) - 1]]);
                } else {
                    const unsigned *row = r.rowsX + (long long)x * W;
                    for (unsigned cm = C; cm && hit; cm &= cm - 1u) {
                        const int col = mem[__ffs(cm) - 1];
                        hit = (row[col >> 5] >> (col & 31)) & 1u;
                    }
                }
            }
            dominated = __any_sync(kFull, hit);
            words += (unsigned long long)c * (unsigned)min(32, lpX - base);
        }
        if (dominated) continue;
        const int size = rsize + c;
        if (lane == 0) {
            if (size >= a.out.hist_len) {                     // cannot happen: size <= d + 1
                set_status(a.g.ctrl, MCE_ERR_INTERNAL);
            } else {
                acc.count++;
                acc.hash += mix64(sum);
                acc.nodes++;
                atomicAdd(&s_hist[size], 1ULL);
            }
        }
    }
    if (lane == 0) acc.words += words;
    __syncwarp();
}

// ------------------------------------------------------------------ worker list (Section 3.3)
//
// Idle warps put their id in a bounded multi-producer multi-consumer ring (one slot per warp,
// so it cannot overflow) and wait on their inbox flag.  A busy warp ("donor") that is about to
// descend into a branch with |P| >= donate_min_p, with other branches left at the same level
// and at an earlier level, pops an idle warp, claims its inbox (idle -> claimed), writes the
// branch into the idle warp's workspace and publishes it (claimed -> full, release).  `busy`
// counts warps holding work; an idle warp leaves when roots are exhausted and busy == 0.  An
// idle warp that waited spin_limit_ns retires (idle -> retired); a donor that pops a retired
// warp keeps the branch.  Ring slots carry sequence numbers, so a slot is never reused before
// its previous value was taken.  Every wait is bounded.

__device__ bool ring_push(const SearchArgs &a, int w)
{
    const int t = dev_int(a.g.ctrl->ring_tail).fetch_add(1, cuda::memory_order_relaxed);
    const int slot = t % a.n_workers;
    dev_uint seq(a.ring_seq[slot]);
    const unsigned long long t0 = globaltimer_ns();
    unsigned ns = 32;
    while (seq.load(cuda::memory_order_acquire) != (unsigned)t) {
        if ((long long)(globaltimer_ns() - t0) > a.spin_limit_ns) {
            set_status(a.g.ctrl, MCE_ERR_DEVICE_TIMEOUT);
            return false;
        }
        __nanosleep(ns);
        if (ns < 1024) ns <<= 1;
    }
    a.ring[slot] = w;
    seq.store((unsigned)t + 1u, cuda::memory_order_release);
    return true;
}

// Pops an idle warp id, or -1 when the ring is empty (never waits).
__device__ int ring_try_pop(const SearchArgs &a)
{
    dev_int head(a.g.ctrl->ring_head), tail(a.g.ctrl->ring_tail);
    int h = head.load(cuda::memory_order_relaxed);
    for (int attempt = 0; attempt < 16; ++attempt) {
        if (h >= tail.load(cuda::memory_order_relaxed)) return -1;
        const int slot = h % a.n_workers;
        dev_uint seq(a.ring_seq[slot]);
        const unsigned sq = seq.load(cuda::memory_order_acquire);
        if (sq == (unsigned)h + 1u) {
            if (head.compare_exchange_strong(h, h + 1, cuda::memory_order_relaxed)) {
                const int w = a.ring[slot];
                seq.store((unsigned)h + (unsigned)a.n_workers, cuda::memory_order_release);
                return w;
            }
        } else if ((int)(sq - ((unsigned)h + 1u)) < 0) {
            return -1;                           // its pusher has not written the slot yet
        } else {
            h = head.load(cuda::memory_order_relaxed);
        }
    }
    return -1;
}

// Copies the branch R u {c} with sets (Pc, XPc, xx[0..k)) into the workspace `dst` of another
// warp: the P rows, the k live X rows (renumbered 0..k-1), the P ids and keys, R's ids.
template <int W>
__device__ void write_branch(unsigned *scratch, const RootCtx &r, unsigned *dst, int L, int c,
                             const Ck<Geo<W>::CH> &Pc, const Ck<Geo<W>::CH> &XPc, int k,
                             unsigned long long Sc, int lane)
{
    constexpr int CH = Geo<W>::CH, G = Geo<W>::G;
    const int q = lane % G;
    const WsLayout lay = ws_layout(r.lay_deg, r.lay_np, kIP, kL2);
    const int rsize = r.rsize + L + 1;
    if (lane == 0) {
        dst[kHdrDeg] = (unsigned)r.deg;
        dst[kHdrNp] = (unsigned)r.np;
        dst[kHdrLayDeg] = (unsigned)r.lay_deg;
        dst[kHdrLayNp] = (unsigned)r.lay_np;
        dst[kHdrK] = (unsigned)k;
        dst[kHdrRsize] = (unsigned)rsize;
        *reinterpret_cast<unsigned long long *>(dst + kHdrS) = Sc;
    }
    if (lane < G) {
        ck_store<CH>(dst + kHdrP + q * CH, Pc);
        ck_store<CH>(dst + kHdrXP + q * CH, XPc);
    }
    // the branch only ever touches rows (and ids, keys) of vertices in P' u X_P'
    const int nl = list_bits<W>(ck_or<CH>(Pc, XPc), r.plist, lane);
    for (long long t = lane; t < (long long)nl * W; t += 32) {
        const long long i = t / W;
        const long long off = (long long)r.plist[i] * W + (t - i * W);
        dst[lay.rowsP + off] = r.rowsP[off];
    }
    int *dxx = reinterpret_cast<int *>(dst + lay.xx);
    if constexpr (kIP) {
        // no X rows: the ids of the live X_X vertices, renumbered
        int *dxi = reinterpret_cast<int *>(dst + lay.xids);
        for (int i = lane; i < k; i += 32) dxi[i] = r.xids[r.xx[i]];
    } else {
        for (long long t = lane; t < (long long)k * W; t += 32) {
            const long long i = t / W;
            const int x = r.xx[i];
            dst[lay.rowsP + (long long)r.np * W + t] = r.rowsX[(long long)x * W + (t - i * W)];
        }
    }
    for (int i = lane; i < k; i += 32) dxx[i] = i;
    int *dp = reinterpret_cast<int *>(dst + lay.pids);
    unsigned long long *dk = reinterpret_cast<unsigned long long *>(dst + lay.pkey);
    for (int t = lane; t < nl; t += 32) {
        const int i = r.plist[t];
        dp[i] = r.pids[i];
        dk[i] = r.pkey[i];
    }
    int *dr = reinterpret_cast<int *>(dst + lay.rids);
    for (int e = lane; e < rsize; e += 32) dr[e] = clique_elem<W>(scratch, r, L, c, e);
    __threadfence();          // every lane's part of the branch is visible GPU-wide ...
    __syncwarp();             // ... before lane 0 publishes it
}

// Depth-first search of one first-level subtree (or donated branch) from the node
// (P, XP, xx[0..lpX)) at level 0 whose clique R has r.rsize vertices and key sum S.
template <int W>
__device__ void dfs(const SearchArgs &a, const RootCtx &r, Ck<Geo<W>::CH> P, Ck<Geo<W>::CH> XP,
                    int lpX, unsigned long long S, Acc &acc, unsigned long long *s_hist,
                    unsigned *scratch, int lane)
{
    constexpr int CH = Geo<W>::CH, G = Geo<W>::G;
    const int q = lane % G;
    int L = 0;
    bool enter = true;
    bool more_below = false;   // some level below L still has branches to explore
    Ck<CH> P0, XP0, C;
    int cursor = -1;
    long long last_check = __shfl_sync(kFull, (long long)clock64(), 0);
    while (true) {
        if (enter) {
            enter = false;
            acc.nodes++;
            PROF_START(t_piv);
            const int npop = subwarp_sum<G>(ck_popc<CH>(P));
            if constexpr (G == 1) {
                if (npop <= a.small_hi && npop >= a.small_lo && a.out.ids == nullptr) {
                    // the whole subtree at once; no stack entry, so the search backs up next
                    solve_small<W>(a, r, P, XP, lpX, S, L, npop, acc, s_hist, scratch, lane);
                    PROF_ADD(acc, kProfSmall, t_piv);
                    C = ck_zero<CH>();
                    cursor = -1;
                    goto next_candidate;
                }
            } else {
                if (npop <= a.small_hi && npop >= a.small_lo && a.out.ids == nullptr) {
                    solve_small_wide<W>(a, r, P, XP, lpX, S, L, npop, acc, s_hist, scratch, lane);
                    PROF_ADD(acc, kProfSmall, t_piv);
                    C = ck_zero<CH>();
                    cursor = -1;
                    goto next_candidate;
                }
            }
            const int piv = choose_pivot<W>(r, P, ck_or<CH>(P, XP), npop, lpX, acc, lane);
            PROF_ADD(acc, kProfPivot, t_piv);
            if (piv < 0) {
                C = ck_zero<CH>();
            } else {
                const unsigned *row = piv < r.np ? r.rowsP + (long long)piv * W
                                                 : r.rowsX + (long long)(piv - r.np) * W;
                C = ck_andnot<CH>(P, ck_load<CH>(row + q * CH));
            }
            P0 = P;
            XP0 = XP;
            cursor = -1;
            unsigned *lv = stack_at<W>(scratch, r, L);
            if (lane < G) {
                ck_store<CH>(lv + 8 + q * CH, P0);
                ck_store<CH>(lv + 8 + W + q * CH, XP0);
                ck_store<CH>(lv + 8 + 2 * W + q * CH, C);
            }
            if (lane == 0) {
                *reinterpret_cast<unsigned long long *>(lv) = S;
                lv[2] = (unsigned)lpX;
                lv[3] = 0xffffffffu;
                lv[4] = more_below ? 1u : 0u;
            }
            __syncwarp();
        }
    next_candidate:
        const int c = lowest_above<W>(C, cursor, q);
        if (c == INT_MAX) {                       // level exhausted: back up
            if (L == 0) return;
            --L;
            const unsigned *lv = stack_at<W>(scratch, r, L);
            P0 = ck_load<CH>(lv + 8 + q * CH);
            XP0 = ck_load<CH>(lv + 8 + W + q * CH);
            C = ck_load<CH>(lv + 8 + 2 * W + q * CH);
            S = *reinterpret_cast<const unsigned long long *>(lv);
            lpX = (int)lv[2];
            cursor = (int)lv[3];
            more_below = lv[4] != 0u;
            continue;
        }
        cursor = c;
        PROF_START(t_child);
        // branch on c: P at this point is P0 minus earlier candidates, X_P gained them
        const Ck<CH> pre = bits_below<W>(C, c, q);
        const Ck<CH> rc = ck_load<CH>(r.rowsP + (long long)c * W + q * CH);
        const Ck<CH> Pc = ck_and<CH>(ck_andnot<CH>(P0, pre), rc);
        const Ck<CH> XPc = ck_and<CH>(ck_or<CH>(XP0, pre), rc);
        const unsigned long long Sc = S + r.pkey[c];
        if (lane == 0) acc.words += 2 * W;
        if (!__any_sync(kFull, ck_nonzero<CH>(Pc))) {
            // leaf: R u {c} is maximal iff X n N(c) is empty (Algorithm 2, lines 2-3)
            if (!__any_sync(kFull, ck_nonzero<CH>(XPc)) && !xx_hits<W>(a.g, r, lpX, c, acc, lane)) {
                report<W>(a, r, L, c, r.rsize + L + 1, Sc, acc, s_hist, lane, scratch);
                acc.nodes++;
            }
            PROF_ADD(acc, kProfChild, t_child);
            continue;
        }
        const bool more_same = lowest_above<W>(C, c, q) != INT_MAX;
        if (lane == 0) stack_at<W>(scratch, r, L)[3] = (unsigned)c;
        PROF_ADD(acc, kProfChild, t_child);
        PROF_START(t_part);
        const int lpXc = xx_partition<W>(a.g, r, lpX, c, lane);
        PROF_ADD(acc, kProfPartition, t_part);
        if (lane == 0) acc.words += (unsigned)lpX;
        // worker list: hand this branch to an idle warp instead of descending (Section 3.3:
        // only when the donor keeps unexplored branches at this level and an earlier one;
        // donate_rule 1 accepts either)
        if (a.worker_list && (a.donate_rule ? (more_same || more_below)
                                            : (more_same && more_below))) {
            const long long now = __shfl_sync(kFull, (long long)clock64(), 0);
            // a branch worth the copy: |P'| at least donate_min_p and a quarter of the root's P
            const int min_p = a.donate_min_p > (r.np >> 2) ? a.donate_min_p : (r.np >> 2);
            if (now - last_check > kDonateCheckCycles &&
                subwarp_sum<G>(ck_popc<CH>(Pc)) >= min_p) {
                last_check = now;
                int recv = -1;
                if (lane == 0) {
                    recv = ring_try_pop(a);
                    if (recv >= 0) {
                        int expect = kInboxIdle;
                        if (!dev_int(a.flag[recv]).compare_exchange_strong(
                                expect, kInboxClaimed, cuda::memory_order_acq_rel))
                            recv = -1;                // it retired meanwhile
                        else
                            dev_int(a.g.ctrl->busy).fetch_add(1, cuda::memory_order_relaxed);
                    }
                }
                recv = __shfl_sync(kFull, recv, 0);
                PROF_START(t_don);
                if (recv >= 0) {
                    unsigned *dst = a.ws + (unsigned long long)recv * a.ws_words;
                    write_branch<W>(scratch, r, dst, L, c, Pc, XPc, lpXc, Sc, lane);
                    if (lane == 0) {
                        __threadfence();
                        dev_int(a.flag[recv]).store(kInboxFull, cuda::memory_order_release);
                        acc.donations++;
                    }
                    PROF_ADD(acc, kProfDonate, t_don);
                    continue;
                }
            }
        }
        more_below = more_below || more_same;
        lpX = lpXc;
        if (L + 1 > r.np) {                       // cannot happen: |P| shrinks at every level
            if (lane == 0) set_status(a.g.ctrl, MCE_ERR_INTERNAL);
            return;
        }
        ++L;
        P = Pc;
        XP = XPc;
        S = Sc;
        enter = true;
    }
}

// Per-warp shared memory of the build: open-addressing hash of P(v) (id -> local index), a
// one-hash bit filter of P(v) in front of it, cursors of the walk, and small roots' rows.
constexpr int kBatch = 8;   // N+ entries a lane loads before probing them

// The same for the normal roots' load-balanced walk, per row width (measured on R-MAT: 2-word
// rows run best with 4 loads in flight, 4-word rows with 12).
template <int W>
struct WalkBatch {
    static constexpr int value = W == 2 ? 4 : (W == 4 ? 12 : kBatch);
};

struct WarpSmem {
    int *hkey, *hval;
    unsigned *filter;            // kFilterWords words: bit f(id) set for every id of P(v)
    int slots;
    int *cur_start, *cur_base;   // build: per group of 32 neighbours, list starts and bases
    unsigned *rows;              // rows of a root small enough for shared memory
    int rows_words;
};

__device__ __forceinline__ unsigned hash_slot(int id, int mask)
{
    return ((unsigned)id * 0x9E3779B1u >> 7) & (unsigned)mask;
}

// The filter's bit of an id (a hash independent of the slot hash).
__device__ __forceinline__ unsigned filter_bit(int id)
{
    return ((unsigned)id * 0x85EBCA6Bu) >> (32 - kFilterLog2Bits);
}

// Local index of id in P(v), or -1.  Most walked ids are not in P: the filter answers for
// almost all of them with one shared-memory load.
__device__ __forceinline__ int hash_find(const WarpSmem &sm, int id)
{
    const unsigned f = filter_bit(id);
    if (!((sm.filter[f >> 5] >> (f & 31)) & 1u)) return -1;
    const int mask = sm.slots - 1;
    unsigned s = hash_slot(id, mask);
    while (true) {
        const int k = sm.hkey[s];
        if (k == id) return sm.hval[s];
        if (k < 0) return -1;
        s = (s + 1) & (unsigned)mask;
    }
}

// Load-balanced build of all rows (normal roots).  The neighbours u_t of v (P first, then X)
// are taken 32 at a time; the warp walks the concatenation of their lists N+(u_t) with
// consecutive lanes on consecutive entries (coalesced), WalkBatch entries per lane in flight.  A
// hit on p_j sets bit j of row t, and, when u_t = p_t is in P, bit t of row j as well.
template <int W, int kB = WalkBatch<W>::value>
__device__ void build_flat(const SearchArgs &a, const RootCtx &r, const WarpSmem &h, int deg,
                           int np, int lane)
{
    unsigned *rows = r.rowsP;   // rowsX follows rowsP directly
    for (int g0 = 0; g0 < deg; g0 += 32) {
        const int t = g0 + lane;
        int base = 0, len = 0;
        if (t < deg) {
            const int u = t < np ? r.pids[t] : r.xids[t - np];
            base = __ldg(a.g.offs + u);
            len = __ldg(a.g.pcount + u);
        }
        int incl = len;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += y;
        }
        const int total = __shfl_sync(kFull, incl, 31);
        h.cur_start[lane] = incl - len;
        h.cur_base[lane] = base;
        if (lane == 0) h.cur_start[32] = total;
        __syncwarp();
        // the list this lane is in, kept in registers for W >= 2: a lane's entries only move
        // forward, and long lists are crossed rarely (measured: the narrowest class, whose roots
        // see many short lists, runs faster reading the cursors from shared memory each time)
        int own = 0, own_start = 0, own_next = h.cur_start[1], own_base = h.cur_base[0];
        for (int f0 = 0; f0 < total; f0 += 32 * kB) {
            int w[kB], ow[kB];
#pragma unroll
            for (int b = 0; b < kB; ++b) {
                const int f = f0 + b * 32 + lane;
                ow[b] = -1;
                w[b] = -1;
                if (f < total) {
                    if constexpr (W == 1) {
                        while (h.cur_start[own + 1] <= f) ++own;
                        own_start = h.cur_start[own];
                        own_base = h.cur_base[own];
                    } else if (own_next <= f) {
                        do {
                            ++own;
                            own_start = own_next;
                            own_next = h.cur_start[own + 1];
                        } while (own_next <= f);
                        own_base = h.cur_base[own];
                    }
                    ow[b] = own;
                    w[b] = __ldg(a.g.padj + own_base + (f - own_start));
                }
            }
#pragma unroll
            for (int b = 0; b < kB; ++b) {
                if (ow[b] < 0) continue;
                const int j = hash_find(h, w[b]);
                if (j < 0) continue;
                const int tt = g0 + ow[b];
                atomicOr(rows + (long long)tt * W + (j >> 5), 1u << (j & 31));
                if (tt < np) atomicOr(rows + (long long)j * W + (tt >> 5), 1u << (tt & 31));
            }
        }
        __syncwarp();
    }
}

// Builds the induced subgraph of root v into the warp's workspace and searches it.
//
// Rows: for u in N(v), row(u) has bit i set iff u is adjacent to the i-th vertex of P (the
// binary-encoded induced subgraph over P u X, Section 3.4's full variant).  Every such
// adjacency u - p with p in P is found by streaming the later-neighbour list N+(u): a vertex of
// X precedes v and so precedes every p in P, hence p is in N+(u); a pair of P vertices is found
// from the earlier of the two.  Membership in P is a shared-memory hash lookup, so the build
// reads the bounded lists N+(u) (each at most d long) with coalesced loads and no search.
// Is some vertex of X adjacent to all of P?  Only an x with |N+(x)| >= |P| can be: per chunk of
// 32 * kBatch vertices of X the candidates are listed (kBatch gathers of |N+(x)| in flight per
// lane) and their lists walked, so a covering vertex early in X ends the test early (big
// roots only).
__device__ __forceinline__ bool x_covers_p(const DevGraph &g, const RootCtx &r, const WarpSmem &h,
                                        int np, int lane)
{
    const unsigned lt = (1u << lane) - 1u;
    bool covered = false;
    for (int base = 0; base < r.nx && !covered; base += 32 * kBatch) {
        int ncand = 0;
        {
            int x[kBatch], c[kBatch];
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
                const int xi = base + b * 32 + lane;
                x[b] = xi < r.nx ? r.xids[xi] : -1;
            }
#pragma unroll
            for (int b = 0; b < kBatch; ++b) c[b] = x[b] >= 0 ? __ldg(g.pcount + x[b]) : 0;
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
                const bool cand = x[b] >= 0 && c[b] >= np;
                const unsigned m = __ballot_sync(kFull, cand);
                if (cand) r.spill[ncand + __popc(m & lt)] = x[b];
                ncand += __popc(m);
            }
        }
        __syncwarp();
        for (int cb = 0; cb < ncand && !covered; cb += 32) {
            const int ci = cb + lane;
            int hits = 0;
            if (ci < ncand) {
                const int u = r.spill[ci];
                const int s0 = __ldg(g.offs + u), s1 = s0 + __ldg(g.pcount + u);
                for (int e0 = s0; e0 < s1; e0 += kBatch) {
                    int w[kBatch];
#pragma unroll
                    for (int b = 0; b < kBatch; ++b) w[b] = e0 + b < s1 ? __ldg(g.padj + e0 + b) : -1;
#pragma unroll
                    for (int b = 0; b < kBatch; ++b) hits += w[b] >= 0 && hash_find(h, w[b]) >= 0;
                }
            }
            covered = __any_sync(kFull, ci < ncand && hits == np);
        }
        __syncwarp();
    }
    return covered;
}

// Builds the induced subgraph of the subtree in r (its P and X ids already in r.pids, r.xids;
// R in r.rids) into the warp's workspace, or into shared memory when the rows fit, and searches
// it from R's key sum S.
template <int W, bool big>
__device__ void build_and_search(const SearchArgs &a, RootCtx r, const WarpSmem &sm,
                                 unsigned long long S, Acc &acc, unsigned long long *s_hist,
                                 int lane)
{
    constexpr int CH = Geo<W>::CH, G = Geo<W>::G;
    PROF_START(t_build);
    const int np = r.np, deg = r.deg;
    const unsigned lt = (1u << lane) - 1u;
    // rows in shared memory when they fit (normal roots only), else in the workspace; zero the
    // rows (the big-root build writes X rows whole when they are at most 4 words wide)
    if (!big && (long long)(kIP ? np : deg) * W <= sm.rows_words) {   // (big: a constant)
        r.rowsP = sm.rows;
        r.rowsX = sm.rows + (long long)np * W;
    }
    {
        const long long words = (long long)(kIP || (big && W <= 4) ? np : deg) * W;
        for (long long t = (long long)lane * CH; t < words; t += 32 * CH)
            ck_store<CH>(r.rowsP + t, ck_zero<CH>());
    }
    PROF_START(t_hash);
    int slots = 32;
    while (slots < 2 * np) slots <<= 1;
    WarpSmem h = sm;
    h.slots = slots;
    for (int i = lane; i < slots; i += 32) h.hkey[i] = -1;
    for (int i = lane; i < kFilterWords; i += 32) h.filter[i] = 0u;
    __syncwarp();
    for (int i = lane; i < np; i += 32) {
        const int id = r.pids[i];
        unsigned sl = hash_slot(id, slots - 1);
        while (atomicCAS(&h.hkey[sl], -1, id) != -1) sl = (sl + 1) & (unsigned)(slots - 1);
        h.hval[sl] = i;
        const unsigned f = filter_bit(id);
        atomicOr(&h.filter[f >> 5], 1u << (f & 31));
    }
    __syncwarp();
    PROF_ADD(acc, kProfHash, t_hash);
    int nxx = 0;
    bool covered = false;
    if constexpr (kIP) {
        // partial induced subgraph: P x P rows only; X_X starts as the whole of X
        build_flat<W>(a, r, h, np, np, lane);
        for (int i = lane; i < r.nx; i += 32) r.xx[i] = i;
        nxx = r.nx;
    } else if constexpr (!big) {
        PROF_START(t_walk);
        build_flat<W>(a, r, h, deg, np, lane);
        PROF_ADD(acc, kProfWalk, t_walk);
        PROF_START(t_xl);
        // X_X and the coverage test: a vertex of X adjacent to all of P makes every clique of
        // this subtree extendable (it is the Tomita pivot of the root with P - N(pivot) empty),
        // so the subtree holds no maximal clique
        for (int base = 0; base < r.nx; base += 32) {
            const int xi = base + lane;
            int cnt = 0;
            if (xi < r.nx)
                for (int k = 0; k < W; ++k) cnt += __popc(r.rowsX[(long long)xi * W + k]);
            covered = covered || __any_sync(kFull, cnt == np);
            const unsigned m = __ballot_sync(kFull, cnt > 0);
            if (cnt > 0) r.xx[nxx + __popc(m & lt)] = xi;
            nxx += __popc(m);
        }
        PROF_ADD(acc, kProfXList, t_xl);
        if (covered) {
            acc.nodes++;
            PROF_ADD(acc, kProfBuild, t_build);
            return;
        }
    } else {
    // A vertex of X adjacent to all of P makes every clique of this subtree extendable (it is
    // the Tomita pivot of the root with P - N(pivot) empty): the subtree holds no maximal
    // clique.  Such a vertex x has all of P in N+(x), so only those with |N+(x)| >= |P| can be
    // one.  A big root's X is mostly vertices with short lists: per chunk of 32 * kBatch
    // vertices of X, the candidates are listed (kBatch gathers of |N+(x)| in flight per lane)
    // and their lists walked, so a covering vertex early in X ends the root early.
    covered = x_covers_p(a.g, r, h, np, lane);
    if (covered) {
        acc.nodes++;
        PROF_ADD(acc, kProfBuild, t_build);
        return;
    }
    // X rows, one vertex per lane
    for (int base = 0; base < r.nx && !covered; base += 32) {
        const int xi = base + lane;
        int hits = 0;
        unsigned reg[W <= 4 ? W : 1];
#pragma unroll
        for (int k = 0; k < (W <= 4 ? W : 1); ++k) reg[k] = 0u;
        unsigned *row = r.rowsX + (long long)xi * W;
        if (xi < r.nx) {
            const int u = r.xids[xi];
            const int s0 = __ldg(a.g.offs + u), s1 = s0 + __ldg(a.g.pcount + u);
            for (int e0 = s0; e0 < s1; e0 += kBatch) {
                int w[kBatch];                           // independent loads in flight
#pragma unroll
                for (int b = 0; b < kBatch; ++b) w[b] = e0 + b < s1 ? __ldg(a.g.padj + e0 + b) : -1;
#pragma unroll
                for (int b = 0; b < kBatch; ++b) {
                    const int j = w[b] < 0 ? -1 : hash_find(h, w[b]);
                    if (j < 0) continue;
                    ++hits;
                    if constexpr (W <= 4) {
#pragma unroll
                        for (int k = 0; k < W; ++k) reg[k] |= (j >> 5) == k ? 1u << (j & 31) : 0u;
                    } else {
                        row[j >> 5] |= 1u << (j & 31);
                    }
                }
            }
            if constexpr (W <= 4) {
                Ck<CH> c;
#pragma unroll
                for (int k = 0; k < CH; ++k) c.w[k] = reg[k];
                ck_store<CH>(row, c);
            }
        }
        covered = __any_sync(kFull, hits == np && xi < r.nx);
        const unsigned m = __ballot_sync(kFull, hits > 0);
        if (hits > 0) r.xx[nxx + __popc(m & lt)] = xi;
        nxx += __popc(m);
    }
    if (covered) {
        acc.nodes++;
        PROF_ADD(acc, kProfBuild, t_build);
        return;
    }
    // P rows, one vertex per lane: the later P neighbours of p_i come from N+(p_i) ...
    for (int base = 0; base < np; base += 32) {
        const int i = base + lane;
        if (i < np) {
            const int u = r.pids[i];
            unsigned *row = r.rowsP + (long long)i * W;
            const int s0 = __ldg(a.g.offs + u), s1 = s0 + __ldg(a.g.pcount + u);
            for (int e0 = s0; e0 < s1; e0 += kBatch) {
                int w[kBatch];
#pragma unroll
                for (int b = 0; b < kBatch; ++b) w[b] = e0 + b < s1 ? __ldg(a.g.padj + e0 + b) : -1;
#pragma unroll
                for (int b = 0; b < kBatch; ++b) {
                    const int j = w[b] < 0 ? -1 : hash_find(h, w[b]);
                    if (j >= 0) row[j >> 5] |= 1u << (j & 31);
                }
            }
        }
    }
    __syncwarp();
    // ... and the earlier ones by symmetry: transpose 32 x 32 bit blocks with ballots
    const int nb = (np + 31) >> 5;
    for (int bi = 0; bi < nb; ++bi) {
        for (int bj = 0; bj < nb; ++bj) {
            const int ri = bi * 32 + lane;                 // this lane's row in block row bi
            const unsigned word = ri < np ? r.rowsP[(long long)ri * W + bj] : 0u;
            unsigned tr = 0;
#pragma unroll 4
            for (int k = 0; k < 32; ++k) {
                const unsigned col = __ballot_sync(kFull, (word >> k) & 1u);
                if (lane == k) tr = col;
            }
            // tr = word bi of row (bj * 32 + lane), as seen from the block (bi, bj)
            const int rj = bj * 32 + lane;
            __syncwarp();
            if (rj < np && tr) r.rowsP[(long long)rj * W + bi] |= tr;
            __syncwarp();
        }
    }
    }
    PROF_START(t_keys);
    for (int i = lane; i < np; i += 32) r.pkey[i] = vertex_key(r.pids[i]);
    __syncwarp();
    PROF_ADD(acc, kProfXList, t_keys);
    PROF_ADD(acc, kProfBuild, t_build);
    const int q = lane % G;
    dfs<W>(a, r, bits_prefix<W>(np, q), ck_zero<CH>(), nxx, S, acc, s_hist, reinterpret_cast<unsigned *>(sm.cur_start), lane);
}

// The split of a wide root's N(v) into P (later) and X (earlier), in id order, with kBatch rank
// gathers in flight per lane (big-workspace roots only).
__device__ __forceinline__ void split_wide(const DevGraph &g, const int *Nv, int deg, int rv, int *pids,
                                        int *xids, int lane)
{
    const unsigned lt = (1u << lane) - 1u;
    int pi = 0, xi = 0;
    for (int base = 0; base < deg; base += 32 * kBatch) {
        int w[kBatch], rk[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int j = base + b * 32 + lane;
            w[b] = j < deg ? __ldg(Nv + j) : -1;
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) rk[b] = w[b] >= 0 ? __ldg(g.rank + w[b]) : 0;
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const bool in = w[b] >= 0;
            const bool isP = in && rk[b] > rv;
            const unsigned mp = __ballot_sync(kFull, isP);
            const unsigned mx = __ballot_sync(kFull, in && !isP);
            if (isP) pids[pi + __popc(mp & lt)] = w[b];
            else if (in) xids[xi + __popc(mx & lt)] = w[b];
            pi += __popc(mp);
            xi += __popc(mx);
        }
    }
    __syncwarp();
}

// First-level subtree of root v (Algorithm 3): P = later neighbours, X = earlier ones.
//
// Rows: for u in N(v), row(u) has bit i set iff u is adjacent to the i-th vertex of P (the
// binary-encoded induced subgraph over P u X, Section 3.4's full variant).  Every such
// adjacency u - p with p in P is found by streaming the later-neighbour list N+(u): a vertex of
// X precedes v and so precedes every p in P, hence p is in N+(u); a pair of P vertices is found
// from the earlier of the two.  Membership in P is a shared-memory hash lookup, so the build
// reads the bounded lists N+(u) (each at most d long) with coalesced loads and no search.
template <int W, bool big>
__device__ void search_root(const SearchArgs &a, unsigned *ws, const WarpSmem &sm, int v, int deg,
                            int np, Acc &acc, unsigned long long *s_hist, int lane)
{
    PROF_START(t_split);
    RootCtx r = make_ctx<W>(ws, deg, np, np, deg - np);
    const int *Nv = a.g.adj + a.g.offs[v];
    const int rv = a.g.rank[v];
    const unsigned lt = (1u << lane) - 1u;
    // split N(v) into P (later) and X (earlier), numbering each part in id order; a wide
    // root keeps kBatch rank gathers in flight per lane
    if (big && deg > 32 * kBatch) {
        split_wide(a.g, Nv, deg, rv, r.pids, r.xids, lane);
    } else {
        int pi = 0, xi = 0;
        for (int base = 0; base < deg; base += 32) {
            const int j = base + lane;
            const bool in = j < deg;
            const int w = in ? __ldg(Nv + j) : 0;
            const bool isP = in && __ldg(a.g.rank + w) > rv;
            const unsigned mp = __ballot_sync(kFull, isP);
            const unsigned mx = __ballot_sync(kFull, in && !isP);
            if (isP) r.pids[pi + __popc(mp & lt)] = w;
            else if (in) r.xids[xi + __popc(mx & lt)] = w;
            pi += __popc(mp);
            xi += __popc(mx);
        }
    }
    if (lane == 0) r.rids[0] = v;
    PROF_ADD(acc, kProfSplit, t_split);
    build_and_search<W, big>(a, r, sm, vertex_key(v), acc, s_hist, lane);
}

// ------------------------------------------------------------------ subtrees built ahead
//
// The default search (full induced subgraphs, first-level subtrees) of the roots of row width
// W <= 4 runs in two launches per launch group: build_kernel builds every root's
// induced subgraph into a record of its own (RecLayout), then the search kernel searches the
// records.  The build is a walk of later-neighbour lists that waits on L2 gathers; in a kernel
// of its own it runs with few registers at 32 warps per SM and kBuildBatch loads in flight per
// lane, where the search kernel of 4-word rows holds 24 warps and 12 loads.  The search kernel
// copies the P rows and only the X rows with a neighbour in P into shared memory when they fit
// (more roots fit than when every X row is copied), and otherwise reads the rows in the
// record.  Records are all or nothing: when they do not fit, every subtree is built by the
// search kernel itself.

// Are the records in use for this launch group?  (The build kernel and both search variants
// read the same total, so exactly one search variant does the work.)
__device__ __forceinline__ bool records_on(const SearchArgs &a)
{
    return a.rec_gate != nullptr && *a.rec_gate <= a.bb_quads;
}

// Does the root at place i of the list have a record?  (Both kernels decide by this alone.)
__device__ __forceinline__ bool has_record(const SearchArgs &a, int i)
{
    return a.bb != nullptr && a.rec_off[i + 1] > a.rec_off[i] && a.rec_off[i + 1] <= a.bb_quads;
}

// Is the record at place i sized for a root of this degree and |P|?  (Always, unless the
// offsets were computed for another arrangement of the list: then the kernels report
// MCE_ERR_INTERNAL instead of writing past the record.)
__device__ __forceinline__ bool record_matches(const SearchArgs &a, int i, int deg, int np, int W)
{
    return a.rec_off[i + 1] - a.rec_off[i] == rec_quads(deg, np, W);
}

// The build kernel's walk (rows of roots built ahead): the walk of build_flat, but an entry
// that passes P's filter (about 6 % on R-MAT) is not looked up at once.  It goes into a queue
// of the warp in shared memory (id, row), appended by ballot, and every 32 queued entries are
// looked up in the hash and set in the rows by the whole warp.  Probing at once would run the
// hash lookup and the row updates for the one or two positive lanes of most 32-entry steps.
__device__ __forceinline__ bool filter_hit(const WarpSmem &h, int id)
{
    const unsigned f = filter_bit(id);
    return (h.filter[f >> 5] >> (f & 31)) & 1u;
}

template <int W>
__device__ __forceinline__ void drain_queue(const WarpSmem &h, unsigned *rows, int np,
                                            const int *qw, const int *qt, int count, int lane)
{
    if (lane < count) {
        const int id = qw[lane], tt = qt[lane];
        const int mask = h.slots - 1;
        unsigned s = hash_slot(id, mask);
        int j = -1;
        while (true) {
            const int k = h.hkey[s];
            if (k == id) { j = h.hval[s]; break; }
            if (k < 0) break;
            s = (s + 1) & (unsigned)mask;
        }
        if (j >= 0) {
            atomicOr(rows + (long long)tt * W + (j >> 5), 1u << (j & 31));
            if (tt < np) atomicOr(rows + (long long)j * W + (tt >> 5), 1u << (tt & 31));
        }
    }
}

template <int W, int kB>
__device__ void build_flat_queued(const SearchArgs &a, const RootCtx &r, const WarpSmem &h,
                                  int *qw, int *qt, int deg, int np, int lane)
{
    unsigned *rows = r.rowsP;
    const unsigned lt = (1u << lane) - 1u;
    int qn = 0;                                   // queued entries (the same in every lane)
    for (int g0 = 0; g0 < deg; g0 += 32) {
        const int t = g0 + lane;
        int base = 0, len = 0;
        if (t < deg) {
            const int u = t < np ? r.pids[t] : r.xids[t - np];
            base = __ldg(a.g.offs + u);
            len = __ldg(a.g.pcount + u);
        }
        int incl = len;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += y;
        }
        const int total = __shfl_sync(kFull, incl, 31);
        h.cur_start[lane] = incl - len;
        h.cur_base[lane] = base;
        if (lane == 0) h.cur_start[32] = total;
        __syncwarp();
        int own = 0, own_start = 0, own_next = h.cur_start[1], own_base = h.cur_base[0];
        for (int f0 = 0; f0 < total; f0 += 32 * kB) {
            int w[kB], ow[kB];
#pragma unroll
            for (int b = 0; b < kB; ++b) {
                const int f = f0 + b * 32 + lane;
                ow[b] = -1;
                w[b] = -1;
                if (f < total) {
                    if (own_next <= f) {
                        do {
                            ++own;
                            own_start = own_next;
                            own_next = h.cur_start[own + 1];
                        } while (own_next <= f);
                        own_base = h.cur_base[own];
                    }
                    ow[b] = own;
                    w[b] = __ldg(a.g.padj + own_base + (f - own_start));
                }
            }
#pragma unroll
            for (int b = 0; b < kB; ++b) {
                const bool pos = ow[b] >= 0 && filter_hit(h, w[b]);
                const unsigned m = __ballot_sync(kFull, pos);
                if (m == 0u) continue;
                if (pos) {
                    const int at = qn + __popc(m & lt);
                    qw[at] = w[b];
                    qt[at] = g0 + ow[b];
                }
                qn += __popc(m);
                if (qn >= 32) {                   // a full warp's worth: look them up
                    __syncwarp();
                    drain_queue<W>(h, rows, np, qw, qt, 32, lane);
                    const int rest = qn - 32;     // at most 31 left: move them to the front
                    int kw = 0, kt = 0;
                    if (lane < rest) {
                        kw = qw[32 + lane];
                        kt = qt[32 + lane];
                    }
                    __syncwarp();
                    if (lane < rest) {
                        qw[lane] = kw;
                        qt[lane] = kt;
                    }
                    __syncwarp();
                    qn = rest;
                }
            }
        }
        __syncwarp();
    }
    if (qn > 0) {
        __syncwarp();
        drain_queue<W>(h, rows, np, qw, qt, qn, lane);
    }
    __syncwarp();
}

// A 1-word root builds its rows by binary search when its neighbours' later-neighbour lists
// hold at least this many entries on average (measured: R-MAT s20's average 227 gains 36 %;
// SBM's 34 loses to the walk, whose loads are independent where a search's are a chain).
#ifndef MCE_SEARCH_MIN_AVG_LIST
#define MCE_SEARCH_MIN_AVG_LIST 64
#endif
constexpr int kSearchMinAvgList = MCE_SEARCH_MIN_AVG_LIST;

// Rows of a 1-word root (|P| <= 32) by binary search: instead of walking N+(u) for each
// u in N(v) (about 225 entries per list on R-MAT), each member p_i of P is looked up in the
// id-sorted N+(u) (about log2 |N+(u)| loads).  The warp takes 32 / S neighbours at a time,
// S = |P| rounded up to a power of two lanes each, lane i of a group searching p_i; the
// group's ballot is row t.  u = p_t in P holds only later vertices in N+(u), so a pair
// (p_t, p_i) is searched only when p_i comes later than p_t, and the earlier one's hit also
// sets bit t of row i (kept per lane, OR-ed into row i at the end).  No atomics.
__device__ void build_rows_w1(const SearchArgs &a, const RootCtx &r, int deg, int np, int lane)
{
    int S = 1;
    while (S < np) S <<= 1;
    const int T = 32 / S;                       // neighbours per step
    const int sub = lane / S, i = lane % S;
    const int p = i < np ? r.pids[i] : -1;
    const int rp = i < np ? __ldg(a.g.rank + p) : 0;
    const unsigned gmask = S == 32 ? 0xffffffffu : ((1u << S) - 1u);
    unsigned sym = 0;                           // bit t: p_t is an earlier P-neighbour of p_i
    for (int t0 = 0; t0 < deg; t0 += T) {
        const int t = t0 + sub;
        bool found = false;
        if (t < deg && i < np) {
            const int u = t < np ? r.pids[t] : r.xids[t - np];
            // p_i can be in N+(u) only if it comes after u (always, for u in X)
            if (t >= np || rp > __ldg(a.g.rank + u)) {
                const int *lst = a.g.padj + __ldg(a.g.offs + u);
                int lo = 0, hi = __ldg(a.g.pcount + u);
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (__ldg(lst + mid) < p) lo = mid + 1;
                    else hi = mid;
                }
                found = lo < __ldg(a.g.pcount + u) && __ldg(lst + lo) == p;
            }
        }
        const unsigned m = __ballot_sync(kFull, found);
        if (found && t < np) sym |= 1u << t;
        if (i == 0 && t < deg) r.rowsP[t] = (m >> (sub * S)) & gmask;
    }
    // row i of P: its later P-neighbours (written above) and its earlier ones (sym, spread over
    // the groups' lanes i)
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
        if (o >= S) sym |= __shfl_xor_sync(kFull, sym, o);
    __syncwarp();
    if (lane < np) r.rowsP[lane] |= sym;
    __syncwarp();
}

// Builds the record of first-level root v (deg neighbours, np of them later) at rec.
template <int W>
__device__ void build_record(const SearchArgs &a, const WarpSmem &sm, int v, int deg, int np,
                             bool big, unsigned *rec, int lane)
{
    constexpr int CH = Geo<W>::CH;
    const RecLayout L = rec_layout(deg, np, W);
    const unsigned lt = (1u << lane) - 1u;
    RootCtx r{};
    r.rowsP = rec + L.rows;
    r.rowsX = r.rowsP + (long long)np * W;
    r.pids = reinterpret_cast<int *>(rec + L.pids);
    r.pkey = reinterpret_cast<unsigned long long *>(rec + L.pkey);
    r.xids = reinterpret_cast<int *>(rec + L.xx);       // X's ids while building
    r.xx = r.xids;                                      // then the live X rows, in place
    r.np = np;
    r.nx = deg - np;
    r.deg = deg;
    // split N(v) into P (later) and X (earlier), each in id order
    const int *Nv = a.g.adj + a.g.offs[v];
    const int rv = a.g.rank[v];
    if (deg > 32 * kBatch) {
        split_wide(a.g, Nv, deg, rv, r.pids, r.xids, lane);
    } else {
        int pi = 0, xi = 0;
        for (int base = 0; base < deg; base += 32) {
            const int j = base + lane;
            const bool in = j < deg;
            const int w = in ? __ldg(Nv + j) : 0;
            const bool isP = in && __ldg(a.g.rank + w) > rv;
            const unsigned mp = __ballot_sync(kFull, isP);
            const unsigned mx = __ballot_sync(kFull, in && !isP);
            if (isP) r.pids[pi + __popc(mp & lt)] = w;
            else if (in) r.xids[xi + __popc(mx & lt)] = w;
            pi += __popc(mp);
            xi += __popc(mx);
        }
    }
    __syncwarp();                                       // P's and X's ids written
    // the hash of P and its filter, for the walk and the covering test
    WarpSmem h = sm;
    auto hash_p = [&]() {
        int slots = 32;
        while (slots < 2 * np) slots <<= 1;
        h.slots = slots;
        for (int i = lane; i < slots; i += 32) h.hkey[i] = -1;
        for (int i = lane; i < kFilterWords; i += 32) h.filter[i] = 0u;
        __syncwarp();
        for (int i = lane; i < np; i += 32) {
            const int id = r.pids[i];
            unsigned sl = hash_slot(id, slots - 1);
            while (atomicCAS(&h.hkey[sl], -1, id) != -1) sl = (sl + 1) & (unsigned)(slots - 1);
            h.hval[sl] = i;
            const unsigned f = filter_bit(id);
            atomicOr(&h.filter[f >> 5], 1u << (f & 31));
        }
        __syncwarp();
    };
    // a root of the big-workspace group (a hub: X of thousands) is first tested for an X vertex
    // adjacent to all of P, which is found early in X when there is one (then no rows are
    // built: the subtree holds no maximal clique); the candidates' list goes in the rows' space
    bool covered = false, hashed = false;
    if (big) {
        hash_p();
        hashed = true;
        RootCtx rc = r;
        rc.spill = reinterpret_cast<int *>(r.rowsP);
        covered = x_covers_p(a.g, rc, h, np, lane);
    }
    int nxx = 0;
    if (!covered) {
        // 1-word roots whose later-neighbour lists are long on average: binary searches (the
        // walk's cost grows with the lists, the searches' with their logarithm)
        bool by_search = false;
        if constexpr (W == 1) {
            int walk = 0;
            for (int t = lane; t < deg; t += 32)
                walk += __ldg(a.g.pcount + (t < np ? r.pids[t] : r.xids[t - np]));
            by_search =
                __reduce_add_sync(kFull, (unsigned)walk) >= (unsigned)(kSearchMinAvgList * deg);
        }
        if (by_search) {
            build_rows_w1(a, r, deg, np, lane);
        } else {
            for (long long t = (long long)lane * CH; t < (long long)deg * W; t += 32 * CH)
                ck_store<CH>(r.rowsP + t, ck_zero<CH>());
            if (!hashed) hash_p();
            __syncwarp();
#ifndef MCE_QUEUED_MIN_W
#define MCE_QUEUED_MIN_W 4
#endif
            if constexpr (W >= MCE_QUEUED_MIN_W)
                build_flat_queued<W, kBuildBatch>(a, r, h, sm.cur_base + 36,
                                                  sm.cur_base + 36 + 64, deg, np, lane);
            else
                build_flat<W, kBuildBatch>(a, r, h, deg, np, lane);
        }
        // the X rows with a neighbour in P, and whether one X vertex is adjacent to all of P
        // (then the subtree holds no maximal clique: that vertex would be the root's Tomita
        // pivot with nothing left to branch on)
        for (int base = 0; base < r.nx; base += 32) {
            const int xi = base + lane;
            int cnt = 0;
            if (xi < r.nx)
                for (int k = 0; k < W; ++k) cnt += __popc(r.rowsX[(long long)xi * W + k]);
            covered = covered || __any_sync(kFull, cnt == np);
            const unsigned m = __ballot_sync(kFull, cnt > 0);
            if (cnt > 0) r.xx[nxx + __popc(m & lt)] = xi;
            nxx += __popc(m);
        }
    }
    for (int i = lane; i < np; i += 32) r.pkey[i] = vertex_key(r.pids[i]);
    if (lane == 0) {
        rec[0] = (unsigned)np;
        rec[1] = (unsigned)r.nx;
        rec[2] = (unsigned)nxx;
        rec[3] = covered ? 1u : 0u;
    }
    __syncwarp();
}

// Searches the subtree of root v from its record (built by build_kernel).
template <int W>
__device__ void search_record(const SearchArgs &a, unsigned *ws, const WarpSmem &sm, int v,
                              int deg, int np, const unsigned *rec, Acc &acc,
                              unsigned long long *s_hist, int lane)
{
    constexpr int CH = Geo<W>::CH, G = Geo<W>::G;
    PROF_START(t_build);
    const RecLayout L = rec_layout(deg, np, W);
    const int nxx = (int)rec[2];
    if (rec[3]) {                                       // an X vertex covers P
        acc.nodes++;
        PROF_ADD(acc, kProfBuild, t_build);
        return;
    }
    RootCtx r = make_ctx<W>(ws, deg, np, np, deg - np);
    r.pids = reinterpret_cast<int *>(const_cast<unsigned *>(rec) + L.pids);
    r.pkey = reinterpret_cast<unsigned long long *>(const_cast<unsigned *>(rec) + L.pkey);
    const int *live = reinterpret_cast<const int *>(rec + L.xx);
    const unsigned *rows = rec + L.rows;
    if ((long long)(np + nxx) * W <= sm.rows_words) {
        // P rows, then the live X rows packed, in shared memory
        for (long long t = (long long)lane * CH; t < (long long)np * W; t += 32 * CH)
            ck_store<CH>(sm.rows + t, ck_load<CH>(rows + t));
        for (long long t = (long long)lane * CH; t < (long long)nxx * W; t += 32 * CH) {
            const long long i = t / W;
            ck_store<CH>(sm.rows + (long long)np * W + t,
                         ck_load<CH>(rows + (long long)(np + live[i]) * W + (t - i * W)));
        }
        for (int i = lane; i < nxx; i += 32) r.xx[i] = i;
        r.rowsP = sm.rows;
        r.rowsX = sm.rows + (long long)np * W;
    } else {
        for (int i = lane; i < nxx; i += 32) r.xx[i] = live[i];
        r.rowsP = const_cast<unsigned *>(rows);
        r.rowsX = r.rowsP + (long long)np * W;
    }
    if (lane == 0) r.rids[0] = v;
    __syncwarp();
    PROF_ADD(acc, kProfBuild, t_build);
    const int q = lane % G;
    dfs<W>(a, r, bits_prefix<W>(np, q), ck_zero<CH>(), nxx, vertex_key(v), acc, s_hist,
           reinterpret_cast<unsigned *>(sm.cur_start), lane);
}

// Second-level subtree of the edge {v, w}, v before w (Algorithm 4): R = {v, w},
// P = N(v) n N(w) after w = N+(v) n N+(w), X = N(v) n N(w) before w.  The workspace keeps the
// layout of root v, which holds any of its second-level subtrees.
template <int W, bool big>
__device__ void search_edge(const SearchArgs &a, unsigned *ws, const WarpSmem &sm, int v, int w,
                            Acc &acc, unsigned long long *s_hist, int lane)
{
    const DevGraph &g = a.g;
    const int degv = g.offs[v + 1] - g.offs[v];
    RootCtx r = make_ctx<W>(ws, degv, g.pcount[v], 0, 0);
    const unsigned lt = (1u << lane) - 1u;
    // P: the later neighbours of v that are later neighbours of w too (both lists id-sorted)
    const int pv0 = g.offs[v], pv1 = pv0 + g.pcount[v];
    const int pw0 = g.offs[w], pw1 = pw0 + g.pcount[w];
    int np = 0;
    for (int j0 = pv0; j0 < pv1; j0 += 32) {
        const int j = j0 + lane;
        const int u = j < pv1 ? __ldg(g.padj + j) : -1;
        const bool in = u >= 0 && sorted_has(g.padj, pw0, pw1, u);
        const unsigned m = __ballot_sync(kFull, in);
        if (in) r.pids[np + __popc(m & lt)] = u;
        np += __popc(m);
    }
    // X: walk the shorter of N(v), N(w) and search the other; keep what comes before w
    const int rw = g.rank[w];
    const int degw = g.offs[w + 1] - g.offs[w];
    const bool walk_v = degv <= degw;
    const int a0 = walk_v ? g.offs[v] : g.offs[w], a1 = walk_v ? g.offs[v + 1] : g.offs[w + 1];
    const int b0 = walk_v ? g.offs[w] : g.offs[v], b1 = walk_v ? g.offs[w + 1] : g.offs[v + 1];
    int nx = 0;
    for (int j0 = a0; j0 < a1; j0 += 32) {
        const int j = j0 + lane;
        const int u = j < a1 ? __ldg(g.adj + j) : -1;
        const bool in = u >= 0 && u != v && u != w && __ldg(g.rank + u) < rw &&
                        sorted_has(g.adj, b0, b1, u);
        const unsigned m = __ballot_sync(kFull, in);
        if (in) r.xids[nx + __popc(m & lt)] = u;
        nx += __popc(m);
    }
    r = make_ctx<W>(ws, degv, g.pcount[v], np, nx);
    r.rsize = 2;
    if (lane == 0) {
        r.rids[0] = v;
        r.rids[1] = w;
    }
    __syncwarp();
    const unsigned long long S = vertex_key(v) + vertex_key(w);
    if (np == 0) {
        // P empty: {v, w} is maximal iff X is empty too
        if (nx == 0) report<W>(a, r, 0, 0, 2, S, acc, s_hist, lane, nullptr);   // level 0
        acc.nodes++;
        return;
    }
    build_and_search<W, big>(a, r, sm, S, acc, s_hist, lane);
}

// Searches a branch that another warp wrote into this warp's workspace.
template <int W>
__device__ void search_inbox(const SearchArgs &a, unsigned *ws, const WarpSmem &sm, Acc &acc,
                             unsigned long long *s_hist, int lane)
{
    constexpr int CH = Geo<W>::CH, G = Geo<W>::G;
    const int q = lane % G;
    const int deg = (int)ws[kHdrDeg], np = (int)ws[kHdrNp];
    const int k = (int)ws[kHdrK], rsize = (int)ws[kHdrRsize];
    const int lay_deg = (int)ws[kHdrLayDeg], lay_np = (int)ws[kHdrLayNp];
    constexpr bool l2 = kL2;
    // a branch always comes from a root of this kernel's class, within its workspace (a
    // second-level subtree is at most as large as its root's first-level one)
    const bool sane = lay_np >= 1 && lay_np <= kMaxP && wclass(lay_np) == W &&
                      lay_deg >= lay_np && np >= 1 && np <= lay_np && deg >= np &&
                      deg <= lay_deg && (l2 || (np == lay_np && deg == lay_deg)) && k >= 0 &&
                      k <= deg - np && rsize >= 2 && rsize <= np + 2 &&
                      (unsigned long long)ws_layout(lay_deg, lay_np, kIP, l2).total <= a.ws_words;
    if (!sane) {
        if (lane == 0) set_status(a.g.ctrl, MCE_ERR_INTERNAL);
        return;
    }
    RootCtx r = make_ctx<W>(ws, lay_deg, lay_np, np, deg - np);
    r.rsize = rsize;
    const unsigned long long S = *reinterpret_cast<const unsigned long long *>(ws + kHdrS);
    const Ck<CH> P = ck_load<CH>(ws + kHdrP + q * CH);
    const Ck<CH> XP = ck_load<CH>(ws + kHdrXP + q * CH);
    dfs<W>(a, r, P, XP, k, S, acc, s_hist, reinterpret_cast<unsigned *>(sm.cur_start), lane);
}

// The last i in [lo, hi) with a[i] <= t, for a non-decreasing a with a[lo] <= t: 32 probes
// per step, so a schedule of n roots takes about log32(n) rounds of loads.
__device__ __forceinline__ int last_at_most(const int *a, int lo, int hi, int t, int lane)
{
    while (hi - lo > 32) {
        const int step = (hi - lo + 31) >> 5;
        const int p = lo + lane * step;
        const unsigned m = __ballot_sync(kFull, p < hi && __ldg(a + p) <= t);
        lo += (31 - __clz(m)) * step;
        hi = min(hi, lo + step);
    }
    const unsigned m = __ballot_sync(kFull, lo + lane < hi && __ldg(a + lo + lane) <= t);
    return lo + 31 - __clz(m);
}

// CTAs per SM the compiler should plan registers for, per row width (more for narrow rows).
#ifndef MCE_MIN_BLOCKS_MID
#define MCE_MIN_BLOCKS_MID 6
#endif
// (measured: 2-word rows run best at 7, which leaves them 72 registers instead of 64)
template <int W>
struct MinBlocks {
    static constexpr int value = W == 1 ? 8 : (W == 2 ? 7 : (W <= 8 ? MCE_MIN_BLOCKS_MID : 4));
};

// First-level subtree of root v (or, with second-level subtrees, the subtree of its edge to w),
// searched with rows of W words.
template <int W, bool Big>
__device__ __forceinline__ void search_unit(const SearchArgs &a, unsigned *ws, const WarpSmem &sm,
                                            int v, int w, int deg, int np, Acc &acc,
                                            unsigned long long *s_hist, int lane)
{
    if constexpr (kL2) {
        if (w >= 0) search_edge<W, Big>(a, ws, sm, v, w, acc, s_hist, lane);
    } else {
        search_root<W, Big>(a, ws, sm, v, deg, np, acc, s_hist, lane);
    }
}

// One persistent launch per row width W and launch group: the roots of that class, heaviest
// first, then donated branches of those roots (Section 3.3).  Big: the group of roots whose
// workspace exceeds kWsCapWords (their build code is compiled into these instances only).
// Rec: the roots' subtrees were built ahead by build_kernel (W <= 4).
template <int W, bool Big, bool Rec = false>
__global__ void __launch_bounds__(128, MinBlocks<W>::value) search_kernel(SearchArgs a)
{
    if constexpr (!kIP && !kL2 && W <= 4) {
        if (a.rec_gate != nullptr && records_on(a) != Rec) return;   // the other variant works
    }
    extern __shared__ __align__(16) unsigned char s_raw[];
    unsigned long long *s_hist = reinterpret_cast<unsigned long long *>(s_raw);
    for (int i = threadIdx.x; i < a.out.hist_len; i += blockDim.x) s_hist[i] = 0ULL;
    const int lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    const int warp = blockIdx.x * wpb + (threadIdx.x >> 5);
    WarpSmem sm;
    {
        constexpr int k = W == 1 ? 0 : W == 2 ? 1 : W == 4 ? 2 : W == 8 ? 3 : W == 16 ? 4 : 5;
        unsigned char *mine = s_raw + smem_hist_bytes(a.out.hist_len) +
                              (size_t)(threadIdx.x >> 5) * warp_smem_bytes(k);
        sm.hkey = reinterpret_cast<int *>(mine);
        sm.hval = sm.hkey + hash_slots(k);
        sm.filter = reinterpret_cast<unsigned *>(sm.hval + hash_slots(k));
        sm.slots = hash_slots(k);
        sm.cur_start = reinterpret_cast<int *>(sm.filter + kFilterWords);
        sm.cur_base = sm.cur_start + 36;
        sm.rows = reinterpret_cast<unsigned *>(sm.cur_base + 36);   // 16-byte aligned
        sm.rows_words = smem_row_words(k);
    }
    __syncthreads();
    unsigned *ws = a.ws + (unsigned long long)warp * a.ws_words;
    const unsigned long long begin = (unsigned long long)a.range[2 * a.group];
    const int end = a.range[2 * a.group + 1];
    // work items: the roots of this launch, or with second-level subtrees their edges
    const int ubase = kL2 ? a.uoff[begin] : 0;
    const unsigned long long n_roots = kL2 ? (unsigned long long)(a.uoff[end] - ubase)
                                           : (unsigned long long)end - begin;
    dev_int busy(a.g.ctrl->busy);
    Acc acc{};
#ifdef MCE_PROFILE
    const long long t_kernel = clock64();
#endif
    // phase 1: first-level subtrees from the shared counter
    while (load_status(a.g.ctrl) == 0) {
        unsigned long long idx = 0;
        if (lane == 0) {
            busy.fetch_add(1, cuda::memory_order_relaxed);
            idx = atomicAdd(&a.g.ctrl->next_root, 1ULL);
            if (idx >= n_roots) busy.fetch_sub(1, cuda::memory_order_acq_rel);
        }
        idx = __shfl_sync(kFull, idx, 0);
        if (idx >= n_roots) break;
        PROF_START(t_root);
        int pos = (int)(begin + idx), w = -1;
        if constexpr (kL2) {
            // the root whose edges hold item idx, and the edge's later end w
            const int t = ubase + (int)idx;
            pos = last_at_most(a.uoff, (int)begin, end, t, lane);
            const int v0 = a.roots[pos];
            if (a.g.pcount[v0] > 0) w = a.g.padj[a.g.offs[v0] + (t - a.uoff[pos])];
        }
        const int v = a.roots[pos];
        const int deg = a.g.offs[v + 1] - a.g.offs[v];
        const int np = a.g.pcount[v];
        if (np == 0) {
            // R = {v}, P empty: maximal iff X is empty too, i.e. v is isolated
            if (deg == 0) {
                RootCtx single{};
                single.rids = reinterpret_cast<int *>(ws);
                single.rsize = 1;
                if (lane == 0) single.rids[0] = v;
                __syncwarp();
                report<W>(a, single, 0, 0, 1, vertex_key(v), acc, s_hist, lane, nullptr);
            }
        } else if (np > kMaxP) {
            if (lane == 0) set_status(a.g.ctrl, MCE_ERR_LIMIT);
        } else {
            if constexpr (Rec) {
                if (has_record(a, pos) && record_matches(a, pos, deg, np, W))
                    search_record<W>(a, ws, sm, v, deg, np, a.bb + a.rec_off[pos] * 4, acc,
                                     s_hist, lane);
                else if (lane == 0)
                    set_status(a.g.ctrl, MCE_ERR_INTERNAL);   // every root has a record
            } else {
                search_unit<W, Big>(a, ws, sm, v, w, deg, np, acc, s_hist, lane);
            }
        }
        __syncwarp();
        if (lane == 0) busy.fetch_sub(1, cuda::memory_order_acq_rel);
#ifdef MCE_PROFILE
        {
            const unsigned long long dt = (unsigned long long)(clock64() - t_root);
            acc.prof[kProfMaxRoot] = dt > acc.prof[kProfMaxRoot] ? dt : acc.prof[kProfMaxRoot];
            acc.prof[kProfRoots]++;
        }
#endif
    }
    // phase 2: receive donated branches until no warp holds work
    while (a.worker_list && load_status(a.g.ctrl) == 0) {
        int state = 0;   // 1: a branch arrived, 2: leave
        PROF_START(t_idle);
        if (lane == 0) {
            if (!ring_push(a, warp)) state = 2;
            dev_int flag(a.flag[warp]);
            const unsigned long long t0 = globaltimer_ns();
            unsigned ns = 64, polls = 0;
            while (state == 0) {
                const int f = flag.load(cuda::memory_order_acquire);
                const long long waited = (long long)(globaltimer_ns() - t0);
                if (f == kInboxFull) {
                    state = 1;
                } else if (f == kInboxIdle) {
                    // the shared counters are read on every 8th poll only (own flag every time)
                    if ((polls++ & 7u) == 0 &&
                        (busy.load(cuda::memory_order_acquire) == 0 || load_status(a.g.ctrl) != 0)) {
                        state = 2;                       // nothing left anywhere
                    } else if (waited > a.spin_limit_ns) {
                        int expect = kInboxIdle;
                        if (flag.compare_exchange_strong(expect, kInboxRetired,
                                                         cuda::memory_order_acq_rel))
                            state = 2;                   // retire; donors skip this warp
                    }
                } else if (waited > a.spin_limit_ns + a.spin_limit_ns) {
                    set_status(a.g.ctrl, MCE_ERR_DEVICE_TIMEOUT);   // claimed, never filled
                    state = 2;
                }
                if (state == 0) {
                    __nanosleep(ns);
                    if (ns < 2048) ns <<= 1;
                }
            }
            if (state == 1) flag.store(kInboxIdle, cuda::memory_order_release);
        }
        state = __shfl_sync(kFull, state, 0);
        PROF_ADD(acc, kProfIdle, t_idle);
        if (state != 1) break;
        __syncwarp();
        cuda::atomic_thread_fence(cuda::memory_order_acquire, cuda::thread_scope_device);
        search_inbox<W>(a, ws, sm, acc, s_hist, lane);
        __syncwarp();
        if (lane == 0) busy.fetch_sub(1, cuda::memory_order_acq_rel);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < a.out.hist_len; i += blockDim.x)
        if (s_hist[i]) atomicAdd(&a.out.hist[i], s_hist[i]);
    if (lane == 0) {
        atomicAdd(&a.g.ctrl->result[0], acc.count);
        atomicAdd(&a.g.ctrl->result[1], acc.hash);
        atomicAdd(&a.g.ctrl->tree_nodes, acc.nodes);
        atomicAdd(&a.g.ctrl->donations, acc.donations);
        atomicAdd(&a.g.ctrl->words[a.cls], acc.words);
#ifdef MCE_PROFILE
        for (int i = 0; i < kProfSlots; ++i) {
            if (i == kProfMaxRoot) atomicMax(&a.g.ctrl->prof[a.cls][i], acc.prof[i]);
            else if (acc.prof[i]) atomicAdd(&a.g.ctrl->prof[a.cls][i], acc.prof[i]);
        }
        // this warp's load: its time in the kernel minus its time waiting in the worker list,
        // added to the slot of the SM it ran on (Section 4.3 compares per-block loads)
        unsigned smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        const unsigned long long span = (unsigned long long)(clock64() - t_kernel);
        const unsigned long long idle = acc.prof[kProfIdle];
        if (a.g.prof_sm && smid < (unsigned)kProfSms)
            atomicAdd(&a.g.prof_sm[a.cls * kProfSms + smid], span > idle ? span - idle : 0ULL);
#endif
    }
}

#if !MCE_SEARCH_IP && !MCE_SEARCH_L2
// The subtree build ahead of the search (see "subtrees built ahead"): the warps take the roots
// of one launch group of row width W <= 4 in turn and build each one's record.
template <int W>
__global__ void __launch_bounds__(kBuildThreads, kBuildMinBlocks) build_kernel(SearchArgs a)
{
    if (!records_on(a)) return;
    extern __shared__ __align__(16) unsigned char s_raw[];
    const int lane = threadIdx.x & 31, wpb = blockDim.x >> 5;
    constexpr int k = W == 1 ? 0 : W == 2 ? 1 : 2;
    WarpSmem sm;
    {
        unsigned char *mine = s_raw + (size_t)(threadIdx.x >> 5) * build_smem_per_warp(k);
        sm.hkey = reinterpret_cast<int *>(mine);
        sm.hval = sm.hkey + hash_slots(k);
        sm.filter = reinterpret_cast<unsigned *>(sm.hval + hash_slots(k));
        sm.slots = hash_slots(k);
        sm.cur_start = reinterpret_cast<int *>(sm.filter + kFilterWords);
        sm.cur_base = sm.cur_start + 36;
        sm.rows = nullptr;
        sm.rows_words = 0;
    }
    const int begin = a.range[2 * a.group], end = a.range[2 * a.group + 1];
    for (int i = begin + blockIdx.x * wpb + (threadIdx.x >> 5); i < end; i += gridDim.x * wpb) {
        if (load_status(a.g.ctrl) != 0) return;
        if (!has_record(a, i)) continue;
        const int v = a.roots[i];
        const int deg = a.g.offs[v + 1] - a.g.offs[v];
        const int np = a.g.pcount[v];
        if (!record_matches(a, i, deg, np, W)) {
            if (lane == 0) set_status(a.g.ctrl, MCE_ERR_INTERNAL);
            continue;
        }
        build_record<W>(a, sm, v, deg, np, (a.group & 1) == 0, a.bb + a.rec_off[i] * 4, lane);
    }
}
#endif

}  // namespace

}  // namespace mce
