// Internal declarations shared by the CUDA sources of libmce_gb300.so (not installed).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "mce.h"

namespace mce {

constexpr int kMaxP = 1024;            // largest |P| of a first-level subtree (32 words per row)
constexpr int kMaxIdxBits = 21;        // pivot codes are packed as count << 21 | ~code
constexpr int kMaxCode = (1 << kMaxIdxBits) - 1;
constexpr int kPeelThreads = 1024;
constexpr int kPeelSoloVertices = 8192;  // the peel finishes in one CTA below this many vertices
constexpr int kDefaultWarpsPerBlock = 4;
constexpr int kNumClasses = 6;           // row widths W = 1, 2, 4, 8, 16, 32 words
constexpr int kNumGroups = 2 * kNumClasses;   // per width: big-workspace roots, then the rest
constexpr long long kWsCapWords = 16384;     // workspace per warp of a "normal" launch (64 KiB)
constexpr long long kBigBudgetWords = 256LL << 20;   // workspace of a "big" launch (1 GiB)
constexpr int kScanBlock = 1024;         // elements per CTA of the exclusive scan
constexpr int kProfSms = 256;            // MCE_PROFILE builds: per-SM load slots per class
constexpr int kProfSlots = 16;           // MCE_PROFILE builds: activity counters per class
constexpr int kSmallP = 10;              // largest |P| of a search-tree node solved whole
constexpr int kSmallPMax = 10;           // ... and the most its bit-sliced test allows
constexpr int kFrontCap = 8192;          // largest round the peel runs from a frontier
constexpr int kRoundUnsorted = 1 << 30;  // rstart flag: places are below 2^30 (n < 2^30)

// Device-resident control block of a handle.
struct DevCtrl {
    int status;                  // first device-side error (mce_status), 0 = none
    int degeneracy;              // peel output
    int rounds;                  // peel output
    long long peel_live;         // peel output: live vertices summed over rounds
    int front_cnt[3];            // peel: frontier sizes, by round modulo 3
    int max_pcount;              // max |P| over first-level subtrees
    unsigned int bar_count;      // grid barrier arrivals (grows by the grid size per barrier)
    unsigned int bar_pad;
    unsigned long long ws_words; // largest per-warp workspace need (words), all classes
    unsigned long long ws_grp[kNumGroups];    // the same per launch group
    unsigned long long next_root;  // search: root claim counter
    unsigned long long n_sched;    // search: number of scheduled roots
    // worker list counters, each on its own 128-byte line: idle warps poll `busy` while donors
    // update the ring
    alignas(128) int busy;       // warps holding work
    alignas(128) int ring_head;  // pops
    alignas(128) int ring_tail;  // pushes
    alignas(128) int n_iso;      // isolated vertices (cliques of size 1)
    int max_degree;              // Delta
    unsigned long long iso_hash; // hash contribution of the isolated vertices
    unsigned long long tree_nodes;
    unsigned long long donations;
    unsigned long long result[2];  // count, hash of the last search
    unsigned long long words[kNumClasses];  // bitset words processed per row-width class
    unsigned long long prof[kNumClasses][kProfSlots];  // MCE_PROFILE builds: cycles per activity
    unsigned long long peel_prof[16];         // MCE_PROFILE builds: peel phases (ns, CTA 0)
    // first-level roots in launch groups g = 2k + b (row width W = 1 << k; b = 0: roots
    // whose workspace exceeds kWsCapWords, b = 1: the others): sched[cls[2g] .. cls[2g+1])
    // for the full schedule, uroots[ucls[2g] .. ucls[2g+1]) for a caller's root list
    int cls[2 * kNumGroups];     // [begin, end) of launch group g at cls[2g], cls[2g+1]
    int ucls[2 * kNumGroups];
};

// Everything the kernels need about a handle's graph (device pointers).
struct DevGraph {
    int n;
    long long nnz;
    const int *offs;
    const int *adj;
    int *rank;        // id -> position in the degeneracy order
    int *core;        // id -> core number
    int *round_of;    // id -> peel round
    int *order;       // position -> id
    int *pcount;      // id -> |P| (later neighbours)
    int *padj;        // [2m] N+(v) in id order at padj[offs[v] .. offs[v] + pcount[v])
                      // (Section 2.4: P of the first-level subtree)
    int *sched;       // first-level roots with |P| > 0, heavy first
    int *deg;         // peel scratch
    int *alive_a, *alive_b;
    int *blk_cnt, *blk_min, *blk_cm;   // peel per-CTA reports [2][grid]
    long long *blk_rd;                 // peel: adjacency entries removed per CTA [grid]
    int *blk_gone;                     // peel per-CTA reports: live entries removed [2][grid]
    int *front;                        // peel: frontiers of three consecutive rounds [3][kFrontCap]
    int *rstart;                       // peel: first place of each round in the order [n + 1]
                                       // (kRoundUnsorted set: a frontier round, sorted at the end)
    int ip;           // search over partial induced subgraphs (rows for P only), Section 3.4
    int l2;           // independent second-level subtrees, one per edge (Section 3.2)
    int *unit_cnt;    // l2: subtrees per root, in schedule order (scan input) [n]
    int *sched_uoff;  // l2: exclusive prefix of subtrees over sched [n+1]
    int *uroots_uoff; // l2: the same over uroots [n+1]
    int *unit_scan;   // l2: exclusive-scan partials of unit_cnt
    int *bucket;      // orient: schedule bucket histogram / cursors [kNumBuckets]
    int *ubucket;     // the same for a caller's root list [kNumBuckets]
    int *uroots;      // a caller's roots, grouped by row width, heaviest first
    unsigned long long *prof_sm;   // MCE_PROFILE builds: busy warp cycles [kNumClasses][kProfSms]
    DevCtrl *ctrl;
};

// Search output descriptors.
struct DevOut {
    unsigned long long *hist;       // [hist_len] histogram by clique size (device, accumulated)
    int hist_len;
    // enumeration (NULL when counting)
    int *ids;
    long long *offsets;
    const long long *region_ids;     // [hist_len] first id slot of each size group
    const long long *region_cl;      // [hist_len] first clique slot of each size group
    unsigned long long *cursor;      // [hist_len] cliques written per size group
};

struct SearchArgs {
    DevGraph g;
    DevOut out;
    const int *roots;        // g.sched or g.uroots
    const int *range;        // roots[range[2 group] .. range[2 group + 1]) are this launch's
    const int *uoff;         // second-level subtrees: prefix of subtree counts over roots[]
    int cls;                 // row-width class of this launch (W = 1 << cls)
    int group;               // launch group (2 cls + 0 for big-workspace roots, + 1 otherwise)
    int small_lo, small_hi;  // nodes with small_lo <= |P| <= small_hi are solved whole
    unsigned *bb;            // records of subtrees built ahead (null: none), bb_quads quads
    long long bb_quads;
    const long long *rec_off;  // quad offset of each root's record, by place in `roots` (+1)
    const long long *rec_gate; // the records' total: they are in use iff it is <= bb_quads
    unsigned int *ws;        // per-warp workspace, ws_words each
    unsigned long long ws_words;
    int *ring;               // worker list: ring of idle warp ids [n_workers]
    unsigned *ring_seq;      // worker list: per-slot sequence numbers [n_workers]
    int *flag;               // worker list: per-warp inbox state [n_workers]
    int n_workers;
    int worker_list;
    int donate_min_p;
    int donate_rule;         // 0: siblings at this level and at an earlier one; 1: either
    long long spin_limit_ns;
};

// Words per bitset row for a first-level subtree with np vertices in P (one bit per P vertex),
// rounded up to 1, 2, 4, 8, 16 or 32 so that rows load as 4-, 8- or 16-byte vectors.
__host__ __device__ inline int wclass(int np)
{
    return np <= 32 ? 1 : np <= 64 ? 2 : np <= 128 ? 4 : np <= 256 ? 8 : np <= 512 ? 16 : 32;
}

// Class index k of a |P| value (W = 1 << k); |P| = 0 joins class 0.
__host__ __device__ inline int wclass_index(int np)
{
    return np <= 32 ? 0 : np <= 64 ? 1 : np <= 128 ? 2 : np <= 256 ? 3 : np <= 512 ? 4 : 5;
}

// Per-warp workspace layout (32-bit word offsets) for a root of degree `deg` with np later
// neighbours.  The same layout serves a branch of such a root donated through the worker list:
// the donor writes the branch into the receiver's workspace at these offsets.
//
// ip: partial induced subgraphs (no X rows).  l2: the layout also holds every second-level
// subtree {v, w} of the root v (Algorithm 4): its P (at most |P(v)|) and X (at most deg(v) - 1
// vertices, some of them later than v) fit once the X lists are sized by deg rather than by
// deg - np; its rows (P rows, then X rows) fit in the deg * W words of rows.
constexpr int kWsHeader = 80;   // inbox: 16 scalar words, then P and X_P bitsets (32 words each)

struct WsLayout {
    long long rowsP, rowsX, pids, pkey, rids, xids, xx, spill, plist, stack, total;
    int W, LV;
};

__host__ __device__ inline WsLayout ws_layout(int deg, int np, bool ip, bool l2)
{
    WsLayout l;
    const int nx = l2 ? deg : deg - np;
    l.W = wclass(np);
    long long o = kWsHeader;
    l.rowsP = o; o += (long long)np * l.W;       // rows of P vertices, columns over P
    l.rowsX = o; o += ip ? 0 : (long long)(deg - np) * l.W;   // X rows (full subgraphs only)
    l.pids = o; o += np;                         // original ids of P vertices (ascending)
    o = (o + 1) & ~1LL;
    l.pkey = o; o += 2LL * np;                   // vertex keys of P vertices (uint64)
    l.rids = o; o += np + 1;                     // ids of R at level 0 (root, or donated R)
    l.xids = o; o += nx;                         // original ids of X vertices (ascending)
    l.xx = o; o += nx;                           // compact X_X list (Section 3.5)
    l.spill = o; o += nx;                        // partition scratch
    l.plist = o; o += np;                        // pivot candidates from P u X_P
    o = (o + 3) & ~3LL;
    l.LV = (8 + 3 * l.W + 3) & ~3;               // level: S(2) lpX cursor more pad(3) | P0 XP0 C
    l.stack = o; o += (long long)(np + 1) * l.LV;
    l.total = (o + 3) & ~3LL;
    return l;
}

// Record of a first-level root built ahead of the search (full induced subgraph; 32-bit word
// offsets from the record's start): header (np, nx, live X rows, covered), rows ((np + nx) * W),
// P's ids (np), P's keys (2 np, 8-byte aligned), X's ids while building and then the indices
// of the live X rows (nx).  Records start on 16-byte boundaries; sizes are kept in quads.
struct RecLayout {
    long long rows, pids, pkey, xx, total;
};

__host__ __device__ inline RecLayout rec_layout(int deg, int np, int W)
{
    RecLayout l;
    long long o = 4;
    l.rows = o; o += (long long)deg * W;
    l.pids = o; o += np;
    o = (o + 1) & ~1LL;
    l.pkey = o; o += 2LL * np;
    l.xx = o; o += deg - np;
    l.total = (o + 3) & ~3LL;
    return l;
}

__host__ __device__ inline long long rec_quads(int deg, int np, int W)
{
    return rec_layout(deg, np, W).total / 4;
}

constexpr long long kRecCapQuads = 1LL << 30;   // records of subtrees built ahead: 16 GiB at most
#ifndef MCE_BUILD_MIN_BLOCKS
#define MCE_BUILD_MIN_BLOCKS 4
#endif
#ifndef MCE_BUILD_BATCH
#define MCE_BUILD_BATCH 16
#endif
constexpr int kBuildThreads = 256;
constexpr int kBuildMinBlocks = MCE_BUILD_MIN_BLOCKS;
constexpr int kBuildBatch = MCE_BUILD_BATCH;   // later-neighbour entries a lane has in flight

// Schedule buckets: launch groups in launch order (widest rows first; per width the roots with
// a big workspace, then the rest) and, inside a group, roots with a larger estimated cost
// (|P| + 1)^2 * (core(v) + 1) first (log2 buckets).  Bucket 0 holds over-limit roots (group of
// W = 32).
constexpr int kCostBuckets = 48;
constexpr int kNumBuckets = 1 + kNumGroups * kCostBuckets;

// Launch position o = 0 .. kNumGroups-1 <-> group g = 2k + b.
__host__ __device__ inline int group_at(int o) { return 2 * (kNumClasses - 1 - o / 2) + (o & 1); }
__host__ __device__ inline int position_of(int g) { return 2 * (kNumClasses - 1 - g / 2) + (g & 1); }

__device__ inline int sched_bucket(int np, int deg, bool ip, bool l2, int core)
{
    if (np > kMaxP) return 0;
    const int k = wclass_index(np);
    const int b = np > 0 && ws_layout(deg, np, ip, l2).total > kWsCapWords ? 0 : 1;
    // the subtree's cost grows with |P| and with how dense the region is (its core number)
    unsigned long long est = (unsigned long long)(np + 1) * (unsigned long long)(np + 1) *
                             (unsigned long long)(core + 1);
#ifdef MCE_EST_X_DIV
    if (MCE_EST_X_DIV > 0) est *= 1ULL + (unsigned long long)(deg - np) / MCE_EST_X_DIV;
#endif
    int lb = est ? 63 - __clzll((long long)est) : 0;
    lb = lb < kCostBuckets - 1 ? lb : kCostBuckets - 1;
    return 1 + position_of(2 * k + b) * kCostBuckets + (kCostBuckets - 1 - lb);
}

// Launchers (each returns the CUDA error of its launch).
cudaError_t launch_ingest_check(const DevGraph &g, int *d_unsorted_list, int *d_stats,
                                int *d_big_list, cudaStream_t s);
cudaError_t launch_ingest_sort(const DevGraph &g, int *adj_mut, const int *d_list, int n_list,
                               int *scratch, long long scratch_len, cudaStream_t s);
cudaError_t launch_ingest_sort_large(const DevGraph &g, int *adj_mut, int v, int *scratch,
                                     cudaStream_t s);
cudaError_t launch_ingest_validate(const DevGraph &g, const int *d_big_list, int n_big,
                                   int max_degree, unsigned long long *d_fb, cudaStream_t s);
// ev_peel (may be null) is recorded on s between the peel and the orientation kernels.
cudaError_t launch_order(const DevGraph &g, int peel_blocks, long long spin_limit_ns,
                         cudaStream_t s, cudaEvent_t ev_peel);
cudaError_t launch_peel(const DevGraph &g, int peel_blocks, long long spin_limit_ns,
                        cudaStream_t s);
// The search launch of launch group a.group; rec selects the variant that searches records.
cudaError_t launch_search(const SearchArgs &a, int blocks, int threads, size_t smem, bool rec,
                          cudaStream_t s);
cudaError_t launch_search_prep(const SearchArgs &a, cudaStream_t s);
// Subtrees built ahead: rec_off[i] = quad offset of the record of the root at place i of
// roots[0 .. n_slots) (the roots of the launch groups of row width <= 4 words have one;
// range = the launch groups' places), rec_off[n_slots] = the total; scan_tmp holds
// n_slots / kScanBlock + 2 partial sums.
cudaError_t launch_record_offsets(const DevGraph &g, const int *roots, const int *range,
                                  int n_slots, long long *scan_tmp, long long *rec_off,
                                  cudaStream_t s);
// The build launch of launch group a.group (row width 1 << a.cls <= 4 words).
cudaError_t launch_build(const SearchArgs &a, int blocks, cudaStream_t s);
// CTAs per SM of that build kernel.
cudaError_t build_occupancy(int cls, int *blocks_per_sm);
const void *build_kernel_full(int cls);
// CTAs per SM of the kernel of launch group `group` (row-width class group / 2).
cudaError_t search_occupancy(int group, int ip, int l2, int threads, size_t smem,
                             int *blocks_per_sm);
// Shared memory of the search kernel of class k: the size histogram, then per warp a hash of
// P(v) (ids and local indices), its bit filter, the build cursors and (W <= 4) a row area.
__host__ __device__ inline int hash_slots(int k) { return 64 << k; }
// Rows of a root with deg * W <= smem_row_words(k) are built and searched in shared memory.
__host__ __device__ inline int smem_row_words(int k) { return k <= 2 ? 1024 : 0; }
// Per warp: hash keys and values, the bit filter in front of the hash, build cursor arrays
// (2 x 36 words), rows.
constexpr int kFilterLog2Bits = 12;
constexpr int kFilterWords = (1 << kFilterLog2Bits) / 32;
__host__ __device__ inline size_t warp_smem_bytes(int k)
{
    return (size_t)hash_slots(k) * 8 + kFilterWords * 4 + 2 * 36 * 4 +
           (size_t)smem_row_words(k) * 4;
}
// Per warp of the build kernel: the hash of P and its filter, the walk's cursors, and a queue
// of 64 walked entries that passed the filter (ids and rows).
__host__ __device__ inline size_t build_smem_per_warp(int k)
{
    return (size_t)hash_slots(k) * 8 + kFilterWords * 4 + 2 * 36 * 4 + 2 * 64 * 4;
}
// The search kernel's size histogram, at the start of its shared memory.
__host__ __device__ inline size_t smem_hist_bytes(int hist_len)
{
    return ((size_t)(hist_len + 1) * 8 + 15) & ~(size_t)15;
}
__host__ __device__ inline size_t search_smem_bytes(int k, int hist_len, int warps)
{
    return smem_hist_bytes(hist_len) + (size_t)warps * warp_smem_bytes(k);
}
cudaError_t search_configure(int cls, int ip, int l2, size_t smem);
cudaError_t launch_bin_roots(const DevGraph &g, const int *roots, int n_roots, cudaStream_t s);
// Second-level subtrees: uoff[i] = number of subtrees of roots[0 .. i) (edges to later
// neighbours; 1 for an isolated root), i <= n_roots; n_roots < 0 reads the schedule length
// from the control block.
cudaError_t launch_unit_offsets(const DevGraph &g, const int *roots, int n_roots, int *uoff,
                                cudaStream_t s);
cudaError_t launch_finalize(const DevGraph &g, const DevOut &o, unsigned long long *d_out,
                            int include_isolated, cudaStream_t s);
cudaError_t launch_enum_layout(const DevGraph &g, const unsigned long long *d_counts,
                               int hist_len, long long *region_ids, long long *region_cl,
                               unsigned long long *cursor, long long *d_totals, cudaStream_t s);
cudaError_t launch_enum_isolated(const DevGraph &g, const DevOut &o, cudaStream_t s);
cudaError_t launch_enum_close(const DevOut &o, const long long *d_totals, cudaStream_t s);

// ------------------------------------------------------------------ device helpers

__device__ __forceinline__ unsigned long long globaltimer_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void set_status(DevCtrl *c, int code)
{
    atomicCAS(&c->status, 0, code);
}

__device__ __forceinline__ int load_status(const DevCtrl *c)
{
    return *(volatile const int *)&c->status;
}

// SplitMix64 output function (Steele, Lea, Flood, "Fast splittable pseudorandom number
// generators", OOPSLA 2014) -- the mixing step of the result hash.
__device__ __forceinline__ unsigned long long mix64(unsigned long long z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

// key(v): the (v+1)-th output of SplitMix64 seeded with 0.
__device__ __forceinline__ unsigned long long vertex_key(int v)
{
    return mix64((unsigned long long)((unsigned)v + 1u) * 0x9E3779B97F4A7C15ULL);
}

}  // namespace mce
