/*
 * mce_oracle.c -- TEST INFRASTRUCTURE, not part of the product.
 *
 * A plain, sequential CPU reference for maximal clique enumeration (MCE).  Only the tests, the
 * smoke check and the timed CPU baseline of the bench load it.  It shares no code, header or
 * table with the CUDA library and must never be linked into it.
 *
 * What it follows (all from "Parallelizing Maximal Clique Enumeration on GPUs",
 * arXiv 2212.01473v2):
 *   - problem statement, Section 2.1: all maximal cliques of a simple undirected graph, exactly;
 *   - Bron-Kerbosch backtracking over (R, P, X), Section 2.2, Algorithm 1;
 *   - pivoting, Section 2.3, Algorithm 2, with the pivot taken over P u X (Tomita's rule,
 *     Section 2.3 last paragraph) maximising |P n N(u)|;
 *   - independent first-level subtrees, Section 2.4, Algorithm 3, in degeneracy order
 *     (Section 2.4, "Degeneracy Ordering"): for the i-th vertex, P = later neighbours and
 *     X = earlier neighbours.
 *
 * Sets are sorted int32 arrays of vertex positions in the degeneracy order.  Nothing here is
 * tuned: no induced subgraphs, no bitsets, no worker list.
 *
 * Readings where the pages are silent (each is repeated in the design notes):
 *   - degeneracy order: the "canonical peel" below -- at level k, every remaining vertex whose
 *     remaining degree is <= k is removed in one round; a vertex's position is its (round, id)
 *     rank.  Any degeneracy order yields the same set of maximal cliques.
 *   - pivot ties: smallest position.  The set of cliques does not depend on the pivot.
 *   - isolated vertices are maximal cliques of size 1 (Algorithm 3 with P = X = {});
 *     the empty graph on zero vertices has no maximal clique.
 *   - result summary (the pages define none): count, histogram by clique size, and
 *     hash = sum over cliques C of mix64( sum_{c in C} key(c) )  (mod 2^64), where
 *     key(c) = mix64((c + 1) * 0x9E3779B97F4A7C15) is the (c+1)-th output of SplitMix64 seeded
 *     with 0 and mix64 is SplitMix64's output function (Steele, Lea, Flood 2014).  The sum is
 *     independent of clique order and of vertex order inside a clique.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum {
    OR_OK = 0,
    OR_ERR_INVALID_ARG = 1,
    OR_ERR_NOT_SIMPLE = 2,     /* self-loop or repeated neighbour */
    OR_ERR_NOT_SYMMETRIC = 3,  /* u in N(v) but v not in N(u) */
    OR_ERR_ID_RANGE = 4,       /* neighbour id outside [0, n) */
    OR_ERR_NOMEM = 5,
    OR_ERR_BUFFER = 6          /* an output buffer is too small */
};

/* Variants of the search, used to cross-check one another. */
enum {
    OR_ALG3_TOMITA = 0,   /* Algorithm 3 over degeneracy order, Algorithm 2 pivot over P u X */
    OR_ALG2_TOMITA = 1,   /* Algorithm 2 from R = {}, P = V, X = {}, pivot over P u X */
    OR_ALG2_PIVOT_P = 2,  /* Algorithm 2 from R = {}, P = V, X = {}, pivot over P only */
    OR_ALG1_PLAIN = 3,    /* Algorithm 1: no pivot */
    OR_ALG4_TOMITA = 4    /* Algorithm 4 over degeneracy order (one subtree per edge), pivot as 0 */
};

/* ------------------------------------------------------------------ hashing */

uint64_t oracle_mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

uint64_t oracle_vertex_key(int32_t id)
{
    return oracle_mix64(((uint64_t)(uint32_t)id + 1ULL) * 0x9E3779B97F4A7C15ULL);
}

uint64_t oracle_clique_hash(const int32_t *ids, int32_t k)
{
    uint64_t s = 0;
    for (int32_t i = 0; i < k; ++i) s += oracle_vertex_key(ids[i]);
    return oracle_mix64(s);
}

/* ------------------------------------------------------------------ validation */

static int cmp_i32(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

static int contains_sorted(const int32_t *a, int64_t n, int32_t key)
{
    int64_t lo = 0, hi = n;
    while (lo < hi) {
        int64_t mid = lo + (hi - lo) / 2;
        if (a[mid] < key) lo = mid + 1;
        else hi = mid;
    }
    return lo < n && a[lo] == key;
}

/* A sorted copy of every adjacency list (the input order is arbitrary). */
static int32_t *sorted_copy(int32_t n, const int32_t *offs, const int32_t *adj)
{
    int64_t total = offs[n];
    int32_t *s = (int32_t *)malloc(sizeof(int32_t) * (size_t)(total > 0 ? total : 1));
    if (!s) return NULL;
    memcpy(s, adj, sizeof(int32_t) * (size_t)total);
    for (int32_t v = 0; v < n; ++v)
        qsort(s + offs[v], (size_t)(offs[v + 1] - offs[v]), sizeof(int32_t), cmp_i32);
    return s;
}

/* Checks that the CSR describes a simple undirected graph (Section 2.1). */
int oracle_validate(int32_t n, const int32_t *offs, const int32_t *adj)
{
    if (n < 0 || !offs) return OR_ERR_INVALID_ARG;
    if (offs[0] != 0) return OR_ERR_INVALID_ARG;
    for (int32_t v = 0; v < n; ++v)
        if (offs[v + 1] < offs[v]) return OR_ERR_INVALID_ARG;
    if (offs[n] > 0 && !adj) return OR_ERR_INVALID_ARG;
    for (int64_t e = 0; e < offs[n]; ++e)
        if (adj[e] < 0 || adj[e] >= n) return OR_ERR_ID_RANGE;
    int32_t *s = sorted_copy(n, offs, adj);
    if (!s) return OR_ERR_NOMEM;
    int rc = OR_OK;
    for (int32_t v = 0; v < n && rc == OR_OK; ++v) {
        for (int64_t e = offs[v]; e < offs[v + 1]; ++e) {
            if (s[e] == v || (e > offs[v] && s[e] == s[e - 1])) { rc = OR_ERR_NOT_SIMPLE; break; }
        }
    }
    for (int32_t v = 0; v < n && rc == OR_OK; ++v) {
        for (int64_t e = offs[v]; e < offs[v + 1]; ++e) {
            int32_t u = s[e];
            if (!contains_sorted(s + offs[u], offs[u + 1] - offs[u], v)) { rc = OR_ERR_NOT_SYMMETRIC; break; }
        }
    }
    free(s);
    return rc;
}

/* ------------------------------------------------------------------ degeneracy order */

/*
 * Canonical peel.  Level k starts at 0.  A round removes, all at once, every remaining vertex
 * whose number of remaining neighbours is <= k; if no vertex qualifies, k grows by one.  The
 * removed vertices get that round's index and core number k; d is the largest k at which a
 * vertex was removed.  The order is by (round, id).  Every vertex has at most k <= d later
 * neighbours, so this is a degeneracy order (Section 2.4, "Degeneracy Ordering").
 */
int oracle_peel(int32_t n, const int32_t *offs, const int32_t *adj,
                int32_t *core, int32_t *rnd, int32_t *rank, int32_t *d_out)
{
    if (n < 0 || !offs || !core || !rnd || !rank || !d_out) return OR_ERR_INVALID_ARG;
    int32_t *curdeg = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n + 1));
    int32_t *alive = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n + 1));
    int32_t *batch = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n + 1));
    if (!curdeg || !alive || !batch) { free(curdeg); free(alive); free(batch); return OR_ERR_NOMEM; }
    for (int32_t v = 0; v < n; ++v) {
        curdeg[v] = offs[v + 1] - offs[v];
        alive[v] = v;
        rnd[v] = -1;
    }
    int32_t n_alive = n, k = 0, r = 0, d = 0;
    while (n_alive > 0) {
        int32_t nb = 0;
        for (int32_t i = 0; i < n_alive; ++i)
            if (curdeg[alive[i]] <= k) batch[nb++] = alive[i];
        if (nb == 0) { ++k; continue; }
        for (int32_t i = 0; i < nb; ++i) { rnd[batch[i]] = r; core[batch[i]] = k; }
        for (int32_t i = 0; i < nb; ++i) {
            int32_t v = batch[i];
            for (int64_t e = offs[v]; e < offs[v + 1]; ++e)
                if (rnd[adj[e]] < 0) curdeg[adj[e]]--;
        }
        int32_t w = 0;
        for (int32_t i = 0; i < n_alive; ++i)
            if (rnd[alive[i]] < 0) alive[w++] = alive[i];
        n_alive = w;
        d = k;
        ++r;
    }
    /* rank by (round, id): counting sort over rounds, ids visited in increasing order */
    int64_t *start = (int64_t *)calloc((size_t)r + 1, sizeof(int64_t));
    if (!start) { free(curdeg); free(alive); free(batch); return OR_ERR_NOMEM; }
    for (int32_t v = 0; v < n; ++v) start[rnd[v] + 1]++;
    for (int32_t i = 0; i < r; ++i) start[i + 1] += start[i];
    for (int32_t v = 0; v < n; ++v) rank[v] = (int32_t)start[rnd[v]]++;
    *d_out = d;
    free(start); free(curdeg); free(alive); free(batch);
    return OR_OK;
}

/*
 * Core numbers by the Batagelj-Zaversnik bucket algorithm ("An O(m) algorithm for cores
 * decomposition of networks", 2003).  A different algorithm from the peel above, used to check
 * the core numbers it produces.
 */
int oracle_core_bz(int32_t n, const int32_t *offs, const int32_t *adj, int32_t *core)
{
    if (n < 0 || !offs || !core) return OR_ERR_INVALID_ARG;
    if (n == 0) return OR_OK;
    int32_t maxdeg = 0;
    for (int32_t v = 0; v < n; ++v) {
        core[v] = offs[v + 1] - offs[v];
        if (core[v] > maxdeg) maxdeg = core[v];
    }
    int32_t *bin = (int32_t *)calloc((size_t)maxdeg + 1, sizeof(int32_t));
    int32_t *pos = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
    int32_t *vert = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
    if (!bin || !pos || !vert) { free(bin); free(pos); free(vert); return OR_ERR_NOMEM; }
    for (int32_t v = 0; v < n; ++v) bin[core[v]]++;
    int32_t startp = 0;
    for (int32_t dg = 0; dg <= maxdeg; ++dg) { int32_t num = bin[dg]; bin[dg] = startp; startp += num; }
    for (int32_t v = 0; v < n; ++v) { pos[v] = bin[core[v]]; vert[pos[v]] = v; bin[core[v]]++; }
    for (int32_t dg = maxdeg; dg >= 1; --dg) bin[dg] = bin[dg - 1];
    bin[0] = 0;
    for (int32_t i = 0; i < n; ++i) {
        int32_t v = vert[i];
        for (int64_t e = offs[v]; e < offs[v + 1]; ++e) {
            int32_t u = adj[e];
            if (core[u] > core[v]) {
                int32_t du = core[u], pu = pos[u], pw = bin[du], w = vert[pw];
                if (u != w) { pos[u] = pw; vert[pu] = w; pos[w] = pu; vert[pw] = u; }
                bin[du]++;
                core[u]--;
            }
        }
    }
    free(bin); free(pos); free(vert);
    return OR_OK;
}

/* ------------------------------------------------------------------ search */

/* A stack of int32 blocks that never moves memory already handed out. */
typedef struct arena_block { struct arena_block *prev; int64_t cap, top; int32_t data[]; } arena_block;
typedef struct { arena_block *cur; } arena;
typedef struct { arena_block *blk; int64_t top; } arena_mark;

static int32_t *arena_alloc(arena *a, int64_t n)
{
    if (n < 1) n = 1;
    if (!a->cur || a->cur->top + n > a->cur->cap) {
        int64_t cap = n > (1 << 20) ? n : (1 << 20);
        arena_block *b = (arena_block *)malloc(sizeof(arena_block) + sizeof(int32_t) * (size_t)cap);
        if (!b) return NULL;
        b->prev = a->cur; b->cap = cap; b->top = 0;
        a->cur = b;
    }
    int32_t *p = a->cur->data + a->cur->top;
    a->cur->top += n;
    return p;
}
static arena_mark arena_save(const arena *a) { arena_mark m = { a->cur, a->cur ? a->cur->top : 0 }; return m; }
static void arena_restore(arena *a, arena_mark m)
{
    while (a->cur && a->cur != m.blk) { arena_block *p = a->cur->prev; free(a->cur); a->cur = p; }
    if (a->cur) a->cur->top = m.top;
}
static void arena_free(arena *a) { arena_mark m = { NULL, 0 }; arena_restore(a, m); }

/* Graph relabelled to degeneracy positions; every list sorted ascending. */
typedef struct {
    int32_t n;
    int64_t *offs;
    int32_t *adj;
    int32_t *orig;   /* position -> original id */
} rgraph;

typedef struct {
    const rgraph *g;
    int variant;
    arena mem;
    int32_t *R;          /* current clique, as positions */
    int32_t r_len;
    int32_t *tmp;        /* scratch for sorting one clique's original ids */
    uint64_t count, hash, nodes;
    uint64_t *hist;
    int32_t hist_len;
    int err;            /* fatal: stops the search */
    int overflow;       /* an output buffer was too small: the search goes on */
    /* enumeration output (NULL when only counting) */
    int32_t *ids; int64_t cap_ids, n_ids;
    int64_t *offsets; int64_t cap_cl, n_cl;
} bk_ctx;

static int64_t intersect(const int32_t *a, int64_t na, const int32_t *b, int64_t nb, int32_t *out)
{
    int64_t k = 0;
    if (na * 16 < nb) {                 /* a much shorter: look each element up in b */
        for (int64_t i = 0; i < na; ++i) if (contains_sorted(b, nb, a[i])) { if (out) out[k] = a[i]; ++k; }
        return k;
    }
    if (nb * 16 < na) {
        for (int64_t j = 0; j < nb; ++j) if (contains_sorted(a, na, b[j])) { if (out) out[k] = b[j]; ++k; }
        return k;
    }
    int64_t i = 0, j = 0;
    while (i < na && j < nb) {
        if (a[i] < b[j]) ++i;
        else if (a[i] > b[j]) ++j;
        else { if (out) out[k] = a[i]; ++k; ++i; ++j; }
    }
    return k;
}

static void report(bk_ctx *c)
{
    int32_t k = c->r_len;
    if (k == 0) return;                 /* the empty set is never reported */
    for (int32_t i = 0; i < k; ++i) c->tmp[i] = c->g->orig[c->R[i]];
    qsort(c->tmp, (size_t)k, sizeof(int32_t), cmp_i32);
    c->count++;
    c->hash += oracle_clique_hash(c->tmp, k);
    if (k >= c->hist_len) c->overflow = 1;
    else c->hist[k]++;
    if (c->offsets) {
        if (c->n_cl + 1 <= c->cap_cl && c->n_ids + k <= c->cap_ids) {
            c->offsets[c->n_cl] = c->n_ids;
            memcpy(c->ids + c->n_ids, c->tmp, sizeof(int32_t) * (size_t)k);
        } else {
            c->overflow = 1;
        }
        c->n_cl++;
        c->n_ids += k;
    }
}

/* BronKerboschPivot(R, P, X) of Algorithm 2 (Algorithm 1 when variant == OR_ALG1_PLAIN). */
static void bk(bk_ctx *c, const int32_t *P, int64_t np, const int32_t *X, int64_t nx)
{
    const rgraph *g = c->g;
    c->nodes++;
    if (np == 0) {                       /* lines 2-3: R is maximal iff P and X are both empty */
        if (nx == 0) report(c);
        return;
    }
    arena_mark mark = arena_save(&c->mem);
    /* line 4: choose the pivot (Tomita: argmax over P u X of |P n N(u)|, ties -> smaller) */
    int32_t pivot = -1;
    if (c->variant != OR_ALG1_PLAIN) {
        int64_t best = -1;
        for (int pass = 0; pass < 2; ++pass) {
            const int32_t *S = pass == 0 ? P : X;
            int64_t ns = pass == 0 ? np : nx;
            if (pass == 1 && c->variant == OR_ALG2_PIVOT_P) break;
            for (int64_t i = 0; i < ns; ++i) {
                int32_t u = S[i];
                int64_t cnt = intersect(P, np, g->adj + g->offs[u], g->offs[u + 1] - g->offs[u], NULL);
                if (cnt > best || (cnt == best && u < pivot)) { best = cnt; pivot = u; }
            }
        }
    }
    /* line 5: branch on P - N(pivot), ascending */
    int32_t *cand = arena_alloc(&c->mem, np);
    int32_t *curP = arena_alloc(&c->mem, np);
    int32_t *curX = arena_alloc(&c->mem, nx + np);
    int32_t *newP = arena_alloc(&c->mem, np);
    int32_t *newX = arena_alloc(&c->mem, nx + np);
    if (!cand || !curP || !curX || !newP || !newX) { c->err = OR_ERR_NOMEM; arena_restore(&c->mem, mark); return; }
    int64_t nc = 0;
    if (pivot < 0) {
        memcpy(cand, P, sizeof(int32_t) * (size_t)np);
        nc = np;
    } else {
        const int32_t *np_ = g->adj + g->offs[pivot];
        int64_t dp = g->offs[pivot + 1] - g->offs[pivot];
        for (int64_t i = 0; i < np; ++i) if (!contains_sorted(np_, dp, P[i])) cand[nc++] = P[i];
    }
    memcpy(curP, P, sizeof(int32_t) * (size_t)np);
    memcpy(curX, X, sizeof(int32_t) * (size_t)nx);
    int64_t ncp = np, ncx = nx;
    for (int64_t ci = 0; ci < nc && !c->err; ++ci) {
        int32_t v = cand[ci];
        const int32_t *nv = g->adj + g->offs[v];
        int64_t dv = g->offs[v + 1] - g->offs[v];
        /* line 6: recurse on (R u {v}, P n N(v), X n N(v)) */
        int64_t nnp = intersect(curP, ncp, nv, dv, newP);
        int64_t nnx = intersect(curX, ncx, nv, dv, newX);
        c->R[c->r_len++] = v;
        bk(c, newP, nnp, newX, nnx);
        c->r_len--;
        /* lines 7-8: P = P - {v}; X = X u {v} (both kept sorted) */
        int64_t w = 0;
        for (int64_t i = 0; i < ncp; ++i) if (curP[i] != v) curP[w++] = curP[i];
        ncp = w;
        int64_t at = ncx;
        while (at > 0 && curX[at - 1] > v) { curX[at] = curX[at - 1]; --at; }
        curX[at] = v;
        ncx++;
    }
    arena_restore(&c->mem, mark);
}

static void rgraph_free(rgraph *g)
{
    free(g->offs); free(g->adj); free(g->orig);
    memset(g, 0, sizeof(*g));
}

/* Relabels the graph to degeneracy positions.  rank_out (optional) receives id -> position. */
static int rgraph_build(int32_t n, const int32_t *offs, const int32_t *adj, rgraph *g,
                        int32_t *d_out)
{
    memset(g, 0, sizeof(*g));
    g->n = n;
    int32_t *core = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n + 1));
    int32_t *rnd = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n + 1));
    int32_t *rank = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n + 1));
    g->offs = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n + 1));
    g->adj = (int32_t *)malloc(sizeof(int32_t) * (size_t)(offs[n] > 0 ? offs[n] : 1));
    g->orig = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n + 1));
    if (!core || !rnd || !rank || !g->offs || !g->adj || !g->orig) {
        free(core); free(rnd); free(rank); rgraph_free(g); return OR_ERR_NOMEM;
    }
    int rc = oracle_peel(n, offs, adj, core, rnd, rank, d_out);
    if (rc == OR_OK) {
        for (int32_t v = 0; v < n; ++v) g->orig[rank[v]] = v;
        g->offs[0] = 0;
        for (int32_t p = 0; p < n; ++p) {
            int32_t v = g->orig[p];
            g->offs[p + 1] = g->offs[p] + (offs[v + 1] - offs[v]);
        }
        for (int32_t p = 0; p < n; ++p) {
            int32_t v = g->orig[p];
            int64_t o = g->offs[p];
            for (int64_t e = offs[v]; e < offs[v + 1]; ++e) g->adj[o++] = rank[adj[e]];
            qsort(g->adj + g->offs[p], (size_t)(g->offs[p + 1] - g->offs[p]), sizeof(int32_t), cmp_i32);
        }
    }
    free(core); free(rnd); free(rank);
    if (rc != OR_OK) rgraph_free(g);
    return rc;
}

static int ctx_init(bk_ctx *c, const rgraph *g, int variant, int32_t hist_len)
{
    memset(c, 0, sizeof(*c));
    c->g = g;
    c->variant = variant;
    c->hist_len = hist_len;
    c->R = (int32_t *)malloc(sizeof(int32_t) * (size_t)(g->n + 1));
    c->tmp = (int32_t *)malloc(sizeof(int32_t) * (size_t)(g->n + 1));
    c->hist = (uint64_t *)calloc((size_t)(hist_len > 0 ? hist_len : 1), sizeof(uint64_t));
    return (c->R && c->tmp && c->hist) ? OR_OK : OR_ERR_NOMEM;
}

static void ctx_free(bk_ctx *c)
{
    free(c->R); free(c->tmp); free(c->hist);
    arena_free(&c->mem);
}

/* Algorithm 3 for one first-level vertex at position p: R = {p}, P = later, X = earlier. */
static void first_level(bk_ctx *c, int32_t p)
{
    const rgraph *g = c->g;
    const int32_t *nv = g->adj + g->offs[p];
    int64_t dv = g->offs[p + 1] - g->offs[p];
    int64_t split = 0;
    while (split < dv && nv[split] < p) ++split;
    c->R[0] = p;
    c->r_len = 1;
    bk(c, nv + split, dv - split, nv, split);
    c->r_len = 0;
}

/*
 * Algorithm 4 for the edges of the vertex at position p to later vertices q: R = {p, q},
 * P = common neighbours after q, X = common neighbours before q.  An isolated vertex has no
 * edge, so Algorithm 4 alone would miss its clique {p}; it is reported here (as Algorithm 3
 * reports it for p).
 */
static void second_level(bk_ctx *c, int32_t p)
{
    const rgraph *g = c->g;
    const int32_t *np_ = g->adj + g->offs[p];
    int64_t dp = g->offs[p + 1] - g->offs[p];
    if (dp == 0) {
        c->R[0] = p;
        c->r_len = 1;
        bk(c, NULL, 0, NULL, 0);
        c->r_len = 0;
        return;
    }
    arena_mark m = arena_save(&c->mem);
    int32_t *common = arena_alloc(&c->mem, dp);
    if (!common) { c->err = OR_ERR_NOMEM; return; }
    for (int64_t e = 0; e < dp && !c->err; ++e) {
        int32_t q = np_[e];
        if (q < p) continue;
        int64_t k = intersect(np_, dp, g->adj + g->offs[q], g->offs[q + 1] - g->offs[q], common);
        int64_t split = 0;
        while (split < k && common[split] < q) ++split;
        c->R[0] = p;
        c->R[1] = q;
        c->r_len = 2;
        bk(c, common + split, k - split, common, split);
    }
    c->r_len = 0;
    arena_restore(&c->mem, m);
}

static void whole_graph(bk_ctx *c)
{
    arena_mark m = arena_save(&c->mem);
    int32_t *all = arena_alloc(&c->mem, c->g->n);
    if (!all) { c->err = OR_ERR_NOMEM; return; }
    for (int32_t i = 0; i < c->g->n; ++i) all[i] = i;
    c->r_len = 0;
    bk(c, all, c->g->n, NULL, 0);
    arena_restore(&c->mem, m);
}

/*
 * Counts the maximal cliques.  out[0] = count, out[1] = hash, out[2 + k] = number of maximal
 * cliques with k vertices for k < hist_len.  roots (original ids, may be NULL = every vertex)
 * restricts Algorithm 3 to those first-level subtrees (Algorithm 4 to those vertices' edges to
 * later ones); it is only meaningful for OR_ALG3_TOMITA and OR_ALG4_TOMITA.  threads > 1 splits
 * the roots over OpenMP threads.
 * nodes_out (optional) receives the number of search-tree nodes visited.
 */
int oracle_count(int32_t n, const int32_t *offs, const int32_t *adj,
                 const int32_t *roots, int64_t n_roots, int32_t variant, int32_t threads,
                 uint64_t *out, int32_t hist_len, uint64_t *nodes_out)
{
    if (!out || hist_len < 1) return OR_ERR_INVALID_ARG;
    int rc = oracle_validate(n, offs, adj);
    if (rc != OR_OK) return rc;
    if (roots) for (int64_t i = 0; i < n_roots; ++i) if (roots[i] < 0 || roots[i] >= n) return OR_ERR_ID_RANGE;
    rgraph g;
    int32_t d = 0;
    rc = rgraph_build(n, offs, adj, &g, &d);
    if (rc != OR_OK) return rc;
    memset(out, 0, sizeof(uint64_t) * (size_t)(2 + hist_len));
    uint64_t nodes = 0;
    int64_t work = roots ? n_roots : n;
    if (variant != OR_ALG3_TOMITA && variant != OR_ALG4_TOMITA) {
        bk_ctx c;
        rc = ctx_init(&c, &g, variant, hist_len);
        if (rc == OR_OK) {
            whole_graph(&c);
            rc = c.err ? c.err : (c.overflow ? OR_ERR_BUFFER : OR_OK);
            out[0] = c.count; out[1] = c.hash; nodes = c.nodes;
            for (int32_t k = 0; k < hist_len; ++k) out[2 + k] = c.hist[k];
        }
        ctx_free(&c);
    } else {
        int32_t *rank = NULL;
        if (roots) {
            rank = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n + 1));
            if (!rank) { rgraph_free(&g); return OR_ERR_NOMEM; }
            for (int32_t p = 0; p < n; ++p) rank[g.orig[p]] = p;
        }
        if (threads < 1) threads = 1;
#ifdef _OPENMP
        #pragma omp parallel num_threads(threads)
#endif
        {
            bk_ctx c;
            int lrc = ctx_init(&c, &g, variant, hist_len);
#ifdef _OPENMP
            #pragma omp for schedule(dynamic, 8)
#endif
            for (int64_t i = 0; i < work; ++i) {
                if (lrc != OR_OK || c.err) continue;
                const int32_t p = roots ? rank[roots[i]] : (int32_t)i;
                if (variant == OR_ALG4_TOMITA) second_level(&c, p);
                else first_level(&c, p);
            }
            if (lrc == OR_OK && c.err) lrc = c.err;
            if (lrc == OR_OK && c.overflow) lrc = OR_ERR_BUFFER;
#ifdef _OPENMP
            #pragma omp critical
#endif
            {
                if (lrc != OR_OK) rc = lrc;
                out[0] += c.count; out[1] += c.hash; nodes += c.nodes;
                if (c.hist) for (int32_t k = 0; k < hist_len; ++k) out[2 + k] += c.hist[k];
            }
            ctx_free(&c);
        }
        free(rank);
    }
    if (nodes_out) *nodes_out = nodes;
    rgraph_free(&g);
    return rc;
}

/*
 * Writes every maximal clique as its original ids sorted ascending: clique i occupies
 * ids[offsets[i] .. offsets[i+1]).  sizes_out[0] = number of cliques, sizes_out[1] = number of
 * ids; both are the full sizes even when a buffer is too small (then OR_ERR_BUFFER is returned
 * and the buffers hold a prefix).  Sequential, Algorithm 3 order.
 */
int oracle_enumerate(int32_t n, const int32_t *offs, const int32_t *adj,
                     const int32_t *roots, int64_t n_roots, int32_t variant,
                     int32_t *ids, int64_t cap_ids, int64_t *offsets, int64_t cap_cliques,
                     int64_t *sizes_out)
{
    if (!sizes_out || (cap_ids > 0 && !ids) || !offsets || cap_cliques < 0 || cap_ids < 0)
        return OR_ERR_INVALID_ARG;
    int rc = oracle_validate(n, offs, adj);
    if (rc != OR_OK) return rc;
    if (roots) for (int64_t i = 0; i < n_roots; ++i) if (roots[i] < 0 || roots[i] >= n) return OR_ERR_ID_RANGE;
    rgraph g;
    int32_t d = 0;
    rc = rgraph_build(n, offs, adj, &g, &d);
    if (rc != OR_OK) return rc;
    bk_ctx c;
    rc = ctx_init(&c, &g, variant, n + 2);
    if (rc == OR_OK) {
        c.ids = ids; c.cap_ids = cap_ids;
        c.offsets = offsets; c.cap_cl = cap_cliques;   /* offsets has cap_cliques + 1 slots */
        if (variant != OR_ALG3_TOMITA && variant != OR_ALG4_TOMITA) {
            whole_graph(&c);
        } else if (roots) {
            int32_t *rank = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n + 1));
            if (!rank) c.err = OR_ERR_NOMEM;
            else {
                for (int32_t p = 0; p < n; ++p) rank[g.orig[p]] = p;
                for (int64_t i = 0; i < n_roots && !c.err; ++i) {
                    if (variant == OR_ALG4_TOMITA) second_level(&c, rank[roots[i]]);
                    else first_level(&c, rank[roots[i]]);
                }
                free(rank);
            }
        } else {
            for (int32_t p = 0; p < n && !c.err; ++p) {
                if (variant == OR_ALG4_TOMITA) second_level(&c, p);
                else first_level(&c, p);
            }
        }
        if (!c.overflow) offsets[c.n_cl] = c.n_ids;
        sizes_out[0] = c.n_cl;
        sizes_out[1] = c.n_ids;
        rc = c.err ? c.err : (c.overflow ? OR_ERR_BUFFER : OR_OK);
    }
    ctx_free(&c);
    rgraph_free(&g);
    return rc;
}
