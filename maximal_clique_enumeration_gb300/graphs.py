"""Seeded synthetic graph generators, shared by the tests, the bench and the oracle runs.

This module only builds inputs: simple undirected graphs stored as a symmetric int32 CSR
(``offsets[n+1]``, ``adj[offsets[n]]``, every adjacency list sorted ascending, no self-loops,
no duplicate edges).  It holds none of the clique-enumeration arithmetic.

The workloads stand in for the real graphs of "Parallelizing Maximal Clique Enumeration on GPUs"
(Table 1), which are not available here.  Families:

* Erdos-Renyi G(n, p)          -- the "Random" family of the GPMA page (Datasets paragraph).
* Barabasi-Albert, m per vertex -- power-law degrees, low degeneracy.
* R-MAT (Graph500 style)        -- the "Graph500" family of the GPMA page (Datasets paragraph).
* planted cliques on G(n, p)    -- extreme subtree imbalance.
* stochastic block model        -- many maximal cliques, large X sets.
* closed-form families (K_n, empty graph, Moon-Moser K_{3,...,3}, complete multipartite,
  cocktail party, path, cycle, bipartite) and disjoint unions, for exact pins.

Every random draw comes from ``numpy.random.Generator(PCG64(seed))``.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

__all__ = [
    "Graph", "csr_from_edges", "er_graph", "ba_graph", "rmat_graph", "planted_graph",
    "sbm_graph", "complete_graph", "empty_graph", "complete_multipartite", "moon_moser",
    "cocktail_party", "path_graph", "cycle_graph", "random_bipartite", "disjoint_union",
    "permute", "sample_roots", "config_graph", "CONFIGS", "edges_of",
]


@dataclass
class Graph:
    """A simple undirected graph as a symmetric, sorted int32 CSR."""

    n: int
    offsets: np.ndarray  # int32[n+1]
    adj: np.ndarray      # int32[offsets[n]]
    name: str = ""

    @property
    def m(self) -> int:
        """Number of undirected edges."""
        return int(self.offsets[-1]) // 2

    def degrees(self) -> np.ndarray:
        return np.diff(self.offsets.astype(np.int64))

    def max_degree(self) -> int:
        return int(self.degrees().max()) if self.n else 0


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def csr_from_edges(n: int, u, v, name: str = "") -> Graph:
    """Build the symmetric sorted CSR of the simple graph spanned by the pairs (u[i], v[i]).

    Self-loops are dropped and duplicate pairs (in either direction) are merged.
    """
    u = np.asarray(u, dtype=np.int64).ravel()
    v = np.asarray(v, dtype=np.int64).ravel()
    if u.size:
        if u.min() < 0 or v.min() < 0 or u.max() >= n or v.max() >= n:
            raise ValueError("edge endpoint out of range")
    keep = u != v
    lo = np.minimum(u[keep], v[keep])
    hi = np.maximum(u[keep], v[keep])
    fwd = lo * n + hi
    fwd.sort()
    if fwd.size:
        fwd = fwd[np.concatenate(([True], fwd[1:] != fwd[:-1]))]     # drop repeated pairs
    lo = fwd // n
    hi = fwd - lo * n
    rev = hi * n + lo
    rev.sort()
    both = np.concatenate([fwd, rev])
    both.sort(kind="stable")                                          # merges two sorted runs
    src = both // n
    dst = both - src * n
    counts = np.bincount(src, minlength=n) if n else np.zeros(0, dtype=np.int64)
    offsets = np.zeros(n + 1, dtype=np.int64)
    np.cumsum(counts, out=offsets[1:])
    if offsets[-1] > np.iinfo(np.int32).max:
        raise ValueError("graph too large for int32 offsets")
    return Graph(n, offsets.astype(np.int32), dst.astype(np.int32), name)


def edges_of(g: Graph):
    """Return (u, v) int64 arrays with u < v, one entry per undirected edge."""
    src = np.repeat(np.arange(g.n, dtype=np.int64), g.degrees())
    dst = g.adj.astype(np.int64)
    keep = src < dst
    return src[keep], dst[keep]


def _unique_pairs_uniform(rng, n: int, count: int, accept=None):
    """Draw `count` distinct unordered pairs {i, j}, i != j, uniformly from the allowed ones."""
    have = np.zeros(0, dtype=np.int64)
    while have.size < count:
        need = count - have.size
        draw = max(1024, int(need * 1.1) + 16)
        i = rng.integers(0, n, draw, dtype=np.int64)
        j = rng.integers(0, n, draw, dtype=np.int64)
        ok = i != j
        if accept is not None:
            ok &= accept(i, j)
        i, j = i[ok], j[ok]
        key = np.minimum(i, j) * n + np.maximum(i, j)
        # keep first occurrences in draw order so the result does not depend on sort ties
        merged = np.concatenate([have, key])
        _, first = np.unique(merged, return_index=True)
        first.sort()
        have = merged[first][:count]
    return have // n, have % n


def er_graph(n: int, p: float, seed: int, name: str = "") -> Graph:
    """G(n, p): every unordered pair independently with probability p.

    For n <= 4096 every pair gets its own Bernoulli draw.  Above that the number of edges is
    drawn from Binomial(n(n-1)/2, p) and that many distinct pairs are drawn uniformly, which
    gives the same distribution.
    """
    rng = _rng(seed)
    if n <= 4096:
        iu, ju = np.triu_indices(n, 1)
        keep = rng.random(iu.size) < p
        return csr_from_edges(n, iu[keep], ju[keep], name or f"er_n{n}_p{p}")
    total = n * (n - 1) // 2
    m = int(rng.binomial(total, p))
    u, v = _unique_pairs_uniform(rng, n, m)
    return csr_from_edges(n, u, v, name or f"er_n{n}_p{p:.3g}")


def ba_graph(n: int, m: int, seed: int, permute_ids: bool = True, name: str = "") -> Graph:
    """Barabasi-Albert preferential attachment.

    Seed graph K_{m+1}; each new vertex attaches to m distinct earlier vertices chosen with
    probability proportional to degree (uniform draws from the list of edge endpoints).  Vertex
    ids are then permuted at random.
    """
    rng = _rng(seed)
    n0 = m + 1
    if n < n0:
        raise ValueError("n must be at least m + 1")
    iu, ju = np.triu_indices(n0, 1)
    n_edges = iu.size + (n - n0) * m
    eu = np.empty(n_edges, dtype=np.int64)
    ev = np.empty(n_edges, dtype=np.int64)
    eu[: iu.size], ev[: iu.size] = iu, ju
    ends = np.empty(2 * n_edges, dtype=np.int64)
    ends[: iu.size] = iu
    ends[iu.size: 2 * iu.size] = ju
    n_ends = 2 * iu.size
    e = iu.size
    pool = rng.random(4 * m * (n - n0) + 64)
    pos = 0
    for t in range(n0, n):
        chosen = []
        seen = set()
        while len(chosen) < m:
            if pos >= pool.size:
                pool = rng.random(pool.size)
                pos = 0
            w = int(ends[int(pool[pos] * n_ends)])
            pos += 1
            if w not in seen:
                seen.add(w)
                chosen.append(w)
        ch = np.asarray(chosen, dtype=np.int64)
        eu[e: e + m] = t
        ev[e: e + m] = ch
        e += m
        ends[n_ends: n_ends + m] = t
        ends[n_ends + m: n_ends + 2 * m] = ch
        n_ends += 2 * m
    if permute_ids:
        perm = rng.permutation(n)
        eu, ev = perm[eu], perm[ev]
    return csr_from_edges(n, eu, ev, name or f"ba_n{n}_m{m}")


def rmat_graph(scale: int, edge_factor: int, abcd=(0.57, 0.19, 0.19, 0.05), seed: int = 1,
               permute_ids: bool = True, name: str = "") -> Graph:
    """R-MAT: edge_factor * 2^scale draws, each picking one quadrant (a, b, c, d) per level.

    No noise is added.  The draws are symmetrised, self-loops and duplicates are removed and
    vertex ids are permuted at random.
    """
    rng = _rng(seed)
    n = 1 << scale
    draws = edge_factor * n
    a, b, c, _ = abcd
    u = np.zeros(draws, dtype=np.int64)
    v = np.zeros(draws, dtype=np.int64)
    chunk = 1 << 22
    for s in range(0, draws, chunk):
        e = min(draws, s + chunk)
        cu = np.zeros(e - s, dtype=np.int64)
        cv = np.zeros(e - s, dtype=np.int64)
        for level in range(scale):
            r = rng.random(e - s)
            bit = np.int64(1) << (scale - 1 - level)
            right = ((r >= a) & (r < a + b)) | (r >= a + b + c)
            down = r >= a + b
            cu |= np.where(down, bit, 0)
            cv |= np.where(right, bit, 0)
        u[s:e], v[s:e] = cu, cv
    if permute_ids:
        perm = rng.permutation(n)
        u, v = perm[u], perm[v]
    return csr_from_edges(n, u, v, name or f"rmat_s{scale}_ef{edge_factor}")


def planted_graph(n: int, avg_degree: float, n_cliques: int, kmin: int, kmax: int, seed: int,
                  name: str = "") -> Graph:
    """G(n, avg_degree/(n-1)) plus `n_cliques` cliques of size uniform in [kmin, kmax].

    Each planted clique is on distinct vertices drawn without replacement; different planted
    cliques may share vertices.
    """
    rng = _rng(seed)
    p = avg_degree / (n - 1)
    total = n * (n - 1) // 2
    m = int(rng.binomial(total, p))
    u, v = _unique_pairs_uniform(rng, n, m)
    us, vs = [u], [v]
    for _ in range(n_cliques):
        k = int(rng.integers(kmin, kmax + 1))
        members = rng.choice(n, size=k, replace=False)
        iu, ju = np.triu_indices(k, 1)
        us.append(members[iu])
        vs.append(members[ju])
    return csr_from_edges(n, np.concatenate(us), np.concatenate(vs),
                          name or f"planted_n{n}_c{n_cliques}")


def sbm_graph(n: int, n_comm: int, smin: int, smax: int, p_in: float, inter_edges: int,
              seed: int, name: str = "") -> Graph:
    """Stochastic block model with `n_comm` contiguous communities summing to n vertices.

    Sizes are drawn uniform in [smin, smax], then random communities are nudged by +-1 (within
    the bounds) until they sum to n.  Inside a community every pair is an edge with probability
    p_in (drawn one community size at a time); `inter_edges` distinct pairs with endpoints in
    different communities are drawn uniformly.
    """
    rng = _rng(seed)
    sizes = rng.integers(smin, smax + 1, n_comm).astype(np.int64)
    total = int(sizes.sum())
    while total != n:
        c = int(rng.integers(0, n_comm))
        if total > n and sizes[c] > smin:
            sizes[c] -= 1
            total -= 1
        elif total < n and sizes[c] < smax:
            sizes[c] += 1
            total += 1
    starts = np.zeros(n_comm + 1, dtype=np.int64)
    np.cumsum(sizes, out=starts[1:])
    comm_of = np.repeat(np.arange(n_comm, dtype=np.int64), sizes)
    us, vs = [], []
    for s in np.unique(sizes):
        s = int(s)
        members = np.nonzero(sizes == s)[0]          # communities of this size, ascending
        iu, ju = np.triu_indices(s, 1)
        keep = rng.random((members.size, iu.size)) < p_in
        ci, pj = np.nonzero(keep)
        base = starts[members][ci]
        us.append(iu[pj] + base)
        vs.append(ju[pj] + base)
    iu, ju = _unique_pairs_uniform(rng, n, inter_edges,
                                   accept=lambda i, j: comm_of[i] != comm_of[j])
    us.append(iu)
    vs.append(ju)
    return csr_from_edges(n, np.concatenate(us), np.concatenate(vs),
                          name or f"sbm_n{n}_k{n_comm}")


# ---------------------------------------------------------------- closed-form families

def complete_graph(n: int) -> Graph:
    iu, ju = np.triu_indices(n, 1)
    return csr_from_edges(n, iu, ju, f"K{n}")


def empty_graph(n: int) -> Graph:
    return csr_from_edges(n, [], [], f"E{n}")


def complete_multipartite(part_sizes) -> Graph:
    """Complete multipartite graph: vertices in different parts are adjacent."""
    part = np.repeat(np.arange(len(part_sizes)), part_sizes)
    n = int(part.size)
    iu, ju = np.triu_indices(n, 1)
    keep = part[iu] != part[ju]
    return csr_from_edges(n, iu[keep], ju[keep], "K_" + "_".join(map(str, part_sizes)))


def moon_moser(k: int) -> Graph:
    """Moon-Moser graph K_{3,3,...,3} on 3k vertices."""
    g = complete_multipartite([3] * k)
    g.name = f"moon_moser_{k}"
    return g


def cocktail_party(k: int) -> Graph:
    """K_{2k} minus a perfect matching (the complete k-partite graph with parts of size 2)."""
    g = complete_multipartite([2] * k)
    g.name = f"cocktail_{k}"
    return g


def path_graph(n: int) -> Graph:
    i = np.arange(max(n - 1, 0))
    return csr_from_edges(n, i, i + 1, f"P{n}")


def cycle_graph(n: int) -> Graph:
    i = np.arange(n)
    return csr_from_edges(n, i, (i + 1) % n, f"C{n}")


def random_bipartite(a: int, b: int, p: float, seed: int) -> Graph:
    rng = _rng(seed)
    iu, ju = np.meshgrid(np.arange(a), np.arange(a, a + b), indexing="ij")
    keep = rng.random(iu.size) < p
    return csr_from_edges(a + b, iu.ravel()[keep.ravel()], ju.ravel()[keep.ravel()],
                          f"bip_{a}_{b}_{p}")


def disjoint_union(graphs) -> Graph:
    us, vs, base = [], [], 0
    for g in graphs:
        u, v = edges_of(g)
        us.append(u + base)
        vs.append(v + base)
        base += g.n
    if not us:
        return empty_graph(0)
    return csr_from_edges(base, np.concatenate(us), np.concatenate(vs), "union")


def permute(g: Graph, seed: int) -> tuple[Graph, np.ndarray]:
    """Relabel vertex i as perm[i] for a seeded random permutation; returns (graph, perm)."""
    perm = _rng(seed).permutation(g.n)
    u, v = edges_of(g)
    return csr_from_edges(g.n, perm[u], perm[v], g.name + "_perm"), perm


def sample_roots(n: int, k: int, seed: int) -> np.ndarray:
    """k distinct vertex ids drawn uniformly without replacement, sorted ascending (int32)."""
    k = min(k, n)
    return np.sort(_rng(seed).choice(n, size=k, replace=False)).astype(np.int32)


# ---------------------------------------------------------------- the five workloads

CONFIGS = {
    "er200": "Erdos-Renyi G(n=200, p=0.10)",
    "ba100k": "Barabasi-Albert n=100,000, m=8, ids permuted",
    "rmat_s20": "R-MAT scale 20, edge factor 16, (0.57, 0.19, 0.19, 0.05), ids permuted",
    "planted50k": "G(50,000, avg degree 20) + 200 planted cliques of size U[30, 60]",
    "sbm1m": "SBM n=1,000,000, 5,000 communities of size U[100, 300], p_in=0.3, "
             "2.5M inter-community edges (about 5 per vertex)",
}


def config_graph(name: str, seed: int) -> Graph:
    """The graph of one named workload at a given seed."""
    if name == "er200":
        return er_graph(200, 0.10, seed, "er200")
    if name == "ba100k":
        return ba_graph(100_000, 8, seed, name="ba100k")
    if name == "rmat_s20":
        return rmat_graph(20, 16, seed=seed, name="rmat_s20")
    if name.startswith("rmat_s"):  # rmat_s<scale>: same parameters at a smaller scale
        return rmat_graph(int(name[6:]), 16, seed=seed, name=name)
    if name == "planted50k":
        return planted_graph(50_000, 20.0, 200, 30, 60, seed, "planted50k")
    if name == "sbm1m":
        return sbm_graph(1_000_000, 5000, 100, 300, 0.3, 2_500_000, seed, "sbm1m")
    if name.startswith("sbm_c"):  # sbm_c<k>: k communities, n = 200 k, 2.5 inter edges/vertex
        k = int(name[5:])
        return sbm_graph(200 * k, k, 100, 300, 0.3, 500 * k, seed, name)
    raise KeyError(name)
