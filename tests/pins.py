"""Independent pure-Python references used to pin the oracle (test-only).

Nothing here calls the oracle or the CUDA library.  The brute-force routines restate the
definition of a maximal clique ("Parallelizing Maximal Clique Enumeration on GPUs",
Section 2.1: a clique that no further vertex can extend) directly; they are exponential and
only used on small graphs.
"""
from __future__ import annotations

import os

import numpy as np

M64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15
HERE = os.path.dirname(os.path.abspath(__file__))


def mix64(z: int) -> int:
    """SplitMix64's output function (Steele, Lea, Flood, OOPSLA 2014)."""
    z &= M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def vertex_key(v: int) -> int:
    return mix64((v + 1) * GOLDEN)


def clique_hash(clique) -> int:
    return mix64(sum(vertex_key(int(c)) for c in clique))


def summary(cliques):
    """(count, hash, hist-tuple) of a collection of cliques, hist trimmed of trailing zeros."""
    hist = {}
    h = 0
    for c in cliques:
        hist[len(c)] = hist.get(len(c), 0) + 1
        h = (h + clique_hash(c)) & M64
    top = max(hist) if hist else -1
    return len(cliques), h, tuple(hist.get(k, 0) for k in range(top + 1))


def neighbour_masks(g):
    masks = [0] * g.n
    for v in range(g.n):
        for u in g.adj[g.offsets[v]: g.offsets[v + 1]]:
            masks[v] |= 1 << int(u)
    return masks


def brute_subsets(g):
    """Every vertex subset tested against the definition (n <= ~16)."""
    n = g.n
    nb = neighbour_masks(g)
    out = []
    for s in range(1, 1 << n):
        members = [v for v in range(n) if s >> v & 1]
        if any((s & ~(1 << v)) & ~nb[v] for v in members):
            continue                                   # not a clique
        if any(not (s >> u & 1) and (s & ~nb[u]) == 0 for u in range(n)):
            continue                                   # some outside vertex extends it
        out.append(tuple(members))
    return sorted(out)


def brute_cliques(g):
    """Every clique, grown in increasing id order, kept when no vertex extends it (n <= ~60)."""
    n = g.n
    nb = neighbour_masks(g)
    full = (1 << n) - 1
    out = []

    def grow(members, common):
        # common = vertices adjacent to every member
        if members and common == 0:
            out.append(tuple(members))
        last = members[-1] if members else -1
        for u in range(last + 1, n):
            if (common >> u) & 1:
                grow(members + [u], common & nb[u])

    grow([], full)
    return sorted(out)


def load_golden(name: str):
    path = os.path.join(HERE, "golden", name)
    edges, cliques, info = [], [], {}
    n = 0
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key == "vertices":
                n = int(vals[0])
            elif key == "edge":
                edges.append((int(vals[0]), int(vals[1])))
            elif key == "clique":
                cliques.append(tuple(sorted(int(x) for x in vals)))
            else:
                info[key] = int(vals[0])
    return n, edges, sorted(cliques), info


def load_peel_golden(name: str):
    """(n, edges, {vertex: (round, core, rank)}, info) of a hand-derived peel fixture."""
    path = os.path.join(HERE, "golden", name)
    edges, peel, info = [], {}, {}
    n = 0
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key == "vertices":
                n = int(vals[0])
            elif key == "edge":
                edges.append((int(vals[0]), int(vals[1])))
            elif key == "peel":
                v, rnd, core, rank = (int(x) for x in vals)
                peel[v] = (rnd, core, rank)
            else:
                info[key] = int(vals[0])
    return n, edges, peel, info


def load_root_golden(name: str):
    """Per-root oracle results written by a committed script under tests/golden/:
    (graph fields, [(root, |P|, (count, hash, hist))], skipped roots)."""
    path = os.path.join(HERE, "golden", name)
    graph, roots, skipped = None, [], []
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key == "graph":
                graph = {"name": vals[0], "seed": int(vals[1]), "n": int(vals[2]),
                         "m": int(vals[3]), "fingerprint": vals[4]}
            elif key == "root":
                hist = tuple(int(x) for x in vals[5:])
                roots.append((int(vals[0]), int(vals[1]),
                              (int(vals[2]), int(vals[3], 16), hist)))
            elif key == "skipped":
                skipped.append((int(vals[0]), int(vals[1])))
    return graph, roots, skipped


def graph_fingerprint(g) -> str:
    """First 16 hex digits of the SHA-256 of a graph's int32 offsets and adjacency."""
    import hashlib
    h = hashlib.sha256()
    h.update(np.ascontiguousarray(g.offsets, np.int32).tobytes())
    h.update(np.ascontiguousarray(g.adj, np.int32).tobytes())
    return h.hexdigest()[:16]


def add_keys(keys):
    """Sum of (count, hash, hist) summaries over disjoint sets of cliques."""
    count, h, hist = 0, 0, []
    for c, hh, hs in keys:
        count += c
        h = (h + hh) & M64
        hist = [x + y for x, y in zip(hist + [0] * (len(hs) - len(hist)),
                                      list(hs) + [0] * (len(hist) - len(hs)))]
    while hist and hist[-1] == 0:
        hist.pop()
    return count, h, tuple(hist)


def csr_arrays(g):
    return np.asarray(g.offsets, np.int32), np.asarray(g.adj, np.int32)
