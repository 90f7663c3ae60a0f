"""Pins for the CPU oracle (no GPU).

Each test checks the oracle against something other than itself: the worked example of the
pages, brute force on tiny graphs, closed forms, a textbook core-number algorithm, an installed
library routine (networkx), or invariants that any correct enumeration satisfies.
"""
import itertools

import numpy as np
import pytest

import oracle as O
from maximal_clique_enumeration_gb300 import graphs as G
from tests import pins


# ---------------------------------------------------------------- the result hash

def test_mix64_matches_published_splitmix64_outputs():
    # SplitMix64 seeded with 0: state advances by the golden gamma, output = mix64(state).
    # The first three outputs are the published test vector of the generator.
    expect = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    for i, e in enumerate(expect):
        assert pins.mix64((i + 1) * pins.GOLDEN) == e
        assert O.vertex_key(i) == e


def test_oracle_hash_equals_independent_python_hash():
    rng = np.random.default_rng(7)
    for _ in range(50):
        x = int(rng.integers(0, 2**63)) * 2 + int(rng.integers(0, 2))
        assert O.mix64(x) == pins.mix64(x)
    for k in range(0, 9):
        ids = rng.choice(10**6, size=k, replace=False)
        assert O.clique_hash(ids) == pins.clique_hash(ids)
        assert O.clique_hash(ids[::-1]) == pins.clique_hash(ids)   # order inside a clique


# ---------------------------------------------------------------- worked example (Figure 1)

def test_worked_example_figure_1():
    n, edges, cliques, info = pins.load_golden("fig1_example.txt")
    u, v = zip(*edges)
    g = G.csr_from_edges(n, u, v)
    assert g.max_degree() == info["max_degree"]
    assert int(np.argmax(g.degrees())) == info["max_degree_vertex"]
    assert sorted(O.enumerate_cliques(g)) == cliques
    assert O.count(g).key() == pins.summary(cliques)
    core, _, rank, d = O.peel(g)
    assert d == info["degeneracy"]
    assert sorted(rank.tolist()) == list(range(n))


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("n", [0, 1, 2, 3, 5, 8, 11, 13])
def test_brute_force_subsets(n):
    for seed, p in itertools.product(range(3), [0.1, 0.3, 0.5, 0.7, 0.9]):
        g = G.er_graph(n, p, seed)
        expect = pins.brute_subsets(g)
        assert sorted(O.enumerate_cliques(g)) == expect
        assert O.count(g).key() == pins.summary(expect)


@pytest.mark.parametrize("n,p", [(20, 0.5), (24, 0.6), (30, 0.4), (40, 0.3), (18, 0.9),
                                 (20, 0.05), (16, 0.95)])
def test_brute_force_clique_growth(n, p):
    for seed in range(3):
        g = G.er_graph(n, p, seed + 100)
        expect = pins.brute_cliques(g)
        if n <= 16:
            assert expect == pins.brute_subsets(g)
        assert sorted(O.enumerate_cliques(g)) == expect
        assert O.count(g).key() == pins.summary(expect)


def test_brute_force_structured_small():
    graphs = [G.er_graph(12, 0.5, 1), G.ba_graph(30, 3, 2), G.rmat_graph(5, 4, seed=3),
              G.planted_graph(40, 3.0, 3, 4, 8, 4), G.sbm_graph(36, 3, 10, 14, 0.5, 10, 5)]
    for g in graphs:
        expect = pins.brute_cliques(g)
        assert sorted(O.enumerate_cliques(g)) == expect, g.name
        assert O.count(g).key() == pins.summary(expect), g.name


# ---------------------------------------------------------------- closed forms

def _hist(size, count):
    return tuple([0] * size + [count])


@pytest.mark.parametrize("n", [1, 2, 3, 7, 33, 64, 65, 100])
def test_complete_graph_has_one_clique(n):
    r = O.count(G.complete_graph(n))
    assert (r.count, r.key()[2]) == (1, _hist(n, 1))
    assert r.hash == pins.clique_hash(range(n))


@pytest.mark.parametrize("n", [1, 2, 10, 1000])
def test_empty_graph_has_n_singletons(n):
    r = O.count(G.empty_graph(n))
    assert (r.count, r.key()[2]) == (n, _hist(1, n))
    assert r.hash == pins.summary([(i,) for i in range(n)])[1]


def test_zero_vertices():
    r = O.count(G.empty_graph(0))
    assert (r.count, r.hash) == (0, 0)


@pytest.mark.parametrize("k", [1, 2, 3, 4, 5, 6, 7, 8])
def test_moon_moser_has_3_to_the_k(k):
    r = O.count(G.moon_moser(k))
    assert (r.count, r.key()[2]) == (3 ** k, _hist(k, 3 ** k))


@pytest.mark.parametrize("parts", [[1, 2, 3], [4, 1, 5, 2], [2, 2, 2, 2, 2, 7], [9, 9]])
def test_complete_multipartite_product(parts):
    r = O.count(G.complete_multipartite(parts))
    assert r.count == int(np.prod(parts))
    assert r.key()[2] == _hist(len(parts), int(np.prod(parts)))


@pytest.mark.parametrize("k", [1, 2, 5, 10])
def test_cocktail_party_2_to_the_k(k):
    r = O.count(G.cocktail_party(k))
    assert (r.count, r.key()[2]) == (2 ** k, _hist(k, 2 ** k))


@pytest.mark.parametrize("n", [2, 3, 10, 257])
def test_path(n):
    r = O.count(G.path_graph(n))
    assert (r.count, r.key()[2]) == (n - 1, _hist(2, n - 1))


@pytest.mark.parametrize("n", [4, 5, 100])
def test_cycle(n):
    r = O.count(G.cycle_graph(n))
    assert (r.count, r.key()[2]) == (n, _hist(2, n))


def test_triangle_free_counts_edges_plus_isolated():
    for seed in range(4):
        g = G.random_bipartite(30, 40, 0.08, seed)
        iso = int((g.degrees() == 0).sum())
        r = O.count(g)
        assert r.count == g.m + iso
        u, v = G.edges_of(g)
        cl = [(int(a), int(b)) for a, b in zip(u, v)] + \
             [(int(i),) for i in np.nonzero(g.degrees() == 0)[0]]
        assert r.key() == pins.summary(cl)


def test_disjoint_union_is_additive():
    parts = [G.moon_moser(3), G.complete_graph(5), G.er_graph(30, 0.3, 9), G.cycle_graph(7),
             G.empty_graph(3)]
    u = G.disjoint_union(parts)
    total, base, hist = [], 0, {}
    for g in parts:
        for c in O.enumerate_cliques(g):
            total.append(tuple(x + base for x in c))
        base += g.n
    assert O.count(u).key() == pins.summary(total)
    assert O.count(u).count == sum(O.count(g).count for g in parts)


# ---------------------------------------------------------------- invariants

def _check_enumeration(g, cliques):
    nb = [set(g.adj[g.offsets[v]: g.offsets[v + 1]].tolist()) for v in range(g.n)]
    assert len(set(cliques)) == len(cliques)                       # no duplicates
    for c in cliques:
        assert list(c) == sorted(set(c))
        for a, b in itertools.combinations(c, 2):
            assert b in nb[a]                                     # a clique
        common = set.intersection(*(nb[x] for x in c))
        assert not common                                         # maximal


@pytest.mark.parametrize("name,seed", [("er200", 1), ("er200", 2), ("rmat_s9", 3)])
def test_enumeration_invariants(name, seed):
    g = G.config_graph(name, seed)
    cl = O.enumerate_cliques(g)
    _check_enumeration(g, cl)
    assert O.count(g).key() == pins.summary(cl)


def test_permutation_invariance():
    g = G.er_graph(120, 0.15, 4)
    cl = O.enumerate_cliques(g)
    for seed in range(3):
        gp, perm = G.permute(g, seed)
        mapped = [tuple(sorted(int(perm[x]) for x in c)) for c in cl]
        assert sorted(O.enumerate_cliques(gp)) == sorted(mapped)
        assert O.count(gp).key() == pins.summary(mapped)


def test_search_variants_agree():
    # Algorithms 1, 2 (pivot from P), 2 (pivot from P u X) and 3 are four traversals of the
    # same problem; they must report the same set of maximal cliques.
    for g in [G.er_graph(40, 0.3, 1), G.er_graph(25, 0.7, 2), G.moon_moser(4),
              G.ba_graph(200, 4, 3), G.planted_graph(200, 4.0, 3, 6, 9, 5)]:
        ref = O.count(g).key()
        for var in (O.ALG2_TOMITA, O.ALG2_PIVOT_P, O.ALG1_PLAIN):
            assert O.count(g, variant=var).key() == ref
        assert sorted(O.enumerate_cliques(g, variant=O.ALG1_PLAIN)) == \
            sorted(O.enumerate_cliques(g))


@pytest.mark.parametrize("n", [0, 1, 2, 5, 9, 13])
def test_second_level_decomposition_brute_force(n):
    # Algorithm 4 (one subtree per edge, plus isolated vertices) reaches exactly the maximal
    # cliques that brute force finds
    for seed, p in itertools.product(range(3), [0.1, 0.4, 0.7, 0.95]):
        g = G.er_graph(n, p, seed + 7)
        expect = pins.brute_subsets(g)
        assert sorted(O.enumerate_cliques(g, variant=O.ALG4_TOMITA)) == expect
        assert O.count(g, variant=O.ALG4_TOMITA).key() == pins.summary(expect)


def test_second_level_decomposition_per_root():
    # per root, Algorithm 4 over the root's edges to later vertices gives the same cliques as
    # the root's first-level subtree (the first level of Algorithm 3 takes no pivot)
    g = G.config_graph("planted50k", 3)
    rng = np.random.default_rng(9)
    roots = np.sort(rng.choice(g.n, 3000, replace=False)).astype(np.int32)
    assert O.count(g, roots=roots, variant=O.ALG4_TOMITA).key() == O.count(g, roots=roots).key()
    for h in [G.moon_moser(5), G.cocktail_party(8), G.empty_graph(7), G.path_graph(30),
              G.complete_graph(12), G.ba_graph(300, 5, 2)]:
        assert sorted(O.enumerate_cliques(h, variant=O.ALG4_TOMITA)) == \
            sorted(O.enumerate_cliques(h))


def test_root_subsets_are_additive_and_threads_agree():
    g = G.config_graph("planted50k", 2)
    full = O.count(g, threads=4)
    assert O.count(g, threads=1).key() == full.key()
    rng = np.random.default_rng(3)
    label = rng.integers(0, 3, g.n)
    parts = [O.count(g, roots=np.nonzero(label == i)[0], hist_len=len(full.hist)) for i in range(3)]
    assert sum(p.count for p in parts) == full.count
    assert sum(p.hash for p in parts) % 2**64 == full.hash
    assert np.array_equal(sum(p.hist for p in parts), full.hist)


def test_networkx_find_cliques_agrees():
    nx = pytest.importorskip("networkx")
    for name, seed in [("er200", 5), ("rmat_s10", 1)]:
        g = G.config_graph(name, seed)
        h = nx.Graph()
        h.add_nodes_from(range(g.n))
        h.add_edges_from(zip(*[x.tolist() for x in G.edges_of(g)]))
        expect = sorted(tuple(sorted(c)) for c in nx.find_cliques(h))
        assert sorted(O.enumerate_cliques(g)) == expect
    g = G.ba_graph(3000, 6, 2)
    h = nx.Graph()
    h.add_nodes_from(range(g.n))
    h.add_edges_from(zip(*[x.tolist() for x in G.edges_of(g)]))
    assert O.count(g).key() == pins.summary([tuple(sorted(c)) for c in nx.find_cliques(h)])


# ---------------------------------------------------------------- degeneracy order

@pytest.mark.parametrize("name,seed", [("er200", 1), ("rmat_s12", 2), ("planted50k", 1),
                                       ("sbm_c20", 3)])
def test_peel_core_numbers_and_order(name, seed):
    g = G.config_graph(name, seed)
    core, rnd, rank, d = O.peel(g)
    assert np.array_equal(core, O.core_bz(g))                 # Batagelj-Zaversnik
    assert d == int(core.max())
    assert np.array_equal(np.sort(rank), np.arange(g.n))
    # order is by (round, id)
    key = rnd.astype(np.int64) * g.n + np.arange(g.n)
    assert np.array_equal(np.argsort(key, kind="stable"), np.argsort(rank, kind="stable"))
    # at most d later neighbours for every vertex, with equality somewhere
    src = np.repeat(np.arange(g.n), g.degrees())
    later = np.bincount(src[rank[g.adj] > rank[src]], minlength=g.n)
    assert later.max() == d
    assert np.all(later <= core)
    nx = pytest.importorskip("networkx")
    if g.n <= 20000:
        h = nx.Graph()
        h.add_nodes_from(range(g.n))
        h.add_edges_from(zip(*[x.tolist() for x in G.edges_of(g)]))
        cn = nx.core_number(h)
        assert all(cn[v] == core[v] for v in range(g.n))


@pytest.mark.parametrize("fixture", ["peel_fig1.txt", "peel_k4_tails.txt"])
def test_peel_rounds_match_hand_derivation(fixture):
    # round, core number and rank of every vertex, derived by hand from the canonical peel's
    # definition (the fixture headers show the derivation)
    n, edges, expect, info = pins.load_peel_golden(fixture)
    g = G.csr_from_edges(n, *zip(*edges))
    core, rnd, rank, d = O.peel(g)
    assert d == info["degeneracy"]
    assert int(rnd.max()) + 1 == info["rounds"]
    for v, (r, c, k) in expect.items():
        assert (int(rnd[v]), int(core[v]), int(rank[v])) == (r, c, k), v


def canonical_peel_violations(g, rnd, core):
    """Checks (round, core) against the definition of the canonical peel, round by round.

    With A_r the vertices whose round is >= r (those left at the start of round r) and deg_r(v)
    the number of neighbours of v in A_r, round r at level k_r must remove exactly
    {v in A_r : deg_r(v) <= k_r}, where k_r = max(k_{r-1}, min over A_r of deg_r) and k_{-1} = 0
    (the level only rises when nothing qualifies, and then to the least remaining degree).
    Returns the list of rounds that break it.
    """
    src = np.repeat(np.arange(g.n), g.degrees())
    dst = g.adj.astype(np.int64)
    bad = []
    k_prev = 0
    for r in range(int(rnd.max()) + 1 if g.n else 0):
        alive = rnd >= r
        keep = alive[src] & alive[dst]
        deg_r = np.bincount(src[keep], minlength=g.n)
        k_r = max(k_prev, int(deg_r[alive].min()))
        removed = alive & (deg_r <= k_r)
        if not np.array_equal(removed, rnd == r) or np.any(core[rnd == r] != k_r):
            bad.append(r)
        k_prev = k_r
    return bad


@pytest.mark.parametrize("name,seed", [("er200", 2), ("rmat_s10", 1), ("ba100k", 1)])
def test_peel_rounds_satisfy_the_definition(name, seed):
    g = G.config_graph(name, seed)
    core, rnd, rank, d = O.peel(g)
    assert canonical_peel_violations(g, rnd, core) == []


# ---------------------------------------------------------------- input checks

def _raw(n, lists):
    offs = np.zeros(n + 1, np.int32)
    offs[1:] = np.cumsum([len(x) for x in lists])
    adj = np.asarray([y for x in lists for y in x], np.int32)
    return G.Graph(n, offs, adj)


def test_validation_errors():
    assert O.validate(_raw(3, [[1], [0, 2], [1]])) == O.OK
    assert O.validate(_raw(3, [[2, 1], [0, 2], [1, 0]])) == O.OK     # unsorted lists are fine
    assert O.validate(_raw(2, [[0, 1], [0]])) == O.NOT_SIMPLE        # self-loop
    assert O.validate(_raw(2, [[1, 1], [0, 0]])) == O.NOT_SIMPLE     # duplicate
    assert O.validate(_raw(3, [[1], [0, 2], []])) == O.NOT_SYMMETRIC
    assert O.validate(_raw(2, [[5], [0]])) == O.ID_RANGE
    assert O.validate(_raw(2, [[-1], [0]])) == O.ID_RANGE
    bad = _raw(2, [[1], [0]])
    bad.offsets = np.asarray([0, 2, 1], np.int32)
    assert O.validate(bad) == O.INVALID_ARG
    with pytest.raises(O.OracleError):
        O.count(_raw(2, [[0, 1], [0]]))
