"""GPU parity: the CUDA library against the CPU oracle, bit-exact on (count, hash, histogram),
the degeneracy order, and the enumerated cliques.  Every call goes through the C ABI
(libmce_gb300.so via the ctypes binding).
"""
import numpy as np
import pytest

import oracle as O
from maximal_clique_enumeration_gb300 import graphs as G
from tests import pins

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from maximal_clique_enumeration_gb300 import build
    build.build()


def _mce():
    import maximal_clique_enumeration_gb300 as mce
    return mce


def gpu_graph(g, **cfg):
    mce = _mce()
    return mce.Graph(torch.from_numpy(g.offsets).cuda(), torch.from_numpy(g.adj).cuda(), g.n,
                     **cfg)


def assert_count_parity(g, roots=None, threads=8, **cfg):
    expect = O.count(g, roots=roots, threads=threads).key()
    with gpu_graph(g, **cfg) as h:
        got = h.count_result() if roots is None else h.count_roots_result(roots)
    assert got == expect, g.name
    return got


# ---------------------------------------------------------------- worked example, closed forms

def test_worked_example_figure_1():
    n, edges, cliques, info = pins.load_golden("fig1_example.txt")
    g = G.csr_from_edges(n, *zip(*edges))
    mce = _mce()
    with gpu_graph(g) as h:
        assert h.count_result() == pins.summary(cliques)
        ids, offs = h.enumerate()
        assert sorted(mce.cliques_from(ids, offs)) == cliques
        assert h.info["degeneracy"] == info["degeneracy"]
        assert h.info["max_degree"] == info["max_degree"]


@pytest.mark.parametrize("n", [1, 2, 3, 32, 33, 64, 65, 128, 129, 256, 257, 512, 513, 1000])
def test_complete_graphs_every_row_width(n):
    # K_n: the first vertex in the order has |P| = n - 1, so n spans every bitset width
    with gpu_graph(G.complete_graph(n)) as h:
        assert h.count_result() == pins.summary([tuple(range(n))])


@pytest.mark.parametrize("g,count,size", [
    (G.empty_graph(1), 1, 1), (G.empty_graph(777), 777, 1),
    (G.moon_moser(1), 3, 1), (G.moon_moser(4), 81, 4), (G.moon_moser(8), 6561, 8),
    (G.cocktail_party(12), 4096, 12), (G.path_graph(2), 1, 2), (G.path_graph(1000), 999, 2),
    (G.cycle_graph(4), 4, 2), (G.cycle_graph(501), 501, 2),
    (G.complete_multipartite([1] * 400 + [2] * 6), 64, 406),
    (G.complete_multipartite([1] * 700 + [2] * 4), 16, 704),
    (G.complete_multipartite([3, 1, 4, 1, 5, 9, 2, 6]), 3 * 4 * 5 * 9 * 2 * 6, 8),
])
def test_closed_forms(g, count, size):
    with gpu_graph(g) as h:
        c, hs, hist = h.count_result()
    assert c == count
    assert hist == tuple([0] * size + [count])
    assert (c, hs, hist) == O.count(g).key()


def test_zero_vertices():
    with gpu_graph(G.empty_graph(0)) as h:
        assert h.count_result() == (0, 0, ())


# ---------------------------------------------------------------- random and structured graphs

@pytest.mark.parametrize("n,p", [(10, 0.5), (40, 0.3), (64, 0.9), (100, 0.05), (100, 0.5),
                                 (300, 0.05), (300, 0.2), (1000, 0.01), (45, 0.97)])
def test_er_vs_oracle(n, p):
    for seed in range(3):
        assert_count_parity(G.er_graph(n, p, seed))


@pytest.mark.parametrize("seed", [1, 2])
def test_large_planted_cliques_wide_rows(seed):
    # a few planted cliques of 300-600 vertices: subtrees with 16- and 32-word rows
    assert_count_parity(G.planted_graph(3000, 6.0, 5, 300, 600, seed))


@pytest.mark.parametrize("name", ["er200", "ba100k", "planted50k", "sbm_c20", "rmat_s10",
                                  "rmat_s12"])
@pytest.mark.parametrize("seed", [1, 2, 3])
def test_workloads_vs_oracle(name, seed):
    assert_count_parity(G.config_graph(name, seed))


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_sbm_full_size_vs_oracle(seed):
    g = G.config_graph("sbm1m", seed)
    assert_count_parity(g, threads=16)


def _light_roots(g, k, seed, max_p):
    """k seeded roots whose first-level P (from the oracle's order) has fewer than max_p vertices."""
    _, _, rank, _ = O.peel(g)
    src = np.repeat(np.arange(g.n), g.degrees())
    pc = np.bincount(src[rank[g.adj] > rank[src]], minlength=g.n)
    cand = np.nonzero(pc < max_p)[0]
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(cand, size=min(k, cand.size), replace=False)).astype(np.int32)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_rmat_s20_sampled_roots_vs_oracle(seed):
    g = G.config_graph("rmat_s20", seed)
    roots = _light_roots(g, 3000, seed, 160)
    assert_count_parity(g, roots=roots, threads=16)


# ---------------------------------------------------------------- root subsets, order, enumerate

def test_root_partition_sums_to_full_count():
    g = G.config_graph("planted50k", 4)
    mce = _mce()
    rng = np.random.default_rng(5)
    label = rng.integers(0, 3, g.n)
    with gpu_graph(g) as h:
        full = mce.Graph.unpack(h.count())
        parts = [h.count_roots(np.nonzero(label == i)[0].astype(np.int32)) for i in range(3)]
        h.check()
        tot = sum(p.cpu().numpy().view(np.uint64).astype(object) for p in parts)
    assert int(tot[0]) == full[0]
    assert int(tot[1]) % 2**64 == full[1]
    assert tuple(int(x) for x in np.trim_zeros(np.array(tot[2:], dtype=np.uint64), "b")) == full[2]
    roots = np.nonzero(label == 1)[0].astype(np.int32)
    with gpu_graph(g) as h:
        assert h.count_roots_result(roots) == O.count(g, roots=roots).key()


@pytest.mark.parametrize("name,seed", [("er200", 1), ("ba100k", 2), ("rmat_s14", 1),
                                       ("sbm_c50", 2), ("rmat_s20", 1)])
def test_degeneracy_order_matches_oracle(name, seed):
    g = G.config_graph(name, seed)
    core, _, rank, d = O.peel(g)
    with gpu_graph(g) as h:
        r, c = h.order_arrays()
        assert np.array_equal(r.cpu().numpy(), rank)
        assert np.array_equal(c.cpu().numpy(), core)
        assert h.info["degeneracy"] == d
        h.order()                       # recomputing gives the same order
        r2, _ = h.order_arrays()
        assert np.array_equal(r2.cpu().numpy(), rank)


@pytest.mark.parametrize("g", [G.config_graph("er200", 3), G.planted_graph(400, 4.0, 4, 8, 20, 1),
                               G.moon_moser(6), G.disjoint_union([G.empty_graph(5),
                                                                  G.er_graph(60, 0.3, 2)])])
def test_enumerate_matches_oracle(g):
    mce = _mce()
    with gpu_graph(g) as h:
        ids, offs = h.enumerate()
        got = mce.cliques_from(ids, offs)
    assert len(got) == len(set(got))
    assert sorted(got) == sorted(O.enumerate_cliques(g))
    sizes = [len(c) for c in got]
    assert sizes == sorted(sizes)           # grouped by size, ascending


def test_repeat_is_deterministic():
    g = G.config_graph("ba100k", 3)
    with gpu_graph(g) as h:
        a = h.count_result()
        h.order()
        b = h.count_result()
    assert a == b


@pytest.mark.parametrize("overlap", [0, 1])
def test_builds_on_either_stream(overlap):
    # subtree builds on the handle's own stream or on the caller's: the same results
    g = G.config_graph("rmat_s12", 2)
    roots = np.arange(0, g.n, 3, dtype=np.int32)
    with gpu_graph(g, overlap_builds=overlap) as h:
        assert h.count_result() == O.count(g, threads=8).key()
        assert h.count_roots_result(roots) == O.count(g, roots=roots, threads=8).key()


@pytest.mark.parametrize("name,seed", [("rmat_s12", 1), ("sbm_c50", 2), ("planted50k", 3),
                                       ("sbm1m", 1)])
def test_count_after_each_reorder(name, seed):
    # each order places the roots of a schedule bucket anew (atomic cursors), and roots of one
    # bucket differ in degree: every count after a new order must still be the oracle's
    g = G.config_graph(name, seed)
    expect = O.count(g, threads=16).key()
    with gpu_graph(g) as h:
        for _ in range(4):
            h.order()
            assert h.count_result() == expect
        if expect[0] > 2_000_000:
            return
        h.order()
        ids, offs = h.enumerate()
    assert len(_mce().cliques_from(ids, offs)) == expect[0]


# ---------------------------------------------------------------- input handling and errors

def _shuffled(g, seed):
    rng = np.random.default_rng(seed)
    adj = g.adj.copy()
    for v in range(g.n):
        lo, hi = g.offsets[v], g.offsets[v + 1]
        adj[lo:hi] = rng.permutation(adj[lo:hi])
    return G.Graph(g.n, g.offsets.copy(), adj, g.name + "_shuffled")


def test_unsorted_adjacency_is_accepted():
    star = G.csr_from_edges(5001, np.zeros(5000, int), np.arange(1, 5001))   # one 5000-list
    for g in [G.config_graph("er200", 1), G.disjoint_union([star, G.er_graph(300, 0.05, 3)])]:
        expect = O.count(g).key()
        with gpu_graph(_shuffled(g, 1)) as h:
            assert h.count_result() == expect


def test_host_input_path():
    mce = _mce()
    g = G.config_graph("er200", 2)
    with mce.Graph(g.offsets, g.adj) as h:          # numpy host arrays: copied by the library
        assert h.count_result() == O.count(g).key()


def _raw(n, lists):
    offs = np.zeros(n + 1, np.int32)
    offs[1:] = np.cumsum([len(x) for x in lists])
    adj = np.asarray([y for x in lists for y in x] or [0], np.int32)[: offs[-1]]
    return G.Graph(n, offs, adj)


@pytest.mark.parametrize("lists,code", [
    ([[0, 1], [0]], "MCE_ERR_NOT_SIMPLE"), ([[1, 1], [0, 0]], "MCE_ERR_NOT_SIMPLE"),
    ([[1], [0, 2], []], "MCE_ERR_NOT_SYMMETRIC"), ([[5], [0]], "MCE_ERR_ID_RANGE"),
    ([[-1], [0]], "MCE_ERR_ID_RANGE"),
    # only a backward entry (1 lists 0, 0 lists nothing): caught by the entry counts
    ([[], [0]], "MCE_ERR_NOT_SYMMETRIC"), ([[2], [0], [1]], "MCE_ERR_NOT_SYMMETRIC"),
])
def test_invalid_graphs_are_rejected(lists, code):
    mce = _mce()
    with pytest.raises(mce.MceError) as e:
        gpu_graph(_raw(len(lists), lists))
    assert e.value.name == code


def _star(n_leaves, centre_last):
    # a star whose centre list is longer than one validation chunk of a warp
    c = n_leaves if centre_last else 0
    leaves = [i for i in range(n_leaves + 1) if i != c]
    lists = [[c] for _ in range(n_leaves + 1)]
    lists[c] = list(leaves)
    return lists


@pytest.mark.parametrize("centre_last", [False, True])
@pytest.mark.parametrize("defect", ["none", "missing_reverse", "repeat"])
def test_long_lists_are_validated(centre_last, defect):
    mce = _mce()
    lists = _star(9000, centre_last)
    c = 9000 if centre_last else 0
    if defect == "missing_reverse":
        leaf = 4097 if not centre_last else 4095     # inside the second chunk of the centre
        lists[leaf] = []
    elif defect == "repeat":
        k = 4096                                      # a repeat across two chunks
        lists[c].insert(k, lists[c][k - 1])
    g = _raw(len(lists), lists)
    if defect == "none":
        with gpu_graph(g) as h:
            assert h.count_result() == O.count(g).key()
        return
    with pytest.raises(mce.MceError) as e:
        gpu_graph(g)
    want = "MCE_ERR_NOT_SIMPLE" if defect == "repeat" else "MCE_ERR_NOT_SYMMETRIC"
    assert e.value.name == want


def test_widest_rows_and_the_p_limit():
    # K_1025: the first vertex has |P| = 1024, the widest rows (32 words); K_1026 is over
    mce = _mce()
    with gpu_graph(G.complete_graph(1025)) as h:
        assert h.count_result() == pins.summary([tuple(range(1025))])
    with pytest.raises(mce.MceError) as e:
        gpu_graph(G.complete_graph(1026))
    assert e.value.name == "MCE_ERR_LIMIT"


def _star_graph(leaves):
    return G.csr_from_edges(leaves + 1, np.zeros(leaves, np.int64), np.arange(1, leaves + 1))


def test_degree_limit():
    # a degree of 2^21 - 1 is the largest a pivot code can hold; one more is refused
    mce = _mce()
    g = _star_graph((1 << 21) - 1)
    with gpu_graph(g) as h:
        got = h.count_result()
    assert got == O.count(g).key()
    assert got[0] == (1 << 21) - 1 and got[2] == (0, 0, (1 << 21) - 1)
    with pytest.raises(mce.MceError) as e:
        gpu_graph(_star_graph(1 << 21))
    assert e.value.name == "MCE_ERR_LIMIT"


def test_duplicate_roots_count_twice():
    g = G.config_graph("planted50k", 2)
    roots = np.arange(0, g.n, 5, dtype=np.int32)
    with gpu_graph(g) as h:
        one = h.count_roots_result(roots)
        two = h.count_roots_result(np.concatenate([roots, roots[::-1]]))
    assert two[0] == 2 * one[0]
    assert two[1] == (2 * one[1]) % (1 << 64)
    assert two[2] == tuple(2 * x for x in one[2])


def test_bad_offsets_rejected():
    mce = _mce()
    g = G.Graph(3, np.asarray([0, 2, 1, 2], np.int32), np.asarray([1, 2], np.int32))
    with pytest.raises(mce.MceError) as e:
        gpu_graph(g)
    assert e.value.name == "MCE_ERR_INVALID_ARG"


def test_bad_root_id_is_reported():
    mce = _mce()
    g = G.config_graph("er200", 1)
    with gpu_graph(g) as h:
        h.count_roots(np.asarray([3, 999], np.int32))
        assert h.last_error() == 4          # MCE_ERR_ID_RANGE
        assert h.last_error() == 0          # cleared
        assert h.count_result() == O.count(g).key()


def test_enumerate_buffer_too_small():
    import ctypes
    mce = _mce()
    g = G.config_graph("er200", 1)
    with gpu_graph(g) as h:
        sizes = np.zeros(2, np.int64)
        ids = torch.empty(10, dtype=torch.int32, device="cuda")
        offs = torch.empty(11, dtype=torch.int64, device="cuda")
        code = mce.library().mce_enumerate(h._h, mce._stream_ptr(None),
                                           ctypes.c_void_p(ids.data_ptr()), 10,
                                           ctypes.c_void_p(offs.data_ptr()), 10,
                                           sizes.ctypes.data_as(ctypes.c_void_p))
        assert code == 6
        r = O.count(g)
        assert sizes[0] == r.count
        assert sizes[1] == sum(k * int(c) for k, c in enumerate(r.hist))


# ---------------------------------------------------------------- worker list and bounded waits

@pytest.mark.parametrize("name", ["rmat_s12", "planted50k", "sbm_c20"])
def test_worker_list_on_off_and_forced_donations(name):
    g = G.config_graph(name, 2)
    expect = O.count(g, threads=8).key()
    for cfg in [dict(worker_list=0), dict(worker_list=1),
                dict(worker_list=1, donate_min_p=1, blocks_per_sm=1),
                dict(worker_list=1, donate_min_p=1, blocks_per_sm=1, donate_rule=1)]:
        with gpu_graph(g, **cfg) as h:
            assert h.count_result() == expect, cfg
            info = h.get_info()
            if not cfg["worker_list"]:
                assert info["donations"] == 0
    # rmat: heavy subtrees must actually be split when donation is forced
    if name == "rmat_s12":
        with gpu_graph(g, donate_min_p=1, blocks_per_sm=1) as h:
            h.count_result()
            assert h.get_info()["donations"] > 0


def test_rmat_s13_with_worker_list():
    g = G.config_graph("rmat_s13", 1)
    expect = O.count(g, threads=16).key()
    with gpu_graph(g) as h:
        assert h.count_result() == expect
        assert h.get_info()["donations"] > 0


def test_enumerate_with_forced_donations():
    mce = _mce()
    g = G.config_graph("rmat_s10", 3)
    with gpu_graph(g, donate_min_p=1, blocks_per_sm=1) as h:
        ids, offs = h.enumerate()
        got = mce.cliques_from(ids, offs)
    assert sorted(got) == sorted(O.enumerate_cliques(g))


def test_device_wait_limit_returns_an_error_not_a_hang():
    # a 1 ns limit makes the grid barrier of the peel give up at once: the kernel records
    # MCE_ERR_DEVICE_TIMEOUT and returns; the context stays usable afterwards
    mce = _mce()
    g = G.config_graph("ba100k", 1)
    with pytest.raises(mce.MceError) as e:
        gpu_graph(g, spin_limit_ns=1)
    assert e.value.name == "MCE_ERR_DEVICE_TIMEOUT"
    with gpu_graph(g) as h:
        assert h.count_result() == O.count(g, threads=8).key()
