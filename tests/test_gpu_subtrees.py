"""GPU parity of the independent second-level subtrees, one per edge {v, w} ordered v before w
("Parallelizing Maximal Clique Enumeration on GPUs", Section 3.2, Algorithm 4), over full and
partial induced subgraphs.  The set of maximal cliques does not depend on how the search is
split, so every result is compared with the oracle bit for bit.
"""
import numpy as np
import pytest

import oracle as O
from maximal_clique_enumeration_gb300 import graphs as G
from tests import pins

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

L2 = dict(subtree_level=2)


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
    return _mce().Graph(torch.from_numpy(g.offsets).cuda(), torch.from_numpy(g.adj).cuda(), g.n,
                        **cfg)


@pytest.mark.parametrize("induced", [1, 2])
@pytest.mark.parametrize("name", ["er200", "ba100k", "planted50k", "sbm_c20", "rmat_s10",
                                  "rmat_s12"])
@pytest.mark.parametrize("seed", [1, 2])
def test_workloads_second_level_vs_oracle(name, seed, induced):
    g = G.config_graph(name, seed)
    with gpu_graph(g, induced=induced, **L2) as h:
        info = h.get_info()
        assert (info["subtree_level"], info["induced"]) == (2, induced)
        assert h.count_result() == O.count(g, threads=8).key()


@pytest.mark.parametrize("n", [1, 2, 3, 33, 65, 129, 257, 513])
def test_second_level_complete_graphs(n):
    with gpu_graph(G.complete_graph(n), **L2) as h:
        assert h.count_result() == pins.summary([tuple(range(n))])


@pytest.mark.parametrize("g", [G.empty_graph(1), G.empty_graph(300), G.moon_moser(6),
                               G.cocktail_party(10), G.path_graph(2), G.path_graph(500),
                               G.cycle_graph(3), G.cycle_graph(99),
                               G.complete_multipartite([1] * 400 + [2] * 6),
                               G.complete_multipartite([3, 1, 4, 1, 5, 9, 2, 6])])
@pytest.mark.parametrize("induced", [1, 2])
def test_second_level_closed_forms(g, induced):
    with gpu_graph(g, induced=induced, **L2) as h:
        assert h.count_result() == O.count(g).key()


def test_second_level_isolated_vertices_and_bare_edges():
    # isolated vertices, edges in no triangle (P and X empty) and one triangle
    src = np.asarray([0, 2, 5, 5, 6])
    dst = np.asarray([1, 3, 6, 7, 7])
    g = G.csr_from_edges(10, src, dst)
    with gpu_graph(g, **L2) as h:
        assert h.count_result() == O.count(g).key()
        roots = np.asarray([4, 8, 9, 0, 5], np.int32)
        assert h.count_roots_result(roots) == O.count(g, roots=roots).key()


@pytest.mark.parametrize("name", ["rmat_s12", "planted50k"])
def test_second_level_with_forced_donations(name):
    g = G.config_graph(name, 2)
    expect = O.count(g, threads=8).key()
    for induced in (1, 2):
        with gpu_graph(g, induced=induced, donate_min_p=1, blocks_per_sm=1, donate_rule=1,
                       **L2) as h:
            assert h.count_result() == expect, induced
            if name == "rmat_s12":
                assert h.get_info()["donations"] > 0


def test_second_level_root_subsets_sum_to_whole():
    g = G.config_graph("planted50k", 3)
    rng = np.random.default_rng(11)
    label = rng.integers(0, 3, g.n)
    whole = O.count(g, threads=8).key()
    with gpu_graph(g, **L2) as h:
        assert h.count_result() == whole
        parts = []
        for k in range(3):
            roots = np.nonzero(label == k)[0].astype(np.int32)
            got = h.count_roots_result(roots)
            assert got == O.count(g, roots=roots, threads=8).key()
            parts.append(got)
    assert sum(p[0] for p in parts) == whole[0]
    assert sum(p[1] for p in parts) % (1 << 64) == whole[1]


def test_second_level_enumerate_matches_oracle():
    mce = _mce()
    g = G.config_graph("rmat_s10", 1)
    with gpu_graph(g, donate_min_p=1, blocks_per_sm=1, **L2) as h:
        ids, offs = h.enumerate()
        got = mce.cliques_from(ids, offs)
    assert sorted(got) == sorted(O.enumerate_cliques(g))
