"""GPU parity of the partial induced subgraphs (rows for P only; P-X adjacencies looked up in
the graph; pivot from P u X_P) and of the rule that picks them ("Parallelizing Maximal Clique
Enumeration on GPUs", Sections 3.4, 3.5 and 4.5).  The set of maximal cliques does not depend
on the variant, so every result is compared with the oracle bit for bit.
"""
import numpy as np
import pytest

import oracle as O
from maximal_clique_enumeration_gb300 import graphs as G
from tests import pins

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

PARTIAL, FULL = 2, 1


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


@pytest.mark.parametrize("name,seed", [("er200", 1), ("ba100k", 1), ("ba100k", 2),
                                       ("planted50k", 1), ("sbm_c20", 1), ("rmat_s12", 1)])
def test_default_rule_picks_partial_iff_delta_over_d_above_200(name, seed):
    g = G.config_graph(name, seed)
    with gpu_graph(g) as h:
        info = h.get_info()
        want = PARTIAL if info["max_degree"] > 200 * info["degeneracy"] else FULL
        assert info["induced"] == want
        assert info["subtree_level"] == 1
        assert h.count_result() == O.count(g, threads=8).key()


@pytest.mark.parametrize("induced", [PARTIAL, FULL])
@pytest.mark.parametrize("name", ["er200", "ba100k", "planted50k", "sbm_c20", "rmat_s10",
                                  "rmat_s12"])
@pytest.mark.parametrize("seed", [1, 2])
def test_workloads_both_variants_vs_oracle(name, seed, induced):
    g = G.config_graph(name, seed)
    with gpu_graph(g, induced=induced) as h:
        assert h.get_info()["induced"] == induced
        assert h.count_result() == O.count(g, threads=8).key()


@pytest.mark.parametrize("n", [1, 2, 33, 65, 129, 257, 513, 1000])
def test_partial_complete_graphs_every_row_width(n):
    with gpu_graph(G.complete_graph(n), induced=PARTIAL) as h:
        assert h.count_result() == pins.summary([tuple(range(n))])


@pytest.mark.parametrize("g", [G.empty_graph(5), G.moon_moser(6), G.cocktail_party(10),
                               G.path_graph(300), G.cycle_graph(77),
                               G.complete_multipartite([1] * 400 + [2] * 6),
                               G.complete_multipartite([3, 1, 4, 1, 5, 9, 2, 6])])
def test_partial_closed_forms(g):
    with gpu_graph(g, induced=PARTIAL) as h:
        assert h.count_result() == O.count(g).key()


def test_partial_star_hub_with_huge_x():
    # a hub adjacent to 5000 leaves and to one triangle: the triangle's late vertices see the
    # hub in X, whose later-neighbour list is searched for every X_X test
    n = 5003
    src = list(np.zeros(5002, int)) + [5001]
    dst = list(range(1, 5003)) + [5002]
    g = G.csr_from_edges(n, np.asarray(src), np.asarray(dst))
    with gpu_graph(g, induced=PARTIAL) as h:
        assert h.count_result() == O.count(g).key()


@pytest.mark.parametrize("name", ["rmat_s12", "planted50k"])
def test_partial_with_forced_donations(name):
    g = G.config_graph(name, 2)
    expect = O.count(g, threads=8).key()
    for rule in (0, 1):
        with gpu_graph(g, induced=PARTIAL, donate_min_p=1, blocks_per_sm=1,
                       donate_rule=rule) as h:
            assert h.count_result() == expect, rule
            if name == "rmat_s12":
                assert h.get_info()["donations"] > 0


def test_partial_root_subsets_sum_to_whole():
    g = G.config_graph("ba100k", 3)
    rng = np.random.default_rng(7)
    label = rng.integers(0, 2, g.n)
    whole = O.count(g, threads=8).key()
    with gpu_graph(g, induced=PARTIAL) as h:
        assert h.count_result() == whole
        parts = [h.count_roots_result(np.nonzero(label == k)[0].astype(np.int32))
                 for k in (0, 1)]
    for k, part in zip((0, 1), parts):
        roots = np.nonzero(label == k)[0].astype(np.int32)
        assert part == O.count(g, roots=roots, threads=8).key()
    assert parts[0][0] + parts[1][0] == whole[0]
    assert (parts[0][1] + parts[1][1]) % (1 << 64) == whole[1]


def test_partial_enumerate_matches_oracle():
    mce = _mce()
    g = G.config_graph("rmat_s10", 2)
    with gpu_graph(g, induced=PARTIAL, donate_min_p=1, blocks_per_sm=1) as h:
        ids, offs = h.enumerate()
        got = mce.cliques_from(ids, offs)
    assert sorted(got) == sorted(O.enumerate_cliques(g))
