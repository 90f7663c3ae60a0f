"""GPU parity of enumeration by root batches (mce_enumerate_roots) and of the streamed
enumeration built on it, whose pieces are copied to pinned host memory while the next batch
runs.  Every clique set is compared with the oracle's enumeration.
"""
import numpy as np
import pytest

import oracle as O
from maximal_clique_enumeration_gb300 import graphs as G

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
    return _mce().Graph(torch.from_numpy(g.offsets).cuda(), torch.from_numpy(g.adj).cuda(), g.n,
                        **cfg)


def _pieces_to_cliques(pieces):
    out = []
    for ids, offs in pieces:
        assert offs[0] == 0 and offs[-1] == len(ids)
        out += [tuple(int(x) for x in ids[offs[i]: offs[i + 1]]) for i in range(len(offs) - 1)]
    return out


@pytest.mark.parametrize("cfg", [{}, dict(induced=2), dict(subtree_level=2)])
def test_enumerate_roots_matches_oracle(cfg):
    mce = _mce()
    g = G.config_graph("planted50k", 2)
    rng = np.random.default_rng(3)
    roots = np.sort(rng.choice(g.n, 5000, replace=False)).astype(np.int32)
    with gpu_graph(g, **cfg) as h:
        ids, offs = h.enumerate_roots(roots)
        got = mce.cliques_from(ids, offs)
        # the counting path agrees with the enumeration
        c, _, _ = h.count_roots_result(roots)
    want = O.enumerate_cliques(g, roots=roots)
    assert sorted(got) == sorted(want)
    assert c == len(want)


def test_enumerate_roots_empty_and_bad_root():
    mce = _mce()
    g = G.config_graph("er200", 1)
    with gpu_graph(g) as h:
        ids, offs = h.enumerate_roots(np.zeros(0, np.int32))
        assert offs.cpu().tolist() == [0] and ids.numel() == 0
    with gpu_graph(g) as h:
        with pytest.raises(mce.MceError) as e:
            h.enumerate_roots(np.asarray([3, g.n + 5], np.int32))
        assert e.value.name == "MCE_ERR_ID_RANGE"


@pytest.mark.parametrize("name,cfg", [("rmat_s10", {}), ("ba100k", {}), ("sbm_c20", {}),
                                      ("rmat_s10", dict(subtree_level=2, induced=2))])
def test_streamed_enumeration_with_small_buffers(name, cfg):
    g = G.config_graph(name, 1)
    want = O.enumerate_cliques(g)
    # the most cliques and ids one root owns (a clique belongs to its earliest vertex)
    rank = O.peel(g)[2]
    owner = np.asarray([min(c, key=lambda v: rank[v]) for c in want])
    per_root = np.bincount(owner, minlength=g.n)
    ids_root = np.bincount(owner, weights=[len(c) for c in want], minlength=g.n)
    # buffers far smaller than the output: many batches, some halved and retried
    max_cl = int(max(per_root.max(), 64, len(want) // 50))
    max_ids = int(max(ids_root.max(), max_cl * 4))
    with gpu_graph(g, **cfg) as h:
        pieces = list(h.enumerate_stream(max_cliques=max_cl, max_ids=max_ids,
                                         batch_roots=4096))
    assert len(pieces) > 10
    got = _pieces_to_cliques(pieces)
    assert sorted(got) == sorted(want)


def test_streamed_enumeration_of_a_root_subset():
    g = G.config_graph("planted50k", 1)
    roots = np.arange(0, g.n, 7, dtype=np.int32)
    with gpu_graph(g) as h:
        got = _pieces_to_cliques(h.enumerate_stream(roots=roots, max_cliques=2000,
                                                    max_ids=120000))
    assert sorted(got) == sorted(O.enumerate_cliques(g, roots=roots))


def test_streamed_enumeration_root_too_large_for_buffers():
    mce = _mce()
    g = G.moon_moser(7)          # 3^7 cliques; the first root's subtree alone holds 3^6
    with gpu_graph(g) as h:
        with pytest.raises(mce.MceError) as e:
            list(h.enumerate_stream(max_cliques=100, max_ids=10000))
    assert e.value.name == "MCE_ERR_BUFFER_TOO_SMALL"
