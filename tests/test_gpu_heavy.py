"""GPU parity on the heavy first-level subtrees of the R-MAT scale-20 workload graph.

The bench's headline leaves out the roots with |P| >= 128 (8-, 16- and 32-word rows); this
suite checks the kernels of those widths on the real graph.  The expected values are the
oracle's, root by root, stored in tests/golden/rmat_s20_heavy_roots.txt by the committed script
tests/golden/make_rmat_s20_heavy.py (the oracle and the seeded generator only): a seeded
sample of the roots with 128 <= |P| < 256 and 256 <= |P| < 512, each one the oracle finished
within its time limit.
"""
import numpy as np
import pytest

from maximal_clique_enumeration_gb300 import graphs as G
from tests import pins

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

torch = pytest.importorskip("torch")

GOLDEN = "rmat_s20_heavy_roots.txt"


@pytest.fixture(scope="module")
def heavy():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from maximal_clique_enumeration_gb300 import build
    build.build()
    info, roots, skipped = pins.load_root_golden(GOLDEN)
    g = G.config_graph(info["name"], info["seed"])
    assert pins.graph_fingerprint(g) == info["fingerprint"], \
        "the seeded generator no longer reproduces the graph the stored results were made on"
    return g, roots


def _handle(g, **cfg):
    import maximal_clique_enumeration_gb300 as mce
    return mce.Graph(torch.from_numpy(g.offsets).cuda(), torch.from_numpy(g.adj).cuda(), g.n,
                     **cfg)


def test_heavy_roots_one_by_one(heavy):
    g, roots = heavy
    assert roots
    widths = set()
    with _handle(g) as h:
        for v, p, key in roots:
            assert h.count_roots_result(np.array([v], np.int32)) == key, (v, p)
            widths.add(8 if p < 256 else 16)
    assert 8 in widths


def test_heavy_roots_together_and_with_forced_donations(heavy):
    g, roots = heavy
    ids = np.array([v for v, _, _ in roots], np.int32)
    expect = pins.add_keys([key for _, _, key in roots])
    with _handle(g) as h:
        assert h.count_roots_result(ids) == expect
    with _handle(g, donate_min_p=1, donate_rule=1) as h:
        assert h.count_roots_result(ids) == expect
        assert h.get_info()["donations"] > 0
