"""The allocation-free ordering entry point (mce_order_noalloc) against the regular one.

Some callers cannot allocate device memory (a framework's allocator owns the GPU, or the call
sits on a path that must not synchronise for cudaMalloc); mce_order_noalloc serves them from a
fixed scratch array.  This test calls it through the C ABI twice in a row, on two different
graphs, and checks that rank, core numbers and degeneracy equal what mce_create +
mce_get_order report -- exactly, as these are integers.  The second call also shows that state
left in the shared scratch array by the first call does not leak into the next result.
"""
import ctypes

import numpy as np
import pytest

from maximal_clique_enumeration_gb300 import graphs as G

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from maximal_clique_enumeration_gb300 import build
    build.build()
    import maximal_clique_enumeration_gb300 as mce
    L = mce.library()
    P = ctypes.c_void_p
    L.mce_order_noalloc.restype = ctypes.c_int
    L.mce_order_noalloc.argtypes = [P, P, ctypes.c_int32, P, P, P, P]
    return L


def _regular(g):
    import maximal_clique_enumeration_gb300 as mce
    with mce.Graph(torch.from_numpy(g.offsets).cuda(), torch.from_numpy(g.adj).cuda(), g.n) as h:
        rank, core = h.order_arrays()
        return rank.cpu().numpy(), core.cpu().numpy(), h.info["degeneracy"]


def _noalloc(lib, g):
    offs = torch.from_numpy(g.offsets).cuda()
    adj = torch.from_numpy(g.adj).cuda()
    rank = torch.full((max(g.n, 1),), -7, dtype=torch.int32, device="cuda")
    core = torch.full((max(g.n, 1),), -7, dtype=torch.int32, device="cuda")
    res = torch.full((2,), -7, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    code = lib.mce_order_noalloc(ctypes.c_void_p(offs.data_ptr()), ctypes.c_void_p(adj.data_ptr()),
                                 g.n, ctypes.c_void_p(rank.data_ptr()),
                                 ctypes.c_void_p(core.data_ptr()), ctypes.c_void_p(res.data_ptr()),
                                 ctypes.c_void_p(stream.cuda_stream))
    assert code == 0
    torch.cuda.synchronize()
    r = res.cpu().numpy()
    assert r[1] == 0, f"device-side status {r[1]}"
    return rank.cpu().numpy()[: g.n], core.cpu().numpy()[: g.n], int(r[0])


def test_noalloc_order_matches_regular_entry_point_twice(lib):
    graphs = [G.config_graph("ba100k", 1), G.config_graph("planted50k", 2)]
    expected = [_regular(g) for g in graphs]
    for g, (rank, core, d) in zip(graphs, expected):          # two calls in a row
        got_rank, got_core, got_d = _noalloc(lib, g)
        assert np.array_equal(got_rank, rank), g.name
        assert np.array_equal(got_core, core), g.name
        assert got_d == d, g.name


def test_noalloc_rejects_oversize_graph(lib):
    res = torch.zeros(2, dtype=torch.int32, device="cuda")
    code = lib.mce_order_noalloc(None, None, (1 << 18) + 1, None, None,
                                 ctypes.c_void_p(res.data_ptr()), None)
    assert code == 8                                           # MCE_ERR_LIMIT
