"""The allocation-free ordering entry point (mce_order_noalloc), through the C ABI.

Some callers cannot allocate device memory: code running under a framework whose caching
allocator owns the GPU, plug-ins that are only handed buffers, or paths that must not stall on
cudaMalloc.  mce_order_noalloc serves them from one fixed scratch array in device memory.

Its rank, core numbers and degeneracy are compared exactly (they are integers) with the CPU
oracle's canonical peel and with the regular entry point (mce_create + mce_get_order), on calls
made back to back, so that anything the shared scratch array keeps from one call cannot leak
into the next result.  The cases cover the largest graph the scratch admits (n = 2^18), a dense
core that the peel must not finish in a single CTA, and the graph with no vertices.
"""
import ctypes

import numpy as np
import pytest

import oracle as O
from maximal_clique_enumeration_gb300 import graphs as G

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

NOALLOC_MAX_N = 1 << 18


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
    adj = torch.from_numpy(g.adj if g.adj.size else np.zeros(1, np.int32)).cuda()
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


def _check_against_oracle(g, got):
    core, _, rank, d = O.peel(g)
    got_rank, got_core, got_d = got
    assert np.array_equal(got_rank, rank), g.name
    assert np.array_equal(got_core, core), g.name
    assert got_d == d, g.name


def test_noalloc_order_matches_oracle_and_regular_entry_point_twice(lib):
    graphs = [G.config_graph("ba100k", 1), G.config_graph("planted50k", 2)]
    expected = [_regular(g) for g in graphs]
    for g, (rank, core, d) in zip(graphs, expected):          # two calls in a row
        got = _noalloc(lib, g)
        _check_against_oracle(g, got)
        assert np.array_equal(got[0], rank), g.name
        assert np.array_equal(got[1], core), g.name
        assert got[2] == d, g.name


def test_noalloc_at_the_size_limit_and_with_a_dense_core(lib):
    # n at the limit fills every per-vertex array of the scratch to its end; the dense core
    # (4,000 vertices, about 1.6M adjacency entries) keeps the peel on the whole grid
    big = G.er_graph(NOALLOC_MAX_N, 8.0 / (NOALLOC_MAX_N - 1), 5, "er_noalloc_max")
    dense = G.er_graph(4000, 0.1, 6, "er_dense_core")
    assert big.n == NOALLOC_MAX_N and dense.offsets[-1] > (1 << 20)
    for g in (big, dense, big):
        _check_against_oracle(g, _noalloc(lib, g))


def test_noalloc_empty_graph(lib):
    g = G.empty_graph(0)
    res = torch.full((2,), -7, dtype=torch.int32, device="cuda")
    offs = torch.zeros(1, dtype=torch.int32, device="cuda")
    code = lib.mce_order_noalloc(ctypes.c_void_p(offs.data_ptr()), None, 0, None, None,
                                 ctypes.c_void_p(res.data_ptr()),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 0
    torch.cuda.synchronize()
    assert res.cpu().tolist() == [0, 0]
    # and a regular graph right after it still comes out right
    g = G.config_graph("er200", 3)
    _check_against_oracle(g, _noalloc(lib, g))


def test_noalloc_rejects_oversize_graph(lib):
    res = torch.zeros(2, dtype=torch.int32, device="cuda")
    code = lib.mce_order_noalloc(None, None, NOALLOC_MAX_N + 1, None, None,
                                 ctypes.c_void_p(res.data_ptr()), None)
    assert code == 8                                           # MCE_ERR_LIMIT
