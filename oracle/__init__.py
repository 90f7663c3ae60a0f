"""TEST INFRASTRUCTURE -- ctypes wrapper around the plain C oracle in ``mce_oracle.c``.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package.  The product (the CUDA library and its Python binding) never touches it.

The oracle follows "Parallelizing Maximal Clique Enumeration on GPUs" (arXiv 2212.01473v2),
Algorithms 2 and 3 (Sections 2.3-2.4) with degeneracy ordering; see the header of
``mce_oracle.c`` for the exact readings.  Results are summarised as
``(count, hash, hist)`` where ``hist[k]`` is the number of maximal cliques of size k.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mce_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None

OK, INVALID_ARG, NOT_SIMPLE, NOT_SYMMETRIC, ID_RANGE, NOMEM, BUFFER = range(7)
ALG3_TOMITA, ALG2_TOMITA, ALG2_PIVOT_P, ALG1_PLAIN, ALG4_TOMITA = range(5)


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: oracle status {code}")
        self.code = code


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH, defines=()) -> str:
    """Compile the oracle C source into a shared library (OpenMP when gcc supports it)."""
    if (not force and not defines and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", *[f"-D{d}" for d in defines],
            "-o", tmp, src]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, out)
    return out


def _bind(path: str):
    lib = ctypes.CDLL(path)
    i32, i64, u64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64
    P = ctypes.c_void_p
    lib.oracle_mix64.restype = u64
    lib.oracle_mix64.argtypes = [u64]
    lib.oracle_vertex_key.restype = u64
    lib.oracle_vertex_key.argtypes = [i32]
    lib.oracle_clique_hash.restype = u64
    lib.oracle_clique_hash.argtypes = [P, i32]
    lib.oracle_validate.restype = ctypes.c_int
    lib.oracle_validate.argtypes = [i32, P, P]
    lib.oracle_peel.restype = ctypes.c_int
    lib.oracle_peel.argtypes = [i32, P, P, P, P, P, P]
    lib.oracle_core_bz.restype = ctypes.c_int
    lib.oracle_core_bz.argtypes = [i32, P, P, P]
    lib.oracle_count.restype = ctypes.c_int
    lib.oracle_count.argtypes = [i32, P, P, P, i64, i32, i32, P, i32, P]
    lib.oracle_enumerate.restype = ctypes.c_int
    lib.oracle_enumerate.argtypes = [i32, P, P, P, i64, i32, P, i64, P, i64, P]
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(build())
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _csr(g):
    return (np.ascontiguousarray(g.offsets, dtype=np.int32),
            np.ascontiguousarray(g.adj if g.adj.size else np.zeros(1, np.int32), dtype=np.int32))


@dataclass
class Result:
    count: int
    hash: int
    hist: np.ndarray          # uint64, hist[k] = cliques with k vertices
    nodes: int = 0            # search-tree nodes visited (a diagnostic, not part of parity)

    def key(self):
        h = np.trim_zeros(np.asarray(self.hist, dtype=np.uint64), "b")
        return int(self.count), int(self.hash), tuple(int(x) for x in h)


def mix64(x: int) -> int:
    return int(_load().oracle_mix64(ctypes.c_uint64(x & (2**64 - 1))))


def vertex_key(v: int) -> int:
    return int(_load().oracle_vertex_key(v))


def clique_hash(ids) -> int:
    a = np.ascontiguousarray(ids, dtype=np.int32)
    return int(_load().oracle_clique_hash(_ptr(a), a.size))


def validate(g) -> int:
    """Status code of the input checks (0 = a simple undirected graph)."""
    offs, adj = _csr(g)
    return int(_load().oracle_validate(g.n, _ptr(offs), _ptr(adj)))


def peel(g):
    """Canonical peel: returns (core, round, rank, d)."""
    offs, adj = _csr(g)
    n = g.n
    core = np.zeros(max(n, 1), np.int32)
    rnd = np.zeros(max(n, 1), np.int32)
    rank = np.zeros(max(n, 1), np.int32)
    d = ctypes.c_int32(0)
    rc = _load().oracle_peel(n, _ptr(offs), _ptr(adj), _ptr(core), _ptr(rnd), _ptr(rank),
                             ctypes.byref(d))
    if rc:
        raise OracleError(rc, "peel")
    return core[:n], rnd[:n], rank[:n], int(d.value)


def core_bz(g) -> np.ndarray:
    offs, adj = _csr(g)
    core = np.zeros(max(g.n, 1), np.int32)
    rc = _load().oracle_core_bz(g.n, _ptr(offs), _ptr(adj), _ptr(core))
    if rc:
        raise OracleError(rc, "core_bz")
    return core[: g.n]


def count(g, roots=None, variant: int = ALG3_TOMITA, threads: int = 1,
          hist_len: int | None = None) -> Result:
    """Count the maximal cliques (optionally only the first-level subtrees of `roots`)."""
    offs, adj = _csr(g)
    if hist_len is None:
        hist_len = (peel(g)[3] + 2) if g.n else 2
    out = np.zeros(2 + hist_len, np.uint64)
    nodes = ctypes.c_uint64(0)
    r = None if roots is None else np.ascontiguousarray(roots, dtype=np.int32)
    rc = _load().oracle_count(g.n, _ptr(offs), _ptr(adj), _ptr(r), 0 if r is None else r.size,
                              variant, threads, _ptr(out), hist_len, ctypes.byref(nodes))
    if rc:
        raise OracleError(rc, "count")
    return Result(int(out[0]), int(out[1]), out[2:].copy(), int(nodes.value))


def enumerate_cliques(g, roots=None, variant: int = ALG3_TOMITA):
    """All maximal cliques as a list of tuples of original ids (each sorted ascending)."""
    offs, adj = _csr(g)
    r = None if roots is None else np.ascontiguousarray(roots, dtype=np.int32)
    nr = 0 if r is None else r.size
    sizes = np.zeros(2, np.int64)
    dummy_o = np.zeros(1, np.int64)
    lib = _load()
    rc = lib.oracle_enumerate(g.n, _ptr(offs), _ptr(adj), _ptr(r), nr, variant, None, 0,
                              _ptr(dummy_o), 0, _ptr(sizes))
    if rc not in (OK, BUFFER):
        raise OracleError(rc, "enumerate (sizing)")
    ncl, nids = int(sizes[0]), int(sizes[1])
    ids = np.zeros(max(nids, 1), np.int32)
    offsets = np.zeros(ncl + 1, np.int64)
    rc = lib.oracle_enumerate(g.n, _ptr(offs), _ptr(adj), _ptr(r), nr, variant, _ptr(ids), nids,
                              _ptr(offsets), ncl, _ptr(sizes))
    if rc:
        raise OracleError(rc, "enumerate")
    return [tuple(int(x) for x in ids[offsets[i]: offsets[i + 1]]) for i in range(ncl)]


class Oracle:
    """The same API bound to a specific build of the oracle source (used by mutation tests)."""

    def __init__(self, path: str):
        self._lib = _bind(path)

    def __getattr__(self, name):
        fn = globals()[name]
        if not callable(fn):
            raise AttributeError(name)

        def call(*a, **k):
            global _lib
            saved = _lib
            _lib = self._lib
            try:
                return fn(*a, **k)
            finally:
                _lib = saved
        return call
