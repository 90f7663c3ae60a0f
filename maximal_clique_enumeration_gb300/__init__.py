"""GB300 maximal clique enumeration: Python binding of libmce_gb300.so (ctypes).

The binding only marshals arguments: every step of the computation runs in the CUDA library
declared in ``include/mce.h``.  PyTorch supplies device memory and streams.  There is no CPU
fallback: if the library is missing, every call raises.

    import maximal_clique_enumeration_gb300 as mce
    g = mce.Graph(offsets, adj)          # CSR as torch tensors (CUDA or CPU) or numpy arrays
    count, hash_, hist = g.count_result()
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import LIB_PATH

__all__ = ["Graph", "MceError", "Config", "Info", "library", "STATUS", "graphs"]

STATUS = {
    0: "MCE_OK", 1: "MCE_ERR_INVALID_ARG", 2: "MCE_ERR_NOT_SIMPLE", 3: "MCE_ERR_NOT_SYMMETRIC",
    4: "MCE_ERR_ID_RANGE", 5: "MCE_ERR_OUT_OF_MEMORY", 6: "MCE_ERR_BUFFER_TOO_SMALL",
    7: "MCE_ERR_DEVICE_TIMEOUT", 8: "MCE_ERR_LIMIT", 9: "MCE_ERR_CUDA", 10: "MCE_ERR_INTERNAL",
}
EXPORTS = ["mce_config_default", "mce_create", "mce_order", "mce_count", "mce_count_roots",
           "mce_enumerate", "mce_get_order", "mce_last_error", "mce_get_info", "mce_get_profile",
           "mce_destroy", "mce_status_str", "mce_order_noalloc", "mce_enumerate_roots",
           "mce_trim_memory"]
PROFILE_ACTIVITIES = ["build", "pivot", "child", "partition", "donate", "idle", "max_root",
                      "roots", "small", "split", "hash", "walk", "xlist"]
PROF_SLOTS = 16


class MceError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = int(code)
        self.name = STATUS.get(self.code, str(code))
        super().__init__(f"{what}: {self.name}" if what else self.name)


NUM_WIDTHS = 6
PROF_SMS = 256


class Config(ctypes.Structure):
    _fields_ = [("worker_list", ctypes.c_int32), ("donate_min_p", ctypes.c_int32),
                ("warps_per_block", ctypes.c_int32), ("blocks_per_sm", ctypes.c_int32),
                ("profile", ctypes.c_int32), ("donate_rule", ctypes.c_int32),
                ("spin_limit_ns", ctypes.c_int64), ("induced", ctypes.c_int32),
                ("subtree_level", ctypes.c_int32), ("overlap_builds", ctypes.c_int32)]


class Info(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int32), ("degeneracy", ctypes.c_int32), ("m", ctypes.c_int64),
                ("max_degree", ctypes.c_int32), ("hist_len", ctypes.c_int32),
                ("peel_rounds", ctypes.c_int32), ("n_workers", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_int64), ("tree_nodes", ctypes.c_uint64),
                ("donations", ctypes.c_uint64), ("words", ctypes.c_uint64 * NUM_WIDTHS),
                ("roots", ctypes.c_int32 * NUM_WIDTHS), ("workers", ctypes.c_int32 * NUM_WIDTHS),
                ("ms_search", ctypes.c_float * NUM_WIDTHS), ("ms_order", ctypes.c_float),
                ("launches", ctypes.c_int32), ("induced", ctypes.c_int32),
                ("subtree_level", ctypes.c_int32), ("ms_peel", ctypes.c_float),
                ("peel_live", ctypes.c_int64), ("ms_build", ctypes.c_float * NUM_WIDTHS)]

    def as_dict(self):
        out = {}
        for k, _ in self._fields_:
            v = getattr(self, k)
            out[k] = list(v) if isinstance(v, ctypes.Array) else v
        return out


_lib = None


def library(path: str | None = None):
    """Loads libmce_gb300.so (raises if it has not been built).

    MCE_LIBRARY in the environment selects another build of the same library (for example the
    MCE_PROFILE variant from build.build(profile=True)).
    """
    global _lib
    if _lib is not None:
        return _lib
    path = path or os.environ.get("MCE_LIBRARY") or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                           "(nvcc, sm_103a); there is no CPU fallback")
    lib = ctypes.CDLL(path)
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    st = ctypes.c_int
    lib.mce_config_default.restype = st
    lib.mce_config_default.argtypes = [ctypes.POINTER(Config)]
    lib.mce_create.restype = st
    lib.mce_create.argtypes = [P, P, i32, ctypes.c_int, ctypes.POINTER(Config), P,
                               ctypes.POINTER(P)]
    lib.mce_order.restype = st
    lib.mce_order.argtypes = [P, P]
    lib.mce_count.restype = st
    lib.mce_count.argtypes = [P, P, P]
    lib.mce_count_roots.restype = st
    lib.mce_count_roots.argtypes = [P, P, P, i32, P]
    lib.mce_enumerate.restype = st
    lib.mce_enumerate.argtypes = [P, P, P, i64, P, i64, P]
    lib.mce_enumerate_roots.restype = st
    lib.mce_enumerate_roots.argtypes = [P, P, P, i32, P, i64, P, i64, P]
    lib.mce_get_order.restype = st
    lib.mce_get_order.argtypes = [P, P, P, P]
    lib.mce_last_error.restype = st
    lib.mce_last_error.argtypes = [P, P]
    lib.mce_get_info.restype = st
    lib.mce_get_info.argtypes = [P, ctypes.POINTER(Info)]
    lib.mce_get_profile.restype = st
    lib.mce_get_profile.argtypes = [P, P]
    lib.mce_destroy.restype = None
    lib.mce_destroy.argtypes = [P]
    lib.mce_trim_memory.restype = st
    lib.mce_trim_memory.argtypes = []
    lib.mce_status_str.restype = ctypes.c_char_p
    lib.mce_status_str.argtypes = [st]
    _lib = lib
    return lib


def _check(code: int, what: str):
    if code != 0:
        raise MceError(code, what)


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def default_config(**overrides) -> Config:
    cfg = Config()
    _check(library().mce_config_default(ctypes.byref(cfg)), "mce_config_default")
    for k, v in overrides.items():
        setattr(cfg, k, v)
    return cfg


def _u64_view(t):
    """uint64 numpy view of an int64 tensor's host copy."""
    return t.detach().cpu().numpy().view(np.uint64)


class Graph:
    """One graph held by the library (mce_create ... mce_destroy)."""

    def __init__(self, offsets, adj, n: int | None = None, config: Config | None = None,
                 stream=None, **config_overrides):
        import torch
        lib = library()
        if isinstance(offsets, np.ndarray):
            offsets = torch.from_numpy(np.ascontiguousarray(offsets, dtype=np.int32))
        if isinstance(adj, np.ndarray):
            adj = torch.from_numpy(np.ascontiguousarray(adj, dtype=np.int32))
        if offsets.dtype != torch.int32 or adj.dtype != torch.int32:
            raise TypeError("offsets and adj must be int32")
        offsets, adj = offsets.contiguous(), adj.contiguous()
        if offsets.is_cuda != adj.is_cuda:
            raise ValueError("offsets and adj must both be on the host or both on the device")
        if n is None:
            n = offsets.numel() - 1
        if config is None:
            config = default_config(**config_overrides)
        self._keep = (offsets, adj)
        self._h = ctypes.c_void_p(0)
        adj_ptr = adj.data_ptr() if adj.numel() else 0
        code = lib.mce_create(ctypes.c_void_p(offsets.data_ptr()), ctypes.c_void_p(adj_ptr),
                              int(n), 1 if offsets.is_cuda else 0, ctypes.byref(config),
                              _stream_ptr(stream), ctypes.byref(self._h))
        self._keep = None
        _check(code, "mce_create")
        self.info = self.get_info()
        self.n = self.info["n"]
        self.hist_len = self.info["hist_len"]

    # -- lifecycle
    def close(self):
        if getattr(self, "_h", None) and self._h.value:
            library().mce_destroy(self._h)
            self._h = ctypes.c_void_p(0)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # -- calls
    def get_info(self) -> dict:
        info = Info()
        _check(library().mce_get_info(self._h, ctypes.byref(info)), "mce_get_info")
        return info.as_dict()

    def profile(self) -> dict:
        """Per row width: cycles per activity of the last search (MCE_PROFILE builds only)."""
        out = np.zeros(PROF_SLOTS * NUM_WIDTHS + 16 + PROF_SMS * NUM_WIDTHS, np.uint64)
        _check(library().mce_get_profile(self._h, out.ctypes.data_as(ctypes.c_void_p)),
               "mce_get_profile")
        res = {1 << k: dict(zip(PROFILE_ACTIVITIES,
                                (int(x) for x in out[PROF_SLOTS * k: PROF_SLOTS * k + 13])))
               for k in range(NUM_WIDTHS)}
        phases = ["scan_ns", "exchange_ns", "write_ns", "edges_ns", "barrier_ns", "rounds"]
        base = PROF_SLOTS * NUM_WIDTHS
        res["peel"] = {"multi": dict(zip(phases, (int(x) for x in out[base: base + 6]))),
                       "single": dict(zip(phases, (int(x) for x in out[base + 8: base + 14]))),
                       "max_removed_degree": int(out[base + 6])}
        sm = out[base + 16:].reshape(NUM_WIDTHS, PROF_SMS)
        for k in range(NUM_WIDTHS):
            res[1 << k]["sm_busy"] = sm[k].astype(np.int64)
        return res

    def order(self, stream=None):
        _check(library().mce_order(self._h, _stream_ptr(stream)), "mce_order")

    def new_output(self):
        import torch
        return torch.zeros(2 + self.hist_len, dtype=torch.int64, device="cuda")

    def count(self, out=None, stream=None):
        """Enqueues mce_count; returns the int64 device tensor holding the uint64 output."""
        out = self.new_output() if out is None else out
        _check(library().mce_count(self._h, _stream_ptr(stream), ctypes.c_void_p(out.data_ptr())),
               "mce_count")
        return out

    def count_roots(self, roots, out=None, stream=None):
        import torch
        out = self.new_output() if out is None else out
        if not isinstance(roots, torch.Tensor):
            roots = torch.as_tensor(np.asarray(roots, dtype=np.int32))
        roots = roots.to(device="cuda", dtype=torch.int32).contiguous()
        self._roots_keep = roots
        _check(library().mce_count_roots(self._h, _stream_ptr(stream),
                                         ctypes.c_void_p(roots.data_ptr()), int(roots.numel()),
                                         ctypes.c_void_p(out.data_ptr())), "mce_count_roots")
        return out

    def last_error(self, stream=None) -> int:
        return int(library().mce_last_error(self._h, _stream_ptr(stream)))

    def check(self, stream=None):
        code = self.last_error(stream)
        if code:
            raise MceError(code, "device-side status")

    @staticmethod
    def unpack(out):
        """(count, hash, hist tuple trimmed of trailing zeros) from an output tensor."""
        u = _u64_view(out)
        hist = np.trim_zeros(u[2:], "b")
        return int(u[0]), int(u[1]), tuple(int(x) for x in hist)

    def count_result(self, stream=None):
        out = self.count(stream=stream)
        self.check(stream)
        return self.unpack(out)

    def count_roots_result(self, roots, stream=None):
        out = self.count_roots(roots, stream=stream)
        self.check(stream)
        return self.unpack(out)

    def enumerate_roots(self, roots, stream=None):
        """The maximal cliques of the given roots' subtrees: (ids, offsets) device tensors."""
        import torch
        roots = torch.as_tensor(np.asarray(roots, dtype=np.int32)).cuda()
        dummy_i = torch.zeros(1, dtype=torch.int32, device="cuda")
        dummy_o = torch.zeros(1, dtype=torch.int64, device="cuda")
        code, (nc, ni) = _enumerate_roots_into(self._h, roots, dummy_i[:0], dummy_o, stream)
        if code not in (0, 6):
            raise MceError(code, "mce_enumerate_roots (sizing)")
        ids = torch.empty(max(ni, 1), dtype=torch.int32, device="cuda")
        offs = torch.empty(nc + 1, dtype=torch.int64, device="cuda")
        code, _ = _enumerate_roots_into(self._h, roots, ids, offs, stream)
        _check(code, "mce_enumerate_roots")
        return ids[:ni], offs

    def enumerate_stream(self, roots=None, max_cliques: int = 1 << 22, max_ids: int = 1 << 25,
                         batch_roots: int = 1 << 16, stream=None):
        """Yields the enumeration in host pieces (ids, offsets), numpy, piece by piece.

        Roots (all vertices by default) are taken in batches whose output fits device buffers of
        max_cliques cliques and max_ids ids; a batch that does not fit is halved, and one that
        fills little of them lets the next batch grow.  Two buffer pairs alternate: while one
        batch is enumerated, the previous one is copied to pinned host memory on a side stream.
        Each piece's offsets start at 0.  A single root whose cliques exceed the buffers raises
        MceError(MCE_ERR_BUFFER_TOO_SMALL).
        """
        import torch
        if roots is None:
            roots = np.arange(self.n, dtype=np.int32)
        roots = np.asarray(roots, dtype=np.int32)
        dev_roots = torch.as_tensor(roots).cuda()
        main = stream if stream is not None else torch.cuda.current_stream()
        side = torch.cuda.Stream()
        bufs = [(torch.empty(max_ids, dtype=torch.int32, device="cuda"),
                 torch.empty(max_cliques + 1, dtype=torch.int64, device="cuda"),
                 torch.empty(max_ids, dtype=torch.int32).pin_memory(),
                 torch.empty(max_cliques + 1, dtype=torch.int64).pin_memory(),
                 torch.cuda.Event()) for _ in range(2)]
        pending = None          # (slot, cliques, ids) being copied to the host
        start, b, slot = 0, max(1, int(batch_roots)), 0
        while start < len(roots):
            n_b = min(b, len(roots) - start)
            d_ids, d_offs, h_ids, h_offs, done = bufs[slot]
            done.synchronize()                       # this slot's last copy has landed
            with torch.cuda.stream(main):
                code, (nc, ni) = _enumerate_roots_into(self._h, dev_roots[start:start + n_b],
                                                       d_ids, d_offs, main)
            if code == 6:
                if n_b == 1:
                    raise MceError(code, f"mce_enumerate_roots: root {int(roots[start])} needs "
                                         f"{nc} cliques / {ni} ids")
                b = max(1, n_b // 2)
                continue
            _check(code, "mce_enumerate_roots")
            ready = torch.cuda.Event()
            ready.record(main)
            with torch.cuda.stream(side):
                side.wait_event(ready)
                h_ids[:ni].copy_(d_ids[:ni], non_blocking=True)
                h_offs[:nc + 1].copy_(d_offs[:nc + 1], non_blocking=True)
                done.record(side)
            if pending is not None:
                p_slot, p_nc, p_ni = pending
                bufs[p_slot][4].synchronize()
                yield bufs[p_slot][2][:p_ni].numpy().copy(), bufs[p_slot][3][:p_nc + 1].numpy().copy()
            pending = (slot, nc, ni)
            slot ^= 1
            start += n_b
            if 4 * nc < max_cliques and 4 * ni < max_ids:
                b = min(2 * b, 1 << 24)
        if pending is not None:
            p_slot, p_nc, p_ni = pending
            bufs[p_slot][4].synchronize()
            yield bufs[p_slot][2][:p_ni].numpy().copy(), bufs[p_slot][3][:p_nc + 1].numpy().copy()

    def enumerate(self, stream=None):
        """All maximal cliques: (ids int32 tensor, offsets int64 tensor) on the device."""
        import torch
        lib = library()
        sizes = np.zeros(2, np.int64)
        dummy = torch.zeros(1, dtype=torch.int64, device="cuda")
        code = lib.mce_enumerate(self._h, _stream_ptr(stream), ctypes.c_void_p(0), 0,
                                 ctypes.c_void_p(dummy.data_ptr()), 0,
                                 sizes.ctypes.data_as(ctypes.c_void_p))
        if code not in (0, 6):
            raise MceError(code, "mce_enumerate (sizing)")
        ids = torch.empty(max(int(sizes[1]), 1), dtype=torch.int32, device="cuda")
        offs = torch.empty(int(sizes[0]) + 1, dtype=torch.int64, device="cuda")
        _check(lib.mce_enumerate(self._h, _stream_ptr(stream), ctypes.c_void_p(ids.data_ptr()),
                                 ids.numel(), ctypes.c_void_p(offs.data_ptr()), int(sizes[0]),
                                 sizes.ctypes.data_as(ctypes.c_void_p)), "mce_enumerate")
        self.check(stream)
        return ids[: int(sizes[1])], offs

    def order_arrays(self, stream=None):
        """(rank, core) int32 device tensors of the current degeneracy order."""
        import torch
        rank = torch.empty(max(self.n, 1), dtype=torch.int32, device="cuda")
        core = torch.empty(max(self.n, 1), dtype=torch.int32, device="cuda")
        _check(library().mce_get_order(self._h, _stream_ptr(stream),
                                       ctypes.c_void_p(rank.data_ptr()),
                                       ctypes.c_void_p(core.data_ptr())), "mce_get_order")
        return rank[: self.n], core[: self.n]


def trim_memory():
    """Hands the device memory cached by the library's pool (current device) back to the driver."""
    _check(library().mce_trim_memory(), "mce_trim_memory")


def _enumerate_roots_into(h, roots, ids, offs, stream):
    """One mce_enumerate_roots call: returns (status code, (cliques, ids) needed or written)."""
    sizes = np.zeros(2, np.int64)
    code = library().mce_enumerate_roots(
        h, _stream_ptr(stream), ctypes.c_void_p(roots.data_ptr() if roots.numel() else 0),
        int(roots.numel()), ctypes.c_void_p(ids.data_ptr()), int(ids.numel()),
        ctypes.c_void_p(offs.data_ptr()), int(offs.numel()) - 1,
        sizes.ctypes.data_as(ctypes.c_void_p))
    return int(code), (int(sizes[0]), int(sizes[1]))


def cliques_from(ids, offsets):
    """List of tuples from an enumeration's (ids, offsets)."""
    ids = ids.cpu().numpy()
    offs = offsets.cpu().numpy()
    return [tuple(int(x) for x in ids[offs[i]: offs[i + 1]]) for i in range(len(offs) - 1)]


from . import graphs  # noqa: E402  (input generators; no CUDA needed)
