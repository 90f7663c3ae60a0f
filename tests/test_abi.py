"""The C-ABI library builds, loads without a GPU, and exports every entry point of include/mce.h.

No compute call is made here (there may be no GPU); only entry points that return before
touching CUDA are called.
"""
import ctypes
import os
import re

import pytest

import maximal_clique_enumeration_gb300 as mce
from maximal_clique_enumeration_gb300 import build as mce_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "mce.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mce_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    mce_build.build()
    return mce.library()


def test_header_declares_the_binding_exports():
    assert _declared() == sorted(mce.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_calls_that_need_no_gpu(lib):
    cfg = mce.Config()
    assert lib.mce_config_default(ctypes.byref(cfg)) == 0
    assert (cfg.worker_list, cfg.donate_min_p) == (1, 10)
    assert cfg.spin_limit_ns > 0
    assert lib.mce_config_default(None) == 1
    for code, name in mce.STATUS.items():
        assert lib.mce_status_str(code)
    out = ctypes.c_void_p(0)
    # argument errors are caught before any CUDA call
    assert lib.mce_create(None, None, 5, 0, None, None, ctypes.byref(out)) == 1
    assert lib.mce_create(None, None, 0, 0, None, None, None) == 1
    assert (cfg.induced, cfg.subtree_level, cfg.overlap_builds) == (0, 1, 1)
    offs = (ctypes.c_int32 * 2)(0, 0)
    for field, value in [("induced", 3), ("induced", -1), ("subtree_level", 0),
                         ("subtree_level", 3), ("overlap_builds", 2), ("overlap_builds", -1)]:
        bad = mce.Config()
        lib.mce_config_default(ctypes.byref(bad))
        setattr(bad, field, value)
        assert lib.mce_create(offs, None, 1, 0, ctypes.byref(bad), None, ctypes.byref(out)) == 1
        assert out.value is None
    assert lib.mce_count(None, None, None) == 1
    assert lib.mce_count_roots(None, None, None, 0, None) == 1
    assert lib.mce_order(None, None) == 1
    assert lib.mce_last_error(None, None) == 1
    lib.mce_destroy(None)


def test_struct_layouts_match_header(tmp_path):
    # compile a probe against the header and compare sizes and offsets with the ctypes mirror
    src = tmp_path / "probe.c"
    fields = [("mce_config", f) for f, _ in mce.Config._fields_] + \
             [("mce_info", f) for f, _ in mce.Info._fields_]
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "mce.h"', 'int main(void){',
             'printf("%zu %zu\\n", sizeof(mce_config), sizeof(mce_info));']
    lines += [f'printf("%zu\\n", offsetof({t}, {f}));' for t, f in fields]
    lines += ['return 0;}']
    src.write_text("\n".join(lines))
    exe = tmp_path / "probe"
    import subprocess
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(src)],
                   check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    assert int(out[0]) == ctypes.sizeof(mce.Config)
    assert int(out[1]) == ctypes.sizeof(mce.Info)
    ct = [getattr(mce.Config, f).offset for f, _ in mce.Config._fields_] + \
         [getattr(mce.Info, f).offset for f, _ in mce.Info._fields_]
    assert [int(x) for x in out[2:]] == ct


def test_missing_library_fails_loudly(tmp_path):
    saved = mce._lib
    mce._lib = None
    try:
        with pytest.raises(RuntimeError, match="no CPU fallback"):
            mce.library(str(tmp_path / "nope.so"))
    finally:
        mce._lib = saved
