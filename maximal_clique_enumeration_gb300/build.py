"""Builds libmce_gb300.so in-tree with nvcc for sm_103a (GB300)."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libmce_gb300.so")
PROBE_PATH = os.path.join(BUILD_DIR, "libmce_probe.so")
SOURCES = ["api.cu", "ingest.cu", "order.cu", "search.cu", "search_full.cu", "search_partial.cu",
           "search_full_l2.cu", "search_partial_l2.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         f"-I{INCLUDE}", f"-I{CSRC}"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmce_gb300.so")


def _stale(*outputs) -> bool:
    outputs = outputs or (LIB_PATH, PROBE_PATH)
    if not all(os.path.exists(o) for o in outputs):
        return True
    t = min(os.path.getmtime(o) for o in outputs)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "mce.h")]
    return any(os.path.getmtime(d) > t for d in deps)


PROFILE_LIB_PATH = os.path.join(BUILD_DIR, "profile", "libmce_gb300.so")


def build(force: bool = False, verbose: bool = False, extra_flags=(), profile: bool = False) -> str:
    """Compile every CUDA source (in parallel) and link the shared library; returns its path.

    profile=True builds the MCE_PROFILE variant (activity cycle counters) into
    _build/profile/ instead; the normal library is left alone.
    """
    if profile:
        if not force and not extra_flags and not _stale(PROFILE_LIB_PATH):
            return PROFILE_LIB_PATH
        return _build_variant(os.path.dirname(PROFILE_LIB_PATH), ["-DMCE_PROFILE", *extra_flags],
                              verbose)
    if not force and not extra_flags and not _stale():
        return LIB_PATH
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    procs, objs = [], []
    probe_tmp = PROBE_PATH + f".tmp{os.getpid()}"
    probe_cmd = [nvcc, *ARCH, *FLAGS, *extra_flags, "-shared", "-cudart", "static",
                 os.path.join(CSRC, "probe.cu"), "-o", probe_tmp]
    procs.append(("probe.cu", subprocess.Popen(probe_cmd, stdout=subprocess.PIPE,
                                               stderr=subprocess.STDOUT)))
    for src in SOURCES:
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [nvcc, *ARCH, *FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    errors = []
    for src, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            errors.append(f"--- {src}\n{out.decode(errors='replace')}")
        elif verbose and out:
            print(out.decode(errors="replace"), file=sys.stderr)
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB_PATH)
    os.replace(probe_tmp, PROBE_PATH)
    return LIB_PATH


def _build_variant(out_dir: str, flags, verbose: bool) -> str:
    nvcc = _nvcc()
    os.makedirs(out_dir, exist_ok=True)
    procs, objs = [], []
    for src in SOURCES:
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [nvcc, *ARCH, *FLAGS, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    outs = [(src, p.communicate()[0], p.returncode) for src, p in procs]
    errors = [f"--- {src}\n{out.decode(errors='replace')}" for src, out, rc in outs if rc != 0]
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
    out = os.path.join(out_dir, "libmce_gb300.so")
    tmp = out + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True,
                extra_flags=["-Xptxas", "-v"] if "--ptxas" in sys.argv else []))
