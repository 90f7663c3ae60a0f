#!/usr/bin/env python3
"""Writes rmat_s20_heavy_roots.txt: the oracle's result for each root of a seeded sample of the
R-MAT scale-20 (seed 1) first-level roots with 128 <= |P| < 256 (8-word rows) and
256 <= |P| < 512 (16-word rows).

Test infrastructure: it calls only the oracle and the seeded graph generator.  Each root is
counted by the oracle alone, in a process of its own with a time limit; roots the oracle does
not finish within it are listed as skipped (the cost of a subtree varies by orders of
magnitude).  The file also records a fingerprint of the generated graph, so that a reader can
tell whether its generator reproduces the same graph.

    python tests/golden/make_rmat_s20_heavy.py [--limit-s 240] [--jobs 8]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

OUT = os.path.join(HERE, "rmat_s20_heavy_roots.txt")
BANDS = [(128, 256, 48, 101), (256, 512, 12, 102)]   # |P| range, roots sampled, sample seed

WORKER = r"""
import json, sys, time
import numpy as np
sys.path.insert(0, %(root)r)
import oracle as O
from maximal_clique_enumeration_gb300.graphs import Graph
z = np.load(sys.argv[1])
g = Graph(int(z["offsets"].size - 1), z["offsets"], z["adj"], "rmat_s20")
v = int(sys.argv[2])
t0 = time.perf_counter()
r = O.count(g, roots=np.array([v], np.int32), threads=1, hist_len=1026)
print(json.dumps({"key": r.key(), "s": time.perf_counter() - t0}))
"""


def fingerprint(g) -> str:
    h = hashlib.sha256()
    h.update(np.ascontiguousarray(g.offsets, np.int32).tobytes())
    h.update(np.ascontiguousarray(g.adj, np.int32).tobytes())
    return h.hexdigest()[:16]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--limit-s", type=float, default=240.0)
    ap.add_argument("--jobs", type=int, default=8)
    a = ap.parse_args()
    import oracle as O
    from maximal_clique_enumeration_gb300 import graphs as G
    g = G.config_graph("rmat_s20", 1)
    core, rnd, rank, d = O.peel(g)
    src = np.repeat(np.arange(g.n), g.degrees())
    pc = np.bincount(src[rank[g.adj] > rank[src]], minlength=g.n)
    todo = []
    for lo, hi, k, seed in BANDS:
        cand = np.nonzero((pc >= lo) & (pc < hi))[0]
        pick = G.sample_roots(cand.size, k, seed)
        todo += [int(v) for v in cand[pick]]
    results = {}
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, "g.npz")
        np.savez(path, offsets=g.offsets, adj=g.adj)
        script = WORKER % {"root": ROOT}
        running = []
        queue = list(todo)
        while queue or running:
            while queue and len(running) < a.jobs:
                v = queue.pop(0)
                p = subprocess.Popen([sys.executable, "-c", script, path, str(v)],
                                     stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                running.append((v, p, time.time()))
            time.sleep(0.5)
            for item in list(running):
                v, p, t0 = item
                if p.poll() is not None:
                    out = p.stdout.read()
                    results[v] = json.loads(out) if p.returncode == 0 else None
                    running.remove(item)
                elif time.time() - t0 > a.limit_s:
                    p.kill()
                    p.wait()
                    results[v] = None
                    running.remove(item)
            print(f"{len(results)}/{len(todo)}", file=sys.stderr, flush=True)
    with open(OUT, "w") as f:
        f.write("# R-MAT scale 20, edge factor 16, (0.57, 0.19, 0.19, 0.05), ids permuted, seed 1:\n")
        f.write("# the oracle's result for each root of a seeded sample of first-level roots with\n")
        f.write("# 128 <= |P| < 256 and 256 <= |P| < 512 (|P| from the oracle's canonical peel),\n")
        f.write("# each counted alone.  Written by make_rmat_s20_heavy.py (oracle only); roots the\n")
        f.write(f"# oracle did not finish within {a.limit_s:.0f} s are listed as skipped.\n")
        f.write("# root <id> <|P|> <count> <hash> <seconds> <hist[0..]>\n")
        f.write(f"graph rmat_s20 1 {g.n} {g.m} {fingerprint(g)}\n")
        for v in todo:
            r = results.get(v)
            if r is None:
                f.write(f"skipped {v} {int(pc[v])}\n")
                continue
            count, h, hist = r["key"]
            f.write(f"root {v} {int(pc[v])} {count} {h:#018x} {r['s']:.2f} "
                    + " ".join(str(x) for x in hist) + "\n")
    print(OUT)


if __name__ == "__main__":
    main()
