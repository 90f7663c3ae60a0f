#!/usr/bin/env python3
"""Benchmark: maximal cliques per second and ms per graph on R-MAT scale 20, edge factor 16.

One step is the whole hot path on one GPU, through the C ABI of libmce_gb300.so:
  mce_order        degeneracy order of the full graph (parallel k-core peel + orientation);
  mce_count_roots  the Bron-Kerbosch/Tomita search over the workload's first-level subtrees
                   (bitset induced subgraphs, compact X, worker list), with count, histogram
                   and hash of the maximal cliques.
The full R-MAT s20 graph has on the order of 1e14 maximal cliques (its ~5.8k densest
first-level subtrees each take minutes to hours), so the workload is every first-level
subtree whose root has fewer than --max-p later neighbours (98% of the roots); the order is
always computed for the whole graph.

Beside the headline the same JSON line carries:
  configs       the other four workloads (ER, BA, planted cliques, SBM), each timed whole
                (order + count) with the oracle timed beside it;
  graph_stages  achieved GB/s of the peel, the orientation and the subtree build against the
                measured HBM bandwidth, from their algorithmic bytes;
  heavy         the R-MAT roots with 128 <= |P| < 512 of a stored seeded sample, with
                parity root by root against the oracle's stored results;
  activity      per-activity split of the search's warp time (MCE_PROFILE build, in a child
                process), which also times the subtree build.

Lines printed: one JSON object (rank 0).  `--impl reference` times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "maximal cliques/sec (R-MAT s20 ef16)"
UNIT = "cliques/s"
OTHER_CONFIGS = ["er200", "ba100k", "planted50k", "sbm1m"]
WIDTHS = [1, 2, 4, 8, 16, 32]

# DRAM traffic of the dominant search launch from an ncu capture of a 10 % root sample of this
# workload (dram bytes read + written per counted bitset word).  It is scaled to a full launch
# by the counted words, and only reported while the kernel sources hash to the version that
# was captured.
TRAFFIC_CAPTURE = {"sources": "9983555e31ede7a6", "width_class": 2,
                   "bytes_per_word": (17.606144e6 + 0.203520e6) / 90368612.0}
KERNEL_SOURCES = ["maximal_clique_enumeration_gb300/csrc/search_impl.cuh",
                  "maximal_clique_enumeration_gb300/csrc/search_full.cu",
                  "maximal_clique_enumeration_gb300/csrc/mce_internal.cuh"]


def kernel_sources_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


_T0 = time.perf_counter()


def progress(msg: str):
    """One line on stderr per bench section (so that a cut-off run shows where it was)."""
    print(f"[bench {time.perf_counter() - _T0:7.1f}s] {msg}", file=sys.stderr, flush=True)


def hbm_peak():
    """(GB/s, source) of the HBM roofline: the measured copy bandwidth, else fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "of measured (MEASURED_PEAKS.json hbm_gbs)"
    except (OSError, KeyError, ValueError):
        return 6800.0, "of fallback (6.8 TB/s)"


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    p.add_argument("--seed", type=int, default=1)
    p.add_argument("--scale", type=int, default=20)
    p.add_argument("--max-p", type=int, default=128,
                   help="first-level subtrees whose root has |P| < max_p form the workload")
    p.add_argument("--root-fraction", type=float, default=1.0,
                   help="profiling aid: keep only this seeded share of the workload roots")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--configs", default=",".join(OTHER_CONFIGS),
                   help="other workloads timed beside the headline ('' for none)")
    p.add_argument("--no-heavy", action="store_true",
                   help="skip the heavy-root tier (stored sample of roots with |P| >= 128)")
    p.add_argument("--no-activity", action="store_true",
                   help="skip the activity profile (MCE_PROFILE build, child process)")
    p.add_argument("--induced", type=int, default=0, choices=[0, 1, 2],
                   help="induced subgraphs: 0 the Delta/d rule (default), 1 full, 2 partial")
    p.add_argument("--subtree-level", type=int, default=1, choices=[1, 2],
                   help="independent subtrees: 1 first-level (default), 2 second-level (per edge)")
    p.add_argument("--imbalance", action="store_true",
                   help="diagnostic: per-SM load max/avg with and without the worker list "
                        "(planted50k, rmat_s14), MCE_PROFILE build; prints one JSON line")
    p.add_argument("--activity-child", default=None, help=argparse.SUPPRESS)
    return p.parse_args(argv)


# ---------------------------------------------------------------- process group (replicas)

def dist_init(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "gb300" else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl"
                     else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- workload

def workload_graph(args):
    from maximal_clique_enumeration_gb300 import graphs as G
    name = "rmat_s20" if args.scale == 20 else f"rmat_s{args.scale}"
    return G.config_graph(name, args.seed)


def later_counts(g, rank):
    """|P(v)| for every v: neighbours later in the order `rank`."""
    src = np.repeat(np.arange(g.n), g.degrees())
    return np.bincount(src[rank[g.adj] > rank[src]], minlength=g.n)


def light_roots(g, rank, max_p):
    """Roots v with |P(v)| < max_p, where P(v) = neighbours later in the order `rank`."""
    pc = later_counts(g, rank)
    return np.nonzero(pc < max_p)[0].astype(np.int32), pc


HEAVY_GOLDEN = os.path.join(ROOT, "tests", "golden", "rmat_s20_heavy_roots.txt")


def graph_fingerprint(g) -> str:
    import hashlib
    h = hashlib.sha256()
    h.update(np.ascontiguousarray(g.offsets, np.int32).tobytes())
    h.update(np.ascontiguousarray(g.adj, np.int32).tobytes())
    return h.hexdigest()[:16]


def heavy_golden(g):
    """Roots of the stored heavy sample that the oracle finished, with its (count, hash, hist)
    for each (written by tests/golden/make_rmat_s20_heavy.py from the oracle alone), or None
    when the file is missing or was made from another graph."""
    try:
        lines = open(HEAVY_GOLDEN).read().splitlines()
    except OSError:
        return None
    roots, keys, pcs = [], [], []
    for line in lines:
        f = line.split()
        if not f or f[0].startswith("#"):
            continue
        if f[0] == "graph" and f[5] != graph_fingerprint(g):
            return None
        if f[0] == "root":
            roots.append(int(f[1]))
            pcs.append(int(f[2]))
            keys.append((int(f[3]), int(f[4], 16), tuple(int(x) for x in f[6:])))
    return np.asarray(roots, np.int32), keys, np.asarray(pcs)


def workload_config(args, g, roots, pc, d):
    return {
        "workload": f"R-MAT scale {args.scale}, edge factor 16, (a,b,c,d)=(0.57,0.19,0.19,0.05), "
                    f"ids permuted, seed {args.seed}: degeneracy order of the whole graph + the "
                    f"first-level subtrees of the {len(roots)} roots with |P| < {args.max_p}",
        "n": g.n, "m": g.m, "max_degree": g.max_degree(), "degeneracy": d,
        "roots": int(len(roots)), "roots_total": g.n, "max_p": args.max_p,
        "roots_left_out": int((pc >= args.max_p).sum()),
        "root_fraction": args.root_fraction,
        "l2": "flushed between steps (256 MiB write, untimed)",
        # the variant in use: the Delta / d > 200 rule resolved as the library resolves it
        "induced": ({1: "full", 2: "partial"}[args.induced] if getattr(args, "induced", 0)
                    else ("partial" if g.max_degree() > 200 * d else "full")),
        "subtree_level": getattr(args, "subtree_level", 1),
    }


# ---------------------------------------------------------------- algorithmic bytes (roofline)

def stage_bytes(g, rank, roots, peel_live):
    """Algorithmic bytes of the graph stages, from the graph (int32 everywhere).

    peel (a1):   8m   every adjacency list read once, when its vertex is removed
               + 8m   one 4-byte degree update per adjacency entry
               + 8 L  id and degree of every live vertex in every round (L = live vertices
                      summed over rounds, counted by the peel)
               + 16n  rank, core number, round and order written
    orient (a2): 8m + 8m + 4m + 16n: adjacency read, the rank of every entry gathered, every
                 edge written once into a later-neighbour list N+; offsets and ranks read,
                 |P| and the schedule written
    build (a3):  per workload root v (|P| > 0), with W(v) words per row:
                 16 deg(v)  N(v) read, the rank of each neighbour, |N+(u)| and offset of each
               + 4 sum_{u in N(v)} |N+(u)|  the later-neighbour lists walked
               + 4 (deg(v) W(v) + deg(v) + 2 |P(v)| + 4)  the record written: rows, P's ids
                                            and keys, the live X list, its header
                 A 1-word root whose lists average >= 64 entries searches instead of walking:
                 its walk term becomes 4 sum_u pairs(u) (ceil(log2(|N+(u)| + 1)) + 1), with
                 pairs(u) = |P| for u in X and (|P| - 1) / 2 on average for u in P.
    """
    n, m = g.n, g.m
    deg = g.degrees()
    pc = later_counts(g, rank)
    src = np.repeat(np.arange(n), deg)
    walk = np.bincount(src, weights=pc[g.adj].astype(np.float64), minlength=n)
    w = np.select([pc <= 32, pc <= 64, pc <= 128, pc <= 256, pc <= 512], [1, 2, 4, 8, 16], 32)
    # 1-word roots on the binary-search path (the build kernel's rule)
    steps = np.ceil(np.log2(pc[g.adj] + 1.0)) + 1.0
    later = rank[g.adj] > rank[src]
    pairs = np.where(later, (pc[src] - 1) / 2.0, pc[src].astype(np.float64))
    probes = np.bincount(src, weights=pairs * steps, minlength=n)
    search = (w == 1) & (walk >= 64.0 * deg)
    read = np.where(search, probes, walk)
    per_root = 16.0 * deg + 4.0 * read + 4.0 * (deg * w + deg + 2.0 * pc + 4.0)
    sel = np.zeros(n, bool)
    sel[roots] = True
    sel &= pc > 0
    k = np.log2(w).astype(int)
    a3_cls = [float(per_root[sel & (k == c)].sum()) for c in range(6)]
    return {"peel": 16.0 * m + 8.0 * peel_live + 16.0 * n,
            "orient": 20.0 * m + 16.0 * n,
            "build": float(sum(a3_cls)), "build_by_width": a3_cls}


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self, device_index=0):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((int(parts[0]), float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        idx = sorted({r[0] for r in rows})
        mine = [r for r in rows if r[0] == (idx[device_index] if device_index < len(idx) else
                                            (idx[0] if idx else 0))]
        if not mine:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in mine for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[1] for r in mine),
                "sm_max_mhz": max(r[2] for r in mine), "samples": len(mine), "reasons": reasons}


# ---------------------------------------------------------------- CPU oracle baseline

def oracle_count_timed(g, roots, threads, hist_len=1026):
    """Times the oracle (as it stands) on the given roots (None = the whole graph)."""
    import oracle
    oracle.build()
    t0 = time.perf_counter()
    res = oracle.count(g, roots=roots, threads=threads, hist_len=hist_len)
    return res, time.perf_counter() - t0


def oracle_preprocessing_s(g):
    """The oracle's own input checks and peel, timed alone (context for its rates)."""
    import oracle
    oracle.build()
    t0 = time.perf_counter()
    oracle.validate(g)
    oracle.peel(g)
    return time.perf_counter() - t0


def cpu_block(value, cores, sample_desc, **extra):
    return dict({"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                 "sample": sample_desc}, **extra)


# ---------------------------------------------------------------- GPU helpers

def timed_steps(step, steps, warmup, flush, stream, info_fn=None):
    """W untimed steps, then K steps each bracketed by CUDA events on `stream` (L2 flushed
    before each, untimed); returns (per-step ms list, summed info deltas)."""
    import torch
    for _ in range(max(warmup, 0)):
        step()
    torch.cuda.synchronize()
    ms, infos = [], []
    for k in range(steps):
        flush.fill_(k & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
        if info_fn is not None:
            infos.append(info_fn())
    return ms, infos


def dominant_class(infos, steps):
    ms_cls = np.sum([np.asarray(i["ms_search"]) for i in infos], axis=0) / steps
    words = np.sum([np.asarray(i["words"], dtype=np.float64) for i in infos], axis=0) / steps
    dom = int(np.argmax(ms_cls))
    return dom, ms_cls, words


def run_other_config(name, seed, args, flush, word_peak, threads, want_cpu, hbm):
    """One of the other workloads, whole: W + K steps of (order + count), oracle beside it."""
    import torch
    import maximal_clique_enumeration_gb300 as mce
    from maximal_clique_enumeration_gb300 import graphs as G
    g = G.config_graph(name, seed)
    h = mce.Graph(torch.from_numpy(g.offsets).cuda(), torch.from_numpy(g.adj).cuda(), g.n,
                  profile=1)
    out = h.new_output()
    stream = torch.cuda.current_stream()

    def step():
        h.order()
        h.count(out=out)

    ms, infos = timed_steps(step, args.steps, args.warmup, flush, stream, h.get_info)
    h.check()
    res = mce.Graph.unpack(out)
    step_ms = float(np.mean(ms))
    dom, ms_cls, words = dominant_class(infos, args.steps)
    order_ms = float(np.mean([i["ms_order"] for i in infos]))
    peel_ms = float(np.mean([i["ms_peel"] for i in infos]))
    info = infos[-1]
    rank, _ = h.order_arrays()
    rank = rank.cpu().numpy()
    entry = {
        "workload": G.CONFIGS[name] + f", seed {seed}",
        "n": g.n, "m": g.m, "max_degree": g.max_degree(), "degeneracy": info["degeneracy"],
        "induced": {1: "full", 2: "partial"}[info["induced"]],
        "cliques": res[0], "hash": f"{res[1]:#018x}", "max_size": len(res[2]) - 1,
        "ms_per_graph": step_ms, "value": res[0] / (step_ms * 1e-3), "unit": UNIT,
        "stage_ms": {"order": order_ms, "peel": peel_ms,
                     "search_by_width": {str(WIDTHS[i]): float(ms_cls[i])
                                         for i in range(6) if ms_cls[i] > 0}},
        "search_roofline": {"bound": "alu", "kernel": f"search_kernel<W={WIDTHS[dom]}>",
                            "achieved_gword_s": words[dom] / max(ms_cls[dom], 1e-9) * 1e-6,
                            "frac": (words[dom] / max(ms_cls[dom], 1e-9) * 1e3) / word_peak},
        "tree_nodes": info["tree_nodes"], "donations": info["donations"],
    }
    sb = stage_bytes(g, rank, np.arange(g.n, dtype=np.int32), info["peel_live"])
    entry["graph_stages"] = {
        "peel": _gbs(sb["peel"], peel_ms, hbm),
        "orient": _gbs(sb["orient"], order_ms - peel_ms, hbm)}
    if want_cpu:
        if name == "sbm1m":
            # a seeded tenth of the roots keeps the oracle near 10 s; the GPU counts the same
            from maximal_clique_enumeration_gb300.graphs import sample_roots
            roots = sample_roots(g.n, g.n // 10, seed + 4000)
            ores, dt = oracle_count_timed(g, roots, threads, hist_len=h.hist_len)
            got = h.count_roots_result(roots)
            desc = (f"oracle on a seeded 10% of the roots ({len(roots)}): {ores.count} cliques "
                    f"in {dt:.1f} s, including its input checks, peel and relabelling")
        else:
            ores, dt = oracle_count_timed(g, None, threads, hist_len=h.hist_len)
            got = res
            desc = (f"oracle on the whole graph: {ores.count} cliques in {dt:.2f} s, including "
                    f"its input checks, peel and relabelling")
        entry["cpu_baseline"] = cpu_block(ores.count / dt, threads, desc)
        entry["parity"] = "ok" if got == ores.key() else f"MISMATCH {got} {ores.key()}"
    h.close()
    return entry


def _gbs(nbytes, ms, hbm):
    if ms <= 0:
        return {"bytes": nbytes, "ms": ms, "achieved_gbs": None, "frac": None}
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"bytes": nbytes, "ms": ms, "achieved_gbs": gbs, "frac": gbs / hbm[0],
            "peak_gbs": hbm[0], "peak": hbm[1]}


# ---------------------------------------------------------------- activity profile (child)

def activity_profile(g, roots, args):
    """Runs the MCE_PROFILE build on the same graph and roots in a child process; returns its
    per-class activity split (SM cycles summed over warps) and per-SM loads."""
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "w.npz")
        np.savez(path, offsets=g.offsets, adj=g.adj, roots=roots)
        cmd = [sys.executable, os.path.abspath(__file__), "--activity-child", path,
               "--induced", str(args.induced), "--subtree-level", str(args.subtree_level)]
        r = subprocess.run(cmd, capture_output=True, text=True, timeout=900)
    if r.returncode != 0:
        return {"error": (r.stderr or r.stdout)[-500:]}
    return json.loads(r.stdout.strip().splitlines()[-1])


def _load_stats(sm_busy, n_sms):
    x = np.asarray(sm_busy[:n_sms], dtype=np.float64)
    if x.sum() <= 0:
        return None
    return {"max_over_avg": float(x.max() / x.mean()), "min_over_avg": float(x.min() / x.mean())}


def activity_child(args):
    """Child process: load the MCE_PROFILE library (MCE_LIBRARY) and profile one search."""
    import torch
    from maximal_clique_enumeration_gb300 import build
    os.environ["MCE_LIBRARY"] = build.build(profile=True)
    import maximal_clique_enumeration_gb300 as mce
    z = np.load(args.activity_child)
    offs, adj, roots = z["offsets"], z["adj"], z["roots"]
    n = len(offs) - 1
    h = mce.Graph(torch.from_numpy(offs).cuda(), torch.from_numpy(adj).cuda(), n, profile=1,
                  induced=args.induced, subtree_level=args.subtree_level)
    r = torch.from_numpy(roots).cuda()
    out = h.count_roots(r)
    torch.cuda.synchronize()
    h.count_roots(r, out=out)
    h.check()
    info = h.get_info()
    prof = h.profile()
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    acts = ["split", "build", "pivot", "small", "child", "partition", "donate", "idle"]
    sub = ["hash", "walk", "xlist"]
    res = {"ms_search": info["ms_search"], "workers": info["workers"], "n_sms": n_sms}
    for k in range(6):
        p = prof[1 << k]
        tot = sum(p[a] for a in acts)
        if tot == 0:
            continue
        res[str(1 << k)] = {"cycles": {a: int(p[a]) for a in acts + sub},
                            "share": {a: p[a] / tot for a in acts},
                            "build_parts_share": {a: p[a] / max(p["build"], 1) for a in sub},
                            "roots": int(p["roots"]), "slowest_root_cycles": int(p["max_root"]),
                            "sm_load": _load_stats(p["sm_busy"], n_sms)}
    h.close()
    print(json.dumps(res), flush=True)


def imbalance_run(args):
    """Per-SM load (max / average) with and without the worker list, per row-width class."""
    import torch
    from maximal_clique_enumeration_gb300 import build
    os.environ["MCE_LIBRARY"] = build.build(profile=True)
    import maximal_clique_enumeration_gb300 as mce
    from maximal_clique_enumeration_gb300 import graphs as G
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    out = {"kind": "imbalance", "n_sms": n_sms, "graphs": {}}
    for name in ["planted50k", "rmat_s14"]:
        g = G.config_graph(name, 1)
        per = {}
        for wl in (0, 1):
            progress(f"imbalance {name} worker_list={wl}")
            h = mce.Graph(torch.from_numpy(g.offsets).cuda(), torch.from_numpy(g.adj).cuda(),
                          g.n, profile=1, worker_list=wl)
            h.count_result()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            o = h.count()
            e1.record()
            torch.cuda.synchronize()
            h.check()
            info = h.get_info()
            prof = h.profile()
            per["worker_list" if wl else "static"] = {
                "ms": e0.elapsed_time(e1), "cliques": int(mce.Graph.unpack(o)[0]),
                "donations": info["donations"], "tree_nodes": info["tree_nodes"],
                "sm_load_by_width": {str(1 << k): _load_stats(prof[1 << k]["sm_busy"], n_sms)
                                     for k in range(6) if prof[1 << k]["sm_busy"].sum() > 0},
                "sm_load_all": _load_stats(sum(prof[1 << k]["sm_busy"] for k in range(6)),
                                           n_sms)}
            h.close()
        out["graphs"][name] = per
    print(json.dumps(out), flush=True)


# ---------------------------------------------------------------- GPU arm

def run_gb300(args, rank, world, local):
    import torch
    import maximal_clique_enumeration_gb300 as mce
    from maximal_clique_enumeration_gb300 import build, probe

    torch.cuda.set_device(local)
    build.build()
    hbm = hbm_peak()
    g = workload_graph(args)
    progress(f"graph n={g.n} m={g.m}")
    dev_offs = torch.from_numpy(g.offsets).cuda()
    dev_adj = torch.from_numpy(g.adj).cuda()
    h = mce.Graph(dev_offs, dev_adj, g.n, profile=1, induced=args.induced,
                  subtree_level=args.subtree_level)
    rank_arr = h.order_arrays()[0].cpu().numpy()
    roots, pc = light_roots(g, rank_arr, args.max_p)
    if args.root_fraction < 1.0:
        rng = np.random.default_rng(args.seed + 3000)
        keep = max(1, int(len(roots) * args.root_fraction))
        roots = np.sort(rng.choice(roots, size=keep, replace=False)).astype(np.int32)
    roots_dev = torch.from_numpy(roots).cuda()
    out = h.new_output()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        h.order()
        h.count_roots(roots_dev, out=out)

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()
    h.check()
    ref = mce.Graph.unpack(out)

    progress("warm-up done")
    sampler = ClockSampler()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    ms_cls = np.zeros(mce.NUM_WIDTHS)
    words_cls = np.zeros(mce.NUM_WIDTHS)
    ms_order = ms_peel = 0.0
    ms_bld = np.zeros(mce.NUM_WIDTHS)
    launches = 0
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    wall0 = time.perf_counter()
    for k in range(args.steps):
        flush.fill_(k & 0xFF)                      # untimed: evict the graph from L2
        ev[k][0].record(stream)
        step()
        ev[k][1].record(stream)
        torch.cuda.synchronize()
        info = h.get_info()
        ms_cls += np.asarray(info["ms_search"])
        words_cls += np.asarray(info["words"], dtype=np.float64)
        ms_order += info["ms_order"]
        ms_peel += info["ms_peel"]
        ms_bld += np.asarray(info["ms_build"])
        launches += info["launches"]
    wall = time.perf_counter() - wall0
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    h.check()
    res = mce.Graph.unpack(out)
    assert res == ref, "result changed between steps"
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(sum(step_ms), world)
    ms_per_step = total_ms / args.steps
    value = world * res[0] * args.steps / (total_ms * 1e-3)
    info = h.get_info()

    progress(f"timed steps done: {ms_per_step:.2f} ms/step")
    # roofline of the dominant kernel: the search launch with the largest device time
    dom = int(np.argmax(ms_cls))
    rate = 0.0
    pr = probe.word_rate()
    if ms_cls[dom] > 0:
        rate = words_cls[dom] / (ms_cls[dom] * 1e-3)
    roofline = {
        "bound": "alu", "kernel": f"search_kernel<W={1 << dom}>",
        "achieved": rate / 1e9, "peak": pr["words_per_s"] / 1e9, "unit": "Gword/s",
        "frac": rate / pr["words_per_s"] if pr["words_per_s"] else None,
        "traffic": (TRAFFIC_CAPTURE["bytes_per_word"] * words_cls[dom] / args.steps
                    if kernel_sources_hash() == TRAFFIC_CAPTURE["sources"]
                    and dom == TRAFFIC_CAPTURE["width_class"] else None),
        "traffic_unit": "bytes per launch (ncu capture, scaled by counted words)",
        "peak_source": "measured: AND+POPC+ADD word rate of a register-only kernel on this GPU "
                       f"({pr['ms']:.2f} ms probe)",
        "share_of_step": float(ms_cls[dom] / max(sum(step_ms), 1e-9)),
        "ms_per_launch": float(ms_cls[dom] / args.steps),
        "words_per_launch": float(words_cls[dom] / args.steps),
    }
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "ms_per_graph": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
        "data": "synthetic (seeded R-MAT generator)",
        "config": dict(workload_config(args, g, roots, pc, h.info["degeneracy"]),
                       induced={1: "full", 2: "partial"}[h.info["induced"]]),
        "result": {"cliques": res[0], "hash": f"{res[1]:#018x}", "max_size": len(res[2]) - 1},
        "stage_ms": {"order": ms_order / args.steps, "peel": ms_peel / args.steps,
                     "search_by_width": {str(1 << i): float(ms_cls[i] / args.steps)
                                         for i in range(mce.NUM_WIDTHS) if ms_cls[i] > 0},
                     "build_span_by_width": {str(1 << i): float(ms_bld[i] / args.steps)
                                             for i in range(mce.NUM_WIDTHS) if ms_bld[i] > 0},
                     "build_span_note": "event spans of the build launches on the handle's "
                                        "own stream, overlapping the wider classes' search"},
        "roofline": roofline, "clocks": clocks, "gpu_launches": launches,
        "wall_s_timed": wall,
    }

    # graph stages against HBM: peel, orientation, and the subtree build launches (rows of 1,
    # 2 and 4 words; device time by CUDA events around each build launch)
    sb = stage_bytes(g, rank_arr, roots, info["peel_live"])
    peel_ms = ms_peel / args.steps
    stages = {"peel": _gbs(sb["peel"], peel_ms, hbm),
              "orient": _gbs(sb["orient"], ms_order / args.steps - peel_ms, hbm),
              "peel_live_vertices": info["peel_live"], "rounds": info["peel_rounds"],
              "bytes_formulas": "see stage_bytes() in bench.py"}
    # the build launches' own times: a second handle whose builds run on the caller's stream,
    # each just before its search (outside the timed region; same roots)
    progress("build stage")
    hb = mce.Graph(dev_offs, dev_adj, g.n, profile=1, induced=args.induced,
                   subtree_level=args.subtree_level, overlap_builds=0)
    bout = hb.new_output()
    _, binfos = timed_steps(lambda: (hb.order(), hb.count_roots(roots_dev, out=bout)),
                            args.steps, args.warmup, flush, stream, hb.get_info)
    hb.check()
    assert mce.Graph.unpack(bout) == ref, "result changed with the builds on the caller's stream"
    hb.close()
    ms_b = np.sum([np.asarray(i["ms_build"]) for i in binfos], axis=0) / args.steps
    built = [c for c in range(mce.NUM_WIDTHS) if ms_b[c] > 0]
    if built:
        stages["build"] = dict(_gbs(sum(sb["build_by_width"][c] for c in built),
                                    float(sum(ms_b[c] for c in built)), hbm),
                               by_width={str(1 << c): _gbs(sb["build_by_width"][c], ms_b[c], hbm)
                                         for c in built},
                               time_source="CUDA events around each build launch, builds on "
                                           "the caller's stream (overlap_builds = 0)")
    if rank == 0 and world == 1 and not args.no_activity:
        progress("activity profile")
        line["activity"] = activity_profile(g, roots, args)
    line["graph_stages"] = stages

    if not args.no_heavy and args.scale == 20 and args.seed == 1:
        # heavy roots (|P| >= 128, left out of the headline): the stored seeded sample that the
        # oracle finished root by root (tests/golden/rmat_s20_heavy_roots.txt); parity root by
        # root against the stored results, timing of the whole sample, and the oracle timed on
        # its 8-word roots (the 16-word ones take it minutes each)
        progress("heavy roots")
        gold = heavy_golden(g)
        if gold is None:
            line["heavy"] = {"error": "stored heavy-root results missing or made on another graph"}
        else:
            groots, gkeys, gpc = gold
            bad = [int(v) for v, key in zip(groots, gkeys)
                   if h.count_roots_result(np.array([v], np.int32)) != key]
            gdev = torch.from_numpy(groots).cuda()
            gout = h.new_output()
            gms, ginfos = timed_steps(lambda: h.count_roots(gdev, out=gout), args.steps,
                                      args.warmup, flush, stream, h.get_info)
            h.check()
            gres = mce.Graph.unpack(gout)
            gdom, gcls, gwords = dominant_class(ginfos, args.steps)
            gstep = float(np.mean(gms))
            entry = {
                "sample": "stored seeded sample of R-MAT s20 roots with 128 <= |P| < 512 that "
                          "the oracle finished (tests/golden/rmat_s20_heavy_roots.txt)",
                "roots": int(len(groots)), "roots_8_word": int((gpc < 256).sum()),
                "roots_16_word": int((gpc >= 256).sum()),
                "cliques": gres[0], "hash": f"{gres[1]:#018x}", "ms": gstep,
                "value": gres[0] / (gstep * 1e-3), "unit": UNIT,
                "search_by_width": {str(WIDTHS[i]): float(gcls[i]) for i in range(6)
                                    if gcls[i] > 0},
                "search_roofline": {"kernel": f"search_kernel<W={WIDTHS[gdom]}>",
                                    "achieved_gword_s": gwords[gdom] / max(gcls[gdom], 1e-9)
                                    * 1e-6,
                                    "frac": gwords[gdom] / max(gcls[gdom], 1e-9) * 1e3
                                    / pr["words_per_s"]},
                "parity_per_root": "ok" if not bad else f"MISMATCH at roots {bad[:8]}"}
            if rank == 0 and world == 1 and not args.no_cpu_baseline:
                keep = gpc < 256
                sub = groots[keep]
                cores = len(os.sched_getaffinity(0))
                ores, dt = oracle_count_timed(g, sub, cores)
                got = h.count_roots_result(sub)
                entry["cpu_baseline"] = cpu_block(
                    ores.count / dt, cores, f"oracle on the sample's {len(sub)} 8-word roots: "
                    f"{ores.count} cliques in {dt:.1f} s, including its input checks, peel and "
                    f"relabelling of the whole graph")
                entry["parity_8_word_roots"] = ("ok" if got == ores.key()
                                                else f"MISMATCH {got} {ores.key()}")
            line["heavy"] = entry

    if not args.no_e2e:
        progress("e2e")
        line["e2e"] = e2e_leg(args, g, roots, world)
    threads = len(os.sched_getaffinity(0))
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        progress("oracle on the workload")
        ores, dt = oracle_count_timed(g, roots, threads)
        pre = oracle_preprocessing_s(g)
        line["cpu_baseline"] = cpu_block(
            ores.count / dt, threads,
            f"oracle on the whole workload ({len(roots)} roots): {ores.count} cliques in "
            f"{dt:.1f} s, including its own input checks, peel and relabelling of the whole "
            f"graph (those alone: {pre:.1f} s)", preprocessing_s=pre, seconds=dt)
        line["parity_on_cpu_sample"] = "ok" if res == ores.key() else \
            f"MISMATCH {res} {ores.key()}"
        line["parity_scope"] = "the whole workload"

    names = [c for c in args.configs.split(",") if c]
    if names:
        line["configs"] = {}
        for name in names:
            progress(f"config {name}")
            line["configs"][name] = run_other_config(
                name, args.seed, args, flush, pr["words_per_s"], threads,
                rank == 0 and world == 1 and not args.no_cpu_baseline, hbm)
    h.close()
    if rank == 0:
        print(json.dumps(line), flush=True)


def e2e_leg(args, g, roots, world):
    """Same metric end to end: pinned host CSR and roots in, result out, through the C ABI."""
    import torch
    import maximal_clique_enumeration_gb300 as mce
    offs = torch.from_numpy(g.offsets).pin_memory()
    adj = torch.from_numpy(g.adj).pin_memory()
    roots_h = torch.from_numpy(roots).pin_memory()
    stream = torch.cuda.current_stream()
    res_h = None
    times = []
    count = 0
    for k in range(1 + args.steps):                   # first pass untimed
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h = mce.Graph(offs, adj, g.n, induced=args.induced,   # host pointers: copied in
                      subtree_level=args.subtree_level)
        r = roots_h.to("cuda", non_blocking=True)
        out = h.count_roots(r)
        res_h = out.to("cpu", non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        h.check()
        h.close()
        if k:
            times.append(e0.elapsed_time(e1))
            count = int(res_h.numpy().view(np.uint64)[0])
    total_ms = max_over_ranks(sum(times), world)
    return {"value": world * count * args.steps / (total_ms * 1e-3), "unit": UNIT,
            "ms_per_step": total_ms / args.steps,
            "h2d_bytes_per_step": int(offs.numel() * 4 + adj.numel() * 4 + roots_h.numel() * 4),
            "d2h_bytes_per_step": int(res_h.numel() * 8),
            "includes": "mce_create from pinned host CSR (copy in, input checks, order, "
                        "workspace allocation), roots copy, search, result copy out, destroy"}


# ---------------------------------------------------------------- reference arm (CPU oracle)

def run_reference(args, rank, world):
    """The oracle, as it stands, on the host cores: each timed step counts the whole workload
    (every root with |P| < max_p, with the oracle's own input checks, peel and relabelling);
    the untimed warm-up steps count a 1 % seeded sample."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    g = workload_graph(args)
    _, _, orank, d = oracle.peel(g)
    roots, pc = light_roots(g, orank, args.max_p)
    threads = len(os.sched_getaffinity(0))
    rng = np.random.default_rng(args.seed + 2000)
    warm = np.sort(rng.choice(roots, size=max(1, len(roots) // 100), replace=False))
    for _ in range(args.warmup):
        oracle_count_timed(g, warm.astype(np.int32), threads)
    total_cl = 0
    total_s = 0.0
    for _ in range(args.steps):
        res, dt = oracle_count_timed(g, roots, threads)
        total_cl += res.count
        total_s += dt
    value = total_cl / total_s
    desc = ("oracle, each step the whole workload (all roots with |P| < max_p), with its own "
            "input checks, peel and relabelling of the whole graph")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
        "data": "synthetic (seeded R-MAT generator)",
        "config": workload_config(args, g, roots, pc, d),
        "cpu_baseline": cpu_block(value, threads, desc),
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    args = parse_args()
    if args.activity_child:
        activity_child(args)
        return
    if args.imbalance:
        imbalance_run(args)
        return
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    rank, world, local = dist_init(args)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_gb300(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
