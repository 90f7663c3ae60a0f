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

# DRAM traffic of the dominant search launch, from the last ncu capture summarised in
# profiles/search_kernel_w4_rmat_s20_sample.md (a 10 % root sample; dram bytes read + written
# = 82.4 MB for 86,953,769 counted words).  It is scaled to a full launch by the counted words
# and only reported while the kernel sources are the ones it was measured on.
TRAFFIC_CAPTURE = {"sources": "b4a4ad260dfd7168", "width_class": 2,
                   "bytes_per_word": 93.36e6 / 86953769.0}
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


def parse_args():
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
    p.add_argument("--cpu-fraction", type=float, default=0.2,
                   help="share of the workload roots the oracle baseline counts")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--induced", type=int, default=0, choices=[0, 1, 2],
                   help="induced subgraphs: 0 the Delta/d rule (default), 1 full, 2 partial")
    p.add_argument("--subtree-level", type=int, default=1, choices=[1, 2],
                   help="independent subtrees: 1 first-level (default), 2 second-level (per edge)")
    return p.parse_args()


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


def light_roots(g, rank, max_p):
    """Roots v with |P(v)| < max_p, where P(v) = neighbours later in the order `rank`."""
    src = np.repeat(np.arange(g.n), g.degrees())
    pc = np.bincount(src[rank[g.adj] > rank[src]], minlength=g.n)
    return np.nonzero(pc < max_p)[0].astype(np.int32), pc


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
        "induced": {0: "Delta/d rule", 1: "full", 2: "partial"}[getattr(args, "induced", 0)],
        "subtree_level": getattr(args, "subtree_level", 1),
    }


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

def oracle_sample(g, roots, fraction, seed, threads):
    """Times the oracle (as it stands) on a seeded sample of the workload roots."""
    import oracle
    oracle.build()
    rng = np.random.default_rng(seed)
    k = max(1, int(len(roots) * fraction))
    sample = np.sort(rng.choice(roots, size=k, replace=False)).astype(np.int32)
    t0 = time.perf_counter()
    res = oracle.count(g, roots=sample, threads=threads, hist_len=1026)
    dt = time.perf_counter() - t0
    return sample, res, dt


def cpu_block(value, cores, sample_desc):
    return {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample_desc}


# ---------------------------------------------------------------- GPU arm

def run_gb300(args, rank, world, local):
    import torch
    import maximal_clique_enumeration_gb300 as mce
    from maximal_clique_enumeration_gb300 import build, probe

    torch.cuda.set_device(local)
    build.build()
    g = workload_graph(args)
    dev_offs = torch.from_numpy(g.offsets).cuda()
    dev_adj = torch.from_numpy(g.adj).cuda()
    h = mce.Graph(dev_offs, dev_adj, g.n, profile=1, induced=args.induced,
                  subtree_level=args.subtree_level)
    rank_arr, _ = h.order_arrays()
    roots, pc = light_roots(g, rank_arr.cpu().numpy(), args.max_p)
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

    sampler = ClockSampler()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    ms_cls = np.zeros(mce.NUM_WIDTHS)
    words_cls = np.zeros(mce.NUM_WIDTHS)
    ms_order = 0.0
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
        "stage_ms": {"order": ms_order / args.steps,
                     "search_by_width": {str(1 << i): float(ms_cls[i] / args.steps)
                                         for i in range(mce.NUM_WIDTHS) if ms_cls[i] > 0}},
        "roofline": roofline, "clocks": clocks, "gpu_launches": launches,
        "wall_s_timed": wall,
    }

    if not args.no_e2e:
        line["e2e"] = e2e_leg(args, g, roots, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = len(os.sched_getaffinity(0))
        sample, ores, dt = oracle_sample(g, roots, args.cpu_fraction, args.seed + 1000, threads)
        got = h.count_roots_result(sample)
        line["cpu_baseline"] = cpu_block(
            ores.count / dt, threads,
            f"oracle on {len(sample)} seeded roots ({args.cpu_fraction:.0%} of the workload "
            f"roots): {ores.count} cliques in {dt:.1f} s, including its own input checks, "
            f"peel and relabelling of the whole graph")
        line["parity_on_cpu_sample"] = "ok" if got == ores.key() else f"MISMATCH {got} {ores.key()}"
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
    if rank != 0:
        return
    import oracle
    oracle.build()
    g = workload_graph(args)
    _, _, orank, d = oracle.peel(g)
    roots, pc = light_roots(g, orank, args.max_p)
    threads = len(os.sched_getaffinity(0))
    frac = min(args.cpu_fraction, 1.0) / 2
    total_cl = 0
    total_s = 0.0
    for k in range(args.warmup + args.steps):
        _, res, dt = oracle_sample(g, roots, frac, args.seed + 2000 + k, threads)
        if k >= args.warmup:
            total_cl += res.count
            total_s += dt
    value = total_cl / total_s
    desc = (f"oracle, each step {frac:.0%} of the workload roots (seeded), with its own input "
            f"checks, peel and relabelling of the whole graph")
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
