"""The multi-GPU path is replicas only (independent copies of the workload, no data-path
collective).  Its host side -- process group set-up, the barrier around the timed region and
the max over ranks of the timed region -- runs here as two gloo ranks on the CPU.
"""
import argparse
import json
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
mp = pytest.importorskip("torch.multiprocessing")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    args = argparse.Namespace(impl="reference")
    r, w, local = bench.dist_init(args)
    bench.barrier(w)
    # each rank times a different amount; every rank must see the slowest
    slowest = bench.max_over_ranks(10.0 + 5.0 * r, w)
    bench.barrier(w)
    # the reference arm does no work on ranks other than 0
    did = None
    if r != 0:
        did = bench.run_reference(argparse.Namespace(), r, w)
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"rank": r, "world": w, "local": local, "slowest": slowest,
                   "ref_return": did}, f)
    import torch.distributed as dist
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_replica_process_group_on_cpu(tmp_path, world):
    port = _free_port()
    mp.spawn(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, join=True)
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    assert [g["rank"] for g in got] == list(range(world))
    assert all(g["world"] == world for g in got)
    assert all(g["slowest"] == 10.0 + 5.0 * (world - 1) for g in got)
    assert got[1]["ref_return"] is None


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    env = {k: os.environ.pop(k) for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK") if k in os.environ}
    try:
        assert bench.dist_init(argparse.Namespace(impl="gb300")) == (0, 1, 0)
        assert bench.max_over_ranks(3.25, 1) == 3.25
    finally:
        os.environ.update(env)
