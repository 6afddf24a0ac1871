"""The N > 1 path of the benchmark on CPU: two ranks over gloo.

The hot path has no exchange step, so N GPUs run N independent replicas
(each draws its own batch); the only collectives are a barrier around each
timed region and the maximum over ranks of the step time, and the whole-job
rate is the units of all ranks over that maximum.  These tests run the same
`Replicas` helper the benchmark uses, with the gloo backend, in two spawned
processes (no GPU).
"""
import json
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str) -> None:
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench
    from lora_adapters_gb300 import workloads

    rep = bench.Replicas("gloo")
    rep.barrier()
    # rank r "measured" (r + 1) ms per step: every rank reports the slowest
    ms = rep.max(1.0 + rank)
    rate = rep.rate(256, ms * 1e-3)
    # each replica draws its own batch
    ta = workloads.make("tiny", seed=rank).token_adapter.tolist()
    objs = [None] * world
    rep.dist.all_gather_object(objs, ta)
    # the reference arm: only rank 0 runs it (the others return at once)
    ref_returned = bench.run_reference(None, None, None) is None if rank != 0 else True
    rep.barrier()
    rep.close()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"world": rep.world, "rank": rep.rank, "max_ms": ms, "rate": rate, "batches": objs,
                   "ref_returned": ref_returned}, f)


def test_two_replicas_over_gloo(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp

    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, d in enumerate(res):
        assert d["world"] == world and d["rank"] == r
        assert d["max_ms"] == 2.0                       # the slowest rank's time, on every rank
        assert d["rate"] == pytest.approx(world * 256 / 2e-3)
        assert d["ref_returned"]
    batches = res[0]["batches"]
    assert batches == res[1]["batches"]
    assert batches[0] != batches[1]                     # independent batches per replica


def test_single_process_needs_no_process_group(monkeypatch):
    for k in ("WORLD_SIZE", "RANK"):
        monkeypatch.delenv(k, raising=False)
    sys.path.insert(0, ROOT)
    import bench

    rep = bench.Replicas("gloo")
    assert rep.world == 1 and rep.rank == 0 and rep.dist is None
    rep.barrier()
    assert rep.max(3.5) == 3.5
    assert rep.rate(10, 2.0) == 5.0
    rep.close()
