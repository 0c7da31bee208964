"""The multi-GPU path of bench.py is replicas only (one process per GPU, no
data-path collective): rank timings are combined as the maximum time over
ranks and the sum of processed units.  Checked here with two gloo ranks on CPU."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import bench
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    d = bench.maybe_init_dist(ws, "gloo")
    t, units = bench.aggregate(d, local_seconds=1.0 + rank, local_units=100.0 * (rank + 1))
    out[rank] = (t, units)
    # the reference arm runs on rank 0 only: other ranks return at once
    if rank != 0:
        out[world + rank] = bench.run_reference(None)
    d.barrier()
    d.destroy_process_group()


def test_two_gloo_ranks_aggregate_max_time_and_summed_units():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:   # no fork of this multi-threaded process
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        for rank in range(world):
            t, units = out[rank]
            assert t == 2.0              # the slowest rank's time
            assert units == 300.0        # every rank's units
        assert out[world + 1] == 0       # rank 1 of the reference arm did nothing


def test_single_process_aggregate_is_identity():
    import bench
    assert bench.aggregate(None, 1.5, 7.0) == (1.5, 7.0)



def test_reference_arm_prints_the_contract_line(monkeypatch, capsys):
    # the reference arm is the oracle on the host cores: one JSON line with the
    # base contract's keys, its cpu_baseline (one thread, plus every core) and
    # an e2e entry with no host/device traffic (a small shape keeps it short)
    import json

    import bench
    from workload import Shape
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    monkeypatch.setattr(bench, "_shape", lambda: Shape(d=256, f=128, f_shared=128, n_experts=8, top_k=2))
    assert bench.main(["--impl", "reference", "--steps", "2", "--warmup", "3", "--cpu-budget", "1"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["warmup"] == 3 and line["value"] > 0
    for key in ("metric", "unit", "n_gpus", "steps", "ms_per_step", "higher_is_better", "scaling", "dtype",
                "data", "config"):
        assert key in line
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == line["value"]
    assert cb["all_cores"]["value"] > 0 and cb["all_cores"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
