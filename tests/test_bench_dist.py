"""The multi-rank host logic of bench.py on CPU: two gloo ranks, as torchrun
would start them.  Every rank runs its own full workload (independent
problems, no data-path collective); the step time reported is the max over
ranks and the value counts the work of all ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      LOCAL_RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    dist = bench.init_dist(ws, "gloo")
    assert dist is not None
    # each rank "measured" a different time; everyone must agree on the max
    t = bench.max_over_ranks(10.0 + rank * 5.0, dist)
    out[rank] = t
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        assert dict(out) == {0: 15.0, 1: 15.0}


def test_single_rank_needs_no_process_group(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    import bench
    assert bench.dist_env() == (1, 0, 0)
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(3.5, None) == 3.5


def test_reference_arm_other_ranks_do_no_work(monkeypatch):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    args = type("A", (), {"steps": 1, "warmup": 3, "reference_budget": 1.0})()
    from tiled_attention_tk_gb300.inputs import WORKLOADS
    assert bench.run_reference(args, WORKLOADS[1]) is None


def test_reference_arm_line_on_rank0(monkeypatch):
    """On rank 0 the reference arm times the oracle on the host and returns
    the contract's line: the metric, a positive value, impl "reference", a
    cpu_baseline describing this run and an e2e entry with no copies."""
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    import bench
    from tiled_attention_tk_gb300.inputs import WORKLOADS
    args = type("A", (), {"steps": 2, "warmup": 3, "reference_budget": 0.5})()
    line = bench.run_reference(args, WORKLOADS[1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["value"] > 0 and line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    assert line["steps"] == 2 and line["warmup"] == 3 and line["gpu_launches"] == 0
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"] == WORKLOADS[1].name
