"""The multi-rank host logic of bench.py on CPU: two gloo ranks, as torchrun
would start them.  The ranks split the B*H heads of one workload into
contiguous slices (no data-path collective); the step time reported is the
max over ranks."""
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


@pytest.mark.parametrize("bh,world", [(512, 8), (32, 2), (7, 2), (5, 8), (1, 2), (64, 3), (100, 7)])
def test_shard_covers_every_head_once(bh, world):
    import bench
    seen = []
    for r in range(world):
        first, count = bench.shard(bh, world, r)
        assert count >= 0
        seen.extend(range(first, first + count))
    assert seen == list(range(bh))  # contiguous, in rank order, each head once
    counts = [bench.shard(bh, world, r)[1] for r in range(world)]
    assert max(counts) - min(counts) <= 1


def _shard_oracle_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      LOCAL_RANK=str(rank), WORLD_SIZE=str(world))
    import numpy as np
    import torch
    import bench
    import oracle
    from tiled_attention_tk_gb300.inputs import make_qkv
    dist = bench.init_dist(world, "gloo")
    B, H, N, D = 1, 5, 40, 16  # 5 heads over 2 ranks: 3 + 2
    q, k, v = make_qkv(B, H, N, D, 9100)
    first, count = bench.shard(B * H, world, rank)
    sl = slice(first, first + count)
    qs = q.reshape(B * H, N, D)[sl].reshape(1, count, N, D)
    ks = k.reshape(B * H, N, D)[sl].reshape(1, count, N, D)
    vs = v.reshape(B * H, N, D)[sl].reshape(1, count, N, D)
    O, L = oracle.attn_fwd(qs, ks, vs, True, 0.25)
    # every rank's slice to every rank (padded to the largest slice)
    cnt = bench.shard(B * H, world, 0)[1]
    o_pad = torch.zeros((cnt, N, D), dtype=torch.float64)
    l_pad = torch.zeros((cnt, N), dtype=torch.float64)
    o_pad[:count] = torch.from_numpy(O[0])
    l_pad[:count] = torch.from_numpy(L[0])
    o_all = [torch.empty_like(o_pad) for _ in range(world)]
    l_all = [torch.empty_like(l_pad) for _ in range(world)]
    dist.all_gather(o_all, o_pad)
    dist.all_gather(l_all, l_pad)
    if rank == 0:
        parts_o, parts_l = [], []
        for r in range(world):
            c = bench.shard(B * H, world, r)[1]
            parts_o.append(o_all[r][:c])
            parts_l.append(l_all[r][:c])
        o_cat = torch.cat(parts_o).numpy().reshape(B, H, N, D)
        l_cat = torch.cat(parts_l).numpy().reshape(B, H, N)
        O_full, L_full = oracle.attn_fwd(q, k, v, True, 0.25)
        out["equal"] = bool(np.array_equal(o_cat, O_full) and np.array_equal(l_cat, L_full))
    dist.barrier()
    dist.destroy_process_group()


def test_sharded_oracle_results_reassemble_bitwise():
    """Per-slice results of two gloo ranks, gathered and put back in head
    order, equal the whole-problem oracle bit for bit."""
    import oracle
    oracle.build()
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_shard_oracle_worker, args=(world, port, out), nprocs=world, join=True)
        assert out["equal"] is True


def test_gpus_without_torchrun_relaunches_ranks(monkeypatch):
    """--gpus N outside torchrun runs the script as N ranks rather than
    printing a one-rank line."""
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    import bench
    cmd = bench.relaunch_cmd(4, ["--gpus", "4", "--steps", "5"], 29500)
    assert cmd[1:3] == ["-m", "torch.distributed.run"]
    assert "--nproc-per-node=4" in cmd and "--master-addr=127.0.0.1" in cmd
    assert cmd[-4:] == ["--gpus", "4", "--steps", "5"]
    calls = []
    monkeypatch.setattr(bench, "relaunch_ranks", lambda n, argv: calls.append((n, list(argv))) or 0)
    with pytest.raises(SystemExit) as e:
        bench.main(["--gpus", "2", "--steps", "3", "--warmup", "3"])
    assert e.value.code == 0 and calls == [(2, ["--gpus", "2", "--steps", "3", "--warmup", "3"])]


def test_parity_rows_cover_edges():
    import bench
    from tiled_attention_tk_gb300.inputs import WORKLOADS
    w = WORKLOADS[5]
    rows = bench.parity_rows(w)
    assert rows[0] == 0 and rows[-1] == w.N - 1 and len(rows) <= 320 and len(set(rows)) == len(rows)
    assert 127 in rows and 128 in rows
    assert bench.parity_rows(WORKLOADS[1]) == list(range(128))
    assert bench.parity_heads(10, 3) == [10, 11, 12]
    h = bench.parity_heads(0, 512)
    assert h[0] == 0 and h[-1] == 511 and len(h) == 4
