"""The N > 1 path of bench.py is replicas only (the chain has no exchange
step): two gloo ranks on the host check the slowest-rank reduction and the
whole-job throughput the rank-0 line reports."""
import json
import os
import socket
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    dt_local = 1.0 + rank          # rank 1 is the slower replica
    dt, per_step, value = bench.replicas_value(dt_local, 100, 3.0e9, world, dist, device="cpu")
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"dt": dt, "per_step": per_step, "value": value}, f)
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank_and_all_bytes(tmp_path):
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    mp.spawn(_rank, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(2)]
    for r in res:
        assert r["dt"] == 2.0                      # max over ranks
        assert r["per_step"] == 2.0 / 100
        assert abs(r["value"] - 2 * 3.0e9 / 0.02 / 1e9) < 1e-9  # both ranks' bytes


def test_one_replica_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    dt, per_step, value = bench.replicas_value(0.5, 10, 1.0e9, 1)
    assert dt == 0.5 and per_step == 0.05 and abs(value - 20.0) < 1e-12
