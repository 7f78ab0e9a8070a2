"""Host logic of bench.py that needs no GPU: the replica aggregation over two
ranks (gloo on CPU, world_size 2), the whole-job µs-per-call arithmetic, and
the rule that recorded DRAM traffic is reported only for the kernel sources
it was measured on."""
import json
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    d = bench.Dist()
    assert d.world == world and d.rank == rank and d.pg is not None
    d.barrier()
    # each rank timed its own replica: 10 ms on rank 0, 25 ms on rank 1
    elapsed = d.max(10.0 if rank == 0 else 25.0)
    us = bench.aggregate_us_per_call(elapsed, calls_per_rank=100, world=d.world)
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"max": elapsed, "us": us}, f)
    d.close()


def test_two_rank_replicas_take_the_max_and_count_every_rank(tmp_path):
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    for r in (0, 1):
        res = json.loads((tmp_path / f"r{r}.json").read_text())
        assert res["max"] == 25.0                       # max over ranks
        assert res["us"] == pytest.approx(25.0 * 1000 / 200)   # all 200 calls of the job


def test_single_rank_needs_no_process_group(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    d = bench.Dist()
    assert d.world == 1 and d.pg is None
    assert d.max(3.5) == 3.5
    assert bench.aggregate_us_per_call(2.0, 4, 1) == 500.0


def test_traffic_record_only_for_the_measured_sources(tmp_path, monkeypatch):
    csrc = tmp_path / "mxfp4_mixture_experts_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in bench.KERNEL_SOURCES["decode"]:
        (csrc / f).write_text(f"// {f}\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_hash("decode")
    rec = {"kernel_hash": h, "dram_over_alg": {"32": 1.007}}
    (tmp_path / "profiles" / "decode_traffic.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic("decode") == rec
    (csrc / "decode.cu").write_text("// changed\n")      # the kernel changed since
    assert bench.kernel_hash("decode") != h
    assert bench.recorded_traffic("decode") is None
    (tmp_path / "profiles" / "decode_traffic.json").unlink()
    assert bench.recorded_traffic("decode") is None
