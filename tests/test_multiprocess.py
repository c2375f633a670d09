"""The multi-rank host path of bench.py on CPU: two gloo ranks over
127.0.0.1.  N GPUs run N independent replicas (no collective on the data
path); the only cross-rank steps are the timing barrier, the max over ranks
and the rank-0 report, which these tests exercise with the real functions."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank, ws, port):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(ws),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})


def _timing_rank(rank, ws, port, out_dir):
    _env(rank, ws, port)
    import bench
    wsz, rk, _ = bench.dist_setup()
    try:
        bench.barrier(wsz)
        local_ms = 10.0 * (rk + 1)                      # rank 1 is the slow one
        m = bench.max_over_ranks(local_ms, wsz, torch.device("cpu"))
        rate = bench.job_rate(100, 64, wsz, m)
        json.dump({"rank": rk, "ws": wsz, "max_ms": m, "rate": rate},
                  open(os.path.join(out_dir, f"r{rk}.json"), "w"))
    finally:
        import torch.distributed as dist
        dist.destroy_process_group()


def _reference_rank(rank, ws, port, out_dir):
    _env(rank, ws, port)
    import argparse
    import bench
    wsz, rk, _ = bench.dist_setup()
    try:
        args = argparse.Namespace(gpus=ws, steps=2, warmup=1, workload="tiny", rot=1, soak=0.0,
                                  cpu_budget=0.1, no_cpu_baseline=True, impl="reference")
        buf = io.StringIO()
        with redirect_stdout(buf):
            rc = bench.run_reference(args, wsz, rk)
        json.dump({"rank": rk, "rc": rc, "stdout": buf.getvalue()}, open(os.path.join(out_dir, f"r{rk}.json"), "w"))
    finally:
        import torch.distributed as dist
        dist.destroy_process_group()


def _run(fn, tmp_path, ws=2):
    mp.start_processes(fn, args=(ws, _free_port(), str(tmp_path)), nprocs=ws, start_method="spawn", join=True)
    return [json.load(open(tmp_path / f"r{r}.json")) for r in range(ws)]


def test_two_ranks_time_by_the_slowest(tmp_path):
    res = _run(_timing_rank, tmp_path)
    for r in res:
        assert r["ws"] == 2
        assert r["max_ms"] == pytest.approx(20.0)
        assert r["rate"] == pytest.approx(100 * 64 * 2 / 0.020)   # all ranks' tokens / slowest time


def test_reference_arm_reports_on_rank0_only(tmp_path):
    pytest.importorskip("numpy")
    res = _run(_reference_rank, tmp_path)
    r0, r1 = sorted(res, key=lambda r: r["rank"])
    assert r0["rc"] == 0 and r1["rc"] == 0
    assert r1["stdout"] == ""
    lines = [l for l in r0["stdout"].splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    required = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"}
    assert required <= set(line), required - set(line)
    assert line["steps"] == 2 and line["warmup"] == 1 and line["higher_is_better"] is True
    assert {"value", "unit", "cores", "kind", "sample"} <= set(line["cpu_baseline"])
    assert line["e2e"]["value"] == line["value"] and line["e2e"]["unit"] == line["unit"]
