"""The multi-rank host logic of bench.py on CPU: two gloo ranks.

The product does not shard (replicas only): every rank runs the whole
workload on its own GPU, the job takes as long as its slowest rank, and the
reported throughput is all ranks' work over that time."""
import json
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, outdir):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # Per-rank step times (ms): rank 1 is the slow one.
        mine = [2.0, 3.0][rank]
        slowest = bench.max_over_ranks(mine, "cpu")
        value = bench.job_tflops(2.0 * 4096 ** 3, world, slowest)
        with open(os.path.join(outdir, f"rank{rank}.json"), "w") as f:
            json.dump({"slowest": slowest, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time(tmp_path):
    port = _free_port()
    mp.spawn(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for g in got:
        assert g["slowest"] == 3.0
        # Both ranks' 137.4 GFLOP over 3 ms.
        assert g["value"] == pytest.approx(2 * 2.0 * 4096 ** 3 / 3e-3 / 1e12)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert not dist.is_initialized()
    assert bench.max_over_ranks(1.25, "cpu") == 1.25
    assert bench.job_tflops(2e12, 1, 1000.0) == pytest.approx(2.0)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    sys.path.insert(0, ROOT)
    import bench
    from fp32_sgemm_gb300 import inputs
    args = type("A", (), {"steps": 1, "warmup": 0})()
    bench.run_reference(args, inputs.WORKLOADS["sgemm_128"], rank=1, world=2)
    assert capsys.readouterr().out == ""


def test_reference_arm_line_on_rank_zero(capsys):
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    from fp32_sgemm_gb300 import inputs
    oracle.build()
    args = type("A", (), {"steps": 2, "warmup": 1})()
    bench.run_reference(args, inputs.WORKLOADS["sgemm_128"], rank=0, world=2)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
