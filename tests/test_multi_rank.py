"""Multi-rank host logic of the benchmark, on CPU with the gloo backend
(world size 2): the job time is the slowest rank's, the job throughput counts
every rank's bytes, and the reference arm does work on rank 0 only."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(1.0 + 2.5 * rank, "cpu")  # rank 1 is slower
        out[rank] = (ms, bench.job_gbs(1_000_000_000, world, ms))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput():
    world, port = 2, _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for rank in range(world):
        ms, gbs = out[rank]
        assert ms == pytest.approx(3.5)
        assert gbs == pytest.approx(2 * 1e9 / 3.5e-3 / 1e9)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(4.25, "cpu") == 4.25
    assert bench.job_gbs(2_000_000_000, 1, 1000.0) == pytest.approx(2.0)


def test_reference_arm_does_nothing_on_other_ranks(capsys):
    class A:
        steps, warmup = 1, 0
    bench.run_reference(A(), rank=1, world=2)
    assert capsys.readouterr().out == ""


def test_reference_arm_json_line():
    # rank 0 runs the CPU oracle on the bounded sample and prints one JSON
    # line with the contract's keys; its value, cpu_baseline and e2e agree
    import json
    import subprocess
    import sys

    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                         cwd=bench.ROOT, capture_output=True, text=True, timeout=600, check=True).stdout
    lines = [ln for ln in out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["vs_baseline"] is None
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["tensors"] == 225


def test_batched_launch_count_matches_the_library():
    # a batched decode of n tensors: ceil(n / 128) launch-table uploads, one decode
    assert [bench.batched_launches(n) for n in (1, 128, 129, 225)] == [2, 2, 3, 3]
    src = open(os.path.join(bench.ROOT, "quantized_weight_block_gb300", "csrc", "ndq_internal.h")).read()
    assert f"constexpr int kUploadChunk = {bench.UPLOAD_CHUNK};" in src
