"""Host-side checks of bench.py: the byte accounting, the max-over-ranks aggregation
on a real two-rank gloo process group, and the reference arm's JSON contract."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

from conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_algorithmic_bytes_of_the_specified_workloads():
    # every input byte read once, every output byte written once (H = 4096)
    assert bench.bytes_fold(4, 2048, 4096, fp8=True, y=False) == 109_076_480
    assert bench.bytes_fold(8, 64, 4096) == 5_783_552
    assert bench.bytes_fold(8, 64, 4096, residual=False) == 5_259_264
    assert bench.bytes_fold(8, 254, 4096) == 22_904_832
    assert bench.bytes_moe(1024, 4096, 8) == 92_356_608
    # FP8 read on the finalize: residual' + codes + scales instead of residual' + y
    assert bench.bytes_moe(1024, 4096, 8, y=False, fp8=True) == 88_166_400
    assert bench.bytes_fold(2, 16, 512) == 83_968


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    d = bench.Dist()
    d.init("gloo")
    # rank r pretends its timed region took r + 1 seconds for 10 steps of 2048 rows
    value, worst = bench.aggregate(float(rank + 1), 2048, 10, d)
    d.barrier()
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"value": value, "worst": worst}, f)
    d.close()


def test_aggregate_takes_the_slowest_rank_over_gloo(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    for r in range(world):
        got = json.load(open(tmp_path / f"r{r}.json"))
        assert got["worst"] == 2.0
        assert got["value"] == world * 2048 * 10 / 2.0


def test_reference_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "4", "--warmup", "3"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line
    assert line["impl"] == "reference" and line["steps"] == 4
    assert line["config"]["workload"] == "prefill_fold_norm_fp8"
    cores = len(os.sched_getaffinity(0))
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert 1 <= line["cpu_baseline"]["cores"] <= cores
    assert line["config"]["rows_per_step"] >= line["cpu_baseline"]["cores"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "4", "--warmup", "3"], capture_output=True,
                       text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_native_arm_refuses_to_run_without_a_gpu():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "4"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode != 0 and "needs a CUDA GPU" in (r.stderr + r.stdout)


def test_oracle_rate_counts_every_thread():
    """The CPU baseline's row-partitioned oracle timing counts the rows of every
    thread and reports a positive rate."""
    sys.path.insert(0, ROOT)
    import bench
    from layer_boundary_fusion_gb300 import workloads as wl
    w = wl.tiny_fold_norm()
    rate, rows, el = bench.oracle_rate(w, 2, 0.2, 8)
    assert rows > 0 and rows % 8 == 0 and rate == rows / el
    cores, model = bench.host_cpu()
    assert cores >= 1 and model
