"""bench.py across ranks, on CPU with the gloo backend (world size 2).

Each rank of a multi-GPU bench run is an independent replica; the only
cross-rank steps are the barriers around the timed region, the max over ranks
of the step time, and rank 0 alone printing the line. These run here as two
processes on 127.0.0.1.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# On a machine with a GPU bench.py picks NCCL and one device per rank; these
# checks are of the CPU (gloo) path.
pytestmark = pytest.mark.skipif(torch.cuda.is_available(), reason="checks the gloo path on a CPU-only host")


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, _ = bench.dist_setup()
    assert (r, w) == (rank, ws) and dist.get_backend() == "gloo"
    bench.barrier(w)
    step_ms = 1.0 + rank                      # rank 1 is the slow one
    res = bench.job_throughput(step_ms, w, 64)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump(res, f)
    dist.destroy_process_group()


def test_job_throughput_takes_the_slowest_rank(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn", join=True)
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    # both ranks see the max step (2 ms) and the job rate 2 ranks x 64 tokens / 2 ms
    for step_ms_max, value in got:
        assert step_ms_max == 2.0
        assert value == pytest.approx(2 * 64 / 2e-3)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_throughput(4.0, 1, 64) == (4.0, 64 / 4e-3)


def test_reference_arm_under_torchrun_prints_once():
    # the reference arm (the oracle on host cores) runs on rank 0 only; rank 1 exits 0 without work
    port = _free_port()
    env = dict(os.environ, PYTHONPATH=ROOT)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "3"]
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [json.loads(l) for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["steps"] == 1 and line["warmup"] == 3
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["value"] > 0


def test_clock_sampler_counts_only_samples_taken_while_timing(tmp_path, monkeypatch):
    """The sampler waits for its tool's first line and summarises only the lines written after it: a slow start
    of the tool must not leave a short timed region unsampled, and its idle first sample must not count."""
    import time
    fake = tmp_path / "nvidia-smi"
    fake.write_text(
        "#!/bin/sh\n"
        "echo '0, 120, 2070, 100.0, 0x0, Not Active, Not Active, Not Active, Not Active'\n"
        "sleep 0.3\n"
        "while true; do\n"
        "  echo '0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Active'\n"
        "  sleep 0.05\n"
        "done\n")
    fake.chmod(0o755)
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ['PATH']}")
    sys.path.insert(0, ROOT)
    import bench
    clk = bench.ClockSampler(0)
    with clk:
        assert clk.skip == 1                      # the idle line written before the region
        time.sleep(0.6)
    out = clk.summary()
    assert out["samples"] >= 3
    assert out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]
