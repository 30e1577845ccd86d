"""The benchmark's multi-rank path on the CPU (gloo, world size 2).

The forward shards over independent (batch, head) slices: every rank runs its own copy of the
workload and no data-path collective exists.  What the ranks share is the timing: the job's
time is the slowest rank's (a MAX all-reduce), the whole-job rate is world x tokens / that
time, and only rank 0 prints.  Those pieces run here as two gloo processes; the reference arm's
rule that ranks other than 0 exit at once without work is checked by running it as rank 1, and
its rank-0 JSON line (the oracle timed on the host cores) against the contract's keys.
"""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, values, out_dir):
    import torch.distributed as tdist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(values[rank], world, "cpu")
    rate = bench.job_rate(world, 25088, ms)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"ms": ms, "rate": rate}, f)
    tdist.barrier()
    tdist.destroy_process_group()


def _free_port():
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def test_max_over_ranks_and_job_rate_gloo(tmp_path):
    values = [0.0731, 0.0795]                       # per-rank mean step times, ms
    mp.start_processes(_rank_main, args=(2, _free_port(), values, str(tmp_path)), nprocs=2,
                       join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for r in res:
        assert r["ms"] == max(values)               # every rank sees the slowest rank's time
        assert r["rate"] == pytest.approx(2 * 25088 / (max(values) / 1e3), rel=1e-12)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(1.25, 1, "cpu") == 1.25
    assert bench.job_rate(1, 1000, 2.0) == pytest.approx(5e5)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "1"], env=env, capture_output=True,
                       text=True, timeout=120)
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""


def test_reference_arm_line_on_rank0():
    """The reference arm (the fp64 oracle on the host cores) prints one JSON line with the
    contract's keys: the same metric and unit as the GPU arm, impl = reference, a cpu_baseline
    describing the run and an e2e object with no host-device bytes."""
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_f32", "--steps", "2", "--warmup", "1"], env=env,
                       capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr
    lines = [l for l in p.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    import bench
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["higher_is_better"] is True and line["value"] > 0
    assert line["steps"] == 2 and line["warmup"] == 1 and line["n_gpus"] == 1
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["cpu_baseline"]["value"] == line["value"] and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"],
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert line["config"]["workload"].startswith("tiny_f32")
