"""The multi-GPU path of bench.py is replicas only (independent problems, no
exchange step): each rank runs the same workload, the job's step time is the
slowest rank's and the whole-job value counts every rank's bytes.  These
tests run that aggregation on world_size-2 gloo groups on the CPU, and check
that the reference arm does its work on rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, step_ms, out):
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(step_ms[rank], dist, "cpu")
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_step_time_is_the_slowest_rank():
    world = 2
    step_ms = [0.25, 0.40]
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank, args=(world, _free_port(), step_ms, out), nprocs=world,
                       join=True, start_method="spawn")
    assert out[0] == out[1] == max(step_ms)


def test_job_value_counts_every_replica():
    import bench
    one = bench.job_value(1, 1_000_000_000, 1000.0)
    assert abs(one - 1.0) < 1e-12
    assert abs(bench.job_value(2, 1_000_000_000, 1000.0) - 2 * one) < 1e-12


def test_single_rank_needs_no_group():
    import bench
    assert bench.max_over_ranks(0.3, None, "cpu") == 0.3


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_recorded_traffic_only_for_unchanged_sources(tmp_path):
    """The roofline's DRAM traffic comes from a committed ncu capture and is
    reported only while the kernel sources are those that were captured."""
    import bench
    kern = "dominant_kernel"
    good = tmp_path / "good.json"
    good.write_text(json.dumps({kern: {"sources_sha": bench.kernel_sources_sha(),
                                       "dram_bytes_per_launch": 123, "profile": "p.md"}}))
    assert bench.recorded_traffic(str(good)) == (123, "p.md")
    stale = tmp_path / "stale.json"
    stale.write_text(json.dumps({kern: {"sources_sha": "0" * 16, "dram_bytes_per_launch": 123}}))
    assert bench.recorded_traffic(str(stale))[0] is None
    assert bench.recorded_traffic(str(tmp_path / "missing.json"))[0] is None


def test_reference_arm_prints_one_complete_json_line():
    """On rank 0 the reference arm (the fp64 oracle on the host cores) prints
    exactly one JSON line with the contract's keys, its own cpu_baseline and
    an e2e entry without host-device copies."""
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_back_to_back_copies_exceed_twice_l2():
    """The back-to-back timing rotates over enough input copies that the
    other copies read between two uses of one copy exceed twice the L2 size."""
    import bench
    l2 = 126 * 2**20
    for nbytes in (4 << 20, 8_135_168, 64_322_048, 134_242_436, 291_030_672, 10**9):
        n = bench.graph_copies(nbytes, l2)
        assert n >= 3
        assert (n - 1) * nbytes > 2 * l2
        assert n == 3 or (n - 2) * nbytes <= 2 * l2  # no more copies than needed
