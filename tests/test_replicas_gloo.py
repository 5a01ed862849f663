"""bench.py's host side on CPU.  Its multi-replica path: one process per
rank over gloo (world size 2), as torch.distributed.run launches it; the
replicas share nothing on the data path (each runs the whole step on its own
GPU), only the timing is reduced -- the slowest rank's time -- and rank 0
alone prints.  Then its clock samplers and the committed DRAM-traffic
figure it reports."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    w, r, _, dist = bench.dist_setup()
    ms = 10.0 + 5.0 * r            # rank 1 is the slower replica
    got = bench.max_over_ranks(ms, dist)
    q.put((r, w, got, bench.whole_job_value(w, 16384, 100, got)))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_two_replicas():
    import torch.multiprocessing as mp

    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, *_ in results] == [0, 1]
    for _, world, got, value in results:
        assert world == 2
        assert got == 15.0            # every rank sees the slowest rank's time
        assert value == pytest.approx(2 * 16384 * 100 / 0.015)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(12.5, None) == 12.5
    assert bench.whole_job_value(1, 1000, 10, 5.0) == pytest.approx(2e6)


def test_reference_arm_under_torchrun():
    """Two ranks launched as the driver launches them: rank 0 alone times the
    oracle and prints one JSON line; rank 1 exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--workload", "tiny", "--gpus", "2", "--steps", "2",
           "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["n_gpus"] == 2 and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["e2e"]["value"] == d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle"


def test_clock_samples_use_nvidia_smi_timestamps():
    """The bench keeps the clock samples whose own nvidia-smi timestamp lies
    in the measured window (a pipe may hand lines over late, in batches)."""
    import bench

    s = bench.ClockSampler(0)
    base = bench.ClockSampler.sample_time("2026/12/02 13:42:01.100", 0.0)
    assert base > 0
    assert abs(bench.ClockSampler.sample_time("2026/12/02 13:42:01.350", 0.0) - base - 0.25) < 1e-6
    assert bench.ClockSampler.sample_time("not a time", 7.5) == 7.5
    line = "{t}, 0, {mhz}, 2070, 500.0, 0x0, Not Active, Not Active, Not Active, {cap}"
    late = base + 10.0   # every line read long after it was sampled
    s.lines = [(late, line.format(t="2026/12/02 13:42:01.000", mhz=1000, cap="Not Active")),
               (late, line.format(t="2026/12/02 13:42:01.150", mhz=2070, cap="Active")),
               (late, line.format(t="2026/12/02 13:42:01.200", mhz=2070, cap="Not Active")),
               (late, line.format(t="2026/12/02 13:42:02.000", mhz=900, cap="Not Active"))]
    out = s.summary(base, base + 0.12)
    assert out["samples"] == 2
    assert out["sm_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]


def test_nvml_clock_samples_inside_the_timed_steps():
    """The in-process NVML sampler keeps the samples taken during the timed
    steps, maps the clock-event reason bits to their names, and gives no
    summary (the nvidia-smi one stands) where the library is not there."""
    import bench
    import torch

    s = bench.NvmlSampler.__new__(bench.NvmlSampler)
    s.max_mhz = 2070
    s.rows = [(0.9, 600, 0x1, 100.0),          # before the window: idle, left out
              (1.0, 2070, 0x0, 700.0),
              (1.2, 2055, 0x4, 1300.0),       # power cap
              (1.4, 2070, 0x8 | 0x40, 800.0),  # hardware slowdowns
              (2.5, 900, 0x20, 200.0)]        # after the window
    out = s.summary(1.0, 2.0)
    assert out["samples"] == 3 and out["sm_mhz"] == 2070 and out["sm_mhz_min"] == 2055
    assert out["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap"]
    assert out["power_w_max"] == 1300.0 and out["sm_max_mhz"] == 2070
    assert s.summary(3.0, 4.0) is None
    if not torch.cuda.is_available():
        n = bench.NvmlSampler(torch, 0)
        n.start()
        n.stop()
        assert n.summary(0.0, 1e12) is None


def test_committed_kv_traffic_matches_the_kernel_source():
    """The KV store's DRAM traffic that the benchmark reports comes from the
    committed ncu summary, which carries a digest of the kernel's sources; a
    change to those sources without a new capture would turn the figure into
    null, so the digest must match the sources as they are."""
    import bench

    per_unit = bench.committed_traffic(1)
    assert per_unit is not None, (
        "profiles/kv_write_large_step.md was captured on another kernel source "
        f"(current digest {bench.kernel_source_digest()})")
    # K and V lines of 1 KiB read and written plus the slot: 4104 bytes of
    # algorithmic traffic per token-layer; DRAM saw no re-reads
    assert 0.9 * 4104 < per_unit < 1.05 * 4104


def test_line_bytes_override_is_checked_and_recorded():
    """--line-bytes (small profiling cases) takes a positive multiple of 16
    and shows in the line's config; anything else is refused before any
    work."""
    base = [sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny",
            "--steps", "1", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    bad = subprocess.run(base + ["--line-bytes", "24"], cwd=ROOT, capture_output=True,
                         text=True, timeout=300, env=env)
    assert bad.returncode == 2 and "--line-bytes" in bad.stderr
    ok = subprocess.run(base + ["--line-bytes", "64"], cwd=ROOT, capture_output=True,
                        text=True, timeout=600, env=env)
    assert ok.returncode == 0, ok.stderr[-2000:]
    d = json.loads([ln for ln in ok.stdout.splitlines() if ln.startswith("{")][-1])
    assert d["config"]["line_bytes"] == 64
