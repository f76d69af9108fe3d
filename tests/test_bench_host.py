"""Host-side logic of bench.py on the CPU: the cross-rank timing of the N-GPU
(replica) runs over a 2-rank gloo group, the whole-job rate, the clock-sample
parser, workload selection and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _rank(rank, world, port, q):
    import torch.distributed as tdist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [3.0, 5.0][rank]            # rank 1 is the slower one
        slowest = bench.max_over_ranks(local_ms)
        rate = bench.job_rate(100.0, world, slowest * 1e-3)
        tdist.barrier()
        q.put((rank, slowest, rate))
    finally:
        tdist.destroy_process_group()


def test_max_over_ranks_and_job_rate_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, slowest, rate in got:
        assert slowest == 5.0                    # every rank sees the slowest rank's time
        assert rate == pytest.approx(2 * 100.0 / 5e-3)   # units of both ranks over that time


def test_max_over_ranks_without_a_group_is_identity():
    assert bench.max_over_ranks(7.5) == 7.5
    assert bench.job_rate(10.0, 1, 2.0) == 5.0


def test_parse_clock_rows():
    rows = "\n".join([
        "0, 1900, 2070, 1200.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 1800, 2070, 1350.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2000, 2070, 900.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ])
    c = bench.parse_clock_rows(rows)
    assert c["sm_mhz"] == 1900 and c["sm_max_mhz"] == 2070 and c["samples"] == 3
    assert c["reasons"] == ["sw_power_cap"] and c["power_w_max"] == 1350.0
    hot = bench.parse_clock_rows("0, 1500, 2070, 1000, 0x40, Active, Active, Not Active, Not Active")
    assert hot["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]


def test_clock_summary_of_nvml_samples():
    """Samples polled in-process while the timed region ran: the median SM
    clock and the clock-event reasons named from their NVML bits (GPU idle and
    other bits are not judged)."""
    samples = [(1900.0, 1200.0, 0x4), (1950.0, 1300.0, 0x0), (1800.0, None, 0x1 | 0x4), (1850.0, 1100.0, 0x0)]
    c = bench.summarize_clock_samples(samples, 2070.0, before=(2000.0, 300.0, 0), after=(1900.0, 800.0, 0))
    assert c["sm_mhz"] == 1875.0 and c["samples"] == 4 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"] and c["power_w_max"] == 1300.0
    assert (c["sm_mhz_min"], c["sm_mhz_max"], c["sm_mhz_before"], c["sm_mhz_after"]) == (1800.0, 1950.0, 2000.0,
                                                                                        1900.0)
    hot = bench.summarize_clock_samples([(1500.0, 1000.0, 0x8 | 0x40)], 2070.0)
    assert hot["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]
    none = bench.summarize_clock_samples([], 2070.0)
    assert none["sm_mhz"] is None and none["samples"] == 0


def test_nvml_sampler_without_a_gpu_is_inert():
    c = bench.NvmlClocks(0)
    if not c.ok:
        assert c.sample() is None


def test_workload_selection():
    class A:
        config, k_group = 3, 128
    assert bench.workload_key(A) == "3g128" and "K group" in bench.describe(A)
    A.k_group = 0
    assert bench.workload_key(A) == "3"
    A.config, A.k_group = 2, 128
    with pytest.raises(SystemExit):
        bench.make_workload(A)


def test_reference_arm_json_line():
    """--impl reference times the oracle on the host: one JSON line with the
    contract's keys, the oracle as its cpu_baseline and no host<->device bytes."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "1",
                        "--steps", "3", "--warmup", "3", "--ref-seconds", "2"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0

    # both arms describe the workload with the same config dict (run details
    # such as the plan go under "setup" in the GPU arm)
    class A:
        config, shape, k_group, b_block = 1, None, 0, 1
    assert d["config"] == bench.config_of(A, bench.make_workload(A))


def test_shape_option():
    class A:
        config, k_group, shape = 2, 0, "64,256,128"
    w = bench.make_workload(A)
    assert (w.M, w.N, w.K, w.b_layout) == (64, 256, 128, "nk") and tuple(w.B.shape) == (256, 128)
    assert bench.workload_key(A) == "2s64x256x128" and "M=64 N=256 K=128" in bench.describe(A)
    A.config = 3
    with pytest.raises(SystemExit):
        bench.make_workload(A)


def test_recorded_traffic_follows_source_hash_and_plan_tile(tmp_path):
    """A DRAM figure from the traffic records is reported only while the device
    code hashes the same and, where the record names a tile, while the plan
    still chooses that tile."""
    sha = bench.kernel_source_hash()
    path = tmp_path / "dram_traffic.txt"
    path.write_text("# test records\n"
                    f"workload=2 kernel_src_sha={sha} tile=256x256x2 dram_bytes_per_launch=1000\n"
                    "workload=3 kernel_src_sha=0000000000000000 tile=256x256x2 dram_bytes_per_launch=2000\n"
                    f"workload=4 kernel_src_sha={sha} dram_bytes_per_launch=3000\n")
    pair = {"tile_m": 256, "tile_n": 256, "cta_group": 2}
    single = {"tile_m": 128, "tile_n": 256, "cta_group": 1}
    assert bench.recorded_traffic("2", pair, str(path)) == 1000
    assert bench.recorded_traffic("2", None, str(path)) == 1000
    assert bench.recorded_traffic("2", single, str(path)) is None   # another tile
    assert bench.recorded_traffic("3", pair, str(path)) is None     # older device code
    assert bench.recorded_traffic("4", single, str(path)) == 3000   # no tile named
    assert bench.recorded_traffic("5", pair, str(path)) is None
