"""Host logic of bench.py, no GPU needed.

* The multi-process path on CPU ranks (gloo): each rank runs its own
  replica (no exchange step on the data path); the reported time is the
  slowest rank's, taken by an all-reduce MAX, and the value aggregates every
  rank's work over that time.  Ranks other than 0 do no work in the
  reference (oracle) arm, and rank 0's line carries the contract's keys.
* The roofline's inputs: algorithmic bytes per launch against hand counts,
  DRAM traffic only from an ncu summary of the current kernel sources.
* The clock record: median SM clock inside the timed window, active
  throttle reasons by name.
"""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

import bench


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    got = bench.max_over_ranks(10.0 + 3 * rank, dist, "cpu")
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"r{rank}"), "w") as f:
        f.write(repr(got))


@pytest.mark.parametrize("world", [2, 3])
def test_max_over_ranks_takes_the_slowest(tmp_path, world):
    import torch.multiprocessing as mp
    mp.spawn(_rank_main, args=(world, free_port(), str(tmp_path)), nprocs=world, join=True)
    for r in range(world):
        assert float((tmp_path / f"r{r}").read_text()) == 10.0 + 3 * (world - 1)


def test_aggregate_counts_every_rank():
    # 2 ranks x 100 steps x 1 Mpix over 50 ms = 4 Gpix/s
    assert bench.aggregate_gpix(1_000_000, 100, 2, 50.0) == pytest.approx(4.0)
    assert bench.aggregate_gpix(1_000_000, 100, 1, 50.0) == pytest.approx(2.0)


def test_reference_arm_other_ranks_do_nothing(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        workload, steps, warmup, cpu_budget = "4k_to_1080p", 1, 0, 0.1

    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.reference_arm(Args()) is None
    assert buf.getvalue() == ""


def test_profile_traffic_only_for_current_sources(tmp_path, monkeypatch):
    # the roofline's traffic comes from a committed ncu summary, and only
    # while the kernel's sources hash to the value recorded in it
    (tmp_path / "profiles").mkdir()
    current = bench.kernel_sources_hash("multi.cu")
    summary = ("kernel sources (multi.cu + headers) sha256[:16]: `{}`\n\n"
               "dram bytes per launch: `123456` (read + write)\n")
    (tmp_path / "profiles" / "ncu_fresh.md").write_text(summary.format(current))
    (tmp_path / "profiles" / "ncu_stale.md").write_text(summary.format("0" * 16))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profile_traffic("fresh") == 123456
    assert bench.profile_traffic("stale") is None
    assert bench.profile_traffic("absent") is None


def test_reference_arm_line_carries_the_contract_keys(monkeypatch):
    # rank 0 of the reference arm times the oracle on the host and prints one
    # JSON line with the keys the driver reads (the oracle needs no GPU)
    import json
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")

    class Args:
        workload, steps, warmup, cpu_budget = "4k_to_1080p", 1, 3, 0.1

    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.reference_arm(Args())
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == "Gpix/s"
    assert line["value"] > 0 and line["higher_is_better"] is True and line["steps"] == 1
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]


@pytest.mark.parametrize("workload, read, write", [
    ("4k_to_1080p", 2160 * 3840 * 3, 1080 * 1920 * 3),             # every source row is a tap
    ("4k_to_1080p_nearest", 1080 * 3840 * 3, 1080 * 1920 * 3),     # the even rows only
    ("1080p_to_4k", 1080 * 1920 * 3, 2160 * 3840 * 3),
    ("4k_to_1080p_gray", 2160 * 3840 * 3, 1080 * 1920),            # one gray byte out per pixel
    # 720 -> 224: taps 3.2 rows apart, two distinct rows per output row
    ("batch64_720p_to_224_norm", 64 * 448 * 1280 * 3, 64 * 3 * 224 * 224 * 4),
    ("f32_8192_to_5980_filter3x3", 8192 * 8192 * 4, 5980 * 5980 * 4),
    # 2160 -> 768: taps 2.8 rows apart, two distinct rows per output row
    ("4k_to_1366x768", 2 * 768 * 3840 * 3, 768 * 1366 * 3),
    ("720p_to_1080p", 720 * 1280 * 3, 1080 * 1920 * 3),             # an upscale taps every row
])
def test_algorithmic_bytes_of_the_workloads(workload, read, write):
    # the roofline's numerator: source rows the taps read plus the output,
    # against counts worked out by hand from the geometry
    desc, kind, H, W, OH, OW, C, mode, batch = bench.WORKLOADS[workload]
    from bilinear_image_resize_gb300 import _build
    _build.build()
    assert bench.algorithmic_bytes(kind, H, W, OH, OW, C, mode, batch) == (read, write)


def test_clock_summary_reads_the_timed_window_and_reasons():
    # nvidia-smi lines (csv, no header, no units) in the sampler's field
    # order; only samples inside [t0, t1] count, and an "Active" throttle
    # field is reported by name
    s = bench.ClockSampler(0)

    def line(sm, hw="Not Active", thermal="Not Active", power="Not Active"):
        return f"2026/01/01 00:00:00.000, 0, {sm}, 2070, 900.0, 0x0, {hw}, {thermal}, Not Active, {power}"

    s.samples = [(0.5, line(600)), (1.0, line(2070)), (1.1, line(2055, power="Active")), (1.2, line(2070)),
                 (2.5, line(1000, hw="Active")), (1.3, "garbage")]
    got = s.summary(0.9, 1.3)
    assert got == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    assert s.summary(2.0, 3.0)["reasons"] == ["hw_slowdown"]
    assert s.summary(5.0, 6.0) == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_trimmed_mean_drops_a_tenth_at_each_end():
    # the Volcanic page's procedure: sort, drop 10% of the samples at each
    # end, average the rest
    xs = [5.0, 1.0, 100.0, 2.0, 3.0, 4.0, 6.0, 7.0, 8.0, 9.0]   # 10 samples: drop one at each end
    assert bench.trimmed_mean(xs) == sum(range(2, 10)) / 8
    assert bench.trimmed_mean([3.0]) == 3.0
    assert bench.trimmed_mean([1.0, 2.0]) == 1.5                  # nothing to drop
    assert bench.trimmed_mean([1.0, 2.0, 30.0], frac=0.4) == 2.0  # keeps the middle one
    ys = list(range(100))
    assert bench.trimmed_mean(ys) == sum(range(10, 90)) / 80
    with pytest.raises(ValueError):
        bench.trimmed_mean([])


def test_host_cpu_reports_cores_and_model():
    h = bench.host_cpu()
    assert h["cpu_count"] == os.cpu_count()
    assert isinstance(h["model"], str) and h["model"]


def test_filter_tc_flops_hand_count():
    # K = 64 on 4096^2: 127 x 32 tiles of 128 x 32 outputs, 3 chunks of 32
    # Toeplitz columns (32 + 63 = 95 <= 96), per filter row 3 products x 12
    # steps of 2 x 128 x 32 x 8 FLOPs
    assert bench.filter_tc_flops(64, 4033, 4033) == 127 * 32 * 64 * 3 * 12 * 2 * 128 * 32 * 8
    # K = 16: 32 + 15 = 47 -> 2 chunks
    assert bench.filter_tc_flops(16, 4081, 4081) == 128 * 32 * 16 * 3 * 8 * 2 * 128 * 32 * 8
    assert bench.FILTER_TC_MIN_K == 48
