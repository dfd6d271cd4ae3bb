"""Host-side logic of bench.py on the CPU: the reference arm's JSON line, the
algorithmic byte count, the roofline bound, and the rule that ties a stored
ncu traffic figure to the kernel source it was taken on."""

import hashlib
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _run_bench(args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)


def test_reference_arm_prints_one_contract_line():
    r = _run_bench(["--impl", "reference", "--steps", "3", "--warmup", "3"])
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 3 and d["warmup"] == 3
    assert d["value"] > 0 and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_are_silent():
    r = _run_bench(["--impl", "reference", "--steps", "3", "--warmup", "3"],
                   {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_warmup_below_three_is_refused():
    r = _run_bench(["--impl", "reference", "--steps", "3", "--warmup", "2"])
    assert r.returncode != 0


def test_gemm_bytes_counted_by_hand():
    import bench
    # dense 128 x 256 x 512: A 65536 + sA 128*4*4 + B 131072 + sB 2*4*4 + D 128*256*2
    assert bench.gemm_bytes(128, 256, 512) == 65536 + 2048 + 131072 + 32 + 65536
    # a partial last K block (K = 144) carries its own scale column
    assert bench.gemm_bytes(1, 128, 144) == 144 + 2 * 4 + 128 * 144 + 2 * 4 + 256
    # grouped: B and its scales once per active expert, A and D for the real rows
    assert bench.gemm_bytes(0, 256, 256, e_active=3, rows=10) == (
        10 * 256 + 10 * 2 * 4 + 3 * (256 * 256 + 2 * 2 * 4) + 10 * 256 * 2)


def test_roof_takes_the_slower_bound():
    import bench
    peaks = {"hbm_gbs": 1000.0, "bf16": 500.0, "bf16_sustained": 400.0, "source": "test"}
    # 1e12 FLOP at 800 TFLOP/s = 1.25 ms; 1e6 B at 1000 GB/s = 1 us: tensor-bound
    r = bench._roof(1e12, 1e6, 2.5, peaks, sustained=True)
    assert r["bound"] == "tensor" and r["roofline_frac"] == pytest.approx(0.5)
    # 1e9 FLOP at the burst-derived 1000 TFLOP/s (1 us) against 1e9 B (1 ms): HBM-bound
    r = bench._roof(1e9, 1e9, 4.0, peaks)
    assert r["bound"] == "hbm" and r["roofline_frac"] == pytest.approx(0.25)
    assert r["gbs"] == pytest.approx(250.0)


def test_traffic_figure_only_for_the_source_it_was_taken_on(tmp_path, monkeypatch):
    import bench
    csrc = tmp_path / "fp8_fine_grained_e4m3_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("kernel v1\n")
    digest = hashlib.sha256(b"kernel v1\n").hexdigest()[:16]
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(
        {"case": {"sources": ["k.cu"], "source_hash": digest, "dram_bytes_per_launch": 1234}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_from_profiles("case") == 1234
    assert bench.traffic_from_profiles("other") is None
    (csrc / "k.cu").write_text("kernel v2\n")
    assert bench.traffic_from_profiles("case") is None


def test_clock_summary_keeps_the_timed_window():
    """Only samples stamped inside the timed interval count; an idle sample
    before it (low clock) and a throttled one after it are left out."""
    import bench
    from datetime import datetime
    rows = [
        "2026/01/05 10:00:00.100, 0, 345, 2070, 120.5, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/01/05 10:00:00.210, 0, 2070, 2070, 900.1, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/01/05 10:00:00.220, 0, 2055, 2070, 910.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/01/05 10:00:00.230, 0, 2070, 2070, 905.2, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/01/05 10:00:00.400, 0, 1500, 2070, 1300.0, 0x20, Not Active, Active, Not Active, Not Active",
        "not a row",
    ]
    t = lambda s: datetime.strptime(s, "%Y/%m/%d %H:%M:%S.%f").timestamp()
    s = bench.ClockSampler.summarise("\n".join(rows), t("2026/01/05 10:00:00.200"),
                                     t("2026/01/05 10:00:00.300"))
    assert s["samples"] == 3 and s["samples_total"] == 5
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    # no sample inside a very short window: the whole record is summarised
    s = bench.ClockSampler.summarise("\n".join(rows), t("2026/01/05 10:00:00.300"),
                                     t("2026/01/05 10:00:00.301"))
    assert s["samples"] == 0 and s["samples_total"] == 5
    assert s["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


def test_end_to_end_gemm_parts_keep_whole_tile_waves():
    """The end-to-end step splits each shape's GEMM into row parts only as far
    as every part keeps a wave of whole 128 x 256 tiles (smaller parts would
    take the split-tile form, whose rounding differs from one call's)."""
    import bench
    assert bench.gemm_parts(4096, 7168, 4, 152) == 4   # 8 x 28 = 224 tiles per part
    assert bench.gemm_parts(4096, 4096, 4, 152) == 2   # 16 x 16 = 256; 4 parts: 128 < 152
    assert bench.gemm_parts(4096, 7168, 8, 152) == 4   # 8 parts: 4 x 28 = 112 < 152
    assert bench.gemm_parts(1024, 4096, 4, 152) == 1   # not even one wave: one call
    assert bench.gemm_parts(4096, 4096, 3, 152) == 3   # 1365 rows: 10 whole M blocks x 16 = 160
    assert bench.gemm_parts(4096, 4096, 3, 168) == 1   # 160 < 168; 2 does not divide 3 blocks
    for M, N, chunks, sms in [(4096, 7168, 4, 160), (8192, 4096, 8, 152), (4096, 4096, 4, 132)]:
        p = bench.gemm_parts(M, N, chunks, sms)
        assert chunks % p == 0
        assert p == 1 or (M // p) // 128 * -(-N // 256) >= sms


def test_clock_rows_summary_and_nvml_fallback():
    """The NVML sampler's rows go through the same window summary; where the
    management library cannot be loaded (no driver here) it declines, and the
    bench falls back to the nvidia-smi sampler."""
    import bench
    rows = [(1.0, 1500.0, 2070.0, []), (2.0, 2070.0, 2070.0, ["sw_power_cap"]),
            (2.5, 2055.0, 2070.0, []), (3.0, 2070.0, 2070.0, []), (9.0, 990.0, 2070.0, ["hw_slowdown"])]
    s = bench.summarise_clock_rows(rows, 1.9, 3.1)
    assert s["samples"] == 3 and s["samples_total"] == 5
    assert s["sm_mhz"] == 2070.0 and s["reasons"] == ["sw_power_cap"]
    s = bench.summarise_clock_rows(rows)
    assert s["samples"] == 0 and s["reasons"] == ["hw_slowdown", "sw_power_cap"]
    import ctypes.util
    if ctypes.util.find_library("nvidia-ml") is None:
        assert bench.NvmlClockSampler(0).start() is False
