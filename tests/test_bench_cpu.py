"""CPU-only checks of bench.py's own arithmetic and bookkeeping: sample spreads, the
per-workload entry, the hash gate on committed ncu traffic records, the clock summary
over sampled nvidia-smi lines, and the CUDA -> nvidia-smi device index."""
import os
import shutil

import pytest

import bench


def test_spread_of_known_samples():
    s = bench._spread([0.3, 0.1, 0.2, 0.4])          # milliseconds
    assert s["n"] == 4
    assert s["mean_us"] == pytest.approx(250.0)
    assert s["median_us"] == pytest.approx(300.0)    # upper median of an even count
    assert s["min_us"] == pytest.approx(100.0) and s["max_us"] == pytest.approx(400.0)
    assert s["stdev_us"] == pytest.approx(111.80339887, rel=1e-9)
    assert bench._spread([0.5])["stdev_us"] == 0.0


def test_entry_turns_bytes_and_time_into_bandwidth():
    # 2 GB in 250 us -> 8000 GB/s: exactly the spec figure, and twice a 4000 GB/s peak
    e = bench._entry("w", "k", 2_000_000_000, 1_000_000, [0.25, 0.25], 4000.0)
    assert e["GBps"] == pytest.approx(8000.0)
    assert e["frac"] == pytest.approx(2.0)
    assert e["pct_of_spec_8000_GBps"] == pytest.approx(100.0)
    assert e["seq_tokens_per_s"] == pytest.approx(4e9)
    assert e["traffic"] is None                       # no record asked for
    assert bench._entry("w", "k", 1, 1, [1.0], 1.0, extra_key=3)["extra_key"] == 3


def _tree_with_record(tmp_path, name):
    """A copy of the sources and of one committed record under tmp_path."""
    root = tmp_path / "repo"
    shutil.copytree(os.path.join(bench.ROOT, "paged_kv_cache_187_gb300", "csrc"),
                    root / "paged_kv_cache_187_gb300" / "csrc")
    (root / "profiles").mkdir(parents=True)
    shutil.copy(os.path.join(bench.ROOT, "profiles", f"{name}_traffic.txt"), root / "profiles")
    return root


@pytest.mark.parametrize("name,family", [("paged_decode_l3_8b", "bf16_d128"),
                                         ("paged_decode_mq4_l3_8b", "mq_tc")])
def test_traffic_record_is_used_only_on_the_sources_it_was_taken_on(tmp_path, monkeypatch,
                                                                    name, family):
    root = _tree_with_record(tmp_path, name)
    monkeypatch.setattr(bench, "ROOT", str(root))
    text = (root / "profiles" / f"{name}_traffic.txt").read_text()
    recorded = [ln.split(":", 1)[1].strip() for ln in text.splitlines()
                if ln.startswith("dram_bytes_per_launch:")][0]
    hash_line = [ln for ln in text.splitlines() if ln.startswith("kernel_sources_sha256_16:")][0]
    # a record stamped with the present hash of its family is reported as is
    current = bench._kernel_hash(family)
    (root / "profiles" / f"{name}_traffic.txt").write_text(
        text.replace(hash_line, f"kernel_sources_sha256_16: {current}"))
    assert bench._traffic_record(name) == float(recorded)
    # a change to any source of the family (a comment counts) makes it stale
    src = root / "paged_kv_cache_187_gb300" / "csrc" / bench.FAMILY_SOURCES[family][-1]
    src.write_text(src.read_text() + "\n// edited\n")
    assert bench._kernel_hash(family) != current
    assert bench._traffic_record(name) is None
    # and a missing record is no record
    assert bench._traffic_record("paged_decode_no_such_workload") is None


def test_kernel_hash_tracks_the_family_sources_only(tmp_path, monkeypatch):
    root = _tree_with_record(tmp_path, "paged_decode_l3_8b")
    monkeypatch.setattr(bench, "ROOT", str(root))
    before = {f: bench._kernel_hash(f) for f in bench.FAMILY_SOURCES}
    fp8 = root / "paged_kv_cache_187_gb300" / "csrc" / "pa_decode_fp8.cu"
    fp8.write_text(fp8.read_text() + "\n")
    after = {f: bench._kernel_hash(f) for f in bench.FAMILY_SOURCES}
    assert after["fp8"] != before["fp8"]
    assert all(after[f] == before[f] for f in bench.FAMILY_SOURCES if f != "fp8")


def _sampler(rows):
    cs = bench.ClockSampler(0)
    # index, clocks.sm, clocks.max.sm, power.draw, active, hw_slowdown, hw_thermal,
    # sw_thermal, sw_power_cap
    cs.lines = [(t, ", ".join(str(x) for x in r)) for t, r in rows]
    return cs


def test_clock_summary_over_the_timed_region():
    quiet = ["0x0", "Not Active", "Not Active", "Not Active", "Not Active"]
    rows = [(float(t), [0, mhz, 2070, 900.0] + quiet) for t, mhz in
            ((1, 1500), (2, 2070), (3, 2070), (4, 2055), (5, 1400))]
    cs = _sampler(rows)
    cs.t_start, cs.t_stop = 1.5, 4.5
    s = cs.summary()
    assert s["window"] == "timed region" and s["samples"] == 3
    assert s["sm_mhz"] == 2070 and s["sm_min_mhz"] == 2055 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == []


def test_clock_summary_names_throttle_reasons_and_widens_a_short_window():
    busy = ["0x4", "Not Active", "Active", "Not Active", "Active"]
    rows = [(float(t), [0, 1800, 2070, 1390.0] + busy) for t in range(1, 6)]
    cs = _sampler(rows)
    cs.t_start, cs.t_stop = 2.9, 3.1          # one sample inside: too few to judge by
    s = cs.summary(phase=(1.0, 5.0))
    assert s["samples"] == 5 and "GPU measurement phase" in s["window"]
    assert s["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert bench.ClockSampler(0).summary()["reasons"] == ["no nvidia-smi samples"]


def test_nvidia_smi_index_follows_cuda_visible_devices(monkeypatch):
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "3,5")
    assert bench._smi_index(0) == "3" and bench._smi_index(1) == "5"
    monkeypatch.delenv("CUDA_VISIBLE_DEVICES")
    assert bench._smi_index(2) == "2"
