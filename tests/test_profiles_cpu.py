"""CPU-only: the committed ncu summaries agree with the workload they describe (the
algorithmic bytes of one decode launch) and were taken without touching the clocks."""
import glob
import os

import numpy as np

from paged_kv_cache_187_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _record(path):
    kv = {}
    with open(path) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
    return kv


def _algorithmic_bytes(name, kv_fp8, q_len):
    """K and V of every context token and kv head of the first decode step (one byte an
    element for fp8 pools, two otherwise), plus q_len query and output rows of 16 bits."""
    w = W.WORKLOADS[name]
    L = W.start_context_lens(w).astype(np.int64)
    elt = 1 if kv_fp8 else 2
    return (int(L.sum()) * w.num_kv_heads * w.head_size * 2 * elt +
            2 * q_len * w.num_seqs * w.num_q_heads * w.head_size * 2)


RECORDS = sorted(glob.glob(os.path.join(ROOT, "profiles", "*_traffic.txt")))


def test_every_workload_has_a_traffic_record():
    names = {os.path.basename(p)[:-len("_traffic.txt")] for p in RECORDS}
    assert {"paged_decode_l3_8b", "paged_decode_l2_7b", "paged_decode_skew",
            "paged_decode_l3_70b", "paged_decode_fp8_l3_8b", "paged_decode_fp8_l3_70b",
            "paged_decode_mq4_l3_8b", "paged_decode_mq4_l3_70b", "paged_decode_mq2_l3_8b"} <= names


def test_traffic_records_match_the_workload_bytes():
    import bench
    assert _algorithmic_bytes("l3_8b", False, 1) == 1_301_938_176
    for path in RECORDS:
        kv = _record(path)
        alg = _algorithmic_bytes(kv["workload"], kv["kv_fp8"] == "1", int(kv["q_len"]))
        assert int(kv["algorithmic_bytes_per_launch"]) == alg, path
        dram = int(kv["dram_bytes_read"]) + int(kv["dram_bytes_write"])
        assert int(float(kv["dram_bytes_per_launch"])) == dram, path
        assert 1.0 <= dram / alg < 1.05, path              # each K/V byte read about once
        assert abs(float(kv["traffic_over_algorithmic"]) - dram / alg) < 1e-3, path
        assert kv["family"] in bench.FAMILY_SOURCES, path
        assert len(kv["kernel_sources_sha256_16"]) == 16, path
        text = open(path).read()
        assert "--clock-control none" in text and "ncu --metrics" in text, path


def test_every_summary_names_its_command_and_leaves_the_clocks_alone():
    files = sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md")))
    assert files
    for path in files:
        text = open(path).read()
        assert "ncu " in text, path
        commands = [ln.strip() for ln in text.splitlines() if ln.strip().startswith("ncu --")]
        assert commands, path
        for line in commands:
            assert "--clock-control none" in line, (path, line)
