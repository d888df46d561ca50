"""CPU-only: the committed ncu summaries agree with the workload they describe (the
algorithmic bytes of one decode launch) and were taken without touching the clocks."""
import glob
import os

import numpy as np

from paged_kv_cache_187_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _record():
    kv = {}
    with open(os.path.join(ROOT, "profiles", "paged_decode_l3_8b_traffic.txt")) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
    return kv


def test_traffic_record_matches_the_workload_bytes():
    kv = _record()
    w = W.WORKLOADS["l3_8b"]
    L = W.start_context_lens(w).astype(np.int64)
    # K and V of every context token and kv head, plus the query and output rows
    alg = int(L.sum()) * w.num_kv_heads * w.head_size * 2 * 2 + \
        2 * w.num_seqs * w.num_q_heads * w.head_size * 2
    assert int(kv["algorithmic_bytes_per_launch"]) == alg == 1_301_938_176
    dram = int(kv["dram_bytes_read"]) + int(kv["dram_bytes_write"])
    assert int(float(kv["dram_bytes_per_launch"])) == dram
    assert 1.0 <= dram / alg < 1.05                      # each K/V byte read about once
    assert abs(float(kv["traffic_over_algorithmic"]) - dram / alg) < 1e-3
    assert len(kv["kernel_sources_sha256_16"]) == 16


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
