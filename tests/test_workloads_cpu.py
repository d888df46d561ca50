"""CPU-only: the synthetic input recipe -- each workload's context lengths, pool size and
seeded value streams are what the design notes state (the lengths and the pool are drawn
on the host; the value streams are checked on the CPU generator)."""
import math

import numpy as np
import pytest

from paged_kv_cache_187_gb300 import workloads as W


def test_tiny_lengths_are_the_stated_ones():
    w = W.WORKLOADS["tiny"]
    assert W.start_context_lens(w).tolist() == [1, 17, 64, 100]
    assert W.pool_blocks(w, W.start_context_lens(w)) == 64


def test_l2_7b_lengths_uniform_in_range():
    w = W.WORKLOADS["l2_7b"]
    L = W.start_context_lens(w)
    assert L.size == 64 and L.min() >= 512 and L.max() <= 2048
    assert 1000 < L.mean() < 1560          # U[512, 2048] has mean 1280


def test_l3_8b_lengths_lognormal_clipped():
    w = W.WORKLOADS["l3_8b"]
    L = W.start_context_lens(w)
    assert L.size == 256 and L.min() >= 16 and L.max() <= 8192
    # lognormal(6.9, 0.8): median e^6.9 ~ 992, mean e^(6.9 + 0.32) ~ 1366
    assert 800 < np.median(L) < 1200 and 1100 < L.mean() < 1650
    # the seeded draw itself (the benchmark's batch: 316,832 context tokens)
    assert int(L.astype(np.int64).sum()) == 316_832
    assert np.array_equal(L, W.start_context_lens(w))          # deterministic


def test_skew_batch_composition():
    w = W.WORKLOADS["skew"]
    L = W.start_context_lens(w)
    assert sorted(set(L.tolist())) == [128, 32768]
    assert int((L == 32768).sum()) == 8 and int((L == 128).sum()) == 248
    assert int(L.astype(np.int64).sum()) == 293_888            # 8 x 32768 + 248 x 128
    assert w.partition_size == 512


def test_l3_70b_start_lengths_and_steps():
    w = W.WORKLOADS["l3_70b"]
    L = W.start_context_lens(w)
    # "start context_lens uniform in [1, 4096]", plus the first step's token
    assert L.size == 512 and L.min() >= 2 and L.max() <= 4097
    assert w.steps == 8 and w.block_size == 32 and w.group == 8


@pytest.mark.parametrize("name", ["l2_7b", "l3_8b", "skew", "l3_70b"])
def test_pool_holds_every_step_plus_ten_percent(name):
    w = W.WORKLOADS[name]
    L = W.start_context_lens(w).astype(np.int64)
    need = int(np.sum((L + w.steps - 1 + w.block_size - 1) // w.block_size))
    assert W.pool_blocks(w, L.astype(np.int32)) == math.ceil(need * 1.1)
    assert W.max_blocks_per_seq(w, L.astype(np.int32)) == \
        (int(L.max()) + w.steps - 1 + w.block_size - 1) // w.block_size


def test_value_streams_are_seeded_and_standard_normal():
    torch = pytest.importorskip("torch")
    a = W.randn_16bit((1 << 16,), "bf16", 123)
    b = W.randn_16bit((1 << 16,), "bf16", 123)
    c = W.randn_16bit((1 << 16,), "bf16", 124)
    assert a.dtype == torch.bfloat16 and torch.equal(a, b) and not torch.equal(a, c)
    x = a.float()
    assert abs(float(x.mean())) < 0.02 and abs(float(x.std()) - 1.0) < 0.02
    assert W.randn_16bit((8,), "f16", 1).dtype == torch.float16


def test_stream_seeds_are_distinct():
    w = W.WORKLOADS["l3_8b"]
    seeds = {W.stream_seed(w, s, step, rank) for s in ("q", "k_new", "v_new", "k_prefill",
                                                       "v_prefill")
             for step in range(8) for rank in range(8)}
    assert len(seeds) == 5 * 8 * 8


def test_poison_patterns_are_nans():
    import oracle
    for dt, bits in W.NAN_BITS.items():
        assert np.isnan(oracle.widen(np.array([bits], np.uint16), dt)[0])
