"""The test-side fan-out of the oracle over host threads (oracle_side.fan_out) gives the
same doubles as one single-threaded call: the ranges cover every sequence once, in
order, and concurrent calls into the oracle share nothing mutable."""
import numpy as np

import oracle
from oracle_side import ErrStats, err_stats, fan_out, seq_ranges


def _batch(lens, Hq, Hkv, D, bs, seed):
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, np.int32)
    S = lens.size
    nb = int(np.sum((lens + bs - 1) // bs)) + 2
    kc = oracle.round_to(rng.standard_normal((nb, Hkv, bs, D)), "bf16")
    vc = oracle.round_to(rng.standard_normal((nb, Hkv, bs, D)), "bf16")
    al = oracle.Alloc(nb, bs, seed)
    for s, L in enumerate(lens):
        al.add_seq(s, int(L))
    bt = al.block_tables(np.arange(S), int((lens.max() + bs - 1) // bs))
    q = oracle.round_to(rng.standard_normal((S, Hq, D)), "bf16")
    return q, kc, vc, bt, lens


def test_seq_ranges_cover_every_sequence_once_in_order():
    rng = np.random.default_rng(3)
    for S in (1, 2, 7, 64, 257):
        lens = rng.integers(0, 5000, size=S)
        for parts in (1, 3, 16, 64, 1000):
            r = seq_ranges(lens, parts)
            assert r[0][0] == 0 and r[-1][1] == S
            assert all(a < b for a, b in r) and all(r[i][1] == r[i + 1][0] for i in range(len(r) - 1))
            assert len(r) <= min(parts, S)


def test_fan_out_equals_one_call_bit_for_bit():
    rng = np.random.default_rng(4)
    lens = rng.integers(1, 300, size=37).astype(np.int32)
    lens[5] = 0
    q, kc, vc, bt, lens = _batch(lens, 8, 2, 32, 16, seed=9)
    scale = np.float32(32 ** -0.5)
    one = oracle.decode_v1(q, kc, vc, bt, lens, scale, "bf16")
    many = fan_out(lambda a, b: oracle.decode_v1(q[a:b], kc, vc, bt[a:b], lens[a:b], scale,
                                                 "bf16"), lens)
    assert np.array_equal(one, many)
    one_v2 = oracle.decode_v2(q, kc, vc, bt, lens, scale, "bf16", 48)
    many_v2 = fan_out(lambda a, b: oracle.decode_v2(q[a:b], kc, vc, bt[a:b], lens[a:b], scale,
                                                    "bf16", 48), lens)
    assert np.array_equal(one_v2, many_v2)
    qm = oracle.round_to(rng.standard_normal((lens.size, 3, 8, 32)), "bf16")
    one_mq = oracle.decode_mq(qm, kc, vc, bt, lens, scale, "bf16")
    many_mq = fan_out(lambda a, b: oracle.decode_mq(qm[a:b], kc, vc, bt[a:b], lens[a:b], scale,
                                                    "bf16"), lens)
    assert np.array_equal(one_mq, many_mq)


def test_err_stats_counts_the_elements_admitted_by_the_ulp_allowance():
    # bf16 outputs: 0.5 (ulp 2^-8 < 1e-2) and 3.0 (ulp 2^-6 > 1e-2)
    ref = np.array([[0.5, 3.0, 3.0, -3.0]])
    gpu = oracle.round_to(np.array([[0.5 + 2 ** -8, 3.0 + 2 ** -6, 3.0, -3.0 - 2 ** -6]]), "bf16")
    e = err_stats(gpu, ref, "bf16")
    assert isinstance(e, ErrStats) and e.n == 4 and e.n_ulp == 2
    assert abs(e.err - 1e-2) < 1e-12 and e.max_abs == 2 ** -6
    assert e.ok("bf16", max_ulp_frac=0.5)
    # the cap: at least 2 elements, else max_ulp_frac of them, may need the allowance
    ref3 = np.full((1, 6), 3.0)
    three = oracle.round_to(np.array([[3.0 + 2 ** -6] * 3 + [3.0] * 3]), "bf16")
    e3 = err_stats(three, ref3, "bf16")
    assert e3.n_ulp == 3 and e3.err <= 1e-2 + 1e-12
    assert e3.ok("bf16", max_ulp_frac=0.5) and not e3.ok("bf16", max_ulp_frac=0.0)
    # two ulps at 3.0 fail the gate
    bad = oracle.round_to(np.array([[0.5, 3.0 + 2 ** -5, 3.0, 3.0]]), "bf16")
    assert not err_stats(bad, ref, "bf16").ok("bf16")
    # a NaN fails
    nan = oracle.round_to(np.array([[np.nan, 3.0, 3.0, 3.0]]), "bf16")
    assert err_stats(nan, ref, "bf16").err == float("inf")
