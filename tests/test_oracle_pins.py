"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each test names what fixes the expected value: a library routine (numpy's binary16
casts, torch's bfloat16 casts, scipy's softmax on a contiguous KV copy), a closed
form, an invariant of the method, a published test vector, or a figure the pages
print.  Together they are chosen so that a plausible slip in the oracle (a wrong
block-table index, a transposed GQA mapping, a dropped LSE term, a wrong scale, a
double rounding) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------- conversions
def test_f16_widen_matches_numpy_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle.widen(bits, "f16")
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_bf16_widen_matches_torch_all_patterns():
    torch = pytest.importorskip("torch")
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle.widen(bits, "bf16")
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def _spread_doubles(n, seed):
    rng = np.random.default_rng(seed)
    mant = rng.random(n) + 1.0
    expo = rng.integers(-30, 20, size=n)
    x = np.ldexp(mant, expo) * rng.choice([-1.0, 1.0], size=n)
    return np.concatenate([x, [0.0, -0.0, 65504.0, 65519.9, 65520.0, 1e6, -1e6,
                               2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -14 * (1 - 2 ** -11)]])


def test_f16_rounding_matches_numpy():
    # numpy's float64 -> float16 cast rounds the double directly, ties to even.
    x = _spread_doubles(200_000, 1)
    ours = oracle.round_to(x, "f16")
    ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_rounding_matches_torch_on_float_inputs():
    torch = pytest.importorskip("torch")
    # For values exact in fp32, torch's fp32 -> bf16 cast (ties to even) is a single
    # rounding, so it is a valid reference.
    x = _spread_doubles(200_000, 2).astype(np.float32).astype(np.float64)
    ours = oracle.round_to(x, "bf16")
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(ours, ref.view(np.uint16))


def test_bf16_rounding_is_single_rounding_of_the_double():
    # Closed-form cases that a double -> float -> bf16 route would get wrong.
    cases = [
        (1.0 + 2.0 ** -8, 0x3F80),                 # exact tie -> even (1.0)
        (1.0 + 2.0 ** -8 + 2.0 ** -40, 0x3F81),    # just above the tie -> up
        (1.0 + 3 * 2.0 ** -8, 0x3F82),             # tie with odd lower neighbour -> up
        (1.0 + 3 * 2.0 ** -8 - 2.0 ** -40, 0x3F81),
        (-2.0, 0xC000),
        (3.0e38 * 1.2, 0x7F80),                    # overflow -> inf
    ]
    for x, bits in cases:
        assert int(oracle.round_to(np.array([x]), "bf16")[0]) == bits, x


# --------------------------------------------------------------------------- splitmix64
def test_splitmix64_published_outputs():
    with open(os.path.join(GOLDEN, "splitmix64_seed0.txt")) as f:
        want = [int(line, 16) for line in f if line.strip() and not line.startswith("#")]
    assert oracle.splitmix64_stream(0, len(want)) == want


# --------------------------------------------------------------------------- helpers
def _paged_batch(lens, Hq, Hkv, D, bs, dtype, seed, alloc_seed, extra_blocks=3):
    """Contiguous per-sequence K/V plus the same data scattered into a NaN-poisoned
    paged pool by the oracle allocator and the oracle's reshape_and_cache."""
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, dtype=np.int32)
    S = lens.size
    nb = int(sum((int(L) + bs - 1) // bs for L in lens)) + extra_blocks
    maxb = max(1, max((int(L) + bs - 1) // bs for L in lens))

    def draw(shape):
        return oracle.round_to(rng.standard_normal(shape), dtype)

    q = draw((S, Hq, D))
    kv = [(draw((int(L), Hkv, D)), draw((int(L), Hkv, D))) for L in lens]
    nan = 0x7E00 if dtype == "f16" else 0x7FC0
    kc = np.full((nb, Hkv, bs, D), nan, dtype=np.uint16)
    vc = np.full((nb, Hkv, bs, D), nan, dtype=np.uint16)
    al = oracle.Alloc(nb, bs, alloc_seed)
    for s, L in enumerate(lens):
        al.add_seq(s, int(L))
        slots = al.slots(s, 0, int(L))
        assert oracle.reshape_and_cache(kv[s][0], kv[s][1], kc, vc, slots, bs) == 0
    bt = al.block_tables(np.arange(S), maxb)
    return q, kv, kc, vc, bt, lens


def _dense_reference(q, kv, lens, Hq, Hkv, scale, dtype):
    """Softmax attention over the contiguous copy, by numpy + scipy.special.softmax."""
    g = Hq // Hkv
    out = []
    for s, L in enumerate(lens):
        qs = oracle.widen(q[s], dtype)                          # [Hq, D]
        k = oracle.widen(kv[s][0], dtype)                      # [L, Hkv, D]
        v = oracle.widen(kv[s][1], dtype)
        k = np.repeat(k, g, axis=1)                            # [L, Hq, D], head h -> kv h//g
        v = np.repeat(v, g, axis=1)
        if L == 0:
            out.append(np.zeros_like(qs))
            continue
        logits = np.einsum("hd,thd->ht", qs, k) * scale
        p = scipy.special.softmax(logits, axis=1)
        out.append(np.einsum("ht,thd->hd", p, v))
    return np.stack(out)


CASES = [
    # lens, Hq, Hkv, D, bs, dtype
    ([1, 17, 64, 100], 4, 4, 64, 16, "f16"),
    ([5, 33, 16, 15, 47], 8, 2, 32, 8, "bf16"),
    ([40, 1, 31, 32, 33], 8, 1, 16, 16, "f16"),
    ([70, 65], 6, 3, 24, 32, "bf16"),
]


@pytest.mark.parametrize("lens,Hq,Hkv,D,bs,dtype", CASES)
def test_v1_equals_dense_bruteforce(lens, Hq, Hkv, D, bs, dtype):
    scale = np.float32(1.0 / math.sqrt(D))
    q, kv, kc, vc, bt, lens = _paged_batch(lens, Hq, Hkv, D, bs, dtype, seed=7, alloc_seed=11)
    got = oracle.decode_v1(q, kc, vc, bt, lens, scale, dtype)
    ref = _dense_reference(q, kv, lens, Hq, Hkv, float(scale), dtype)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("lens,Hq,Hkv,D,bs,dtype", CASES)
def test_block_placement_invariance(lens, Hq, Hkv, D, bs, dtype):
    scale = np.float32(1.0 / math.sqrt(D))
    a = _paged_batch(lens, Hq, Hkv, D, bs, dtype, seed=7, alloc_seed=11)
    b = _paged_batch(lens, Hq, Hkv, D, bs, dtype, seed=7, alloc_seed=12345, extra_blocks=9)
    assert not np.array_equal(a[4], b[4][:, :a[4].shape[1]]) or len(lens) == 0
    oa = oracle.decode_v1(a[0], a[2], a[3], a[4], a[5], scale, dtype)
    ob = oracle.decode_v1(b[0], b[2], b[3], b[4], b[5], scale, dtype)
    assert np.array_equal(oa, ob)


def test_context_len_one_returns_that_v_row():
    D, bs = 64, 16
    q, kv, kc, vc, bt, lens = _paged_batch([1, 1, 1], 4, 2, D, bs, "bf16", seed=3, alloc_seed=5)
    got = oracle.decode_v1(q, kc, vc, bt, lens, np.float32(0.125), "bf16")
    for s in range(3):
        v0 = oracle.widen(kv[s][1][0], "bf16")              # [Hkv, D]
        assert np.array_equal(got[s], np.repeat(v0, 2, axis=0))


def test_identical_keys_give_mean_of_v():
    D, bs, L = 32, 16, 45
    q, kv, kc, vc, bt, lens = _paged_batch([L], 2, 1, D, bs, "f16", seed=4, alloc_seed=6)
    kv[0][0][:] = kv[0][0][0]                               # every key equal to the first
    kc[:] = 0x7E00
    vc[:] = 0x7E00
    al = oracle.Alloc(kc.shape[0], bs, 6)
    al.add_seq(0, L)
    oracle.reshape_and_cache(kv[0][0], kv[0][1], kc, vc, al.slots(0, 0, L), bs)
    bt = al.block_tables([0], bt.shape[1])
    got = oracle.decode_v1(q, kc, vc, bt, lens, np.float32(0.3), "f16")
    mean_v = oracle.widen(kv[0][1], "f16").mean(axis=0)     # [Hkv, D]
    np.testing.assert_allclose(got[0], np.repeat(mean_v, 2, axis=0), rtol=1e-13, atol=1e-14)


def test_scale_zero_gives_mean_of_v():
    q, kv, kc, vc, bt, lens = _paged_batch([9, 30], 4, 4, 16, 8, "f16", seed=8, alloc_seed=9)
    got = oracle.decode_v1(q, kc, vc, bt, lens, np.float32(0.0), "f16")
    for s, L in enumerate(lens):
        np.testing.assert_allclose(got[s], oracle.widen(kv[s][1], "f16").mean(axis=0),
                                   rtol=1e-13, atol=1e-14)


def test_dominant_key_selects_its_value_row():
    D, bs, L = 16, 8, 20
    q, kv, kc, vc, bt, lens = _paged_batch([L], 1, 1, D, bs, "f16", seed=10, alloc_seed=2)
    qv = np.zeros(D)
    qv[0] = 1.0
    q[0, 0] = oracle.round_to(qv, "f16")
    k = np.zeros((L, 1, D))
    k[13, 0, 0] = 64.0                                      # logit 64 * scale vs 0 elsewhere
    kv[0] = (oracle.round_to(k, "f16"), kv[0][1])
    kc[:] = 0
    al = oracle.Alloc(kc.shape[0], bs, 2)
    al.add_seq(0, L)
    oracle.reshape_and_cache(kv[0][0], kv[0][1], kc, vc, al.slots(0, 0, L), bs)
    got = oracle.decode_v1(q, kc, vc, al.block_tables([0], bt.shape[1]), lens,
                           np.float32(1.0), "f16")
    v = oracle.widen(kv[0][1][:, 0], "f16")
    # weight of every other token is exp(-64) / (1 + 19 exp(-64)) < 2e-27
    np.testing.assert_allclose(got[0, 0], v[13], rtol=0, atol=1e-25)


def test_empty_context_gives_zeros():
    q, kv, kc, vc, bt, lens = _paged_batch([0, 3], 2, 2, 8, 8, "bf16", seed=1, alloc_seed=1)
    got = oracle.decode_v1(q, kc, vc, bt, lens, np.float32(0.5), "bf16")
    assert np.all(got[0] == 0.0)
    assert np.all(np.isfinite(got[1]))


@pytest.mark.parametrize("lens,Hq,Hkv,D,bs,dtype", CASES)
def test_v2_equals_v1(lens, Hq, Hkv, D, bs, dtype):
    scale = np.float32(1.0 / math.sqrt(D))
    q, kv, kc, vc, bt, lens = _paged_batch(lens, Hq, Hkv, D, bs, dtype, seed=21, alloc_seed=22)
    v1 = oracle.decode_v1(q, kc, vc, bt, lens, scale, dtype)
    for P in (bs, 2 * bs, 512, int(max(lens)) + 1):
        v2 = oracle.decode_v2(q, kc, vc, bt, lens, scale, dtype, P)
        np.testing.assert_allclose(v2, v1, rtol=1e-12, atol=1e-13)


def test_only_mask_computes_selected_rows():
    q, kv, kc, vc, bt, lens = _paged_batch([10, 20, 30], 4, 2, 16, 8, "f16", seed=2, alloc_seed=3)
    full = oracle.decode_v1(q, kc, vc, bt, lens, np.float32(0.25), "f16")
    only = np.zeros((3, 4), dtype=np.uint8)
    only[1, 2] = only[2, 0] = 1
    part = oracle.decode_v1(q, kc, vc, bt, lens, np.float32(0.25), "f16", only=only)
    assert np.array_equal(part[1, 2], full[1, 2]) and np.array_equal(part[2, 0], full[2, 0])
    assert np.all(part[0] == 0)


# --------------------------------------------------------------------------- reshape_and_cache
def test_reshape_and_cache_matches_numpy_scatter():
    rng = np.random.default_rng(0)
    NB, Hkv, bs, D, T = 9, 3, 8, 16, 20
    key = rng.integers(0, 1 << 16, size=(T, Hkv, D), dtype=np.uint16)
    val = rng.integers(0, 1 << 16, size=(T, Hkv, D), dtype=np.uint16)
    slots = rng.permutation(NB * bs)[:T].astype(np.int32)
    slots[[3, 11]] = -1                                        # padding tokens
    kc = rng.integers(0, 1 << 16, size=(NB, Hkv, bs, D), dtype=np.uint16)
    vc = kc.copy()
    ref_k, ref_v = kc.copy(), vc.copy()
    keep = slots >= 0
    ref_k[slots[keep] // bs, :, slots[keep] % bs, :] = key[keep]
    ref_v[slots[keep] // bs, :, slots[keep] % bs, :] = val[keep]
    assert oracle.reshape_and_cache(key, val, kc, vc, slots, bs) == 0
    assert np.array_equal(kc, ref_k) and np.array_equal(vc, ref_v)


def test_reshape_and_cache_skips_out_of_range_slots():
    NB, Hkv, bs, D = 2, 1, 4, 8
    kc = np.zeros((NB, Hkv, bs, D), dtype=np.uint16)
    vc = kc.copy()
    key = np.ones((2, Hkv, D), dtype=np.uint16)
    bad = oracle.reshape_and_cache(key, key, kc, vc, np.array([NB * bs, 1], np.int32), bs)
    assert bad == 1
    assert kc.sum() == D and kc[0, 0, 1].tolist() == [1] * D


# --------------------------------------------------------------------------- allocator
def test_allocator_invariants():
    NB, bs = 50, 16
    al = oracle.Alloc(NB, bs, seed=99)
    lens = [1, 16, 17, 100, 0]
    for s, L in enumerate(lens):
        al.add_seq(s, L)
    used = sum((L + bs - 1) // bs for L in lens)
    assert al.num_free == NB - used
    bt = al.block_tables(np.arange(5), 8)
    ids = bt[bt >= 0]
    assert len(set(ids.tolist())) == ids.size == used
    assert np.all((ids >= 0) & (ids < NB))
    # slots = block * bs + offset, unique over the whole pool
    all_slots = np.concatenate([al.slots(s, 0, L) for s, L in enumerate(lens)])
    assert len(set(all_slots.tolist())) == all_slots.size
    for s, L in enumerate(lens):
        sl = al.slots(s, 0, L)
        t = np.arange(L)
        assert np.array_equal(sl, bt[s, t // bs] * bs + t % bs)
    # append crosses a block boundary exactly at multiples of bs
    before = al.num_free
    slot = al.append(1)                                  # len 16 -> 17 pops a block
    assert al.num_free == before - 1 and slot == al.block_tables([1], 8)[0, 1] * bs
    slot = al.append(2)                                  # len 17 -> 18 pops nothing
    assert al.num_free == before - 1 and slot % bs == 1
    assert list(al.context_lens([0, 1, 2, 3, 4])) == [1, 17, 18, 100, 0]


def test_allocator_oom_changes_nothing_and_free_reuses():
    al = oracle.Alloc(4, 8, seed=1)
    al.add_seq(0, 24)                                    # 3 blocks
    with pytest.raises(oracle.OracleAllocError):
        al.add_seq(1, 9)                                 # needs 2, 1 free
    assert al.num_free == 1
    al.add_seq(1, 8)
    with pytest.raises(oracle.OracleAllocError):
        al.append(1)                                     # len 8 -> new block, none free
    assert al.num_free == 0 and list(al.context_lens([1])) == [8]
    blocks0 = al.block_tables([0], 3)[0].tolist()
    al.free_seq(0)
    assert al.num_free == 3
    al.add_seq(2, 8)                                     # pops the last pushed block
    assert al.block_tables([2], 1)[0, 0] == blocks0[-1]


def test_allocator_is_a_seeded_permutation():
    a = oracle.Alloc(64, 16, seed=5)
    b = oracle.Alloc(64, 16, seed=5)
    c = oracle.Alloc(64, 16, seed=6)
    for x in (a, b, c):
        x.add_seq(0, 64 * 16)
    ta, tb, tc = (x.block_tables([0], 64)[0] for x in (a, b, c))
    assert np.array_equal(ta, tb) and not np.array_equal(ta, tc)
    assert sorted(ta.tolist()) == list(range(64))
    # Fisher-Yates with splitmix64: the first block popped is the entry swapped into the
    # last position, i.e. index r0 % 64 of the identity.
    r0 = oracle.splitmix64_stream(5, 1)[0]
    assert ta[0] == r0 % 64


# --------------------------------------------------------------------------- byte accounting
def test_kv_bytes_per_token_matches_the_quoted_llama13b_figure():
    vals = {}
    with open(os.path.join(GOLDEN, "llama13b_kv_bytes.txt")) as f:
        for line in f:
            if "=" in line and not line.startswith("#"):
                k, v = line.split("=")
                vals[k.strip()] = float(v)
    # one token of one layer occupies one row of the K pool and one of the V pool
    per_token_layer = 2 * vals["kv_heads"] * vals["head_size"] * vals["elem_bytes"]
    per_seq = per_token_layer * vals["layers"] * vals["max_context"]
    assert per_token_layer == 20480
    assert abs(per_seq - vals["quoted_bytes_per_sequence"]) / vals["quoted_bytes_per_sequence"] < 0.02


def test_allocator_reserve_then_appends_pop_nothing():
    bs = 8
    al = oracle.Alloc(20, bs, seed=3)
    al.add_seq(0, 7)                                     # 1 block
    al.reserve(0, 10)                                    # 7 + 10 = 17 tokens -> 3 blocks
    assert al.num_free == 17
    table = al.block_tables([0], 3)[0]
    assert (table >= 0).all()
    for i in range(10):                                  # positions 7 .. 16
        slot = al.append(0)
        pos = 7 + i
        assert slot == table[pos // bs] * bs + pos % bs
    assert al.num_free == 17
    al.append(0)                                         # position 17: still block 2
    assert al.num_free == 17
    for _ in range(7):                                   # positions 18 .. 24 -> block 3 popped
        al.append(0)
    assert al.num_free == 16


# --------------------------------------------------------------------------- shared prefixes
def test_fork_shares_blocks_and_copy_on_write_keeps_the_parent_intact():
    bs = 8
    al = oracle.Alloc(32, bs, seed=9)
    al.add_seq(0, 20)                                    # blocks b0 b1 b2 (b2 partial: 4 rows)
    parent = al.block_tables([0], 3)[0].copy()
    free0 = al.num_free
    al.fork(0, 1, 20)                                    # child shares all three
    assert al.num_free == free0
    assert np.array_equal(al.block_tables([1], 3)[0], parent)
    assert [al.refcount(int(b)) for b in parent] == [2, 2, 2]
    slot = al.append(1)                                  # position 20 lands in shared b2 -> COW
    child = al.block_tables([1], 3)[0]
    assert np.array_equal(child[:2], parent[:2]) and child[2] != parent[2]
    assert al.refcount(int(parent[2])) == 1 and al.refcount(int(child[2])) == 1
    assert slot == child[2] * bs + 4
    assert al.take_copies().tolist() == [[int(parent[2]), int(child[2])]]
    assert al.take_copies().shape == (0, 2)
    assert np.array_equal(al.block_tables([0], 3)[0], parent)        # parent untouched
    al.append(0)                                         # parent's b2 is private again: no COW
    assert al.take_copies().shape == (0, 2)
    al.fork(0, 2, 16)                                    # block-aligned prefix: b0 b1 only
    al.append(2)                                         # position 16 needs a fresh block
    assert al.take_copies().shape == (0, 2)
    for s in (0, 1, 2):
        al.free_seq(s)
    assert al.num_free == 32                             # every block back exactly once


def test_decode_over_a_fork_equals_dense_attention_over_its_tokens():
    D, bs, Hq, Hkv = 16, 8, 4, 2
    rng = np.random.default_rng(12)
    draw = lambda shape: oracle.round_to(rng.standard_normal(shape), "f16")
    nb = 16
    kc = np.full((nb, Hkv, bs, D), 0x7E00, np.uint16)
    vc = kc.copy()
    al = oracle.Alloc(nb, bs, seed=4)
    prefix_k, prefix_v = draw((13, Hkv, D)), draw((13, Hkv, D))
    al.add_seq(0, 13)
    oracle.reshape_and_cache(prefix_k, prefix_v, kc, vc, al.slots(0, 0, 13), bs)
    al.fork(0, 1, 11)                                    # child keeps 11 prefix tokens
    own_k, own_v = draw((5, Hkv, D)), draw((5, Hkv, D))
    slots = np.array([al.append(1) for _ in range(5)], np.int32)
    pairs = al.take_copies()
    assert pairs.shape == (1, 2)                         # block 1 (rows 8..12) was shared
    oracle.copy_blocks(kc, vc, pairs)
    oracle.reshape_and_cache(own_k, own_v, kc, vc, slots, bs)
    q = draw((2, Hq, D))
    bt = al.block_tables([0, 1], 3)
    lens = np.array([13, 16], np.int32)
    got = oracle.decode_v1(q, kc, vc, bt, lens, np.float32(0.25), "f16")
    kv = [(prefix_k, prefix_v),
          (np.concatenate([prefix_k[:11], own_k]), np.concatenate([prefix_v[:11], own_v]))]
    ref = _dense_reference(q, kv, lens, Hq, Hkv, 0.25, "f16")
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------- fp8 E4M3
def test_e4m3_widen_matches_torch_all_patterns():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    bits = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_widen(bits)
    ref = torch.from_numpy(bits).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan) and nan.sum() == 2
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9


def test_e4m3_rounding_matches_torch_in_range_and_saturates_beyond():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    rng = np.random.default_rng(5)
    x = np.ldexp(rng.random(100_000) + 1.0, rng.integers(-12, 9, size=100_000))
    x *= rng.choice([-1.0, 1.0], size=x.size)
    x = x[np.abs(x) < 464.0].astype(np.float32).astype(np.float64)   # below the overflow tie
    ours = oracle.e4m3_round(x)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)
    # closed forms: ties to even, saturation, NaN
    cases = [(1.0 + 1 / 16, 0x38), (1.0 + 3 / 16, 0x3A), (448.0, 0x7E), (460.0, 0x7E),
             (1e6, 0x7E), (-1e6, 0xFE), (2.0 ** -10, 0x00), (3 * 2.0 ** -10, 0x02), (3 * 2.0 ** -11, 0x01)]
    for v, b in cases:
        assert int(oracle.e4m3_round(np.array([v]))[0]) == b, v
    assert int(oracle.e4m3_round(np.array([np.nan]))[0]) & 0x7F == 0x7F


def test_fp8_cache_decode_equals_dense_attention_over_dequantised_values():
    D, bs, Hq, Hkv = 32, 16, 8, 2
    rng = np.random.default_rng(19)
    lens = np.array([3, 16, 40], np.int32)
    S = lens.size
    nb = 8
    ks, vs = np.float32(0.07), np.float32(0.05)
    k16 = [oracle.round_to(rng.standard_normal((int(L), Hkv, D)), "bf16") for L in lens]
    v16 = [oracle.round_to(rng.standard_normal((int(L), Hkv, D)), "bf16") for L in lens]
    kc = np.zeros((nb, Hkv, bs, D), np.uint8)
    vc = kc.copy()
    al = oracle.Alloc(nb, bs, 2)
    for s, L in enumerate(lens):
        al.add_seq(s, int(L))
        assert oracle.reshape_and_cache_fp8(k16[s], v16[s], kc, vc, al.slots(s, 0, int(L)), bs,
                                            "bf16", ks, vs) == 0
    bt = al.block_tables(np.arange(S), 3)
    q = oracle.round_to(rng.standard_normal((S, Hq, D)), "bf16")
    got = oracle.decode_fp8(q, kc, vc, bt, lens, np.float32(D ** -0.5), ks, vs, "bf16")
    # dense reference on the dequantised contiguous rows: e4m3(x * (1/scale)) * scale
    inv_k, inv_v = np.float32(1) / ks, np.float32(1) / vs
    def deq(x16, inv, sc):
        xf = oracle.widen(x16, "bf16").astype(np.float32)
        return oracle.e4m3_widen(oracle.e4m3_round((xf * inv).astype(np.float64))) * float(sc)
    g = Hq // Hkv
    for s, L in enumerate(lens):
        k = np.repeat(deq(k16[s], inv_k, ks), g, axis=1)
        v = np.repeat(deq(v16[s], inv_v, vs), g, axis=1)
        logits = np.einsum("hd,thd->ht", oracle.widen(q[s], "bf16"), k) * float(np.float32(D ** -0.5))
        p = scipy.special.softmax(logits, axis=1)
        np.testing.assert_allclose(got[s], np.einsum("ht,thd->hd", p, v), rtol=1e-12, atol=1e-13)


def test_fp8_decode_context_past_its_table_row_reads_zeros_and_flags():
    """A context longer than its block-table row: the tokens past the row have no block,
    so they read as zeros (logit 0, no V contribution) and the call is flagged -- the
    same reading as the 16-bit decode and the GPU (an out-of-pool tile reads as zeros).
    The entry that physically follows the row belongs to the next sequence and points at
    a NaN-poisoned block; reading it would turn the output into NaN."""
    D, bs, Hq, Hkv = 32, 16, 4, 2
    rng = np.random.default_rng(23)
    ks, vs = np.float32(0.05), np.float32(0.04)
    nb = 3
    kc = np.full((nb, Hkv, bs, D), 0x7F, np.uint8)     # E4M3 NaN everywhere
    vc = kc.copy()
    k16 = oracle.round_to(rng.standard_normal((bs, Hkv, D)), "f16")
    v16 = oracle.round_to(rng.standard_normal((bs, Hkv, D)), "f16")
    slots = np.arange(2 * bs, 3 * bs, dtype=np.int32)  # block 2 holds sequence 0's 16 tokens
    assert oracle.reshape_and_cache_fp8(k16, v16, kc, vc, slots, bs, "f16", ks, vs) == 0
    bt = np.array([[2], [0]], np.int32)                # one block per row; block 0 is poison
    lens = np.array([bs + 3, 0], np.int32)             # 3 tokens past sequence 0's row
    q = oracle.round_to(rng.standard_normal((2, Hq, D)), "f16")
    scale = np.float32(D ** -0.5)
    got, flagged = oracle.decode_fp8(q, kc, vc, bt, lens, scale, ks, vs, "f16", strict=False)
    assert flagged and np.all(np.isfinite(got))
    with pytest.raises(IndexError):
        oracle.decode_fp8(q, kc, vc, bt, lens, scale, ks, vs, "f16")
    inv_k, inv_v = np.float32(1) / ks, np.float32(1) / vs
    def deq(x16, inv, sc):
        xf = oracle.widen(x16, "f16").astype(np.float32)
        return oracle.e4m3_widen(oracle.e4m3_round((xf * inv).astype(np.float64))) * float(sc)
    g = Hq // Hkv
    k = np.concatenate([np.repeat(deq(k16, inv_k, ks), g, axis=1), np.zeros((3, Hq, D))])
    v = np.concatenate([np.repeat(deq(v16, inv_v, vs), g, axis=1), np.zeros((3, Hq, D))])
    logits = np.einsum("hd,thd->ht", oracle.widen(q[0], "f16"), k) * float(scale)
    ref = np.einsum("ht,thd->hd", scipy.special.softmax(logits, axis=1), v)
    np.testing.assert_allclose(got[0], ref, rtol=1e-12, atol=1e-13)
    assert np.all(got[1] == 0)                         # empty context: zero rows


# --------------------------------------------------------------------------- multi-query
def test_multi_query_rows_equal_single_query_decodes_over_their_prefixes():
    D, bs, Hq, Hkv, QL = 16, 8, 4, 2, 3
    lens = np.array([3, 10, 17], np.int32)
    q_single, kv, kc, vc, bt, lens = _paged_batch(lens, Hq, Hkv, D, bs, "bf16", seed=40,
                                                  alloc_seed=41)
    rng = np.random.default_rng(42)
    q = oracle.round_to(rng.standard_normal((lens.size, QL, Hq, D)), "bf16")
    got = oracle.decode_mq(q, kc, vc, bt, lens, np.float32(0.3), "bf16")
    for j in range(QL):
        # row j equals an ordinary decode whose context stops at L - QL + j + 1
        ref = oracle.decode_v1(q[:, j], kc, vc, bt, lens - QL + j + 1, np.float32(0.3), "bf16")
        assert np.array_equal(got[:, j], ref)
    # and the dense reference with a causal mask, for the longest sequence
    s = 2
    k = np.repeat(oracle.widen(kv[s][0], "bf16"), Hq // Hkv, axis=1)
    v = np.repeat(oracle.widen(kv[s][1], "bf16"), Hq // Hkv, axis=1)
    for j in range(QL):
        limit = int(lens[s]) - QL + j + 1
        logits = np.einsum("hd,thd->ht", oracle.widen(q[s, j], "bf16"), k[:limit]) * float(np.float32(0.3))
        ref = np.einsum("ht,thd->hd", scipy.special.softmax(logits, axis=1), v[:limit])
        np.testing.assert_allclose(got[s, j], ref, rtol=1e-12, atol=1e-13)
