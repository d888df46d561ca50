"""CPU-only checks of the C ABI library: it loads, exports every symbol include/pa.h
declares, and its host block allocator matches the oracle allocator byte for byte
(no GPU call is made here)."""
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pa():
    from paged_kv_cache_187_gb300 import build
    build.build()
    import paged_kv_cache_187_gb300 as pkg
    return pkg


def _declared_functions():
    with open(os.path.join(ROOT, "include", "pa.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_boundary_calls():
    names = _declared_functions()
    for must in ("pa_reshape_and_cache", "pa_decode_v1", "pa_decode_v2", "pa_decode_auto",
                 "pa_decode_v2_workspace_size", "pa_alloc_create", "pa_alloc_block_tables",
                 "pa_alloc_append"):
        assert must in names


def test_library_exports_every_declared_symbol(pa):
    lib = pa.raw()
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_workspace_size_is_host_only_and_monotone(pa):
    a = pa.pa_decode_v2_workspace_size(256, 32, 128, 8192, 512)
    b = pa.pa_decode_v2_workspace_size(256, 32, 128, 8192, 256)
    assert 0 < a < b
    # partials: parts * Hq * (D floats + (m, l)) dominate
    parts = 256 * 16
    assert a >= parts * 32 * (128 * 4 + 8)


def test_multi_query_workspace_size(pa):
    # partial rows per partition are q_len * num_q_heads: the same bytes as an ordinary V2
    # decode with q_len times the query heads
    assert (pa.pa_decode_mq_workspace_size(64, 4, 32, 8, 128, 16, 4096, 256) ==
            pa.pa_decode_v2_workspace_size(64, 128, 128, 4096, 256))
    # 0: the automatic choice (V2 here, whose smallest partition is 256 tokens)
    assert (pa.pa_decode_mq_workspace_size(64, 4, 32, 8, 128, 16, 4096, 0) ==
            pa.pa_decode_v2_workspace_size(64, 128, 128, 4096, 256))
    assert pa.pa_decode_mq_workspace_size(64, 0, 32, 8, 128, 16, 4096, 256) == 0
    assert pa.pa_decode_mq_workspace_size(64, 2, 32, 0, 128, 16, 4096, 256) == 0


def test_auto_plan_choices(pa):
    v, P = pa.pa_decode_auto_plan(256, 40, 40, 128, 16, 32768)
    assert v == 2 and P % 16 == 0 and P > 0
    v, P = pa.pa_decode_auto_plan(4096, 32, 8, 128, 16, 128)
    assert v == 1 and P == 0
    assert pa.pa_decode_auto_workspace_size(4096, 32, 8, 128, 16, 128) == 0


@pytest.mark.parametrize("seed", [0, 1, 123456789, 2**63 + 5])
def test_allocator_matches_oracle_allocator(pa, seed):
    NB, bs = 97, 16
    prod = pa.PagedAllocator(NB, bs, seed)
    ref = oracle.Alloc(NB, bs, seed)
    rng = np.random.default_rng(seed % 1000)
    lens = rng.integers(0, 200, size=6)
    for s, L in enumerate(lens):
        prod.pa_alloc_add_seq(s, int(L))
        ref.add_seq(s, int(L))
    ids = np.arange(6)
    for _ in range(40):
        a = prod.pa_alloc_append_batch(ids)
        b = np.array([ref.append(int(s)) for s in ids], np.int32)
        assert np.array_equal(a, b)
    assert np.array_equal(prod.pa_alloc_block_tables(ids, 20), ref.block_tables(ids, 20))
    assert np.array_equal(prod.pa_alloc_context_lens(ids), ref.context_lens(ids))
    for s, L in enumerate(lens):
        assert np.array_equal(prod.pa_alloc_slots(s, 0, int(L)), ref.slots(s, 0, int(L)))
    prod.pa_alloc_free_seq(3)
    ref.free_seq(3)
    prod.pa_alloc_add_seq(9, 40)
    ref.add_seq(9, 40)
    assert np.array_equal(prod.pa_alloc_block_tables([9], 5), ref.block_tables([9], 5))
    assert prod.num_free == ref.num_free


def test_allocator_errors_and_all_or_nothing_batch(pa):
    prod = pa.PagedAllocator(3, 8, 7)
    prod.pa_alloc_add_seq(0, 8)
    prod.pa_alloc_add_seq(1, 8)
    prod.pa_alloc_add_seq(2, 1)
    with pytest.raises(pa.PANoBlocks):
        prod.pa_alloc_append_batch([0, 1])          # needs 2 new blocks, 0 free
    assert list(prod.pa_alloc_context_lens([0, 1, 2])) == [8, 8, 1]
    with pytest.raises(pa.PAError):
        prod.pa_alloc_append_batch([2, 2])          # duplicate id
    with pytest.raises(pa.PAError):
        prod.pa_alloc_add_seq(0, 1)                 # already live
    with pytest.raises(pa.PAError):
        prod.pa_alloc_append(42)                    # unknown id
    slots = prod.pa_alloc_append_batch([2])
    assert slots.shape == (1,) and slots[0] % 8 == 1


def test_reserve_matches_oracle_and_appends_use_reserved_blocks(pa):
    NB, bs = 64, 16
    prod = pa.PagedAllocator(NB, bs, 42)
    ref = oracle.Alloc(NB, bs, 42)
    lens = [15, 16, 1, 40]
    for s, L in enumerate(lens):
        prod.pa_alloc_add_seq(s, L)
        ref.add_seq(s, L)
    ids = np.arange(4)
    prod.pa_alloc_reserve_batch(ids, 8)
    for s in ids:
        ref.reserve(int(s), 8)
    free_after_reserve = prod.num_free
    assert free_after_reserve == ref.num_free
    assert np.array_equal(prod.pa_alloc_block_tables(ids, 4), ref.block_tables(ids, 4))
    for _ in range(8):
        a = prod.pa_alloc_append_batch(ids)
        b = np.array([ref.append(int(s)) for s in ids], np.int32)
        assert np.array_equal(a, b)
    assert prod.num_free == free_after_reserve          # no pops inside the reservation
    with pytest.raises(pa.PANoBlocks):
        prod.pa_alloc_reserve_batch(ids, 10_000)        # all or nothing
    assert prod.num_free == free_after_reserve


def test_sharing_allocator_matches_oracle_under_random_requests(pa):
    rng = np.random.default_rng(77)
    NB, bs = 200, 16
    prod = pa.PagedAllocator(NB, bs, 5)
    ref = oracle.Alloc(NB, bs, 5)
    live = {}
    next_id = 0
    for step in range(600):
        op = int(rng.integers(0, 5))
        if op == 0 or not live:                               # new sequence
            n = int(rng.integers(0, 70))
            try:
                prod.pa_alloc_add_seq(next_id, n)
            except pa.PANoBlocks:
                with pytest.raises(oracle.OracleAllocError):
                    ref.add_seq(next_id, n)
                continue
            ref.add_seq(next_id, n)
            live[next_id] = n
            next_id += 1
        elif op == 1:                                         # fork a prefix
            src = int(rng.choice(list(live)))
            n = int(rng.integers(0, live[src] + 1))
            prod.pa_alloc_fork(src, next_id, n)
            ref.fork(src, next_id, n)
            live[next_id] = n
            next_id += 1
        elif op == 2:                                         # append to some sequences
            ids = rng.choice(list(live), size=min(len(live), 4), replace=False).astype(np.int32)
            try:
                a = prod.pa_alloc_append_batch(ids)
            except pa.PANoBlocks:
                continue
            b = np.array([ref.append(int(s)) for s in ids], np.int32)
            assert np.array_equal(a, b)
            for s in ids:
                live[int(s)] += 1
        elif op == 3:                                         # free one
            s = int(rng.choice(list(live)))
            prod.pa_alloc_free_seq(s)
            ref.free_seq(s)
            del live[s]
        else:                                                 # reserve ahead (with COW)
            ids = rng.choice(list(live), size=min(len(live), 3), replace=False).astype(np.int32)
            extra = int(rng.integers(1, 20))
            try:
                prod.pa_alloc_reserve_batch(ids, extra)
            except pa.PANoBlocks:
                continue
            for s in ids:
                ref.reserve(int(s), extra)
        assert prod.num_free == ref.num_free, step
        if step % 50 == 0:
            assert np.array_equal(prod.pa_alloc_take_copies(), ref.take_copies())
    assert np.array_equal(prod.pa_alloc_take_copies(), ref.take_copies())
    ids = np.array(sorted(live), np.int32)
    if ids.size:
        width = max(8, max((live[int(s)] + 40) // bs for s in ids))
        assert np.array_equal(prod.pa_alloc_block_tables(ids, width), ref.block_tables(ids, width))
        assert np.array_equal(prod.pa_alloc_context_lens(ids), ref.context_lens(ids))
    for b in range(NB):
        assert prod.pa_alloc_refcount(b) == ref.refcount(b)
    used = sum(1 for b in range(NB) if prod.pa_alloc_refcount(b) > 0)
    assert used + prod.num_free == NB
