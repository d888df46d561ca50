"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Bars (stated by the workload specification):
  * reshape_and_cache, the allocator's slots and block tables: bit-exact;
  * decode: max |gpu - round_to_dtype(oracle)| <= 2e-3 (fp16) and <= 1e-2 (bf16), with
    the one-ulp allowance for outputs whose ulp exceeds that bound, and a cap on how
    many elements may need it (oracle_side.ErrStats.ok).
Every (sequence, head) row is compared, at full size too: the oracle's sequences are
fanned out over the host's cores (each range runs the plain single-threaded oracle).
The middle steps of the multi-step loop compare sampled rows.
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

import oracle
from oracle_side import OracleState, StepRecord, TOL, bits, err_stats, max_err, record_step

pytestmark = pytest.mark.gpu

W = pytest.importorskip("paged_kv_cache_187_gb300.workloads")


def _pa():
    import paged_kv_cache_187_gb300 as pa
    return pa


def _runner(w, **kw):
    from paged_kv_cache_187_gb300.runner import DecodeRunner
    return DecodeRunner(w, device="cuda", **kw)


def _sample_rows(r, n_seq=12, seed=0):
    rng = np.random.default_rng(seed)
    lens = r.context_lens
    S, Hq = r.w.num_seqs, r.w.num_q_heads
    seqs = {int(np.argmin(lens)), int(np.argmax(lens))}
    seqs |= set(int(x) for x in rng.choice(S, size=min(S, n_seq), replace=False))
    rows = []
    for s in sorted(seqs):
        heads = {0, Hq - 1, int(rng.integers(Hq))}
        rows += [(s, h) for h in sorted(heads)]
    return sorted(seqs), rows


def _status_ok(r):
    torch.cuda.synchronize()
    assert int(r.status.item()) == 0, f"device status {int(r.status.item())}"


# ----------------------------------------------------------------------------- reshape
@pytest.mark.parametrize("name", ["tiny", "l2_7b", "l3_8b"])
def test_reshape_and_cache_bit_exact_full_pool(cuda_device, name):
    w = W.WORKLOADS[name]
    r = _runner(w).next_step()
    r.run_reshape()
    _status_ok(r)
    st = record_step(r)
    o = OracleState(r, [st])
    assert np.array_equal(o.prefill_slots, r.prefill_slots)
    assert np.array_equal(o.step_slots[0], r.slots)
    assert np.array_equal(o.step_tables[0], r.block_tables)
    assert np.array_equal(o.step_lens[0], r.context_lens)
    assert np.array_equal(bits(r.key_cache), o.k_cache)
    assert np.array_equal(bits(r.value_cache), o.v_cache)


@pytest.mark.parametrize("name", ["skew", "l3_70b"])
def test_reshape_and_cache_bit_exact_sampled(cuda_device, name):
    w = W.WORKLOADS[name]
    r = _runner(w).next_step()
    r.run_reshape()
    _status_ok(r)
    st = record_step(r)
    seqs, _ = _sample_rows(r, n_seq=6)
    o = OracleState(r, [st], seqs=seqs)
    assert np.array_equal(o.step_slots[0], r.slots)
    assert np.array_equal(o.step_tables[0], r.block_tables)
    used = torch.from_numpy(o.used_blocks).to(cuda_device)
    assert np.array_equal(bits(r.key_cache.index_select(0, used)), o.k_cache)
    assert np.array_equal(bits(r.value_cache.index_select(0, used)), o.v_cache)
    # blocks no sequence owns are still the poison pattern
    owned = np.zeros(r.num_blocks, bool)
    owned[r.block_tables[r.block_tables >= 0]] = True
    free = torch.from_numpy(np.nonzero(~owned)[0]).to(cuda_device)
    if free.numel():
        nan = W.NAN_BITS[w.dtype]
        nan = nan - 65536 if nan >= 32768 else nan
        assert bool((r.key_cache.index_select(0, free).view(torch.int16) == nan).all())
        assert bool((r.value_cache.index_select(0, free).view(torch.int16) == nan).all())


def test_reshape_padding_and_bad_slots(cuda_device):
    pa = _pa()
    NB, Hkv, bs, D = 4, 2, 16, 64
    kc = torch.zeros((NB, Hkv, bs, D), dtype=torch.float16, device=cuda_device)
    vc = torch.zeros_like(kc)
    key = torch.ones((3, Hkv, D), dtype=torch.float16, device=cuda_device)
    slots = torch.tensor([-1, NB * bs + 5, 7], dtype=torch.int32, device=cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    pa.pa_reshape_and_cache(key, key * 2, kc, vc, slots, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == pa.PA_DEVERR_BAD_SLOT
    assert float(kc.sum()) == Hkv * D and float(vc.sum()) == 2 * Hkv * D
    assert bool((kc[0, :, 7] == 1).all()) and bool((vc[0, :, 7] == 2).all())


# ----------------------------------------------------------------------------- decode
def _check_full(r, o, step_rec, variant, partition_size=None, step=0):
    r.run_decode(variant, partition_size=partition_size)
    _status_ok(r)
    ref = o.decode(step, step_rec)
    err = max_err(bits(r.out), ref, r.w.dtype)
    assert err <= TOL[r.w.dtype], f"{variant} P={partition_size}: max err {err}"
    return ref


def test_decode_tiny_all_variants(cuda_device):
    w = W.WORKLOADS["tiny"]
    r = _runner(w).next_step()
    r.run_reshape()
    st = record_step(r)
    o = OracleState(r, [st])
    ref = _check_full(r, o, st, "v1")
    for P in (16, 32, 64, 512):
        _check_full(r, o, st, "v2", P)
    _check_full(r, o, st, "auto")
    # context_len 1 -> exactly that token's V row (p = 1, l = 1)
    s1 = int(np.nonzero(r.context_lens == 1)[0][0])
    for variant, P in (("v1", None), ("v2", 16)):
        r.run_decode(variant, partition_size=P)
        torch.cuda.synchronize()
        assert np.array_equal(bits(r.out[s1]), st.v_new[s1])
    # the V2 oracle agrees with V1 on this input (pin, repeated at this workload)
    np.testing.assert_allclose(o.decode(0, st, partition_size=16), ref, rtol=1e-12, atol=1e-13)


def test_decode_step_single_call_tiny(cuda_device):
    w = W.WORKLOADS["tiny"]
    r = _runner(w).next_step()
    r.run_step()
    _status_ok(r)
    st = record_step(r)
    o = OracleState(r, [st])
    assert np.array_equal(bits(r.key_cache), o.k_cache)
    err = max_err(bits(r.out), o.decode(0, st), w.dtype)
    assert err <= TOL[w.dtype]


@pytest.mark.parametrize("name", ["l2_7b", "l3_8b", "skew"])
def test_decode_full_size_every_row(cuda_device, name):
    """The whole batch of one full-size decode step: every output element of every
    (sequence, head) row against the oracle, for the auto choice, V1, and V2 at the
    workload's partition size and at 256 tokens; the whole pools bit for bit."""
    w = W.WORKLOADS[name]
    r = _runner(w).next_step()
    r.run_reshape()
    _status_ok(r)
    st = record_step(r)
    o = OracleState(r, [st])
    assert np.array_equal(o.step_slots[0], r.slots)
    assert np.array_equal(o.step_tables[0], r.block_tables)
    assert np.array_equal(bits(r.key_cache), o.k_cache)
    assert np.array_equal(bits(r.value_cache), o.v_cache)
    ref = o.decode(0, st)
    for variant, P in (("auto", None), ("v1", None), ("v2", w.partition_size), ("v2", 256)):
        r.out.fill_(7.0)
        r.run_decode(variant, partition_size=P)
        _status_ok(r)
        e = err_stats(bits(r.out), ref, w.dtype)
        print(f"{name} {variant} P={P}: {e}")
        assert e.ok(w.dtype), f"{name} {variant} P={P}: {e}"


def test_multistep_loop_l3_70b(cuda_device):
    """Eight steps of the Llama-3-70B-shaped loop (append, reshape_and_cache, auto decode
    per step): slots, tables and lengths bit-exact at every step; every row of the
    first and the last step against the oracle, sampled rows of the steps between; the
    pools bit for bit after the loop."""
    w = W.WORKLOADS["l3_70b"]
    r = _runner(w)
    recs, outs = [], []
    for k in range(w.steps):
        r.next_step()
        r.run_step()
        recs.append(record_step(r))
        outs.append(bits(r.out))
    _status_ok(r)
    _, rows = _sample_rows(r, n_seq=8)
    o = OracleState(r, recs)
    for k in range(w.steps):
        assert np.array_equal(o.step_slots[k], recs[k].slots)
        assert np.array_equal(o.step_tables[k], recs[k].block_tables)
        assert np.array_equal(o.step_lens[k], recs[k].context_lens)
        every = k in (0, w.steps - 1)
        ref = o.decode(k, recs[k]) if every else o.decode(k, recs[k], rows=rows)
        e = err_stats(outs[k], ref, w.dtype, rows=None if every else rows)
        print(f"l3_70b step {k} ({'every row' if every else 'sampled rows'}): {e}")
        assert e.ok(w.dtype), f"step {k}: {e}"
    assert np.array_equal(bits(r.key_cache), o.k_cache)
    assert np.array_equal(bits(r.value_cache), o.v_cache)


# ----------------------------------------------------------------------------- GPU pins
def test_block_placement_invariance_bit_identical(cuda_device):
    w = W.WORKLOADS["l3_8b"]
    w = dataclasses.replace(w, num_seqs=24)
    lens = W.start_context_lens(W.WORKLOADS["l3_8b"])[:24]
    outs = []
    for seed in (5, 77):
        r = _runner(w, start_lens=lens, alloc_seed=seed, num_blocks=int(
            np.sum((lens + 15) // 16) * 1.5)).next_step()
        r.run_reshape()
        res = []
        for variant, P in (("v1", None), ("v2", 128), ("auto", None)):
            r.run_decode(variant, partition_size=P)
            torch.cuda.synchronize()
            res.append(bits(r.out))
        _status_ok(r)
        outs.append((res, r.block_tables.copy()))
    assert not np.array_equal(outs[0][1], outs[1][1])
    for a, b in zip(outs[0][0], outs[1][0]):
        assert np.array_equal(a, b)


def test_gqa_tensor_core_and_cuda_core_paths(cuda_device):
    pa = _pa()
    base = W.WORKLOADS["l3_8b"]
    w = dataclasses.replace(base, num_seqs=16)
    lens = np.array([1, 15, 16, 17, 31, 33, 100, 255, 256, 257, 511, 512, 513, 700, 1025, 2000],
                    np.int32)
    r = _runner(w, start_lens=lens).next_step()
    r.run_reshape()
    st = record_step(r)
    o = OracleState(r, [st])
    ref = o.decode(0, st)
    try:
        for mma in (True, False):
            pa.pa_set_gqa_tensor_cores(mma)
            for variant, P in (("v1", None), ("v2", 64)):
                r.run_decode(variant, partition_size=P)
                _status_ok(r)
                err = max_err(bits(r.out), ref, w.dtype)
                assert err <= TOL[w.dtype], f"mma={mma} {variant}: {err}"
    finally:
        pa.pa_set_gqa_tensor_cores(True)


def test_kernel_choice_belongs_to_the_calling_thread(cuda_device):
    """pa_set_gqa_tensor_cores(0) in one thread leaves another thread's calls on the
    tensor-core path: the main thread's output stays bit-identical to its own earlier
    tensor-core result while the other thread's setting is off."""
    import threading
    pa = _pa()
    w = dataclasses.replace(W.WORKLOADS["l3_8b"], num_seqs=8)
    lens = np.array([3, 40, 200, 513, 999, 1500, 64, 17], np.int32)
    r = _runner(w, start_lens=lens).next_step()
    r.run_reshape()
    r.run_decode("v1")
    _status_ok(r)
    mma = bits(r.out)
    done = threading.Event()
    release = threading.Event()

    def other():
        pa.pa_set_gqa_tensor_cores(False)
        done.set()
        release.wait(30)

    t = threading.Thread(target=other)
    t.start()
    assert done.wait(30)
    try:
        r.out.zero_()
        r.run_decode("v1")
        _status_ok(r)
        assert np.array_equal(bits(r.out), mma)
    finally:
        release.set()
        t.join()
    # in the main thread the same switch does take effect (both paths meet the bound)
    st = record_step(r)
    ref = OracleState(r, [st]).decode(0, st)
    try:
        pa.pa_set_gqa_tensor_cores(False)
        r.run_decode("v1")
        _status_ok(r)
        core = bits(r.out)
    finally:
        pa.pa_set_gqa_tensor_cores(True)
    assert max_err(core, ref, w.dtype) <= TOL[w.dtype]
    assert max_err(mma, ref, w.dtype) <= TOL[w.dtype]


EDGE = []
for D in (64, 128):
    for bs in (16, 32):
        for Hq, Hkv in ((4, 4), (8, 4), (12, 4), (16, 2), (32, 2)):
            for dt in ("f16", "bf16"):
                EDGE.append((D, bs, Hq, Hkv, dt))


@pytest.mark.parametrize("D,bs,Hq,Hkv,dt", EDGE)
def test_edge_contexts(cuda_device, D, bs, Hq, Hkv, dt):
    P = 4 * bs
    lens = np.array(sorted({1, bs - 1, bs, bs + 1, P - 1, P, P + 1, 2 * P + 3, 5 * P - 2}),
                    np.int32)
    w = W.Workload("edge", len(lens), Hq, Hkv, D, bs, dt, seed=4242 + D + bs + Hq + len(dt))
    r = _runner(w, start_lens=lens).next_step()
    r.run_reshape()
    st = record_step(r)
    o = OracleState(r, [st])
    assert np.array_equal(bits(r.key_cache), o.k_cache)
    ref = o.decode(0, st)
    for variant, psize in (("v1", None), ("v2", P), ("v2", bs), ("auto", None)):
        r.out.fill_(7.0)
        r.run_decode(variant, partition_size=psize)
        _status_ok(r)
        err = max_err(bits(r.out), ref, dt)
        assert err <= TOL[dt], f"{variant} P={psize}: {err}"


def test_empty_context_gives_zero_row(cuda_device):
    w = dataclasses.replace(W.WORKLOADS["l3_8b"], num_seqs=4)
    r = _runner(w, start_lens=np.array([5, 40, 600, 1], np.int32)).next_step()
    r.run_reshape()
    r.context_lens_d[1] = 0
    lens = r.context_lens.copy()
    lens[1] = 0
    st = record_step(r)
    o = OracleState(r, [st])
    ref = o.decode(0, st, context_lens=lens)
    assert np.all(ref[1] == 0)
    for variant, P in (("v1", None), ("v2", 32), ("v2", 512)):
        r.out.fill_(3.0)
        r.run_decode(variant, partition_size=P)
        _status_ok(r)
        assert max_err(bits(r.out), ref, w.dtype) <= TOL[w.dtype]
        assert bool((r.out[1] == 0).all())


def test_device_error_flags_without_fault(cuda_device):
    pa = _pa()
    w = dataclasses.replace(W.WORKLOADS["l3_8b"], num_seqs=3)
    r = _runner(w, start_lens=np.array([20, 70, 33], np.int32)).next_step()
    r.run_reshape()
    _status_ok(r)
    # a block-table entry outside the pool: flagged, the tile reads as zeros, no fault
    r.block_tables_d[1, 2] = r.num_blocks + 1000
    for variant, P in (("v1", None), ("v2", 32)):
        r.status.zero_()
        r.run_decode(variant, partition_size=P)
        torch.cuda.synchronize()
        assert int(r.status.item()) & pa.PA_DEVERR_BAD_BLOCK
        assert bool(torch.isfinite(r.out.float()).all())
    r.block_tables_d[1, 2] = int(r.block_tables[1, 2])
    # a context longer than max_context_len: clamped and flagged
    for variant, P in (("v1", None), ("v2", 32)):
        r.status.zero_()
        r.run_decode(variant, partition_size=P, max_context_len=40)
        torch.cuda.synchronize()
        assert int(r.status.item()) & pa.PA_DEVERR_BAD_LEN


def test_host_argument_errors(cuda_device):
    pa = _pa()
    w = dataclasses.replace(W.WORKLOADS["tiny"], num_seqs=2)
    r = _runner(w, start_lens=np.array([3, 9], np.int32)).next_step()
    with pytest.raises(pa.PAError):
        r.run_decode("v2", partition_size=24)          # not a multiple of block_size
    small = torch.empty(16, dtype=torch.uint8, device=cuda_device)
    with pytest.raises(pa.PAError):
        pa.pa_decode_v2(r.out, r.q, r.key_cache, r.value_cache, r.block_tables_d,
                        r.context_lens_d, 9, w.scale, 16, small)
    bad = torch.empty((2, 4, 48), dtype=torch.float16, device=cuda_device)
    kc = torch.empty((4, 4, 16, 48), dtype=torch.float16, device=cuda_device)
    with pytest.raises(pa.PAError):
        pa.pa_decode_v1(bad, bad, kc, kc, r.block_tables_d, r.context_lens_d, 9, 0.1)


def test_back_to_back_calls_on_one_workspace(cuda_device):
    """Calls queued back to back on one stream and one workspace, nothing synchronised in
    between, each with its own queries, lengths and output: the next call's plan / reshape
    launch while the previous decode finishes its last tiles, on the other half of the
    workspace.  Every output must still equal the oracle's decode of its own inputs.  Small
    fixed partitions force many split sequences, and with them partial results and merges
    in both halves."""
    pa = _pa()
    base = W.WORKLOADS["l3_8b"]
    w = dataclasses.replace(base, num_seqs=48)
    lens = W.start_context_lens(base)[:48]
    r = _runner(w, start_lens=lens).next_step()
    r.run_reshape()
    _status_ok(r)
    st = record_step(r)
    o = OracleState(r, [st])
    S, Hq, D = w.num_seqs, w.num_q_heads, w.head_size
    mcl = r.step_max_context_len()
    ws = torch.empty(max(pa.pa_decode_v2_workspace_size(S, Hq, D, mcl, 64),
                         pa.pa_decode_auto_workspace_size(S, Hq, w.num_kv_heads, D, w.block_size, mcl)),
                     dtype=torch.uint8, device=cuda_device)
    calls = []
    for k in range(6):
        # each call attends over a prefix of every context (at least one token) with its
        # own queries
        lens_k = np.maximum(r.context_lens - 97 * k, 1).astype(np.int32)
        q_k = W.randn_16bit((S, Hq, D), w.dtype, 5000 + k, cuda_device)
        calls.append((lens_k, torch.from_numpy(lens_k).to(cuda_device), q_k, torch.empty_like(q_k)))
    torch.cuda.synchronize()
    for k, (lens_k, lens_d, q_k, out_k) in enumerate(calls):
        if k % 3 == 0:
            pa.pa_decode_v2(out_k, q_k, r.key_cache, r.value_cache, r.block_tables_d, lens_d, mcl,
                            w.scale, 64, ws, status=r.status)
        elif k % 3 == 1:
            pa.pa_decode_auto(out_k, q_k, r.key_cache, r.value_cache, r.block_tables_d, lens_d,
                              mcl, w.scale, workspace=ws, status=r.status)
        else:
            pa.pa_decode_step(out_k, q_k, r.k_new, r.v_new, r.key_cache, r.value_cache,
                              r.slots_d, r.block_tables_d, lens_d, mcl, w.scale, workspace=ws,
                              status=r.status)
    _status_ok(r)
    for k, (lens_k, _, q_k, out_k) in enumerate(calls):
        stq = dataclasses.replace(st, q=bits(q_k))
        ref = o.decode(0, stq, context_lens=lens_k)
        e = err_stats(bits(out_k), ref, w.dtype)
        assert e.ok(w.dtype), f"call {k}: {e}"
