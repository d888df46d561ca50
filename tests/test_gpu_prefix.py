"""GPU parity for shared prefixes: forked sequences share their parent's blocks, the
first append into a shared partial block copies it (pa_copy_blocks), and decode over
parents and children matches the oracle, which runs the same requests on its own
allocator, copies and pools."""
import numpy as np
import pytest
import torch

import oracle
from oracle_side import TOL, bits, max_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,Hq,Hkv,bs", [("bf16", 32, 8, 16), ("f16", 8, 8, 32)])
def test_forked_prefixes_copy_on_write_and_decode(cuda_device, dtype, Hq, Hkv, bs):
    import paged_kv_cache_187_gb300 as pa
    from paged_kv_cache_187_gb300 import workloads as W
    D = 128
    rng = np.random.default_rng(21)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    parent_lens = rng.integers(40, 700, size=6)
    NB = int(sum((L + 2 * bs) // bs for L in parent_lens) * 3)
    seed = 8
    prod = pa.PagedAllocator(NB, bs, seed)
    ref = oracle.Alloc(NB, bs, seed)
    shape = (NB, Hkv, bs, D)
    kc = torch.full(shape, float("nan"), dtype=tdt, device=cuda_device)
    vc = torch.full(shape, float("nan"), dtype=tdt, device=cuda_device)
    okc = np.full(shape, W.NAN_BITS[dtype], np.uint16)
    ovc = okc.copy()
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    gen = lambda n, s: W.randn_16bit((n, Hkv, D), dtype, s, cuda_device)
    # parents: prefill through both allocators and both scatters
    sid = 0
    lens = {}
    for L in parent_lens:
        L = int(L)
        prod.pa_alloc_add_seq(sid, L)
        ref.add_seq(sid, L)
        k, v = gen(L, 100 + sid), gen(L, 200 + sid)
        slots = prod.pa_alloc_slots(sid, 0, L)
        assert np.array_equal(slots, ref.slots(sid, 0, L))
        pa.pa_reshape_and_cache(k, v, kc, vc, torch.from_numpy(slots).to(cuda_device), status=status)
        oracle.reshape_and_cache(bits(k), bits(v), okc, ovc, slots, bs)
        lens[sid] = L
        sid += 1
    # children: forks at block-aligned, partial and full prefixes
    for p in range(len(parent_lens)):
        L = lens[p]
        for n in (L, L - 3, (L // bs) * bs, 1):
            prod.pa_alloc_fork(p, sid, n)
            ref.fork(p, sid, n)
            lens[sid] = n
            sid += 1
    ids = np.arange(sid, dtype=np.int32)
    # one decode step for everyone: append (copy-on-write where shared), copy, scatter
    slots = prod.pa_alloc_append_batch(ids)
    assert np.array_equal(slots, np.array([ref.append(int(s)) for s in ids], np.int32))
    pairs = prod.pa_alloc_take_copies()
    opairs = ref.take_copies()
    assert np.array_equal(pairs, opairs) and pairs.shape[0] > 0
    pa.pa_copy_blocks(kc, vc, torch.from_numpy(pairs).to(cuda_device), status=status)
    oracle.copy_blocks(okc, ovc, opairs)
    knew, vnew = gen(sid, 900), gen(sid, 901)
    pa.pa_reshape_and_cache(knew, vnew, kc, vc, torch.from_numpy(slots).to(cuda_device),
                            status=status)
    oracle.reshape_and_cache(bits(knew), bits(vnew), okc, ovc, slots, bs)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(bits(kc), okc) and np.array_equal(bits(vc), ovc)
    maxb = max(lens.values()) // bs + 2
    tables = prod.pa_alloc_block_tables(ids, maxb)
    assert np.array_equal(tables, ref.block_tables(ids, maxb))
    ctx = prod.pa_alloc_context_lens(ids)
    q = W.randn_16bit((sid, Hq, D), dtype, 777, cuda_device)
    refout = oracle.decode_v1(bits(q), okc, ovc, tables, ctx, np.float32(D ** -0.5), dtype)
    out = torch.empty_like(q)
    tables_d = torch.from_numpy(tables).to(cuda_device)
    ctx_d = torch.from_numpy(ctx).to(cuda_device)
    ws = torch.empty(pa.pa_decode_v2_workspace_size(sid, Hq, D, int(ctx.max()), 64) + 
                     pa.pa_decode_auto_workspace_size(sid, Hq, Hkv, D, bs, int(ctx.max())),
                     dtype=torch.uint8, device=cuda_device)
    for variant in ("auto", "v1", "v2"):
        if variant == "auto":
            pa.pa_decode_auto(out, q, kc, vc, tables_d, ctx_d, int(ctx.max()), D ** -0.5,
                              workspace=ws, status=status)
        elif variant == "v1":
            pa.pa_decode_v1(out, q, kc, vc, tables_d, ctx_d, int(ctx.max()), D ** -0.5, status=status)
        else:
            pa.pa_decode_v2(out, q, kc, vc, tables_d, ctx_d, int(ctx.max()), D ** -0.5, 64, ws,
                            status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        err = max_err(bits(out), refout, dtype)
        assert err <= TOL[dtype], f"{variant}: {err}"
