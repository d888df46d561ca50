"""GPU parity for the fp8 E4M3 KV cache: the quantising scatter is bit-exact with the
oracle's definition, and decode over fp8 pools matches the oracle's fp8 decode."""
import numpy as np
import pytest
import torch

import oracle
from oracle_side import TOL, bits, max_err

pytestmark = pytest.mark.gpu


def _u8(t):
    return t.detach().cpu().numpy().astype(np.uint8, copy=False)


def _batch(dev, lens, Hq, Hkv, bs, dtype, seed):
    """Per-sequence K/V scattered into NaN-poisoned fp8 pools by the product and the oracle."""
    import paged_kv_cache_187_gb300 as pa
    from paged_kv_cache_187_gb300 import workloads as W
    D = 128
    lens = np.asarray(lens, np.int32)
    S = lens.size
    NB = int(np.sum((lens + bs - 1) // bs) * 1.3) + 4
    maxb = int((lens.max() + bs - 1) // bs)
    ks, vs = np.float32(0.02), np.float32(0.015)   # N(0,1) data spans about +-5 / scale
    prod = pa.PagedAllocator(NB, bs, seed)
    ref = oracle.Alloc(NB, bs, seed)
    kc = torch.full((NB, Hkv, bs, D), 0x7F, dtype=torch.uint8, device=dev)    # E4M3 NaN
    vc = kc.clone()
    okc = np.full((NB, Hkv, bs, D), 0x7F, np.uint8)
    ovc = okc.copy()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for s, L in enumerate(lens):
        L = int(L)
        prod.pa_alloc_add_seq(s, L)
        ref.add_seq(s, L)
        slots = prod.pa_alloc_slots(s, 0, L)
        assert np.array_equal(slots, ref.slots(s, 0, L))
        k = W.randn_16bit((L, Hkv, D), dtype, seed * 1000 + 2 * s, dev)
        v = W.randn_16bit((L, Hkv, D), dtype, seed * 1000 + 2 * s + 1, dev)
        pa.pa_reshape_and_cache_fp8(k, v, kc, vc, torch.from_numpy(slots).to(dev), ks, vs,
                                    status=status)
        oracle.reshape_and_cache_fp8(bits(k), bits(v), okc, ovc, slots, bs, dtype, ks, vs)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    tables = prod.pa_alloc_block_tables(np.arange(S), maxb)
    q = W.randn_16bit((S, Hq, D), dtype, seed * 1000 + 999, dev)
    return dict(kc=kc, vc=vc, okc=okc, ovc=ovc, tables=tables, lens=lens, q=q, ks=ks, vs=vs)


CASES = [
    ("bf16", 32, 8, 16),    # GQA 4
    ("bf16", 64, 8, 32),    # GQA 8, 32-token blocks
    ("f16", 16, 16, 16),    # MHA
    ("bf16", 16, 1, 16),    # GQA 16 (two n-tiles; tensor cores either way)
]


@pytest.fixture(params=[True, False], ids=["tensor_cores", "cuda_cores"])
def fp8_path(request):
    import paged_kv_cache_187_gb300 as pa
    pa.pa_set_gqa_tensor_cores(request.param)
    yield request.param
    pa.pa_set_gqa_tensor_cores(True)


@pytest.mark.parametrize("dtype,Hq,Hkv,bs", CASES)
def test_fp8_cache_scatter_bit_exact_and_decode(cuda_device, fp8_path, dtype, Hq, Hkv, bs):
    import paged_kv_cache_187_gb300 as pa
    lens = [1, bs - 1, bs, bs + 1, 100, 257, 511, 513, 1500, 3000]
    b = _batch(cuda_device, lens, Hq, Hkv, bs, dtype, seed=31 + Hq + bs)
    assert np.array_equal(_u8(b["kc"]), b["okc"]) and np.array_equal(_u8(b["vc"]), b["ovc"])
    scale = 128 ** -0.5
    ref = oracle.decode_fp8(bits(b["q"]), b["okc"], b["ovc"], b["tables"], b["lens"],
                            np.float32(scale), b["ks"], b["vs"], dtype)
    S = len(lens)
    out = torch.empty_like(b["q"])
    tables = torch.from_numpy(b["tables"]).to(cuda_device)
    lens_d = torch.from_numpy(b["lens"]).to(cuda_device)
    mcl = int(b["lens"].max())
    ws = torch.empty(max(pa.pa_decode_auto_workspace_size(S, Hq, Hkv, 128, bs, mcl),
                         pa.pa_decode_v2_workspace_size(S, Hq, 128, mcl, 3 * bs), 256),
                     dtype=torch.uint8, device=cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    # with 16-token blocks, partitions of 4 blocks take the two-block tiles; of 3, one-block
    for variant, P in (("auto", 0), ("v1", 0), ("v2", 4 * bs), ("v2", 3 * bs)):
        out.fill_(5.0)
        pa.pa_decode_fp8(out, b["q"], b["kc"], b["vc"], tables, lens_d, mcl, scale, b["ks"],
                         b["vs"], variant=variant, partition_size=P, workspace=ws, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        err = max_err(bits(out), ref, dtype)
        assert err <= TOL[dtype], f"{variant}: {err}"


def test_fp8_copy_blocks_and_padding_slots(cuda_device):
    import paged_kv_cache_187_gb300 as pa
    NB, Hkv, bs, D = 6, 2, 16, 128
    kc = torch.randint(0, 255, (NB, Hkv, bs, D), dtype=torch.uint8, device=cuda_device)
    vc = torch.randint(0, 255, (NB, Hkv, bs, D), dtype=torch.uint8, device=cuda_device)
    before_k, before_v = kc.clone(), vc.clone()
    pairs = torch.tensor([[1, 4], [2, 5]], dtype=torch.int32, device=cuda_device)
    pa.pa_copy_blocks(kc, vc, pairs)
    torch.cuda.synchronize()
    assert torch.equal(kc[4], before_k[1]) and torch.equal(vc[5], before_v[2])
    assert torch.equal(kc[:4], before_k[:4])
    key = torch.ones((2, Hkv, D), dtype=torch.float16, device=cuda_device)
    slots = torch.tensor([-1, 3], dtype=torch.int32, device=cuda_device)
    pa.pa_reshape_and_cache_fp8(key, key, kc, vc, slots, 0.5, 0.25)
    torch.cuda.synchronize()
    assert bool((kc[0, :, 3] == 0x40).all()) and bool((vc[0, :, 3] == 0x48).all())   # 2.0, 4.0


@pytest.mark.parametrize("name", ["l3_8b", "l3_70b"])
def test_fp8_full_size_every_row(cuda_device, name):
    """A full-size batch over fp8 pools (Llama-3-8B heads with 16-token blocks, and
    Llama-3-70B heads with 32-token blocks): the prefill and the step's rows quantised by
    the product's scatter equal the oracle's whole pools bit for bit, and every output
    row of the automatic choice (the device-sized V2 plan) and of V1 meets the bound."""
    import paged_kv_cache_187_gb300 as pa
    from paged_kv_cache_187_gb300 import workloads as W
    from paged_kv_cache_187_gb300.runner import DecodeRunner
    from oracle_side import OracleState, err_stats, record_step
    w = W.WORKLOADS[name]
    r = DecodeRunner(w, device="cuda", kv_fp8=True).next_step()
    r.run_reshape()
    torch.cuda.synchronize()
    assert int(r.status.item()) == 0
    st = record_step(r)
    o = OracleState(r, [st])
    assert np.array_equal(_u8(r.key_cache), o.k_cache)
    assert np.array_equal(_u8(r.value_cache), o.v_cache)
    del r.k_prefill, r.v_prefill
    ref = o.decode(0, st)
    for variant in ("auto", "v1"):
        r.out.fill_(5.0)
        r.run_decode(variant)
        torch.cuda.synchronize()
        assert int(r.status.item()) == 0
        e = err_stats(bits(r.out), ref, w.dtype)
        print(f"fp8 {name} {variant}: {e}")
        assert e.ok(w.dtype), f"fp8 {name} {variant}: {e}"
