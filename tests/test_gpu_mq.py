"""GPU parity for multi-query decode (several causal query tokens per sequence, the
attention that verifies speculative tokens): every (sequence, token, head) row against
the oracle's fp64 multi-query decode, over pools the product's reshape_and_cache filled
and the oracle's reshape_and_cache rebuilt bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from oracle_side import TOL, bits, err_stats, max_err

pytestmark = pytest.mark.gpu


@pytest.fixture(params=[True, False], ids=["tcgen05", "mma_sync"])
def mq_kernel(request, cuda_device):
    """Runs a test with the tcgen05 multi-query kernel (head_size 128) or the mma.sync one."""
    import paged_kv_cache_187_gb300 as pa
    pa.pa_set_mq_tcgen05(request.param)
    yield request.param
    pa.pa_set_mq_tcgen05(True)


def _batch(dev, lens, QL, Hq, Hkv, D, bs, dtype, seed, k_ramp=None):
    """Pools for `lens` filled through the product's reshape_and_cache, and their oracle
    copy.  k_ramp(t, L): optional factor on the K row of token t of a length-L context."""
    import paged_kv_cache_187_gb300 as pa
    from paged_kv_cache_187_gb300 import workloads as W
    lens = np.asarray(lens, np.int32)
    S = lens.size
    NB = int(np.sum((lens + bs - 1) // bs) * 1.3) + 4
    maxb = max(int((lens.max() + bs - 1) // bs), 1)
    prod = pa.PagedAllocator(NB, bs, seed)
    ref = oracle.Alloc(NB, bs, seed)
    poison = W.NAN_BITS[dtype]
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    kc = torch.from_numpy(np.full((NB, Hkv, bs, D), poison, np.uint16).view(np.int16)).to(dev).view(tdt)
    vc = kc.clone()
    okc = np.full((NB, Hkv, bs, D), poison, np.uint16)
    ovc = okc.copy()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for s, L in enumerate(lens):
        L = int(L)
        prod.pa_alloc_add_seq(s, L)
        ref.add_seq(s, L)
        if L == 0:
            continue
        slots = prod.pa_alloc_slots(s, 0, L)
        assert np.array_equal(slots, ref.slots(s, 0, L))
        k = W.randn_16bit((L, Hkv, D), dtype, seed * 1000 + 2 * s, dev)
        if k_ramp is not None:
            f = torch.tensor([k_ramp(t, L) for t in range(L)], dtype=torch.float32, device=dev)
            k = (k.float() * f[:, None, None]).to(k.dtype)
        v = W.randn_16bit((L, Hkv, D), dtype, seed * 1000 + 2 * s + 1, dev)
        pa.pa_reshape_and_cache(k, v, kc, vc, torch.from_numpy(slots).to(dev), status=status)
        assert oracle.reshape_and_cache(bits(k), bits(v), okc, ovc, slots, bs) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(bits(kc), okc) and np.array_equal(bits(vc), ovc)
    tables = prod.pa_alloc_block_tables(np.arange(S), maxb)
    q = W.randn_16bit((S, QL, Hq, D), dtype, seed * 1000 + 999, dev)
    return dict(kc=kc, vc=vc, okc=okc, ovc=ovc, tables=tables, lens=lens, q=q)


# (dtype, q_len, Hq, Hkv, D, bs): rows per (sequence, kv head) = q_len * group.  With
# head_size 128 the tcgen05 kernel takes cases above 8 rows (16 or 32 rows per unit),
# unless the test switches it off; otherwise the mma.sync kernel (up to 4 row groups of 8
# rows per unit).
CASES = [
    ("bf16", 4, 32, 8, 128, 16),   # 16 rows: one 16-row unit (Llama-3-8B heads)
    ("f16", 2, 32, 8, 128, 32),    # 8 rows, 32-token blocks
    ("bf16", 5, 8, 8, 64, 16),     # MHA: 5 rows on the tensor cores, head_size 64
    ("f16", 3, 16, 2, 128, 16),    # 24 rows: one unit, row groups of 16 + 8
    ("bf16", 2, 16, 1, 64, 32),    # 32 rows: one unit, two full row groups
    ("f16", 7, 4, 4, 128, 16),     # 7 rows
    ("bf16", 5, 16, 2, 128, 16),   # 40 rows: two units, the second with an empty row group
    ("f16", 8, 8, 1, 64, 32),      # 64 rows: two units of two full row groups
    ("f16", 4, 16, 2, 128, 32),    # 32 rows, 32-token blocks
    ("bf16", 3, 32, 8, 128, 32),   # 12 rows, 32-token blocks
    ("bf16", 3, 32, 8, 128, 16),   # 12 rows, 16-token blocks
    ("f16", 2, 64, 8, 128, 16),    # 16 rows, fp16 (one P term on tcgen05)
]


@pytest.mark.parametrize("dtype,QL,Hq,Hkv,D,bs", CASES)
def test_multi_query_decode_matches_oracle(cuda_device, mq_kernel, dtype, QL, Hq, Hkv, D, bs):
    import paged_kv_cache_187_gb300 as pa
    # lengths below q_len give zero rows for the earliest query tokens; 0 is an empty context
    lens = [0, 1, QL - 1, QL, bs - 1, bs, bs + 1, 100, 257, 511, 513, 1500, 3000]
    lens = [max(L, 0) for L in lens]
    b = _batch(cuda_device, lens, QL, Hq, Hkv, D, bs, dtype, seed=71 + QL + Hq + bs)
    scale = D ** -0.5
    ref = oracle.decode_mq(bits(b["q"]), b["okc"], b["ovc"], b["tables"], b["lens"],
                           np.float32(scale), dtype)
    S = len(lens)
    out = torch.empty_like(b["q"])
    tables = torch.from_numpy(b["tables"]).to(cuda_device)
    lens_d = torch.from_numpy(b["lens"]).to(cuda_device)
    mcl = int(b["lens"].max())
    # 128-token partitions suit both kernels; 2 x block_size ones only the mma.sync kernel
    ws = torch.empty(max(pa.pa_decode_mq_workspace_size(S, QL, Hq, Hkv, D, bs, mcl, 0),
                         pa.pa_decode_mq_workspace_size(S, QL, Hq, Hkv, D, bs, mcl, 2 * bs), 256),
                     dtype=torch.uint8, device=cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    for variant, psize in (("auto", 0), ("v1", 0), ("v2", 128), ("v2", 2 * bs)):
        out.fill_(5.0)
        pa.pa_decode_mq(out, b["q"], b["kc"], b["vc"], tables, lens_d, mcl, scale,
                        variant=variant, partition_size=psize, workspace=ws, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        err = max_err(bits(out), ref, dtype)
        assert err <= TOL[dtype], f"{variant}: {err}"
        # rows with nothing to attend to are exactly zero
        for s, L in enumerate(lens):
            for j in range(QL):
                if L - QL + j + 1 <= 0:
                    assert not bits(out[s, j]).any(), (variant, s, j)


@pytest.mark.parametrize("dtype,QL,Hq,Hkv", [("bf16", 4, 32, 8), ("f16", 4, 64, 8)])
def test_multi_query_runs_of_empty_contexts(cuda_device, mq_kernel, dtype, QL, Hq, Hkv):
    """Units without a tile (empty contexts) in runs, between and after ordinary ones, on
    every variant: each such unit still passes its output rows (zero) through the kernel's
    hand-over in order, so runs of them must neither stall nor disturb their neighbours."""
    import paged_kv_cache_187_gb300 as pa
    D, bs = 128, 16
    lens = [0, 0, 0, 300, 0, 0, 0, 0, 5, 0, 0, 2000, 0, 0, 0, 0, 0, 0, 130, 0, 0, 0]
    b = _batch(cuda_device, lens, QL, Hq, Hkv, D, bs, dtype, seed=301 + Hq)
    scale = D ** -0.5
    ref = oracle.decode_mq(bits(b["q"]), b["okc"], b["ovc"], b["tables"], b["lens"],
                           np.float32(scale), dtype)
    S = len(lens)
    out = torch.empty_like(b["q"])
    tables = torch.from_numpy(b["tables"]).to(cuda_device)
    lens_d = torch.from_numpy(b["lens"]).to(cuda_device)
    mcl = int(b["lens"].max())
    ws = torch.empty(max(pa.pa_decode_mq_workspace_size(S, QL, Hq, Hkv, D, bs, mcl, 0),
                         pa.pa_decode_mq_workspace_size(S, QL, Hq, Hkv, D, bs, mcl, 128), 256),
                     dtype=torch.uint8, device=cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    for variant, psize in (("auto", 0), ("v1", 0), ("v2", 128)):
        out.fill_(5.0)
        pa.pa_decode_mq(out, b["q"], b["kc"], b["vc"], tables, lens_d, mcl, scale,
                        variant=variant, partition_size=psize, workspace=ws, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, variant
        assert max_err(bits(out), ref, dtype) <= TOL[dtype], variant
        for s, L in enumerate(lens):
            if L == 0:
                assert not bits(out[s]).any(), (variant, s)


@pytest.mark.parametrize("dtype,Hq,ramp", [("bf16", 32, "up"), ("bf16", 64, "up"),
                                           ("f16", 32, "up"), ("bf16", 64, "down")])
def test_multi_query_moving_references(cuda_device, mq_kernel, dtype, Hq, ramp):
    """Scores that keep growing along each context (K scaled up token by token, to about
    13x the first tokens' spread), so that every row's softmax reference moves again in
    later tiles and the kernels rescale their accumulators in the middle of a unit; and
    scores that shrink instead (the first tokens dominate, later weights underflow).  16
    and 32 query rows per kv head, every variant, against the oracle."""
    import paged_kv_cache_187_gb300 as pa
    QL, Hkv, D, bs = 4, 8, 128, 16
    lens = [130, 700, 2100, 4000, 257, 1029]
    if ramp == "up":
        k_ramp = lambda t, L: 0.5 + 6.0 * t / L
    else:
        k_ramp = lambda t, L: 6.5 - 6.0 * t / L
    b = _batch(cuda_device, lens, QL, Hq, Hkv, D, bs, dtype, seed=401 + Hq, k_ramp=k_ramp)
    scale = D ** -0.5
    ref = oracle.decode_mq(bits(b["q"]), b["okc"], b["ovc"], b["tables"], b["lens"],
                           np.float32(scale), dtype)
    S = len(lens)
    out = torch.empty_like(b["q"])
    tables = torch.from_numpy(b["tables"]).to(cuda_device)
    lens_d = torch.from_numpy(b["lens"]).to(cuda_device)
    mcl = int(b["lens"].max())
    ws = torch.empty(max(pa.pa_decode_mq_workspace_size(S, QL, Hq, Hkv, D, bs, mcl, 0),
                         pa.pa_decode_mq_workspace_size(S, QL, Hq, Hkv, D, bs, mcl, 128), 256),
                     dtype=torch.uint8, device=cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    for variant, psize in (("auto", 0), ("v1", 0), ("v2", 128)):
        out.fill_(5.0)
        pa.pa_decode_mq(out, b["q"], b["kc"], b["vc"], tables, lens_d, mcl, scale,
                        variant=variant, partition_size=psize, workspace=ws, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, variant
        st = err_stats(bits(out), ref, dtype)
        assert st.ok(dtype), (variant, st)


@pytest.mark.parametrize("dtype,Hq,Hkv,D,bs,ramp", [
    ("bf16", 32, 8, 128, 16, "up"),    # grouped-query heads: tensor-core path
    ("f16", 64, 8, 128, 32, "up"),
    ("bf16", 32, 8, 128, 16, "down"),
    ("f16", 8, 8, 128, 16, "up"),      # one head per kv head: CUDA-core path
    ("bf16", 16, 16, 64, 32, "down"),
])
def test_single_query_decode_moving_references(cuda_device, dtype, Hq, Hkv, D, bs, ramp):
    """The ordinary (single-query) decode on contexts whose scores grow, or shrink, along
    the sequence, so that the running maxima keep moving within a unit and across
    partitions: V1, V2 with two partition sizes and the automatic choice against the
    oracle (its multi-query decode with one query token is the ordinary decode)."""
    import paged_kv_cache_187_gb300 as pa
    lens = [130, 700, 2100, 4000, 257, 1029]
    if ramp == "up":
        k_ramp = lambda t, L: 0.5 + 6.0 * t / L
    else:
        k_ramp = lambda t, L: 6.5 - 6.0 * t / L
    b = _batch(cuda_device, lens, 1, Hq, Hkv, D, bs, dtype, seed=433 + Hq + D, k_ramp=k_ramp)
    scale = D ** -0.5
    ref = oracle.decode_mq(bits(b["q"]), b["okc"], b["ovc"], b["tables"], b["lens"],
                           np.float32(scale), dtype)[:, 0]
    S = len(lens)
    q = b["q"][:, 0].contiguous()
    out = torch.empty_like(q)
    tables = torch.from_numpy(b["tables"]).to(cuda_device)
    lens_d = torch.from_numpy(b["lens"]).to(cuda_device)
    mcl = int(b["lens"].max())
    ws = torch.empty(max(pa.pa_decode_v2_workspace_size(S, Hq, D, mcl, 2 * bs),
                         pa.pa_decode_auto_workspace_size(S, Hq, Hkv, D, bs, mcl), 256),
                     dtype=torch.uint8, device=cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    calls = {
        "v1": lambda: pa.pa_decode_v1(out, q, b["kc"], b["vc"], tables, lens_d, mcl, scale,
                                      status=status),
        "v2_512": lambda: pa.pa_decode_v2(out, q, b["kc"], b["vc"], tables, lens_d, mcl, scale,
                                          512, ws, status=status),
        "v2_2bs": lambda: pa.pa_decode_v2(out, q, b["kc"], b["vc"], tables, lens_d, mcl, scale,
                                          2 * bs, ws, status=status),
        "auto": lambda: pa.pa_decode_auto(out, q, b["kc"], b["vc"], tables, lens_d, mcl, scale,
                                          workspace=ws, status=status),
    }
    for name, call in calls.items():
        out.fill_(5.0)
        call()
        torch.cuda.synchronize()
        assert int(status.item()) == 0, name
        st = err_stats(bits(out), ref, dtype)
        assert st.ok(dtype), (name, st)


def test_multi_query_q_len_one_is_the_ordinary_decode(cuda_device):
    import paged_kv_cache_187_gb300 as pa
    lens = [5, 40, 300, 1000]
    b = _batch(cuda_device, lens, 1, 32, 8, 128, 16, "bf16", seed=91)
    tables = torch.from_numpy(b["tables"]).to(cuda_device)
    lens_d = torch.from_numpy(b["lens"]).to(cuda_device)
    out_mq = torch.empty_like(b["q"])
    out_v1 = torch.empty(b["q"].shape[0], 32, 128, dtype=b["q"].dtype, device=cuda_device)
    pa.pa_decode_mq(out_mq, b["q"], b["kc"], b["vc"], tables, lens_d, 1000, 0.088, variant="v1")
    pa.pa_decode_v1(out_v1, b["q"][:, 0].contiguous(), b["kc"], b["vc"], tables, lens_d, 1000, 0.088)
    torch.cuda.synchronize()
    assert torch.equal(out_mq[:, 0].view(torch.int16), out_v1.view(torch.int16))


def test_multi_query_full_size_llama3_8b_verify(cuda_device, mq_kernel):
    """Llama-3-8B heads (32 query, 8 kv, head_size 128), 16-token blocks, 4 tokens to
    verify per sequence, 24 sequences with contexts up to 4096: every row against the
    oracle, through the launch pa_decode_mq picks by itself."""
    import paged_kv_cache_187_gb300 as pa
    rng = np.random.default_rng(5)
    lens = rng.integers(1, 4097, size=24).astype(np.int32)
    lens[0], lens[1] = 4096, 3
    b = _batch(cuda_device, lens, 4, 32, 8, 128, 16, "bf16", seed=93)
    ref = oracle.decode_mq(bits(b["q"]), b["okc"], b["ovc"], b["tables"], b["lens"],
                           np.float32(128 ** -0.5), "bf16")
    S = lens.size
    tables = torch.from_numpy(b["tables"]).to(cuda_device)
    lens_d = torch.from_numpy(b["lens"]).to(cuda_device)
    ws = torch.empty(max(pa.pa_decode_mq_workspace_size(S, 4, 32, 8, 128, 16, 4096, 0), 256),
                     dtype=torch.uint8, device=cuda_device)
    out = torch.empty_like(b["q"])
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    pa.pa_decode_mq(out, b["q"], b["kc"], b["vc"], tables, lens_d, 4096, 128 ** -0.5,
                    workspace=ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert max_err(bits(out), ref, "bf16") <= TOL["bf16"]


def test_multi_query_host_errors(cuda_device):
    import paged_kv_cache_187_gb300 as pa
    b = _batch(cuda_device, [20], 2, 8, 8, 128, 16, "f16", seed=95)
    tables = torch.from_numpy(b["tables"]).to(cuda_device)
    lens_d = torch.from_numpy(b["lens"]).to(cuda_device)
    out = torch.empty_like(b["q"])
    with pytest.raises(pa.PAError):
        pa.pa_decode_mq(out, b["q"], b["kc"], b["vc"], tables, lens_d, 20, 0.1, variant="v2",
                        partition_size=24)    # not a multiple of block_size
    with pytest.raises(pa.PAError):
        pa.pa_decode_mq(out, b["q"], b["kc"], b["vc"], tables, lens_d, 20, 0.1, variant="v2",
                        partition_size=32, workspace=None)


@pytest.mark.parametrize("name,q_lens", [("l3_8b", (4,)), ("l3_70b", (2, 4))])
def test_multi_query_full_size_every_row(cuda_device, name, q_lens):
    """Multi-query decode over a full-size batch's pools (the last q_len tokens of every
    context are the new ones), through the launch pa_decode_mq picks by itself: Llama-3-8B
    heads with 4 tokens (16 rows per kv head), Llama-3-70B heads with 2 tokens (16 rows,
    32-token blocks) and 4 tokens (32 rows), all on the tcgen05 kernel.  Every
    (sequence, token, head) row against the oracle."""
    import paged_kv_cache_187_gb300 as pa
    from paged_kv_cache_187_gb300 import workloads as W
    from paged_kv_cache_187_gb300.runner import DecodeRunner
    from oracle_side import OracleState, err_stats, record_step
    w = W.WORKLOADS[name]
    r = DecodeRunner(w, device="cuda").next_step()
    r.run_reshape()
    torch.cuda.synchronize()
    assert int(r.status.item()) == 0
    st = record_step(r)
    o = OracleState(r, [st])
    del r.k_prefill, r.v_prefill
    S, Hq, Hkv, D = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_size
    mcl = r.step_max_context_len()
    for QL in q_lens:
        q = W.randn_16bit((S, QL, Hq, D), w.dtype, W.stream_seed(w, "q", 1 + QL), r.device)
        out = torch.full_like(q, 5.0)
        need = pa.pa_decode_mq_workspace_size(S, QL, Hq, Hkv, D, w.block_size, mcl, 0)
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=r.device)
        pa.pa_decode_mq(out, q, r.key_cache, r.value_cache, r.block_tables_d, r.context_lens_d,
                        mcl, w.scale, workspace=ws, status=r.status)
        torch.cuda.synchronize()
        assert int(r.status.item()) == 0
        ref = o.decode_mq(0, bits(q))
        e = err_stats(bits(out), ref, w.dtype)
        print(f"mq {name} q_len {QL}: {e}")
        assert e.ok(w.dtype), f"mq {name} q_len {QL}: {e}"
