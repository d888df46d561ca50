"""pa_decode_v2_noalloc: the V2 decode for callers that may not allocate device memory
(for example an inference runtime's plugin enqueue path, which owns all device memory,
or code that must not call cudaMalloc during stream capture).  Its scratch is a fixed
static device array inside the library instead of a caller workspace.

This file sorts last so that a run stopping at its first failure has run every other
test first.  It passes alone in a fresh process and after the rest of the suite.
"""
import dataclasses

import numpy as np
import pytest
import torch

from oracle_side import bits

pytestmark = pytest.mark.gpu


def _setup():
    from paged_kv_cache_187_gb300 import workloads as W
    from paged_kv_cache_187_gb300.runner import DecodeRunner
    base = W.WORKLOADS["l3_8b"]
    w = dataclasses.replace(base, num_seqs=64)
    lens = W.start_context_lens(base)[:64]
    r = DecodeRunner(w, device="cuda", start_lens=lens).next_step()
    r.run_reshape()
    return r


def _existing(pa, r, P):
    out = torch.empty_like(r.out)
    mcl = r.step_max_context_len()
    ws = torch.empty(pa.pa_decode_v2_workspace_size(r.w.num_seqs, r.w.num_q_heads,
                                                    r.w.head_size, mcl, P),
                     dtype=torch.uint8, device=r.device)
    pa.pa_decode_v2(out, r.q, r.key_cache, r.value_cache, r.block_tables_d, r.context_lens_d,
                    mcl, r.w.scale, P, ws, status=r.status)
    return out


def test_noalloc_matches_workspace_entry_point_on_two_calls(cuda_device):
    """Two calls in a row, the second reusing the scratch the first left behind: each is
    bit-identical to pa_decode_v2 with a caller workspace (the same kernels on the same
    inputs), allocates no device memory, and meets the oracle's bound."""
    import paged_kv_cache_187_gb300 as pa
    from oracle_side import OracleState, err_stats, record_step
    r = _setup()
    mcl = r.step_max_context_len()
    ref64 = OracleState(r, [record_step(r)]).decode(0, record_step(r))
    for P in (512, 128):
        need = pa.pa_decode_v2_workspace_size(r.w.num_seqs, r.w.num_q_heads, r.w.head_size,
                                              mcl, P)
        assert need <= pa.PA_NOALLOC_SCRATCH_BYTES
        ref = _existing(pa, r, P)
        got = torch.full_like(r.out, float("nan"))
        torch.cuda.synchronize()
        before = (torch.cuda.memory_allocated(cuda_device), torch.cuda.memory_reserved(cuda_device))
        pa.pa_decode_v2_noalloc(got, r.q, r.key_cache, r.value_cache, r.block_tables_d,
                                r.context_lens_d, mcl, r.w.scale, P, status=r.status)
        torch.cuda.synchronize()
        after = (torch.cuda.memory_allocated(cuda_device), torch.cuda.memory_reserved(cuda_device))
        assert before == after
        assert int(r.status.item()) == 0
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), f"P={P}"
        e = err_stats(bits(got), ref64, r.w.dtype)
        assert e.ok(r.w.dtype), f"P={P}: {e}"


def test_noalloc_rejects_sizes_beyond_its_scratch(cuda_device):
    import paged_kv_cache_187_gb300 as pa
    r = _setup()
    huge = 1 << 22            # a max_context_len whose partials cannot fit the scratch
    assert pa.pa_decode_v2_workspace_size(r.w.num_seqs, r.w.num_q_heads, r.w.head_size,
                                          huge, 16) > pa.PA_NOALLOC_SCRATCH_BYTES
    before = r.out.clone()
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode_v2_noalloc(r.out, r.q, r.key_cache, r.value_cache, r.block_tables_d,
                                r.context_lens_d, huge, r.w.scale, 16, status=r.status)
    assert e.value.status == pa.PA_ERR_WORKSPACE and "scratch" in str(e.value)
    # a bad argument is reported as such, before the scratch size, as pa_decode_v2 does
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode_v2_noalloc(r.out, r.q, r.key_cache, r.value_cache, r.block_tables_d,
                                r.context_lens_d, huge, r.w.scale, 24, status=r.status)
    assert e.value.status == pa.PA_ERR_INVALID_ARG and "partition_size" in str(e.value)
    torch.cuda.synchronize()
    assert torch.equal(r.out.view(torch.int16), before.view(torch.int16))
