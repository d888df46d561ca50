"""GPU tests of the host-buffer entry point and of the bounded-wait failure path."""
import dataclasses

import numpy as np
import pytest
import torch

from oracle_side import OracleState, TOL, bits, max_err, record_step

pytestmark = pytest.mark.gpu


def _runner(w, **kw):
    from paged_kv_cache_187_gb300.runner import DecodeRunner
    return DecodeRunner(w, device="cuda", **kw)


def test_decode_step_host_matches_device_step_and_oracle(cuda_device):
    import paged_kv_cache_187_gb300 as pa
    from paged_kv_cache_187_gb300 import workloads as W
    base = W.WORKLOADS["l3_8b"]
    w = dataclasses.replace(base, num_seqs=32)
    lens = W.start_context_lens(base)[:32]
    # two runners with identical state: one steps from device buffers, one from host
    ra = _runner(w, start_lens=lens).next_step()
    rb = _runner(w, start_lens=lens).next_step()
    ra.run_step()
    mcl = rb.step_max_context_len()
    pin = lambda t: t.cpu().pin_memory()
    out_h = torch.empty(rb.out.shape, dtype=rb.out.dtype).pin_memory()
    staging = torch.empty(pa.pa_decode_step_host_staging_size(w.num_seqs, w.num_q_heads,
                                                              w.num_kv_heads, w.head_size,
                                                              rb.max_blocks),
                          dtype=torch.uint8, device=cuda_device)
    pa.pa_decode_step_host(out_h, pin(rb.q), pin(rb.k_new), pin(rb.v_new),
                           torch.from_numpy(rb.slots).pin_memory(),
                           torch.from_numpy(rb.block_tables).pin_memory(),
                           torch.from_numpy(rb.context_lens).pin_memory(),
                           rb.key_cache, rb.value_cache, mcl, w.scale, staging,
                           workspace=rb.workspace, status=rb.status)
    torch.cuda.current_stream().synchronize()
    assert int(rb.status.item()) == 0
    assert torch.equal(rb.key_cache.view(torch.int16), ra.key_cache.view(torch.int16))
    assert torch.equal(out_h.view(torch.int16), ra.out.cpu().view(torch.int16))
    st = record_step(rb)
    o = OracleState(rb, [st])
    assert max_err(out_h.view(torch.int16).numpy().view(np.uint16), o.decode(0, st),
                   w.dtype) <= TOL[w.dtype]


def test_decode_step_host_overlapped_matches_device_steps(cuda_device):
    """Four steps through pa_decode_step_host_overlapped (copies on their own streams, a ring
    of two staging areas, each step queued before the previous one's output is read) give
    the same bits as the same four steps taken from device buffers."""
    import paged_kv_cache_187_gb300 as pa
    from paged_kv_cache_187_gb300 import workloads as W
    base = W.WORKLOADS["l3_8b"]
    w = dataclasses.replace(base, num_seqs=32, steps=4)
    lens = W.start_context_lens(base)[:32]
    ra = _runner(w, start_lens=lens)
    rb = _runner(w, start_lens=lens)
    compute = torch.cuda.current_stream()
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ring = 2
    size = pa.pa_decode_step_host_staging_size(w.num_seqs, w.num_q_heads, w.num_kv_heads,
                                               w.head_size, rb.max_blocks)
    staging = [torch.empty(size, dtype=torch.uint8, device=cuda_device) for _ in range(ring)]
    staged = [torch.cuda.Event() for _ in range(ring)]
    done = [torch.cuda.Event() for _ in range(ring)]
    fin = [torch.cuda.Event() for _ in range(ring)]
    for e in staged + done + fin:
        e.record(d2h)
    pin = lambda t: t.cpu().pin_memory()
    pending = [None] * ring
    checked = 0

    def check(j):
        nonlocal checked
        if pending[j] is None:
            return
        out_h, ref = pending[j]
        fin[j].synchronize()
        assert torch.equal(out_h.view(torch.int16), ref.view(torch.int16))
        pending[j] = None
        checked += 1

    for i in range(4):
        ra.next_step()
        ra.run_step()
        ref = ra.out.cpu()
        rb.next_step()
        j = i % ring
        check(j)          # the slot's previous step has been read back
        out_h = torch.empty(rb.out.shape, dtype=rb.out.dtype).pin_memory()
        pa.pa_decode_step_host_overlapped(
            out_h, pin(rb.q), pin(rb.k_new), pin(rb.v_new),
            torch.from_numpy(rb.slots).pin_memory(), torch.from_numpy(rb.block_tables).pin_memory(),
            torch.from_numpy(rb.context_lens).pin_memory(), rb.key_cache, rb.value_cache,
            rb.step_max_context_len(), w.scale, staging[j], compute, h2d, d2h, staged[j], done[j],
            workspace=rb.workspace, status=rb.status)
        fin[j].record(d2h)
        pending[j] = (out_h, ref)
    for j in range(ring):
        check(j)
    assert checked == 4
    torch.cuda.synchronize()
    assert int(rb.status.item()) == 0
    assert torch.equal(rb.key_cache.view(torch.int16), ra.key_cache.view(torch.int16))
    with pytest.raises(pa.PAError):   # the copies on the compute stream
        pa.pa_decode_step_host_overlapped(
            out_h, pin(rb.q), pin(rb.k_new), pin(rb.v_new),
            torch.from_numpy(rb.slots).pin_memory(), torch.from_numpy(rb.block_tables).pin_memory(),
            torch.from_numpy(rb.context_lens).pin_memory(), rb.key_cache, rb.value_cache,
            rb.step_max_context_len(), w.scale, staging[0], compute, compute, d2h, staged[0], done[0],
            workspace=rb.workspace, status=rb.status)


def test_bounded_wait_reports_timeout_and_context_survives(cuda_device):
    import paged_kv_cache_187_gb300 as pa
    from paged_kv_cache_187_gb300 import workloads as W
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    pa.pa_selftest_wait_timeout(status, 20000)          # 20 ms on a barrier nobody completes
    torch.cuda.synchronize()
    assert int(status.item()) == pa.PA_DEVERR_TIMEOUT
    with pytest.raises(pa.PAError):
        pa.pa_selftest_wait_timeout(status, 0)
    # the context is still usable: a normal decode runs and matches the oracle
    r = _runner(W.WORKLOADS["tiny"]).next_step()
    r.run_step()
    torch.cuda.synchronize()
    assert int(r.status.item()) == 0
    st = record_step(r)
    o = OracleState(r, [st])
    assert max_err(bits(r.out), o.decode(0, st), "f16") <= TOL["f16"]
