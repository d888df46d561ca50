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
