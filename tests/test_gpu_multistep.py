"""GPU: the multi-step decode loop run on the device (pa_advance_step between steps, blocks
reserved up front) and its CUDA-graph replay, against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from oracle_side import OracleState, StepRecord, TOL, bits, max_err

pytestmark = pytest.mark.gpu


def test_device_multistep_loop_and_graph_replay(cuda_device):
    from paged_kv_cache_187_gb300 import workloads as W
    from paged_kv_cache_187_gb300.runner import DecodeRunner
    w = W.WORKLOADS["l3_70b"]
    k = w.steps
    r = DecodeRunner(w, device="cuda").setup_multistep(k)
    dev_slots, dev_lens = [], []

    def on_step(j):
        dev_slots.append(r.slots_d.cpu().numpy().copy())
        dev_lens.append(r.context_lens_d.cpu().numpy().copy())

    r.run_multistep(on_step=on_step)
    torch.cuda.synchronize()
    assert int(r.status.item()) == 0
    eager = [bits(o) for o in r.ms_out]
    host_slots = r.finish_multistep()
    # the device advanced exactly as the host allocator does, step by step
    for j in range(k):
        assert np.array_equal(dev_slots[j], host_slots[j])
        assert np.array_equal(dev_lens[j], r.ms_lens0 + j + 1)
    # the oracle replays the same requests: reserve, then one append per step
    recs = [StepRecord(bits(r.ms_q[j]), bits(r.ms_k_new[j]), bits(r.ms_v_new[j]), dev_slots[j],
                       dev_lens[j], r.block_tables) for j in range(k)]
    rng = np.random.default_rng(3)
    seqs = sorted({int(np.argmin(r.ms_lens0)), int(np.argmax(r.ms_lens0))} |
                  set(int(x) for x in rng.choice(w.num_seqs, 6, replace=False)))
    rows = [(s, h) for s in seqs for h in (0, w.num_q_heads - 1)]
    o = OracleState(r, recs, seqs=seqs, reserve=k)
    for j in range(k):
        assert np.array_equal(o.step_slots[j], dev_slots[j])
        assert np.array_equal(o.step_tables[j], r.block_tables)
        err = max_err(eager[j], o.decode(j, recs[j], rows=rows), w.dtype, rows=rows)
        assert err <= TOL[w.dtype], f"step {j}: {err}"
    # CUDA graph of the whole loop: replays give the same bits
    r.run_multistep()          # one more eager pass: identical inputs, idempotent writes
    g = r.capture_multistep()
    for o_ in r.ms_out:
        o_.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert int(r.status.item()) == 0
    for j in range(k):
        assert np.array_equal(bits(r.ms_out[j]), eager[j])


def test_advance_step_flags_missing_block(cuda_device):
    import paged_kv_cache_187_gb300 as pa
    lens = torch.tensor([15, 16], dtype=torch.int32, device=cuda_device)
    slots = torch.zeros(2, dtype=torch.int32, device=cuda_device)
    tables = torch.tensor([[3, -1], [5, -1]], dtype=torch.int32, device=cuda_device)
    pos = torch.zeros(2, dtype=torch.int64, device=cuda_device)
    tok = torch.zeros(2, dtype=torch.int64, device=cuda_device)
    sampled = torch.tensor([11, 22], dtype=torch.int64, device=cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    pa.pa_advance_step(lens, slots, tables, 16, 8, input_positions=pos, input_tokens=tok,
                       sampled_token_ids=sampled, status=status)
    torch.cuda.synchronize()
    # seq 0: position 15 in block 3 -> slot 63; seq 1: position 16 needs a block it lacks
    assert lens.tolist() == [16, 17] and slots.tolist() == [63, -1]
    assert pos.tolist() == [15, 16] and tok.tolist() == [11, 22]
    assert int(status.item()) == pa.PA_DEVERR_BAD_BLOCK
