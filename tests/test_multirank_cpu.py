"""The bench's multi-rank logic on CPU: two gloo ranks, each timing its own replica of
the step (weak scaling, no data-path collective).  Checks the rank environment, that the
job time is the slowest rank's, that the whole-job value counts every rank's bytes, and
that the ranks draw distinct synthetic inputs of the same shapes."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, ws: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        _checks(rank, ws, dist, out)
    except BaseException as e:   # report instead of leaving the parent waiting
        out.put((rank, repr(e), False, ()))
        raise
    finally:
        dist.destroy_process_group()


def _checks(rank, ws, dist, out):
    import bench
    from paged_kv_cache_187_gb300 import workloads as W
    cpu = torch.device("cpu")
    assert bench._dist() == (ws, rank, rank)
    # rank r took 10 * (r + 1) ms for 10 steps of 1 GB and 1000 sequence-tokens each
    tot = bench._job_totals(1e9, 1000, 10.0 * (rank + 1), 10, ws, cpu)
    bench._barrier(ws)
    # each rank's replica draws its own query stream
    w = W.WORKLOADS["tiny"]
    q = W.randn_16bit((w.num_seqs, w.num_q_heads, w.head_size), w.dtype,
                      W.stream_seed(w, "q", 0, rank), cpu)
    bits = q.view(torch.int16).to(torch.int32)      # gloo gathers 32-bit integers
    qs = [torch.empty_like(bits) for _ in range(ws)]
    dist.all_gather(qs, bits)
    distinct = all(not torch.equal(qs[i], qs[j]) for i in range(ws) for j in range(i + 1, ws))
    out.put((rank, tot, distinct, tuple(q.shape)))


def test_two_gloo_ranks_weak_scaling_totals():
    ws = 2
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, out)) for r in range(ws)]
    for p in procs:
        p.start()
    res = [out.get(timeout=120) for _ in range(ws)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort(key=lambda x: x[0])
    for rank, tot, distinct, shape in res:
        assert isinstance(tot, dict), f"rank {rank}: {tot}"
        # the slowest rank (rank 1: 20 ms / 10 steps) sets the job time on every rank
        assert tot["ms_per_step"] == pytest.approx(2.0)
        # 2 ranks x 1 GB per step in 2 ms
        assert tot["value"] == pytest.approx(1000.0)
        assert tot["seq_tokens_per_s"] == pytest.approx(2 * 1000 / 2e-3)
        assert distinct
        assert shape == res[0][3]
