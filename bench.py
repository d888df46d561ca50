"""Benchmark of one paged-attention decode step on GB300.

A step is the whole hot path for one batch: reshape_and_cache of every sequence's new
K/V row, then the paged decode (pa_decode_step = reshape + pa_decode_auto), on the
Llama-3-8B-shaped GQA workload (256 sequences, 32 query / 8 kv heads, head size 128,
block size 16, bf16, lognormal contexts).  Prints ONE JSON line.

  value    device-resident throughput: algorithmic bytes (K+V of every context token
           and kv head, plus Q and out) per second, inputs already in HBM;
  e2e      the same metric through the public API with the step's inputs copied from
           pinned host memory (host allocator append, H2D of q/k/v/metadata, the step,
           D2H of out, synchronise) -- every step;
  roofline the decode kernel alone (CUDA events recorded by the library around that
           launch, in a kernel-only pass of its own after the timed steps) against the
           measured HBM copy bandwidth;
  per_config  the other workloads of the suite, each timed the same way: the
           Llama-2-7B MHA batch, the skewed long-context batch under V1, V2 and the
           automatic choice, the 8-step Llama-3-70B loop (issued eagerly and as one CUDA
           graph), fp8 KV caches on the Llama-3-8B and Llama-3-70B batches, and multi-query
           decode with 4 query tokens on the Llama-3-8B batch.

--impl reference times the fp64 CPU oracle (the baseline arm) on a bounded sample of
the same workload.  Under torchrun every rank runs its own replica (weak scaling);
rank 0 prints the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn effective KV HBM GB/s (% of GB300 peak); seq-tokens/s per layer"
WORKLOAD = "l3_8b"
SPEC_HBM_GBS = 8000.0


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# The sources that decide what a measured decode kernel does and how it is launched: the
# kernel templates, the instantiation unit of its family, the plan kernel and the host side.
_COMMON_SOURCES = ("pa_decode.cuh", "pa_decode_family.cuh", "pa_device.cuh", "pa_internal.h",
                   "pa_once.h", "pa_aux.cu", "pa_host.cpp")
FAMILY_SOURCES = {
    "bf16_d128": _COMMON_SOURCES + ("pa_decode_bf16_d128.cu",),
    "f16_d128": _COMMON_SOURCES + ("pa_decode_f16_d128.cu",),
    "fp8": _COMMON_SOURCES + ("pa_decode_fp8.cu",),
    "mq_tc": _COMMON_SOURCES + ("pa_decode_tc.cuh", "pa_decode_tc.cu"),
    "mq_mma": _COMMON_SOURCES + ("pa_decode_mq_bf16.cu", "pa_decode_mq_f16.cu"),
}
KERNEL_SOURCES = FAMILY_SOURCES["bf16_d128"]


def _kernel_hash(family: str = "bf16_d128") -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_187_gb300", "csrc")
    for f in FAMILY_SOURCES[family]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def _traffic_record(record: str = "paged_decode_l3_8b"):
    """dram bytes per decode launch from the committed ncu record profiles/<record>_traffic.txt,
    if it was taken on the current sources of its kernel family (same hash); else None."""
    path = os.path.join(ROOT, "profiles", f"{record}_traffic.txt")
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_sources_sha256_16") != _kernel_hash(kv.get("family", "bf16_d128")):
            return None
        return float(kv["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t_start = self.t_stop = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        def reader():
            for line in self.proc.stdout:
                self.lines.append((time.time(), line.strip()))
        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def _rows(self, t0=None, t1=None):
        rows = []
        for t, line in self.lines:
            if t0 is not None and not (t0 <= t <= (t1 or 1e30)):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((t, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        return rows

    def summary(self, phase=None):
        """Clocks over the timed steps, or -- when that region is shorter than the sampling
        period -- over the whole GPU measurement phase (`phase` = (t0, t1): the timed steps,
        the kernel-only passes and the other workloads, all under the same load)."""
        if not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
        inside = self._rows(self.t_start, self.t_stop) if self.t_start else []
        window = "timed region"
        use = inside
        if len(inside) < 3 and phase is not None:
            use = self._rows(*phase)
            window = (f"GPU measurement phase ({phase[1] - phase[0]:.1f} s: timed steps, kernel "
                      f"passes, other workloads); {len(inside)} sample(s) inside the timed steps")
        if not use:
            use = self._rows()
            window = "whole run"
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unparsed nvidia-smi output"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "sm_min_mhz": min(r[1] for r in use),
                "reasons": reasons, "samples": len(use), "window": window}


def _smi_index(cuda_index: int) -> str:
    """nvidia-smi's id of the CUDA device (CUDA_VISIBLE_DEVICES renumbers devices)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").strip()
    if vis:
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        if cuda_index < len(ids):
            return ids[cuda_index]
    return str(cuda_index)


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _max_over_ranks(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def _job_totals(bytes_step: float, tokens_step: float, ms_total_local: float, steps: int,
                ws: int, device) -> dict:
    """Whole-job figures of a weak-scaling run: every rank processed its own replica of
    the step `steps` times; the job took as long as the slowest rank."""
    ms_step = _max_over_ranks(ms_total_local, ws, device) / steps
    return {"ms_per_step": ms_step,
            "value": ws * bytes_step / (ms_step * 1e-3) / 1e9,
            "seq_tokens_per_s": ws * tokens_step / (ms_step * 1e-3)}


# ----------------------------------------------------------------------------- CPU oracle
def time_oracle(r, budget_s: float = 15.0):
    """Times the fp64 oracle (single thread) on whole sequences of the runner's current
    step, in batch order, until about `budget_s` of CPU work has been spent."""
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle
    from oracle_side import OracleState, record_step
    st = record_step(r)
    w = r.w
    chosen, spent, nbytes, ntok = [], 0.0, 0, 0
    # estimate per-token cost on a short prefix first
    for s in range(w.num_seqs):
        chosen.append(s)
        o = OracleState(r, [st], seqs=[s])
        only = np.zeros((w.num_seqs, w.num_q_heads), np.uint8)
        only[s, :] = 1
        t0 = time.perf_counter()
        oracle.decode_v1(st.q, o.k_cache, o.v_cache, o.tables(0), o.step_lens[0],
                         np.float32(w.scale), w.dtype, only=only)
        spent += time.perf_counter() - t0
        L = int(r.context_lens[s])
        nbytes += L * w.num_kv_heads * w.head_size * 2 * 2 + 2 * w.num_q_heads * w.head_size * 2
        ntok += L
        if spent >= budget_s:
            break
    return {"seconds": spent, "bytes": nbytes, "tokens": ntok, "seqs": len(chosen)}


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import torch
    from paged_kv_cache_187_gb300 import workloads as W
    from paged_kv_cache_187_gb300.runner import DecodeRunner
    w = W.WORKLOADS[WORKLOAD]
    r = DecodeRunner(w, device="cuda").next_step()
    r.run_reshape()
    torch.cuda.synchronize()
    per_step_budget = max(1.0, 60.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        time_oracle(r, per_step_budget)
    samples = [time_oracle(r, per_step_budget) for _ in range(args.steps)]
    sec = sum(x["seconds"] for x in samples)
    byt = sum(x["bytes"] for x in samples)
    tok = sum(x["tokens"] for x in samples)
    gbs = byt / sec / 1e9
    sample = (f"each step: the fp64 oracle (one thread) over whole sequences of the {w.name} "
              f"batch in order until ~{per_step_budget:.1f} s; {samples[0]['seqs']} seqs, "
              f"{samples[0]['tokens']} context tokens in step 1")
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": _config(w, r),
        "seq_tokens_per_s": tok / sec,
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _config(w, r):
    return {
        "workload": f"{w.name}: {w.description}: {w.num_seqs} seqs, {w.num_q_heads} q / "
                    f"{w.num_kv_heads} kv heads, head_size {w.head_size}, block_size "
                    f"{w.block_size}, {w.dtype}, contexts lognormal(6.9, 0.8) clipped [16, 8192]",
        "num_seqs": w.num_seqs, "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
        "head_size": w.head_size, "block_size": w.block_size,
        "context_tokens": int(r.context_lens.sum()), "max_context_len": int(r.context_lens.max()),
        "step": "pa_decode_step: reshape_and_cache of the new tokens + pa_decode_auto",
        "l2": f"no flush: {r.kv_bytes() / 1e9:.2f} GB of K/V per step read once vs 129 MB L2",
        "seed": w.seed,
    }


# ----------------------------------------------------------------------------- GPU arm
def _spread(samples_ms):
    """mean / median / min / max / stdev in microseconds of a list of durations in ms."""
    s = sorted(samples_ms)
    n = len(s)
    return {"n": n, "mean_us": 1e3 * sum(s) / n, "median_us": 1e3 * s[n // 2],
            "min_us": 1e3 * s[0], "max_us": 1e3 * s[-1],
            "stdev_us": 1e3 * (statistics.pstdev(s) if n > 1 else 0.0)}


def kernel_samples(pa, fn, n, device):
    """Durations (ms) of the decode kernel alone over n calls of fn: the library records a
    pair of CUDA events on the launching stream right around its decode launch."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    for a, b in evs:            # materialise the CUDA events before handing them over
        a.record()
        b.record()
    torch.cuda.synchronize(device)
    try:
        for a, b in evs:
            pa.pa_set_kernel_events(a, b)
            fn()
    finally:
        pa.pa_set_kernel_events(None, None)
    torch.cuda.synchronize(device)
    return [a.elapsed_time(b) for a, b in evs]


def steps_ms(fn, n, device):
    """Mean time (ms) of one call of fn over n back-to-back calls, CUDA events around all."""
    import torch
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    torch.cuda._sleep(2_000_000)      # the GPU is busy while the host queues the calls
    a.record()
    for _ in range(n):
        fn()
    b.record()
    torch.cuda.synchronize(device)
    return a.elapsed_time(b) / n


def _entry(desc, kernel, bytes_launch, tokens, samples, peak, family=None, record=None, **extra):
    k = _spread(samples)
    gbs = bytes_launch / (k["mean_us"] * 1e-6) / 1e9
    e = {"workload": desc, "kernel": kernel, "bytes_per_launch": int(bytes_launch),
         "seq_tokens": int(tokens), "kernel_us": k, "GBps": gbs, "frac": gbs / peak,
         "pct_of_spec_8000_GBps": 100.0 * gbs / SPEC_HBM_GBS,
         "seq_tokens_per_s": tokens / (k["mean_us"] * 1e-6),
         "traffic": _traffic_record(record) if record else None}
    e.update(extra)
    return e


def run_per_config(args, device, peak):
    """The suite's other workloads, one at a time (each freed before the next): the decode
    kernel's duration over >= 20 launches (events around that launch only), its bytes and
    roofline fraction, and where a step has more to it, the step's own time."""
    import torch
    import paged_kv_cache_187_gb300 as pa
    from paged_kv_cache_187_gb300 import workloads as W
    from paged_kv_cache_187_gb300.runner import DecodeRunner
    n = max(20, args.kernel_samples)
    out = {}

    def runner(name, **kw):
        r = DecodeRunner(W.WORKLOADS[name], device=device, **kw).next_step()
        r.run_reshape()
        del r.k_prefill, r.v_prefill           # only the pools are needed from here on
        torch.cuda.empty_cache()
        return r

    def warm(fn, k=3):
        for _ in range(k):
            fn()
        torch.cuda.synchronize(device)

    def mq_entry(r, QL, desc, record, single_samples,
                 kernel="paged_decode_tc_kernel (tcgen05, auto)"):
        """Multi-query decode (QL causal query tokens per sequence) over r's pools, with its
        time over the single-query decode kernel's on the same pools."""
        w = r.w
        S, Hq, D = w.num_seqs, w.num_q_heads, w.head_size
        mcl = r.step_max_context_len()
        q = W.randn_16bit((S, QL, Hq, D), w.dtype, W.stream_seed(w, "q", 1), r.device)
        o = torch.empty_like(q)
        wsz = pa.pa_decode_mq_workspace_size(S, QL, Hq, w.num_kv_heads, D, w.block_size, mcl, 0)
        wsb = torch.empty(max(wsz, 256), dtype=torch.uint8, device=r.device)
        fn = lambda: pa.pa_decode_mq(o, q, r.key_cache, r.value_cache, r.block_tables_d,
                                     r.context_lens_d, mcl, w.scale, workspace=wsb, status=r.status)
        warm(fn)
        e = _entry(desc, kernel,
                   r.kv_bytes() + 2 * (QL - 1) * S * Hq * D * 2, r.seq_tokens(),
                   kernel_samples(pa, fn, n, device), peak, record=record,
                   rows_per_kv_head=QL * Hq // w.num_kv_heads)
        e["over_single_query_time"] = e["kernel_us"]["mean_us"] / _spread(single_samples)["mean_us"]
        torch.cuda.synchronize(device)
        assert int(r.status.item()) == 0
        return e

    # Llama-2-7B MHA, fp16 (CUDA-core path)
    r = runner("l2_7b")
    fn = lambda: r.run_decode("auto")
    warm(fn)
    v, P = pa.pa_decode_auto_plan(r.w.num_seqs, r.w.num_q_heads, r.w.num_kv_heads,
                                  r.w.head_size, r.w.block_size, r.step_max_context_len())
    out["l2_7b"] = _entry("Llama-2-7B-shaped MHA decode: 64 seqs, 32/32 heads, head_size 128, "
                          "block 16, fp16, contexts U[512, 2048]", "paged_decode_kernel (auto)",
                          r.kv_bytes(), r.seq_tokens(), kernel_samples(pa, fn, n, device), peak,
                          record="paged_decode_l2_7b", variant=f"v{v}",
                          step_us=1e3 * steps_ms(lambda: r.run_step(), n, device))
    del r, fn
    torch.cuda.empty_cache()

    # skewed batch: 8 x 32768 + 248 x 128 tokens, 40/40 heads, fp16 -- V1 against V2
    r = runner("skew")
    res = {}
    for name, variant, P in (("v1", "v1", None), ("v2_p512", "v2", 512), ("auto", "auto", None)):
        fn = (lambda variant=variant, P=P: r.run_decode(variant, partition_size=P))
        warm(fn)
        res[name] = kernel_samples(pa, fn, n, device)
    e = _entry("Skewed long-context batch, LLaMA-13B-shaped: 8 seqs at 32768 + 248 at 128 "
               "tokens, 40/40 heads, head_size 128, block 16, fp16", "paged_decode_kernel (auto)",
               r.kv_bytes(), r.seq_tokens(), res["auto"], peak, record="paged_decode_skew")
    e["variants"] = {k: _entry(e["workload"], f"paged_decode_kernel ({k})", r.kv_bytes(),
                               r.seq_tokens(), x, peak) for k, x in res.items() if k != "auto"}
    for k in e["variants"].values():
        del k["workload"]
    e["v1_over_v2_time"] = (e["variants"]["v1"]["kernel_us"]["mean_us"] /
                            e["variants"]["v2_p512"]["kernel_us"]["mean_us"])
    e["v1_over_auto_time"] = (e["variants"]["v1"]["kernel_us"]["mean_us"] /
                              e["kernel_us"]["mean_us"])
    out["skew"] = e
    del r, res
    torch.cuda.empty_cache()

    # Llama-3-70B 8-step loop: decode kernel of step 0, and the whole loop eager / graph
    r = runner("l3_70b")
    fn = lambda: r.run_decode("auto")
    warm(fn)
    ks = kernel_samples(pa, fn, n, device)
    bytes0, tok0 = r.kv_bytes(), r.seq_tokens()
    # multi-query decode over the same pools, 4 query tokens per sequence: 32 query rows
    # per kv head (the tcgen05 kernel's 32-row units)
    out["mq4_l3_70b"] = mq_entry(r, 4, "Llama-3-70B-shaped batch (first step), 4 query tokens "
                                 "per sequence (causal within them): 32 query rows per kv head",
                                 "paged_decode_mq4_l3_70b", ks)
    del r, fn
    torch.cuda.empty_cache()
    # the loop starts from the pre-loop lengths: a runner of its own, no step taken yet
    r = DecodeRunner(W.WORKLOADS["l3_70b"], device=device)
    del r.k_prefill, r.v_prefill
    torch.cuda.empty_cache()
    k = r.w.steps
    r.setup_multistep(k)
    lens0 = r.ms_lens0.astype(np.int64)
    w = r.w
    tokens = sum(int((lens0 + j + 1).sum()) for j in range(k))
    loop_bytes = tokens * w.num_kv_heads * w.head_size * 4 + k * 4 * w.num_seqs * w.num_q_heads * w.head_size
    r.run_multistep()
    torch.cuda.synchronize(device)
    graph = r.capture_multistep()
    loops = max(5, n // 4)
    warm(r.run_multistep, 2)
    warm(graph.replay, 2)
    eager = [steps_ms(r.run_multistep, 1, device) for _ in range(loops)]
    replay = [steps_ms(graph.replay, 1, device) for _ in range(loops)]
    assert int(r.status.item()) == 0
    e = _entry("Llama-3-70B-shaped layer: 512 seqs, 64 q / 8 kv heads, head_size 128, block 32, "
               "bf16, start contexts U[1, 4096]; decode kernel of the first step",
               "paged_decode_kernel (auto)", bytes0, tok0, ks, peak, record="paged_decode_l3_70b")
    for name, t in (("eager", eager), ("graph", replay)):
        ms = sorted(t)[len(t) // 2]
        e["loop_" + name] = {"steps": k, "loops": loops, "loop_ms_median": ms,
                             "loop_ms_min": min(t), "loop_ms_max": max(t),
                             "us_per_step": 1e3 * ms / k, "GBps": loop_bytes / (ms * 1e-3) / 1e9,
                             "frac": loop_bytes / (ms * 1e-3) / 1e9 / peak,
                             "seq_tokens_per_s": tokens / (ms * 1e-3)}
    e["loop_bytes"] = loop_bytes
    e["loop_step"] = ("per step: pa_advance_step, then pa_decode_step (reshape_and_cache of the "
                      "512 new tokens + auto decode) on the device")
    out["l3_70b_loop"] = e
    del r, graph
    torch.cuda.empty_cache()

    # fp8 E4M3 KV caches
    for name, desc in (("l3_8b", "Llama-3-8B-shaped GQA batch over fp8 E4M3 pools (block 16)"),
                       ("l3_70b", "Llama-3-70B-shaped GQA batch over fp8 E4M3 pools (block 32)")):
        r = runner(name, kv_fp8=True)
        fn = lambda: r.run_decode("auto")
        warm(fn)
        out["fp8_" + name] = _entry(desc, "paged_decode_kernel (fp8 cache, auto)", r.kv_bytes(),
                                    r.seq_tokens(), kernel_samples(pa, fn, n, device), peak,
                                    record=f"paged_decode_fp8_{name}")
        del r, fn
        torch.cuda.empty_cache()

    # multi-query decode, 4 query tokens per sequence, over the Llama-3-8B batch's pools
    r = runner("l3_8b")
    fn = lambda: r.run_decode("auto")
    warm(fn)
    ks = kernel_samples(pa, fn, n, device)
    out["mq4_l3_8b"] = mq_entry(r, 4, "Llama-3-8B-shaped batch, 4 query tokens per sequence "
                                "(causal within them): 16 query rows per kv head",
                                "paged_decode_mq4_l3_8b", ks)
    # 2 query tokens: 8 rows per kv head, the mma.sync multi-query kernel
    out["mq2_l3_8b"] = mq_entry(r, 2, "Llama-3-8B-shaped batch, 2 query tokens per sequence "
                                "(causal within them): 8 query rows per kv head",
                                "paged_decode_mq2_l3_8b", ks, kernel="paged_decode_kernel (mma.sync multi-query, auto)")
    del r, fn
    torch.cuda.empty_cache()
    return out


def run_gpu(args):
    import torch
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(device)
    import paged_kv_cache_187_gb300 as pa
    from paged_kv_cache_187_gb300 import workloads as W
    from paged_kv_cache_187_gb300.runner import DecodeRunner

    w = W.WORKLOADS[WORKLOAD]
    r = DecodeRunner(w, device=device, rank=rank).next_step()
    stream = torch.cuda.current_stream(device)
    variant, psize = pa.pa_decode_auto_plan(w.num_seqs, w.num_q_heads, w.num_kv_heads,
                                            w.head_size, w.block_size, r.step_max_context_len())
    # reshape_and_cache, then the decode (V1) or the plan and the decode (V2: the
    # partition merge runs inside the decode kernel)
    launches_per_step = 2 if variant == 1 else 3
    bytes_step = r.kv_bytes()
    tokens_step = r.seq_tokens()
    peak, peak_kind = _peaks()

    # ---- device-resident timing: K steps of reshape + decode, nothing else in the stream
    for _ in range(args.warmup):
        r.run_step()
    K = args.steps
    clocks = ClockSampler(_smi_index(device.index or 0))
    clocks.start()
    time.sleep(0.3)
    phase0 = time.time()
    t_start = torch.cuda.Event(enable_timing=True)
    t_stop = torch.cuda.Event(enable_timing=True)
    _barrier(ws)
    torch.cuda.synchronize(device)
    # A sleeping kernel ahead of the start event keeps the GPU busy while the host queues
    # the first steps, so the timed region starts with work queued, as in a running server.
    torch.cuda._sleep(2_000_000)
    clocks.t_start = time.time()
    t_start.record(stream)
    for i in range(K):
        r.run_step()
    t_stop.record(stream)
    torch.cuda.synchronize(device)
    clocks.t_stop = time.time()
    _barrier(ws)
    job = _job_totals(bytes_step, tokens_step, t_start.elapsed_time(t_stop), K, ws, device)
    ms_step, value, seq_tok_s = job["ms_per_step"], job["value"], job["seq_tokens_per_s"]
    assert int(r.status.item()) == 0, f"device status {int(r.status.item())}"

    # ---- the decode kernel alone, in a pass of its own: the library records events
    # around that launch, which keeps it from starting early under the plan kernel
    kern_ms = kernel_samples(pa, r.run_step, max(args.kernel_samples, K), device)
    kern = _spread(kern_ms)
    kern_avg_ms = kern["mean_us"] * 1e-3
    assert int(r.status.item()) == 0

    per_config = None
    if ws == 1 and not args.no_per_config:
        per_config = run_per_config(args, device, peak)
    phase1 = time.time()
    time.sleep(0.15)
    clocks.stop()

    # ---- end-to-end through the public API from pinned host memory
    e2e = run_e2e(args, w, device, rank, pa, W, DecodeRunner)
    e2e_val = _max_over_ranks(-e2e["value"], ws, device)   # slowest rank
    e2e["value"] = -e2e_val * ws

    achieved = bytes_step / (kern_avg_ms * 1e-3) / 1e9
    traffic = _traffic_record()
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": _config(w, r),
        "seq_tokens_per_s": seq_tok_s,
        "pct_of_spec_8000_GBps": 100.0 * value / ws / SPEC_HBM_GBS,
        f"pct_of_{peak_kind}_hbm": 100.0 * value / ws / peak,
        "decode_variant": {"variant": f"v{variant}", "partition_size": psize},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "paged_decode_kernel (persistent V2 decode; CUDA events around "
                               "its launch, in a kernel-only pass after the timed steps)",
                     "bytes_per_launch": bytes_step, "kernel_ms": kern_avg_ms,
                     "kernel_us": kern, "step_over_kernel": ms_step / kern_avg_ms,
                     "peak_source": f"{peak_kind} HBM copy bandwidth"},
        "e2e": e2e,
        "gpu_launches": launches_per_step * K,
        "clocks": clocks.summary((phase0, phase1)),
    }
    if per_config is not None:
        line["per_config"] = per_config
    if ws == 1 and rank == 0 and not args.no_cpu_baseline:
        cb = time_oracle(r, args.cpu_budget)
        line["cpu_baseline"] = {
            "value": cb["bytes"] / cb["seconds"] / 1e9, "unit": "GB/s", "cores": 1,
            "kind": "oracle",
            "sample": f"fp64 oracle, one thread, first {cb['seqs']} sequences of one {w.name} "
                      f"step ({cb['tokens']} context tokens, {cb['seconds']:.1f} s)",
            "seq_tokens_per_s": cb["tokens"] / cb["seconds"],
            "host_cpu_count": os.cpu_count(),
        }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_e2e(args, w, device, rank, pa, W, DecodeRunner):
    """Serving loop through the public C ABI from host memory, pipelined the way a
    server runs it: while the GPU runs step i, the host allocator appends step i+1's
    tokens and writes its slots / block tables / lengths straight into the next slot of
    a ring of pinned buffers, and pa_decode_step_host_overlapped queues step i+1 (H2D of
    its q/k/v/metadata on an H2D stream, reshape_and_cache + decode on the compute stream,
    D2H of out on a D2H stream), so that a step's copies overlap its neighbours' kernels.  Before a ring slot is reused, the host waits for that step's output to have
    arrived in host memory.  Every step's copies lie inside the timed region."""
    import dataclasses
    import torch
    # A fixed number of steps whatever --steps is: every step appends a token to each
    # sequence, so the contexts drift from the configured workload by K tokens (200 by
    # default: about 8 % of the average context over the loop) while the pipeline's fill
    # is amortised.
    K = args.e2e_steps
    warm = 3
    we = dataclasses.replace(w, steps=K + warm + 1)
    r = DecodeRunner(we, device=device, rank=rank)
    S, Hq, Hkv, D = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_size
    tdt = W.torch_dtype(w)
    ring = 3
    qh = [W.randn_16bit((S, Hq, D), w.dtype, 900 + i, "cpu").pin_memory() for i in range(ring)]
    kh = [W.randn_16bit((S, Hkv, D), w.dtype, 910 + i, "cpu").pin_memory() for i in range(ring)]
    vh = [W.randn_16bit((S, Hkv, D), w.dtype, 920 + i, "cpu").pin_memory() for i in range(ring)]
    slots_h = [torch.empty(S, dtype=torch.int32).pin_memory() for _ in range(ring)]
    lens_h = [torch.empty(S, dtype=torch.int32).pin_memory() for _ in range(ring)]
    tables_h = [torch.empty((S, r.max_blocks), dtype=torch.int32).pin_memory() for _ in range(ring)]
    out_h = [torch.empty((S, Hq, D), dtype=tdt).pin_memory() for _ in range(ring)]
    # per ring slot: staging area, copies-landed / step-done / output-back events
    ssize = pa.pa_decode_step_host_staging_size(S, Hq, Hkv, D, r.max_blocks)
    staging = [torch.empty(ssize, dtype=torch.uint8, device=device) for _ in range(ring)]
    h2d_stream = torch.cuda.Stream(device)
    d2h_stream = torch.cuda.Stream(device)
    staged = [torch.cuda.Event() for _ in range(ring)]
    stepped = [torch.cuda.Event() for _ in range(ring)]
    done = [torch.cuda.Event() for _ in range(ring)]
    for e in staged + stepped + done:
        e.record(d2h_stream)           # the CUDA events exist from here on
    need = pa.pa_decode_auto_workspace_size(S, Hq, Hkv, D, w.block_size,
                                            r.max_context_len + K + warm)
    if need > r.workspace.numel():
        r.workspace = torch.empty(need, dtype=torch.uint8, device=device)
    ids = r.seq_ids
    stream = torch.cuda.current_stream(device)
    pending = [None] * ring          # per slot: context tokens of the step in flight
    stats = {"bytes": 0, "tokens": 0, "checksum": 0.0}

    def retire(j, count):
        if pending[j] is None:
            return
        done[j].synchronize()        # that step's output is in host memory now
        stats["checksum"] += float(out_h[j][0, 0, 0])
        if count:
            L = pending[j]
            stats["bytes"] += L * Hkv * D * 2 * 2 + 2 * S * Hq * D * 2
            stats["tokens"] += L
        pending[j] = None

    def issue(i, count):
        j = i % ring
        retire(j, count)
        r.alloc.pa_alloc_append_batch(ids, out=slots_h[j].numpy())
        r.alloc.pa_alloc_block_tables(ids, r.max_blocks, out=tables_h[j].numpy())
        lens_np = lens_h[j].numpy()
        r.alloc.pa_alloc_context_lens(ids, out=lens_np)
        mcl = int(lens_np.max())
        pa.pa_decode_step_host_overlapped(out_h[j], qh[j], kh[j], vh[j], slots_h[j], tables_h[j],
                                          lens_h[j], r.key_cache, r.value_cache, mcl, w.scale,
                                          staging[j], stream, h2d_stream, d2h_stream, staged[j],
                                          stepped[j], workspace=r.workspace, status=r.status)
        done[j].record(d2h_stream)     # after the step's D2H
        pending[j] = int(lens_np.astype(np.int64).sum())

    for i in range(warm):
        issue(i, False)
    for j in range(ring):
        retire(j, False)
    torch.cuda.synchronize(device)
    t0 = time.perf_counter()
    for i in range(K):
        issue(warm + i, True)
    for i in range(K, K + ring):
        retire((warm + i) % ring, True)
    dt = time.perf_counter() - t0
    assert int(r.status.item()) == 0
    h2d = (qh[0].numel() + kh[0].numel() + vh[0].numel()) * 2 + (2 * S + S * r.max_blocks) * 4
    d2h = out_h[0].numel() * 2
    return {"value": stats["bytes"] / dt / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": K, "ms_per_step": 1e3 * dt / K,
            "seq_tokens_per_s": stats["tokens"] / dt,
            "path": "per step: pa_alloc_append_batch / block tables / lengths into pinned host "
                    "buffers, pa_decode_step_host_overlapped (H2D of q/k/v/metadata on an H2D "
                    "stream, reshape + decode on the compute stream, D2H of out on a D2H "
                    "stream); the host prepares step i+1 while the GPU runs step i and waits "
                    "for each step's output before reusing its buffers (ring of 3); wall clock"}


def run_multistep_case(args):
    """The k-step decode loop of one workload on the device (per step: pa_advance_step,
    reshape_and_cache of the step's new tokens, decode), timed with CUDA events as issued
    from Python and as one CUDA-graph replay.  Prints the whole loop's time and the mean
    per step; bytes per step are the decode's algorithmic bytes at that step's lengths."""
    import numpy as np
    import torch
    from paged_kv_cache_187_gb300 import workloads as W
    from paged_kv_cache_187_gb300.runner import DecodeRunner
    w = W.WORKLOADS[args.profile_workload]
    k = args.multistep
    r = DecodeRunner(w, device="cuda").setup_multistep(k)
    lens0 = r.ms_lens0.astype(np.int64)
    kv_per_token = w.num_kv_heads * w.head_size * 2 * 2
    qo = 2 * w.num_seqs * w.num_q_heads * w.head_size * 2
    tokens = sum(int((lens0 + j + 1).sum()) for j in range(k))
    loop_bytes = tokens * kv_per_token + k * qo
    r.run_multistep()
    torch.cuda.synchronize()
    graph = r.capture_multistep()

    def timed(fn, n):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        for a, b in evs:
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return sorted(a.elapsed_time(b) for a, b in evs)

    for _ in range(args.warmup):
        r.run_multistep()
        graph.replay()
    torch.cuda.synchronize()
    res = {}
    for name, fn in (("eager", r.run_multistep), ("graph", graph.replay)):
        t = timed(fn, args.steps)
        ms = t[len(t) // 2]
        res[name] = {"loop_ms": ms, "us_per_step": 1e3 * ms / k,
                     "GBps": loop_bytes / (ms * 1e-3) / 1e9,
                     "seq_tokens_per_s": tokens / (ms * 1e-3)}
    assert int(r.status.item()) == 0
    print(json.dumps({"multistep_case": w.name, "steps_per_loop": k, "loops_timed": args.steps,
                      "warmup": args.warmup, "loop_bytes": loop_bytes, "loop_seq_tokens": tokens,
                      "step": "pa_advance_step + pa_decode_step (reshape_and_cache + auto decode)",
                      **res}))


def run_profile_case(args):
    """Small, self-contained case for ncu: decode steps of one workload only."""
    import torch
    import paged_kv_cache_187_gb300 as pa
    from paged_kv_cache_187_gb300 import workloads as W
    from paged_kv_cache_187_gb300.runner import DecodeRunner
    import dataclasses
    w = W.WORKLOADS[args.profile_workload]
    start_lens = None
    if args.num_seqs:
        # the first num_seqs sequences of the workload, with their own context lengths
        start_lens = W.start_context_lens(w)[:args.num_seqs]
        w = dataclasses.replace(w, num_seqs=args.num_seqs)
    r = DecodeRunner(w, device="cuda", kv_fp8=args.kv_fp8, start_lens=start_lens).next_step()
    r.run_reshape()
    del r.k_prefill, r.v_prefill          # not needed for decoding: keep the footprint small
    torch.cuda.empty_cache()
    if args.gqa_cuda_cores:
        pa.pa_set_gqa_tensor_cores(False)
    variant = args.variant
    if args.q_len > 1:
        # multi-query decode over the same pools: the last q_len tokens of every context
        # are the new ones, each with its own query rows
        S, Hq, D = w.num_seqs, w.num_q_heads, w.head_size
        mcl = r.step_max_context_len()
        q = W.randn_16bit((S, args.q_len, Hq, D), w.dtype, W.stream_seed(w, "q", 1), r.device)
        out = torch.empty_like(q)
        need = pa.pa_decode_mq_workspace_size(S, args.q_len, Hq, w.num_kv_heads, D,
                                              w.block_size, mcl, args.partition_size or 0)
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=r.device)

        def decode():
            pa.pa_decode_mq(out, q, r.key_cache, r.value_cache, r.block_tables_d,
                            r.context_lens_d, mcl, w.scale, variant=variant,
                            partition_size=args.partition_size or 0, workspace=ws,
                            status=r.status)
    else:
        def decode():
            r.run_decode(variant, partition_size=args.partition_size)
    for _ in range(args.warmup + args.steps):
        decode()
    torch.cuda.synchronize()
    assert int(r.status.item()) == 0
    print(json.dumps({"profile_case": w.name, "num_seqs": w.num_seqs,
                      "context_tokens": r.seq_tokens(), "kv_fp8": bool(args.kv_fp8), "variant": variant,
                      "q_len": args.q_len, "steps": args.steps,
                      "warmup": args.warmup, "gqa_cuda_cores": bool(args.gqa_cuda_cores),
                      # K/V once, plus q_len query and output rows per (sequence, head)
                      "bytes_per_decode": r.kv_bytes() + 2 * (args.q_len - 1) * w.num_seqs *
                      w.num_q_heads * w.head_size * 2}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the other workloads (per_config)")
    ap.add_argument("--kernel-samples", type=int, default=40,
                    help="decode-kernel launches timed per workload (at least 20)")
    ap.add_argument("--profile-workload", default=None,
                    help="run only decode steps of this workload (a small case for ncu)")
    ap.add_argument("--variant", default="auto", choices=["auto", "v1", "v2"])
    ap.add_argument("--partition-size", type=int, default=None)
    ap.add_argument("--gqa-cuda-cores", action="store_true",
                    help="profile case: force the CUDA-core path for grouped-query heads")
    ap.add_argument("--kv-fp8", action="store_true",
                    help="profile case: keep the KV pools in fp8 E4M3")
    ap.add_argument("--num-seqs", type=int, default=0,
                    help="profile case: only the first N sequences of the workload")
    ap.add_argument("--q-len", type=int, default=1,
                    help="profile case: multi-query decode with this many query tokens per sequence")
    ap.add_argument("--multistep", type=int, default=0,
                    help="with --profile-workload: time the k-step device loop (eager and "
                         "as a CUDA graph)")
    args = ap.parse_args()
    if args.profile_workload:
        if args.multistep > 0:
            run_multistep_case(args)
        else:
            run_profile_case(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
