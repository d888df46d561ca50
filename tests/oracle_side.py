"""Rebuilds, with the oracle only, what a DecodeRunner holds after its steps.

The oracle side gets the same seeded INPUTS the GPU side drew (per-token K/V of the
prefill and of each step, the step's queries) and the same allocator seed and
requests; everything derived from them -- block placement, slots, pools, decode
outputs -- is recomputed by ``oracle/`` alone and never read back from the CUDA path.
"""
from __future__ import annotations

import concurrent.futures
import dataclasses
import os

import numpy as np
import torch

import oracle


def host_threads() -> int:
    return max(1, os.cpu_count() or 1)


def seq_ranges(lens: np.ndarray, parts: int) -> list[tuple[int, int]]:
    """Contiguous sequence ranges [a, b) covering 0..S-1, each holding about the same
    number of context tokens (the oracle's cost grows with the tokens)."""
    S = int(lens.size)
    if S == 0:
        return []
    cost = np.maximum(lens.astype(np.int64), 1)
    edges = np.searchsorted(np.cumsum(cost), np.linspace(0, cost.sum(), parts + 1)[1:-1],
                            side="right")
    cuts = sorted(set([0] + [int(e) for e in edges if 0 < e < S] + [S]))
    return list(zip(cuts[:-1], cuts[1:]))


def fan_out(call, lens: np.ndarray) -> np.ndarray:
    """Runs call(a, b) -> the oracle's rows of sequences [a, b) over sequence ranges on a
    thread pool and stacks the results in sequence order.  Each call runs the plain,
    single-threaded oracle; ctypes releases the GIL while it runs, so the ranges proceed
    on separate host cores."""
    n = host_threads()
    ranges = seq_ranges(lens, 4 * n)
    if len(ranges) <= 1:
        return call(0, int(lens.size))
    with concurrent.futures.ThreadPoolExecutor(max_workers=n) as ex:
        parts = list(ex.map(lambda ab: call(*ab), ranges))
    return np.concatenate(parts, axis=0)


def bits(t: torch.Tensor) -> np.ndarray:
    """16-bit tensor (any device) -> host uint16 bit patterns."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@dataclasses.dataclass
class StepRecord:
    q: np.ndarray          # [S, Hq, D] uint16
    k_new: np.ndarray      # [S, Hkv, D]
    v_new: np.ndarray
    slots: np.ndarray      # GPU-side slots of this step (compared, never used)
    context_lens: np.ndarray
    block_tables: np.ndarray


def record_step(r) -> StepRecord:
    return StepRecord(bits(r.q), bits(r.k_new), bits(r.v_new), r.slots.copy(),
                      r.context_lens.copy(), r.block_tables.copy())


class OracleState:
    """Oracle allocator + (optionally compacted) oracle pools for a runner's workload."""

    def __init__(self, r, steps: list[StepRecord], seqs=None, reserve: int = 0):
        """`reserve` > 0 replays a multi-step loop whose blocks were reserved up front
        (the allocator's reserve, then one append per sequence per step).  A runner with
        fp8 pools gets uint8 E4M3 pools filled by the oracle's quantising scatter."""
        w = r.w
        self.w = w
        self.kv8 = bool(getattr(r, "kv_fp8", False))
        self.k_scale, self.v_scale = np.float32(r.k_scale), np.float32(r.v_scale)
        S, bs = w.num_seqs, w.block_size
        self.alloc = oracle.Alloc(r.num_blocks, bs, r.alloc_seed, max_seqs=max(S, 1))
        for s in range(S):
            self.alloc.add_seq(s, int(r.prefill_lens[s]))
        if reserve:
            for s in range(S):
                self.alloc.reserve(s, reserve)
        self.prefill_slots = np.concatenate(
            [self.alloc.slots(s, 0, int(r.prefill_lens[s])) for s in range(S)] +
            [np.zeros(0, np.int32)])
        self.step_slots = []
        self.step_tables = []
        self.step_lens = []
        ids = np.arange(S, dtype=np.int32)
        for st in steps:
            self.step_slots.append(np.array([self.alloc.append(s) for s in range(S)], np.int32))
            self.step_tables.append(self.alloc.block_tables(ids, r.max_blocks))
            self.step_lens.append(self.alloc.context_lens(ids))
        self.seqs = np.arange(S) if seqs is None else np.asarray(sorted(set(int(s) for s in seqs)))
        # pools over the blocks of the selected sequences only (all of them when seqs is
        # None), renumbered densely; block tables renumbered the same way
        final_tables = self.step_tables[-1] if steps else self.alloc.block_tables(ids, r.max_blocks)
        used = np.unique(final_tables[self.seqs][final_tables[self.seqs] >= 0])
        if seqs is None:
            self.remap = np.arange(r.num_blocks, dtype=np.int64)
            nb = r.num_blocks
        else:
            self.remap = np.full(r.num_blocks, -1, dtype=np.int64)
            self.remap[used] = np.arange(used.size)
            nb = max(int(used.size), 1)
        self.used_blocks = used
        shape = (nb, w.num_kv_heads, bs, w.head_size)
        from paged_kv_cache_187_gb300 import workloads as W
        if self.kv8:
            self.k_cache = np.full(shape, 0x7F, dtype=np.uint8)     # E4M3 NaN
            self.v_cache = np.full(shape, 0x7F, dtype=np.uint8)
        else:
            self.k_cache = np.full(shape, W.NAN_BITS[w.dtype], dtype=np.uint16)
            self.v_cache = np.full(shape, W.NAN_BITS[w.dtype], dtype=np.uint16)
        # prefill rows of the selected sequences (runs of consecutive sequences at once)
        sel = self.seqs
        runs = np.split(sel, np.nonzero(np.diff(sel) != 1)[0] + 1) if sel.size else []
        for run in runs:
            a, b = int(r.prefill_offsets[run[0]]), int(r.prefill_offsets[run[-1] + 1])
            for c in range(a, b, 1 << 18):
                d = min(b, c + (1 << 18))
                sl = self._map_slots(self.prefill_slots[c:d])
                self._scatter(bits(r.k_prefill[c:d]), bits(r.v_prefill[c:d]), sl)
        for st, slots in zip(steps, self.step_slots):
            sl = self._map_slots(slots[sel])
            self._scatter(st.k_new[sel], st.v_new[sel], sl)

    def _scatter(self, k_bits, v_bits, slots):
        bs = self.w.block_size
        if self.kv8:
            bad = oracle.reshape_and_cache_fp8(k_bits, v_bits, self.k_cache, self.v_cache, slots,
                                               bs, self.w.dtype, self.k_scale, self.v_scale)
        else:
            bad = oracle.reshape_and_cache(k_bits, v_bits, self.k_cache, self.v_cache, slots, bs)
        assert bad == 0

    def _map_slots(self, slots):
        bs = self.w.block_size
        blk = slots // bs
        return (self.remap[blk] * bs + slots % bs).astype(np.int32)

    def tables(self, step: int) -> np.ndarray:
        t = self.step_tables[step]
        out = np.where(t >= 0, self.remap[np.maximum(t, 0)], -1)
        return out.astype(np.int32)

    def decode(self, step: int, st: StepRecord, rows=None, partition_size=None,
               context_lens=None) -> np.ndarray:
        """fp64 decode of `step`; rows = list of (seq, head) to compute (others zero).
        Without `rows`, every row, the sequences fanned out over the host's cores."""
        w = self.w
        lens = self.step_lens[step] if context_lens is None else np.asarray(context_lens, np.int32)
        tables = self.tables(step)
        scale = np.float32(w.scale)

        def run(q, bt, cl, only):
            if self.kv8:
                return oracle.decode_fp8(q, self.k_cache, self.v_cache, bt, cl, scale,
                                         self.k_scale, self.v_scale, w.dtype, only=only)
            args = (q, self.k_cache, self.v_cache, bt, cl, scale, w.dtype)
            if partition_size:
                return oracle.decode_v2(*args, partition_size, only=only)
            return oracle.decode_v1(*args, only=only)

        if rows is not None:
            only = np.zeros((w.num_seqs, w.num_q_heads), np.uint8)
            for s, h in rows:
                only[s, h] = 1
            return run(st.q, tables, lens, only)
        return fan_out(lambda a, b: run(st.q[a:b], tables[a:b], lens[a:b], None), lens)

    def decode_mq(self, step: int, q_bits: np.ndarray) -> np.ndarray:
        """fp64 multi-query decode over the pools after `step`: q [S, q_len, Hq, D]; the
        last q_len tokens of each context are the new ones (every row, fanned out)."""
        w = self.w
        lens = self.step_lens[step]
        tables = self.tables(step)
        return fan_out(lambda a, b: oracle.decode_mq(q_bits[a:b], self.k_cache, self.v_cache,
                                                     tables[a:b], lens[a:b],
                                                     np.float32(w.scale), w.dtype), lens)


# Decode tolerances: max |gpu - round_to_dtype(oracle)|, fp16 2e-3, bf16 1e-2.  Where an
# output is so large that one unit in the last place of the dtype exceeds that bound
# (|out| >= 2 in bf16, >= 4 in fp16), a correctly rounded GPU result that lies within a
# hair of a rounding boundary can land one ulp away from the rounded oracle value; there
# the bound is one ulp of the rounded oracle value instead.
TOL = {"f16": 2e-3, "bf16": 1e-2}
_FRAC_BITS = {"f16": 10, "bf16": 7}


def _ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, np.exp2(e - _FRAC_BITS[dtype]), 0.0)


@dataclasses.dataclass
class ErrStats:
    err: float        # the gated error (see max_err)
    n: int            # elements compared
    n_ulp: int        # elements beyond the stated bound, admitted only as one ulp
    max_abs: float    # max |gpu - round(oracle)| over all compared elements

    def ok(self, dtype: str, max_ulp_frac: float = 1e-5) -> bool:
        """The gate, plus a bound on how often the one-ulp allowance was needed."""
        return self.err <= TOL[dtype] and self.n_ulp <= max(2, max_ulp_frac * self.n)


def err_stats(gpu_bits: np.ndarray, ref64: np.ndarray, dtype: str, rows=None) -> ErrStats:
    """Compares the GPU output with the oracle's fp64 result rounded to the output dtype,
    over the given (seq, head) rows (all if None).  `err` is scaled so that the gate is
    `err <= TOL[dtype]`: elements whose one-ulp spacing exceeds the tolerance are
    measured in units of (their ulp / TOL).  `n_ulp` counts the elements that pass only
    through that allowance (|gpu - round(oracle)| > TOL)."""
    ref_bits = oracle.round_to(ref64, dtype)
    g = oracle.widen(gpu_bits, dtype)
    r = oracle.widen(ref_bits, dtype)
    if rows is not None:
        idx = tuple(np.array(rows).T)
        g, r = g[idx], r[idx]
    if not g.size:
        return ErrStats(0.0, 0, 0, 0.0)
    if not np.all(np.isfinite(g)):
        return ErrStats(float("inf"), int(g.size), int(g.size), float("inf"))
    diff = np.abs(g - r)
    bound = np.maximum(TOL[dtype], _ulp(r, dtype))
    return ErrStats(float(np.max(diff / bound) * TOL[dtype]), int(g.size),
                    int(np.count_nonzero(diff > TOL[dtype])), float(diff.max()))


def max_err(gpu_bits: np.ndarray, ref64: np.ndarray, dtype: str, rows=None) -> float:
    """err_stats(...).err: the gated error, `<= TOL[dtype]` passes."""
    return err_stats(gpu_bits, ref64, dtype, rows).err
