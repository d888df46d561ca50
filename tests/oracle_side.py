"""Rebuilds, with the oracle only, what a DecodeRunner holds after its steps.

The oracle side gets the same seeded INPUTS the GPU side drew (per-token K/V of the
prefill and of each step, the step's queries) and the same allocator seed and
requests; everything derived from them -- block placement, slots, pools, decode
outputs -- is recomputed by ``oracle/`` alone and never read back from the CUDA path.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import oracle


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
        (the allocator's reserve, then one append per sequence per step)."""
        w = r.w
        self.w = w
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
        self.k_cache = np.full(shape, W.NAN_BITS[w.dtype], dtype=np.uint16)
        self.v_cache = np.full(shape, W.NAN_BITS[w.dtype], dtype=np.uint16)
        # prefill rows of the selected sequences
        for s in self.seqs:
            a, b = int(r.prefill_offsets[s]), int(r.prefill_offsets[s + 1])
            if b > a:
                sl = self._map_slots(self.prefill_slots[a:b])
                bad = oracle.reshape_and_cache(bits(r.k_prefill[a:b]), bits(r.v_prefill[a:b]),
                                               self.k_cache, self.v_cache, sl, bs)
                assert bad == 0
        for st, slots in zip(steps, self.step_slots):
            sel = self.seqs
            sl = self._map_slots(slots[sel])
            bad = oracle.reshape_and_cache(st.k_new[sel], st.v_new[sel], self.k_cache,
                                           self.v_cache, sl, bs)
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
        """fp64 decode of `step`; rows = list of (seq, head) to compute (others zero)."""
        w = self.w
        lens = self.step_lens[step] if context_lens is None else context_lens
        only = None
        if rows is not None:
            only = np.zeros((w.num_seqs, w.num_q_heads), np.uint8)
            for s, h in rows:
                only[s, h] = 1
        args = (st.q, self.k_cache, self.v_cache, self.tables(step), lens, np.float32(w.scale),
                w.dtype)
        if partition_size:
            return oracle.decode_v2(*args, partition_size, only=only)
        return oracle.decode_v1(*args, only=only)


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


def max_err(gpu_bits: np.ndarray, ref64: np.ndarray, dtype: str, rows=None) -> float:
    """max over the given (seq, head) rows (all if None) of |gpu - round(oracle)|, scaled so
    that the gate is `<= TOL[dtype]`: elements whose one-ulp spacing exceeds the tolerance
    are measured in units of (their ulp / TOL)."""
    ref_bits = oracle.round_to(ref64, dtype)
    g = oracle.widen(gpu_bits, dtype)
    r = oracle.widen(ref_bits, dtype)
    if rows is not None:
        idx = tuple(np.array(rows).T)
        g, r = g[idx], r[idx]
    if not np.all(np.isfinite(g)):
        return float("inf")
    if not g.size:
        return 0.0
    bound = np.maximum(TOL[dtype], _ulp(r, dtype))
    return float(np.max(np.abs(g - r) / bound) * TOL[dtype])
