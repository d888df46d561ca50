"""A decode batch resident on the GPU, driven through the C ABI.

``DecodeRunner`` is the serving loop of one attention layer for a synthetic workload:
  1. the host allocator ("[core] Multi Step Scheduling #7000": the v2 block manager
     hands out blocks and the slot_mapping / block_tables / seq_lens metadata) places
     every sequence's prefill tokens, and pa_reshape_and_cache writes their K/V rows
     into NaN-poisoned pools;
  2. each decode step appends one token per sequence on the host (pa_alloc_append_batch),
     copies the step's metadata to the device, scatters the new K/V rows and runs the
     decode (pa_decode_step = reshape_and_cache + pa_decode_auto), or a chosen variant.

torch provides device memory and streams only; every step of the path runs in
libpa.so.
"""
from __future__ import annotations

import numpy as np
import torch

from . import _binding as B
from . import workloads as W


class DecodeRunner:
    def __init__(self, w: W.Workload, device="cuda", rank: int = 0, poison: bool = True,
                 prefill_chunk_tokens: int = 65536, start_lens=None, num_blocks=None,
                 alloc_seed=None, kv_fp8: bool = False, k_scale: float = 0.02,
                 v_scale: float = 0.02):
        """``start_lens`` / ``num_blocks`` / ``alloc_seed`` override the workload's own
        (first-step context lengths including the new token, pool size, allocator seed).
        ``kv_fp8`` keeps the pools in fp8 E4M3 with per-pool scales ``k_scale`` /
        ``v_scale`` (queries, new rows and outputs stay in the workload's 16-bit type)."""
        self.w = w
        self.kv_fp8 = kv_fp8
        self.k_scale, self.v_scale = float(k_scale), float(v_scale)
        self.device = torch.device(device)
        self.rank = rank
        S, bs = w.num_seqs, w.block_size
        self.start_lens = (W.start_context_lens(w) if start_lens is None
                           else np.asarray(start_lens, dtype=np.int32))
        assert self.start_lens.shape == (S,) and int(self.start_lens.min()) >= 1
        self.num_blocks = (W.pool_blocks(w, self.start_lens) if num_blocks is None
                           else int(num_blocks))
        self.alloc_seed = (w.seed + rank) if alloc_seed is None else int(alloc_seed)
        self.max_blocks = W.max_blocks_per_seq(w, self.start_lens)
        self.max_context_len = int(self.start_lens.max()) + w.steps - 1
        self.tdtype = W.torch_dtype(w)
        self.alloc = B.PagedAllocator(self.num_blocks, bs, seed=self.alloc_seed)
        self.seq_ids = np.arange(S, dtype=np.int32)
        self.prefill_lens = (self.start_lens - 1).astype(np.int64)
        for s in range(S):
            self.alloc.pa_alloc_add_seq(s, int(self.prefill_lens[s]))
        shape = (self.num_blocks, w.num_kv_heads, bs, w.head_size)
        cdt = torch.uint8 if kv_fp8 else self.tdtype
        self.key_cache = torch.empty(shape, dtype=cdt, device=self.device)
        self.value_cache = torch.empty(shape, dtype=cdt, device=self.device)
        if poison:
            if kv_fp8:
                self.key_cache.fill_(0x7F)          # E4M3 NaN
                self.value_cache.fill_(0x7F)
            else:
                nan = W.NAN_BITS[w.dtype]
                nan = nan - 65536 if nan >= 32768 else nan
                self.key_cache.view(torch.int16).fill_(nan)
                self.value_cache.view(torch.int16).fill_(nan)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        # prefill: tokens in sequence order, positions 0 .. L-2 of every sequence
        self.prefill_offsets = np.concatenate([[0], np.cumsum(self.prefill_lens)]).astype(np.int64)
        total = int(self.prefill_offsets[-1])
        self.k_prefill = W.randn_16bit((total, w.num_kv_heads, w.head_size), w.dtype,
                                       W.stream_seed(w, "k_prefill", 0, rank), self.device)
        self.v_prefill = W.randn_16bit((total, w.num_kv_heads, w.head_size), w.dtype,
                                       W.stream_seed(w, "v_prefill", 0, rank), self.device)
        slots = np.concatenate([self.alloc.pa_alloc_slots(s, 0, int(self.prefill_lens[s]))
                                for s in range(S)] + [np.zeros(0, np.int32)])
        self.prefill_slots = slots
        slots_d = torch.from_numpy(slots).to(self.device)
        for i in range(0, total, prefill_chunk_tokens):
            j = min(total, i + prefill_chunk_tokens)
            self._scatter(self.k_prefill[i:j], self.v_prefill[i:j], slots_d[i:j])
        self.step_index = -1
        self.out = torch.empty((S, w.num_q_heads, w.head_size), dtype=self.tdtype,
                               device=self.device)
        ws = max(B.pa_decode_auto_workspace_size(S, w.num_q_heads, w.num_kv_heads, w.head_size,
                                                 bs, self.max_context_len),
                 B.pa_decode_v2_workspace_size(S, w.num_q_heads, w.head_size,
                                               self.max_context_len, w.partition_size), 256)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=self.device)

    # ------------------------------------------------------------------ one step
    def next_step(self):
        """Host side of a decode step: append one token per sequence, build the
        metadata, draw the step's q / k / v, and stage everything on the device."""
        w = self.w
        self.step_index += 1
        k = self.step_index
        self.slots = self.alloc.pa_alloc_append_batch(self.seq_ids)
        self.block_tables = self.alloc.pa_alloc_block_tables(self.seq_ids, self.max_blocks)
        self.context_lens = self.alloc.pa_alloc_context_lens(self.seq_ids)
        self.slots_d = torch.from_numpy(self.slots).to(self.device)
        self.block_tables_d = torch.from_numpy(self.block_tables).to(self.device)
        self.context_lens_d = torch.from_numpy(self.context_lens).to(self.device)
        S, Hq, Hkv, D = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_size
        self.q = W.randn_16bit((S, Hq, D), w.dtype, W.stream_seed(w, "q", k, self.rank), self.device)
        self.k_new = W.randn_16bit((S, Hkv, D), w.dtype, W.stream_seed(w, "k_new", k, self.rank),
                                   self.device)
        self.v_new = W.randn_16bit((S, Hkv, D), w.dtype, W.stream_seed(w, "v_new", k, self.rank),
                                   self.device)
        return self

    def step_max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.context_lens.size else 0

    def _scatter(self, k, v, slots_d, stream=None):
        if self.kv_fp8:
            B.pa_reshape_and_cache_fp8(k, v, self.key_cache, self.value_cache, slots_d,
                                       self.k_scale, self.v_scale, status=self.status,
                                       stream=stream)
        else:
            B.pa_reshape_and_cache(k, v, self.key_cache, self.value_cache, slots_d,
                                   status=self.status, stream=stream)

    def run_reshape(self, stream=None):
        self._scatter(self.k_new, self.v_new, self.slots_d, stream)

    def run_decode(self, variant: str = "auto", partition_size: int | None = None, stream=None,
                   max_context_len: int | None = None):
        mcl = self.step_max_context_len() if max_context_len is None else max_context_len
        args = (self.out, self.q, self.key_cache, self.value_cache, self.block_tables_d,
                self.context_lens_d, mcl, self.w.scale)
        if self.kv_fp8:
            P = partition_size or (self.w.partition_size if variant == "v2" else 0)
            if variant == "v2":
                need = B.pa_decode_v2_workspace_size(self.w.num_seqs, self.w.num_q_heads,
                                                     self.w.head_size, mcl, P)
                if need > self.workspace.numel():
                    self.workspace = torch.empty(need, dtype=torch.uint8, device=self.device)
            B.pa_decode_fp8(*args, self.k_scale, self.v_scale, variant=variant, partition_size=P,
                            workspace=self.workspace, status=self.status, stream=stream)
            return
        if variant == "v1":
            B.pa_decode_v1(*args, status=self.status, stream=stream)
        elif variant == "v2":
            P = partition_size or self.w.partition_size
            need = B.pa_decode_v2_workspace_size(self.w.num_seqs, self.w.num_q_heads,
                                                 self.w.head_size, mcl, P)
            if need > self.workspace.numel():
                self.workspace = torch.empty(need, dtype=torch.uint8, device=self.device)
            B.pa_decode_v2(*args, P, self.workspace, status=self.status, stream=stream)
        elif variant == "auto":
            B.pa_decode_auto(*args, workspace=self.workspace, status=self.status, stream=stream)
        else:
            raise ValueError(variant)

    def run_step(self, stream=None):
        """reshape_and_cache + pa_decode_auto through the single pa_decode_step call (for
        fp8 pools: the fp8 scatter, then pa_decode_fp8's automatic choice)."""
        if self.kv_fp8:
            self.run_reshape(stream)
            self.run_decode("auto", stream=stream)
            return
        B.pa_decode_step(self.out, self.q, self.k_new, self.v_new, self.key_cache,
                         self.value_cache, self.slots_d, self.block_tables_d, self.context_lens_d,
                         self.step_max_context_len(), self.w.scale, workspace=self.workspace,
                         status=self.status, stream=stream)

    # ------------------------------------------------------------------ accounting
    def kv_bytes(self) -> int:
        """Algorithmic bytes of one decode step: every context token's K and V row of
        every kv head, plus the query and output rows."""
        w = self.w
        elt = 1 if self.kv_fp8 else 2
        lens = self.context_lens.astype(np.int64)
        kv = int(lens.sum()) * w.num_kv_heads * w.head_size * 2 * elt
        qo = 2 * w.num_seqs * w.num_q_heads * w.head_size * 2
        return kv + qo

    def seq_tokens(self) -> int:
        return int(self.context_lens.astype(np.int64).sum())

    # ------------------------------------------------------------------ multi-step loop
    def setup_multistep(self, k: int):
        """Host side of a k-step decode loop run entirely on the device ("[core] Multi Step
        Scheduling #7000": k decode steps between scheduler visits, metadata advanced on
        the GPU).  Reserves every block the loop will touch, builds the block tables once,
        and stages k steps of q / k / v inputs; the device lengths start at the pre-loop
        values and pa_advance_step moves them one token per step."""
        w = self.w
        S, Hq, Hkv, D = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_size
        ids = self.seq_ids
        self.alloc.pa_alloc_reserve_batch(ids, k)
        self.ms_k = k
        self.ms_lens0 = self.alloc.pa_alloc_context_lens(ids)
        self.block_tables = self.alloc.pa_alloc_block_tables(ids, self.max_blocks)
        self.block_tables_d = torch.from_numpy(self.block_tables).to(self.device)
        self.ms_lens0_d = torch.from_numpy(self.ms_lens0).to(self.device)
        self.context_lens_d = self.ms_lens0_d.clone()
        self.slots_d = torch.empty(S, dtype=torch.int32, device=self.device)
        self.ms_max_context_len = int(self.ms_lens0.max()) + k
        base = self.step_index + 1
        self.ms_q = [W.randn_16bit((S, Hq, D), w.dtype, W.stream_seed(w, "q", base + j, self.rank),
                                   self.device) for j in range(k)]
        self.ms_k_new = [W.randn_16bit((S, Hkv, D), w.dtype,
                                       W.stream_seed(w, "k_new", base + j, self.rank), self.device)
                         for j in range(k)]
        self.ms_v_new = [W.randn_16bit((S, Hkv, D), w.dtype,
                                       W.stream_seed(w, "v_new", base + j, self.rank), self.device)
                         for j in range(k)]
        self.ms_out = [torch.empty((S, Hq, D), dtype=self.tdtype, device=self.device)
                       for _ in range(k)]
        need = B.pa_decode_auto_workspace_size(S, Hq, Hkv, D, w.block_size,
                                               self.ms_max_context_len)
        if need > self.workspace.numel():
            self.workspace = torch.empty(need, dtype=torch.uint8, device=self.device)
        return self

    def run_multistep(self, stream=None, on_step=None):
        """The k-step loop on the device: per step pa_advance_step (lengths and slots move
        one token), then pa_decode_step (reshape_and_cache + decode).  Starts from the
        pre-loop lengths every time, so it can be captured once and replayed."""
        w = self.w
        self.context_lens_d.copy_(self.ms_lens0_d)
        for j in range(self.ms_k):
            B.pa_advance_step(self.context_lens_d, self.slots_d, self.block_tables_d,
                              w.block_size, self.num_blocks, status=self.status, stream=stream)
            B.pa_decode_step(self.ms_out[j], self.ms_q[j], self.ms_k_new[j], self.ms_v_new[j],
                             self.key_cache, self.value_cache, self.slots_d, self.block_tables_d,
                             self.context_lens_d, self.ms_max_context_len, w.scale,
                             workspace=self.workspace, status=self.status, stream=stream)
            if on_step is not None:
                on_step(j)

    def capture_multistep(self):
        """CUDA graph of run_multistep (call run_multistep once before, so that every
        kernel is loaded and configured outside the capture)."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run_multistep()
        return g

    def finish_multistep(self):
        """Brings the host allocator to the state after the loop (k appends per sequence,
        on the reserved blocks) and returns the slots it assigns per step, [k][S]."""
        return np.stack([self.alloc.pa_alloc_append_batch(self.seq_ids) for _ in range(self.ms_k)])
