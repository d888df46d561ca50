"""Seeded synthetic workloads shaped like serving decode batches.

This module only draws random inputs: context lengths, pool sizes, and the
query / key / value values.  It holds none of the attention arithmetic and no
block placement (the block allocator owns that), so both the CUDA path and the
CPU oracle can take their inputs from here.

The five workloads are decode steps of one attention layer:

=====  ===========================================================================
tiny   4 seqs, 4/4 heads, head_size 64, block 16, fp16, contexts {1, 17, 64, 100},
       pool of 64 blocks
l2_7b  Llama-2-7B-shaped: 64 seqs, 32/32 heads, head_size 128, block 16, fp16,
       contexts uniform in [512, 2048]
l3_8b  Llama-3-8B-shaped GQA: 256 seqs, 32 q / 8 kv heads, head_size 128, block 16,
       bf16, contexts lognormal(mu=6.9, sigma=0.8) rounded and clipped to [16, 8192]
skew   LLaMA-13B-shaped skewed batch: 40/40 heads, head_size 128, block 16, fp16,
       8 seqs at 32768 plus 248 at 128 (order shuffled), partition size 512
l3_70b Llama-3-70B-shaped multi-step loop: 512 seqs, 64 q / 8 kv heads,
       head_size 128, block 32, bf16, start contexts uniform in [1, 4096],
       8 steps of one new token per sequence
=====  ===========================================================================

Values are N(0, 1) drawn in fp32 and rounded to the workload's 16-bit type.
Pools hold the blocks the batch needs (after all of its steps) plus 10 %, rounded
up, except ``tiny`` whose pool is fixed at 64 blocks.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    dtype: str                 # "f16" or "bf16"
    steps: int = 1             # decode steps (one new token per sequence per step)
    partition_size: int = 512  # V2 partition size the workload names (512 if unstated)
    fixed_pool_blocks: int = 0  # 0: size the pool from the contexts
    seed: int = 0
    description: str = field(default="", compare=False)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_size)


WORKLOADS = {
    "tiny": Workload("tiny", 4, 4, 4, 64, 16, "f16", fixed_pool_blocks=64, seed=1001,
                     description="Tiny MHA paged decode"),
    "l2_7b": Workload("l2_7b", 64, 32, 32, 128, 16, "f16", seed=1002,
                      description="Llama-2-7B-shaped layer decode"),
    "l3_8b": Workload("l3_8b", 256, 32, 8, 128, 16, "bf16", seed=1003,
                      description="Llama-3-8B-shaped GQA decode"),
    "skew": Workload("skew", 256, 40, 40, 128, 16, "f16", partition_size=512, seed=1004,
                     description="Skewed long-context batch (V2 partition path)"),
    "l3_70b": Workload("l3_70b", 512, 64, 8, 128, 32, "bf16", steps=8, seed=1005,
                       description="Multi-step decode loop, Llama-3-70B-shaped layer"),
}


def start_context_lens(w: Workload, seed: int | None = None) -> np.ndarray:
    """Context lengths (int32) of the FIRST decode step, counting the step's new token.

    Step k (0-based) of a multi-step workload decodes over ``start + k`` tokens."""
    rng = np.random.Generator(np.random.PCG64(w.seed if seed is None else seed))
    if w.name == "tiny":
        lens = np.array([1, 17, 64, 100], dtype=np.int64)
    elif w.name == "l2_7b":
        lens = rng.integers(512, 2048, size=w.num_seqs, endpoint=True)
    elif w.name == "l3_8b":
        lens = np.clip(np.rint(rng.lognormal(6.9, 0.8, size=w.num_seqs)), 16, 8192)
    elif w.name == "skew":
        lens = np.array([32768] * 8 + [128] * 248, dtype=np.int64)
        rng.shuffle(lens)
    elif w.name == "l3_70b":
        # "start context_lens uniform in [1, 4096]" are the lengths before the loop;
        # the first step appends one token to each.
        lens = rng.integers(1, 4096, size=w.num_seqs, endpoint=True) + 1
    else:
        raise KeyError(w.name)
    return lens.astype(np.int32)


def pool_blocks(w: Workload, start_lens: np.ndarray) -> int:
    """Physical blocks in the pool: enough for every step, plus 10 % free."""
    if w.fixed_pool_blocks:
        return w.fixed_pool_blocks
    final = start_lens.astype(np.int64) + (w.steps - 1)
    need = int(np.sum((final + w.block_size - 1) // w.block_size))
    return int(math.ceil(need * 1.1))


def max_blocks_per_seq(w: Workload, start_lens: np.ndarray) -> int:
    final = int(start_lens.max()) + (w.steps - 1)
    return (final + w.block_size - 1) // w.block_size


def torch_dtype(w: Workload):
    import torch
    return torch.float16 if w.dtype == "f16" else torch.bfloat16


def randn_16bit(shape, dtype: str, seed: int, device="cpu"):
    """N(0, 1) values drawn in fp32 from a seeded torch generator, rounded to the
    16-bit type.  Returns a torch tensor on ``device``."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    tdt = torch.float16 if dtype == "f16" else torch.bfloat16
    n = int(np.prod(shape)) if len(shape) else 1
    out = torch.empty(shape, dtype=tdt, device=device)
    flat = out.view(-1)
    chunk = 1 << 26
    for i in range(0, n, chunk):
        m = min(chunk, n - i)
        flat[i:i + m] = torch.randn(m, generator=g, device=device, dtype=torch.float32).to(tdt)
    return out


def stream_seed(w: Workload, stream: str, step: int = 0, rank: int = 0) -> int:
    """A distinct seed per (workload, value stream, step, rank)."""
    names = {"q": 1, "k_new": 2, "v_new": 3, "k_prefill": 4, "v_prefill": 5}
    return (w.seed * 1_000_003 + names[stream] * 10_007 + step * 101 + rank * 7_919) & 0x7FFFFFFF


NAN_BITS = {"f16": 0x7E00, "bf16": 0x7FC0}   # quiet NaN patterns used to poison pools
