"""ctypes binding of libpa.so: the C ABI of include/pa.h with the same names.

Argument marshalling only.  Every function takes torch tensors (for device buffers)
or numpy arrays (for the host allocator), checks dtype / shape / device / contiguity,
derives the sizes the C call needs, and passes raw pointers.  All arithmetic happens
in the CUDA library; there is no fallback.  Importing this module on a machine
without the built library raises immediately.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_PKG = os.path.dirname(os.path.abspath(__file__))

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_NO_BLOCKS = 3
PA_ERR_CUDA = 4
PA_ERR_WORKSPACE = 5

PA_F16 = 0
PA_BF16 = 1
PA_FP8_E4M3 = 2

PA_DEVERR_BAD_SLOT = 1
PA_DEVERR_BAD_BLOCK = 2
PA_DEVERR_BAD_LEN = 4
PA_DEVERR_TIMEOUT = 8


class PAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"pa status {status}: {message}")
        self.status = status


class PANoBlocks(PAError):
    pass


def _load():
    path = _build.LIB
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with paged_kv_cache_187_gb300.build.build() "
            "(nvcc for sm_103a); this package has no CPU fallback")
    lib = ctypes.CDLL(path)
    P, i32, u64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint64, ctypes.c_float,
                            ctypes.c_size_t)
    sig = {
        "pa_last_error": ([], ctypes.c_char_p),
        "pa_version": ([], i32),
        "pa_set_gqa_tensor_cores": ([i32], i32),
        "pa_set_mq_tcgen05": ([i32], i32),
        "pa_set_kernel_events": ([P, P], i32),
        "pa_selftest_wait_timeout": ([P, ctypes.c_uint32, P], i32),
        "pa_reshape_and_cache": ([P, P, P, P, P, i32, i32, i32, i32, i32, i32, P, P], i32),
        "pa_decode_v1": ([P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, i32, f32, i32, P, P],
                         i32),
        "pa_decode_v2_workspace_size": ([i32, i32, i32, i32, i32], sz),
        "pa_decode_v2": ([P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, i32, f32, i32, i32,
                          P, sz, P, P], i32),
        "pa_decode_v2_noalloc": ([P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, i32, f32,
                                  i32, i32, P, P], i32),
        "pa_decode_auto_plan": ([i32, i32, i32, i32, i32, i32, ctypes.POINTER(i32),
                                 ctypes.POINTER(i32)], i32),
        "pa_decode_auto_workspace_size": ([i32, i32, i32, i32, i32, i32], sz),
        "pa_decode_auto": ([P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, i32, f32, i32, P,
                            sz, P, P], i32),
        "pa_reshape_and_cache_fp8": ([P, P, P, P, P, i32, i32, i32, i32, i32, i32, f32, f32, P, P],
                                     i32),
        "pa_decode_fp8": ([P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, i32, f32, f32, f32,
                           i32, i32, i32, P, sz, P, P], i32),
        "pa_decode_mq_workspace_size": ([i32, i32, i32, i32, i32, i32, i32, i32], sz),
        "pa_decode_mq": ([P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, i32, i32, f32, i32,
                          i32, i32, P, sz, P, P], i32),
        "pa_decode_step": ([P, P, P, P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, i32, f32,
                            i32, P, sz, P, P], i32),
        "pa_decode_step_host_staging_size": ([i32, i32, i32, i32, i32], sz),
        "pa_decode_step_host": ([P, P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32,
                                 f32, i32, P, sz, P, sz, P, P], i32),
        "pa_decode_step_host_overlapped": ([P, P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                            i32, i32, f32, i32, P, sz, P, sz, P, P, P, P, P, P],
                                           i32),
        "pa_alloc_create": ([i32, i32, u64, ctypes.POINTER(P)], i32),
        "pa_alloc_destroy": ([P], None),
        "pa_alloc_num_free": ([P], i32),
        "pa_alloc_add_seq": ([P, i32, i32], i32),
        "pa_alloc_append": ([P, i32, ctypes.POINTER(i32)], i32),
        "pa_alloc_append_batch": ([P, P, i32, P], i32),
        "pa_alloc_free_seq": ([P, i32], i32),
        "pa_alloc_reserve_batch": ([P, P, i32, i32], i32),
        "pa_alloc_fork": ([P, i32, i32, i32], i32),
        "pa_alloc_num_pending_copies": ([P], i32),
        "pa_alloc_take_copies": ([P, P, i32, ctypes.POINTER(i32)], i32),
        "pa_alloc_refcount": ([P, i32], i32),
        "pa_copy_blocks": ([P, P, P, i32, i32, i32, i32, i32, i32, P, P], i32),
        "pa_advance_step": ([P, P, P, i32, i32, i32, i32, P, P, P, P, P], i32),
        "pa_alloc_slots": ([P, i32, i32, i32, P], i32),
        "pa_alloc_block_tables": ([P, P, i32, i32, P], i32),
        "pa_alloc_context_lens": ([P, P, i32, P], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_lib = _load()


def _check(status: int):
    if status != PA_OK:
        msg = (_lib.pa_last_error() or b"").decode()
        if status == PA_ERR_NO_BLOCKS:
            raise PANoBlocks(status, msg)
        raise PAError(status, msg)


def library_path() -> str:
    return _build.LIB


def raw():
    """The ctypes handle of libpa.so (all C symbols)."""
    return _lib


# --------------------------------------------------------------------------- helpers
def _dt(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return PA_F16
    if t.dtype == torch.bfloat16:
        return PA_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float16 or bfloat16)")


def _dev(t, name, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _opt_dev(t, name):
    import torch
    if t is None:
        return None
    return _dev(t, name, torch.int32)


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


# --------------------------------------------------------------------------- kernels
def pa_reshape_and_cache(key, value, key_cache, value_cache, slot_mapping, status=None,
                         stream=None):
    """key/value [T, Hkv, D]; key_cache/value_cache [NB, Hkv, bs, D]; slot_mapping [T] int32."""
    import torch
    T, Hkv, D = key.shape
    NB, Hkv2, bs, D2 = key_cache.shape
    if value.shape != key.shape or value_cache.shape != key_cache.shape or (Hkv2, D2) != (Hkv, D):
        raise ValueError("reshape_and_cache: inconsistent shapes")
    if slot_mapping.shape != (T,):
        raise ValueError("reshape_and_cache: slot_mapping must be [num_tokens]")
    dt = _dt(key)
    for t, n in ((value, "value"), (key_cache, "key_cache"), (value_cache, "value_cache")):
        if t.dtype != key.dtype:
            raise TypeError(f"{n} dtype differs from key")
    _check(_lib.pa_reshape_and_cache(
        _dev(key, "key"), _dev(value, "value"), _dev(key_cache, "key_cache"),
        _dev(value_cache, "value_cache"), _dev(slot_mapping, "slot_mapping", torch.int32),
        T, Hkv, D, bs, NB, dt, _opt_dev(status, "status"), _stream(stream)))


def _decode_common(out, query, key_cache, value_cache, block_tables, context_lens):
    import torch
    S, Hq, D = query.shape
    NB, Hkv, bs, D2 = key_cache.shape
    if out.shape != query.shape or value_cache.shape != key_cache.shape or D2 != D:
        raise ValueError("decode: inconsistent shapes")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("decode: block_tables [S, max_blocks] and context_lens [S] expected")
    dt = _dt(query)
    for t, n in ((out, "out"), (key_cache, "key_cache"), (value_cache, "value_cache")):
        if t.dtype != query.dtype:
            raise TypeError(f"{n} dtype differs from query")
    ptrs = (_dev(out, "out"), _dev(query, "query"), _dev(key_cache, "key_cache"),
            _dev(value_cache, "value_cache"), _dev(block_tables, "block_tables", torch.int32),
            int(block_tables.shape[1]), _dev(context_lens, "context_lens", torch.int32))
    return ptrs, (S, Hq, Hkv, D, bs, NB), dt


def pa_decode_v1(out, query, key_cache, value_cache, block_tables, context_lens,
                 max_context_len: int, scale: float, status=None, stream=None):
    ptrs, (S, Hq, Hkv, D, bs, NB), dt = _decode_common(out, query, key_cache, value_cache,
                                                       block_tables, context_lens)
    _check(_lib.pa_decode_v1(*ptrs, S, Hq, Hkv, D, bs, NB, int(max_context_len), float(scale), dt,
                             _opt_dev(status, "status"), _stream(stream)))


def pa_decode_v2_workspace_size(num_seqs, num_q_heads, head_size, max_context_len,
                                partition_size) -> int:
    return int(_lib.pa_decode_v2_workspace_size(num_seqs, num_q_heads, head_size,
                                                max_context_len, partition_size))


def _ws(workspace):
    if workspace is None:
        return None, 0
    return _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()


def pa_decode_v2(out, query, key_cache, value_cache, block_tables, context_lens,
                 max_context_len: int, scale: float, partition_size: int, workspace,
                 status=None, stream=None):
    ptrs, (S, Hq, Hkv, D, bs, NB), dt = _decode_common(out, query, key_cache, value_cache,
                                                       block_tables, context_lens)
    wp, wb = _ws(workspace)
    _check(_lib.pa_decode_v2(*ptrs, S, Hq, Hkv, D, bs, NB, int(max_context_len), float(scale), dt,
                             int(partition_size), wp, wb, _opt_dev(status, "status"),
                             _stream(stream)))


def _header_scratch_bytes() -> int:
    """PA_NOALLOC_SCRATCH_BYTES as include/pa.h defines it (the one source of the size)."""
    import re
    with open(os.path.join(os.path.dirname(_PKG), "include", "pa.h")) as f:
        m = re.search(r"#define\s+PA_NOALLOC_SCRATCH_BYTES\s+\(\(size_t\)(\d+)\s*<<\s*(\d+)\)",
                      f.read())
    if not m:
        raise ImportError("include/pa.h: PA_NOALLOC_SCRATCH_BYTES not found")
    return int(m.group(1)) << int(m.group(2))


PA_NOALLOC_SCRATCH_BYTES = _header_scratch_bytes()


def pa_decode_v2_noalloc(out, query, key_cache, value_cache, block_tables, context_lens,
                         max_context_len: int, scale: float, partition_size: int, status=None,
                         stream=None):
    """pa_decode_v2 without a workspace argument: the library's fixed device scratch is
    used instead, and nothing is allocated.  For callers that may not allocate device
    memory; calls that overlap on the GPU share that scratch and must be serialised."""
    ptrs, (S, Hq, Hkv, D, bs, NB), dt = _decode_common(out, query, key_cache, value_cache,
                                                       block_tables, context_lens)
    _check(_lib.pa_decode_v2_noalloc(*ptrs, S, Hq, Hkv, D, bs, NB, int(max_context_len),
                                     float(scale), dt, int(partition_size),
                                     _opt_dev(status, "status"), _stream(stream)))


def pa_decode_auto_plan(num_seqs, num_q_heads, num_kv_heads, head_size, block_size,
                        max_context_len):
    v, p = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(_lib.pa_decode_auto_plan(num_seqs, num_q_heads, num_kv_heads, head_size, block_size,
                                    max_context_len, ctypes.byref(v), ctypes.byref(p)))
    return int(v.value), int(p.value)


def pa_decode_auto_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_size, block_size,
                                  max_context_len) -> int:
    return int(_lib.pa_decode_auto_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_size,
                                                  block_size, max_context_len))


def pa_decode_auto(out, query, key_cache, value_cache, block_tables, context_lens,
                   max_context_len: int, scale: float, workspace=None, status=None, stream=None):
    ptrs, (S, Hq, Hkv, D, bs, NB), dt = _decode_common(out, query, key_cache, value_cache,
                                                       block_tables, context_lens)
    wp, wb = _ws(workspace)
    _check(_lib.pa_decode_auto(*ptrs, S, Hq, Hkv, D, bs, NB, int(max_context_len), float(scale),
                               dt, wp, wb, _opt_dev(status, "status"), _stream(stream)))


def _u8(t, name):
    """An fp8 E4M3 pool: a uint8 (or float8_e4m3fn) CUDA tensor."""
    import torch
    if t.dtype not in (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8)):
        raise TypeError(f"{name} must be uint8 / float8_e4m3fn (fp8 E4M3 bytes), got {t.dtype}")
    return _dev(t, name)


def pa_reshape_and_cache_fp8(key, value, key_cache, value_cache, slot_mapping, k_scale: float,
                             v_scale: float, status=None, stream=None):
    """Quantising scatter: key/value [T, Hkv, D] fp16/bf16 -> fp8 E4M3 pools [NB, Hkv, bs, D]."""
    import torch
    T, Hkv, D = key.shape
    NB, Hkv2, bs, D2 = key_cache.shape
    if value.shape != key.shape or value_cache.shape != key_cache.shape or (Hkv2, D2) != (Hkv, D):
        raise ValueError("reshape_and_cache_fp8: inconsistent shapes")
    if slot_mapping.shape != (T,):
        raise ValueError("reshape_and_cache_fp8: slot_mapping must be [num_tokens]")
    _check(_lib.pa_reshape_and_cache_fp8(
        _dev(key, "key"), _dev(value, "value"), _u8(key_cache, "key_cache"),
        _u8(value_cache, "value_cache"), _dev(slot_mapping, "slot_mapping", torch.int32), T, Hkv, D,
        bs, NB, _dt(key), float(k_scale), float(v_scale), _opt_dev(status, "status"),
        _stream(stream)))


_VARIANTS = {"auto": 0, "v1": 1, "v2": 2}


def pa_decode_fp8(out, query, key_cache, value_cache, block_tables, context_lens,
                  max_context_len: int, scale: float, k_scale: float, v_scale: float,
                  variant: str = "auto", partition_size: int = 0, workspace=None, status=None,
                  stream=None):
    """Paged decode over fp8 E4M3 pools; query/out fp16 or bf16 [S, Hq, D]."""
    import torch
    S, Hq, D = query.shape
    NB, Hkv, bs, D2 = key_cache.shape
    if out.shape != query.shape or value_cache.shape != key_cache.shape or D2 != D:
        raise ValueError("decode_fp8: inconsistent shapes")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("decode_fp8: block_tables [S, max_blocks] and context_lens [S] expected")
    wp, wb = _ws(workspace)
    _check(_lib.pa_decode_fp8(
        _dev(out, "out"), _dev(query, "query"), _u8(key_cache, "key_cache"),
        _u8(value_cache, "value_cache"), _dev(block_tables, "block_tables", torch.int32),
        int(block_tables.shape[1]), _dev(context_lens, "context_lens", torch.int32), S, Hq, Hkv, D,
        bs, NB, int(max_context_len), float(scale), float(k_scale), float(v_scale), _dt(query),
        _VARIANTS[variant], int(partition_size or 0), wp, wb, _opt_dev(status, "status"),
        _stream(stream)))


def pa_decode_mq_workspace_size(num_seqs, q_len, num_q_heads, num_kv_heads, head_size, block_size,
                                max_context_len, partition_size=0) -> int:
    return int(_lib.pa_decode_mq_workspace_size(num_seqs, q_len, num_q_heads, num_kv_heads,
                                                head_size, block_size, max_context_len,
                                                int(partition_size or 0)))


def pa_decode_mq(out, query, key_cache, value_cache, block_tables, context_lens,
                 max_context_len: int, scale: float, variant: str = "auto", partition_size: int = 0,
                 workspace=None, status=None, stream=None):
    """Multi-query paged decode: query/out [S, q_len, Hq, D]; new token j of a sequence of
    length L attends to tokens t < L - q_len + j + 1."""
    import torch
    S, QL, Hq, D = query.shape
    NB, Hkv, bs, D2 = key_cache.shape
    if out.shape != query.shape or value_cache.shape != key_cache.shape or D2 != D:
        raise ValueError("decode_mq: inconsistent shapes")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("decode_mq: block_tables [S, max_blocks] and context_lens [S] expected")
    wp, wb = _ws(workspace)
    _check(_lib.pa_decode_mq(
        _dev(out, "out"), _dev(query, "query"), _dev(key_cache, "key_cache"),
        _dev(value_cache, "value_cache"), _dev(block_tables, "block_tables", torch.int32),
        int(block_tables.shape[1]), _dev(context_lens, "context_lens", torch.int32), S, QL, Hq,
        Hkv, D, bs, NB, int(max_context_len), float(scale), _dt(query), _VARIANTS[variant],
        int(partition_size or 0), wp, wb, _opt_dev(status, "status"), _stream(stream)))


def pa_decode_step(out, query, key, value, key_cache, value_cache, slot_mapping, block_tables,
                   context_lens, max_context_len: int, scale: float, workspace=None, status=None,
                   stream=None):
    import torch
    S, Hq, D = query.shape
    NB, Hkv, bs, D2 = key_cache.shape
    if key.shape != (S, Hkv, D) or value.shape != key.shape or slot_mapping.shape != (S,):
        raise ValueError("decode_step: key/value [S, Hkv, D] and slot_mapping [S] expected")
    if out.shape != query.shape or value_cache.shape != key_cache.shape or D2 != D:
        raise ValueError("decode_step: inconsistent shapes")
    dt = _dt(query)
    wp, wb = _ws(workspace)
    _check(_lib.pa_decode_step(
        _dev(out, "out"), _dev(query, "query"), _dev(key, "key"), _dev(value, "value"),
        _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"),
        _dev(slot_mapping, "slot_mapping", torch.int32),
        _dev(block_tables, "block_tables", torch.int32), int(block_tables.shape[1]),
        _dev(context_lens, "context_lens", torch.int32), S, Hq, Hkv, D, bs, NB,
        int(max_context_len), float(scale), dt, wp, wb, _opt_dev(status, "status"),
        _stream(stream)))


def pa_decode_step_host_staging_size(num_seqs, num_q_heads, num_kv_heads, head_size,
                                     max_blocks_per_seq) -> int:
    return int(_lib.pa_decode_step_host_staging_size(num_seqs, num_q_heads, num_kv_heads,
                                                     head_size, max_blocks_per_seq))


def _host(a, name, dtype=None):
    """Host buffer pointer: a CPU torch tensor or a numpy array, contiguous."""
    if hasattr(a, "is_cuda"):
        if a.is_cuda or not a.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CPU tensor")
        if dtype is not None and a.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}")
        return ctypes.c_void_p(a.data_ptr())
    arr = a
    if not arr.flags.c_contiguous:
        raise ValueError(f"{name} must be contiguous")
    return arr.ctypes.data_as(ctypes.c_void_p)


def pa_decode_step_host(out_host, query_host, key_host, value_host, slot_mapping_host,
                        block_tables_host, context_lens_host, key_cache, value_cache,
                        max_context_len: int, scale: float, staging, workspace=None,
                        status=None, stream=None):
    """One decode step from host buffers (pinned CPU tensors): H2D of the inputs,
    reshape_and_cache + decode, D2H of out, all enqueued on the stream (no wait)."""
    import torch
    S, Hq, D = query_host.shape
    NB, Hkv, bs, D2 = key_cache.shape
    if key_host.shape != (S, Hkv, D) or value_host.shape != key_host.shape or D2 != D:
        raise ValueError("decode_step_host: key/value [S, Hkv, D] expected")
    if out_host.shape != query_host.shape or tuple(slot_mapping_host.shape) != (S,):
        raise ValueError("decode_step_host: out [S, Hq, D] and slot_mapping [S] expected")
    maxb = int(block_tables_host.shape[1])
    dt = _dt(key_cache)
    wp, wb = _ws(workspace)
    sp, sb = _ws(staging)
    _check(_lib.pa_decode_step_host(
        _host(out_host, "out_host"), _host(query_host, "query_host"), _host(key_host, "key_host"),
        _host(value_host, "value_host"), _host(slot_mapping_host, "slot_mapping_host"),
        _host(block_tables_host, "block_tables_host"), _host(context_lens_host, "context_lens_host"),
        _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"), maxb, S, Hq, Hkv, D, bs, NB,
        int(max_context_len), float(scale), dt, sp, sb, wp, wb, _opt_dev(status, "status"),
        _stream(stream)))


def pa_decode_step_host_overlapped(out_host, query_host, key_host, value_host,
                                   slot_mapping_host, block_tables_host, context_lens_host,
                                   key_cache, value_cache, max_context_len: int, scale: float,
                                   staging, compute_stream, h2d_stream, d2h_stream, staged_event,
                                   done_event, workspace=None, status=None):
    """pa_decode_step_host with the copies on `h2d_stream` / `d2h_stream` (see pa.h); the
    events are torch.cuda.Event objects already recorded once (so that the CUDA events
    exist)."""
    S, Hq, D = query_host.shape
    NB, Hkv, bs, D2 = key_cache.shape
    if key_host.shape != (S, Hkv, D) or value_host.shape != key_host.shape or D2 != D:
        raise ValueError("decode_step_host: key/value [S, Hkv, D] expected")
    if out_host.shape != query_host.shape or tuple(slot_mapping_host.shape) != (S,):
        raise ValueError("decode_step_host: out [S, Hq, D] and slot_mapping [S] expected")
    maxb = int(block_tables_host.shape[1])
    wp, wb = _ws(workspace)
    sp, sb = _ws(staging)
    _check(_lib.pa_decode_step_host_overlapped(
        _host(out_host, "out_host"), _host(query_host, "query_host"), _host(key_host, "key_host"),
        _host(value_host, "value_host"), _host(slot_mapping_host, "slot_mapping_host"),
        _host(block_tables_host, "block_tables_host"), _host(context_lens_host, "context_lens_host"),
        _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"), maxb, S, Hq, Hkv, D, bs, NB,
        int(max_context_len), float(scale), _dt(key_cache), sp, sb, wp, wb,
        _opt_dev(status, "status"), _stream(compute_stream), _stream(h2d_stream),
        _stream(d2h_stream), ctypes.c_void_p(staged_event.cuda_event),
        ctypes.c_void_p(done_event.cuda_event)))


def pa_set_kernel_events(start_event, stop_event):
    """torch.cuda.Event pair (already recorded once, so that the CUDA event exists) or
    (None, None) to switch the hook off."""
    if start_event is None or stop_event is None:
        _check(_lib.pa_set_kernel_events(None, None))
        return
    _check(_lib.pa_set_kernel_events(ctypes.c_void_p(start_event.cuda_event),
                                     ctypes.c_void_p(stop_event.cuda_event)))


def pa_advance_step(context_lens, slot_mapping, block_tables, block_size: int, num_blocks: int,
                    input_positions=None, input_tokens=None, sampled_token_ids=None,
                    status=None, stream=None):
    """Device-side move of every sequence to its next token (multi-step decode loop)."""
    import torch
    S = int(context_lens.shape[0])
    if slot_mapping.shape != (S,) or block_tables.dim() != 2 or block_tables.shape[0] != S:
        raise ValueError("advance_step: context_lens / slot_mapping [S], block_tables [S, max]")
    def opt64(t, name):
        return None if t is None else _dev(t, name, torch.int64)
    _check(_lib.pa_advance_step(
        _dev(context_lens, "context_lens", torch.int32), _dev(slot_mapping, "slot_mapping", torch.int32),
        _dev(block_tables, "block_tables", torch.int32), int(block_tables.shape[1]), S,
        int(block_size), int(num_blocks), opt64(input_positions, "input_positions"),
        opt64(input_tokens, "input_tokens"), opt64(sampled_token_ids, "sampled_token_ids"),
        _opt_dev(status, "status"), _stream(stream)))


def pa_copy_blocks(key_cache, value_cache, block_pairs, status=None, stream=None):
    """Device copy of whole blocks old -> new for each row (old, new) of block_pairs
    (int32 [n, 2] on the device), in both pools."""
    import torch
    NB, Hkv, bs, D = key_cache.shape
    if value_cache.shape != key_cache.shape or block_pairs.dim() != 2 or block_pairs.shape[1] != 2:
        raise ValueError("copy_blocks: pools [NB, Hkv, bs, D] and pairs [n, 2] expected")
    dt = PA_FP8_E4M3 if key_cache.element_size() == 1 else _dt(key_cache)
    _check(_lib.pa_copy_blocks(_dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"),
                               _dev(block_pairs, "block_pairs", torch.int32),
                               int(block_pairs.shape[0]), Hkv, D, bs, NB, dt,
                               _opt_dev(status, "status"), _stream(stream)))


def pa_selftest_wait_timeout(status, limit_us: int, stream=None):
    """Runs the bounded-wait self-test kernel; sets PA_DEVERR_TIMEOUT in `status`."""
    import torch
    _check(_lib.pa_selftest_wait_timeout(_dev(status, "status", torch.int32), int(limit_us),
                                         _stream(stream)))


def pa_set_gqa_tensor_cores(enable: bool):
    """Process-wide: True (default) decodes grouped-query heads and fp8 caches on the
    tensor cores, False on the CUDA cores (groups above 8 stay on the tensor cores)."""
    _check(_lib.pa_set_gqa_tensor_cores(1 if enable else 0))


def pa_set_mq_tcgen05(enable: bool):
    """Process-wide: True (default) lets multi-query decode with many rows per kv head
    use the tcgen05 kernel, False keeps it on the mma.sync kernel."""
    _check(_lib.pa_set_mq_tcgen05(1 if enable else 0))


# --------------------------------------------------------------------------- allocator
def _np_i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _nptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


class PagedAllocator:
    """Host block allocator (pa_alloc_* calls): builds block tables and slot mappings."""

    def __init__(self, num_blocks: int, block_size: int, seed: int):
        h = ctypes.c_void_p()
        _check(_lib.pa_alloc_create(int(num_blocks), int(block_size),
                                    int(seed) & (2**64 - 1), ctypes.byref(h)))
        self._h = h
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)

    def close(self):
        if self._h:
            _lib.pa_alloc_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def num_free(self) -> int:
        return int(_lib.pa_alloc_num_free(self._h))

    def pa_alloc_add_seq(self, seq_id: int, num_tokens: int):
        _check(_lib.pa_alloc_add_seq(self._h, int(seq_id), int(num_tokens)))

    def pa_alloc_append(self, seq_id: int) -> int:
        s = ctypes.c_int32(0)
        _check(_lib.pa_alloc_append(self._h, int(seq_id), ctypes.byref(s)))
        return int(s.value)

    @staticmethod
    def _out(out, shape):
        if out is None:
            return np.empty(shape, dtype=np.int32)
        if out.dtype != np.int32 or out.shape != tuple(shape) or not out.flags.c_contiguous:
            raise ValueError(f"out must be a contiguous int32 array of shape {tuple(shape)}")
        return out

    def pa_alloc_append_batch(self, seq_ids, out=None) -> np.ndarray:
        ids = _np_i32(seq_ids)
        out = self._out(out, (ids.size,))
        _check(_lib.pa_alloc_append_batch(self._h, _nptr(ids), ids.size, _nptr(out)))
        return out

    def pa_alloc_reserve_batch(self, seq_ids, extra_tokens: int):
        ids = _np_i32(seq_ids)
        _check(_lib.pa_alloc_reserve_batch(self._h, _nptr(ids), ids.size, int(extra_tokens)))

    def pa_alloc_fork(self, src_seq: int, dst_seq: int, num_tokens: int):
        _check(_lib.pa_alloc_fork(self._h, int(src_seq), int(dst_seq), int(num_tokens)))

    def pa_alloc_take_copies(self) -> np.ndarray:
        """Pending copy-on-write pairs [n, 2] (old, new), cleared."""
        n = int(_lib.pa_alloc_num_pending_copies(self._h))
        out = np.zeros((max(n, 1), 2), dtype=np.int32)
        got = ctypes.c_int32(0)
        _check(_lib.pa_alloc_take_copies(self._h, _nptr(out), n, ctypes.byref(got)))
        return out[:got.value]

    def pa_alloc_refcount(self, block: int) -> int:
        return int(_lib.pa_alloc_refcount(self._h, int(block)))

    def pa_alloc_free_seq(self, seq_id: int):
        _check(_lib.pa_alloc_free_seq(self._h, int(seq_id)))

    def pa_alloc_slots(self, seq_id: int, start: int, n: int) -> np.ndarray:
        out = np.empty(int(n), dtype=np.int32)
        _check(_lib.pa_alloc_slots(self._h, int(seq_id), int(start), int(n), _nptr(out)))
        return out

    def pa_alloc_block_tables(self, seq_ids, max_blocks_per_seq: int, out=None) -> np.ndarray:
        ids = _np_i32(seq_ids)
        out = self._out(out, (ids.size, int(max_blocks_per_seq)))
        _check(_lib.pa_alloc_block_tables(self._h, _nptr(ids), ids.size, int(max_blocks_per_seq),
                                          _nptr(out)))
        return out

    def pa_alloc_context_lens(self, seq_ids, out=None) -> np.ndarray:
        ids = _np_i32(seq_ids)
        out = self._out(out, (ids.size,))
        _check(_lib.pa_alloc_context_lens(self._h, _nptr(ids), ids.size, _nptr(out)))
        return out
