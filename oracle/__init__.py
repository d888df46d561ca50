"""Plain fp64 CPU oracle for the paged-attention decode step (TEST INFRASTRUCTURE).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the package
``paged_kv_cache_187_gb300`` and its CUDA library) never imports it, and this
package imports nothing from the product.

The arithmetic lives in ``oracle.c`` (plain C, single-threaded, fp64, built with
``-ffp-contract=off``); this module compiles it with gcc and wraps it with ctypes
for numpy arrays.  16-bit float tensors travel as ``np.uint16`` bit patterns so
the conversions are the oracle's own, not numpy's or torch's.

Each routine follows the pages it cites in ``oracle.c``:
  * "vLLM Project Update" talk: PagedAttention over blocks of KV cache, and the
    V2 kernel that partitions a sequence and merges like flash decoding;
  * "vLLM: Easy, Fast, and Cheap LLM Serving with PagedAttention" thread: exact
    attention, 1.7 GB of KV per LLaMA-13B sequence;
  * "[core] Multi Step Scheduling #7000": slot_mapping / block_tables / seq_lens
    and the v2 block manager.

Parity is pinned by ``tests/test_oracle_pins.py``; the only unpinned quantity is
the exact fp32 rounding the GPU takes inside its tolerance.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# PA_ORACLE_SRC points the wrapper at another copy of oracle.c (the planted-mistake
# tests compile altered copies in a scratch folder); the library is built next to it.
_SRC = os.environ.get("PA_ORACLE_SRC") or os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(_SRC)), "liboracle.so")
_lock = threading.Lock()
_lib = None

F16 = 0
BF16 = 1
_DTYPES = {"f16": F16, "fp16": F16, "float16": F16, "bf16": BF16, "bfloat16": BF16}


def dtype_code(dtype) -> int:
    if isinstance(dtype, int):
        return dtype
    return _DTYPES[str(dtype).replace("torch.", "")]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, -O2, no FP contraction)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, u64, f32, f64 = (ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64,
                                   ctypes.c_float, ctypes.c_double)
        lib.or_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.or_f16_to_f64.restype = f64
        lib.or_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.or_bf16_to_f64.restype = f64
        lib.or_f64_to_f16.argtypes = [f64]
        lib.or_f64_to_f16.restype = ctypes.c_uint16
        lib.or_f64_to_bf16.argtypes = [f64]
        lib.or_f64_to_bf16.restype = ctypes.c_uint16
        lib.or_widen_array.argtypes = [P, P, i64, i32]
        lib.or_round_array.argtypes = [P, P, i64, i32]
        lib.or_reshape_and_cache.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32]
        lib.or_reshape_and_cache.restype = i32
        dec = [P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, f32, i32, P]
        lib.or_paged_decode_v1.argtypes = dec
        lib.or_paged_decode_v1.restype = i32
        lib.or_paged_decode_v2.argtypes = dec + [i32]
        lib.or_paged_decode_v2.restype = i32
        lib.or_paged_decode_mq.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32,
                                           i32, f32, i32]
        lib.or_paged_decode_mq.restype = i32
        lib.or_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.or_e4m3_to_f64.restype = f64
        lib.or_f64_to_e4m3.argtypes = [f64]
        lib.or_f64_to_e4m3.restype = ctypes.c_uint8
        lib.or_e4m3_widen_array.argtypes = [P, P, i64]
        lib.or_e4m3_round_array.argtypes = [P, P, i64]
        lib.or_reshape_and_cache_fp8.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, f32, f32]
        lib.or_reshape_and_cache_fp8.restype = i32
        lib.or_paged_decode_fp8.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32,
                                            f32, f32, f32, i32, P]
        lib.or_paged_decode_fp8.restype = i32
        lib.or_splitmix64_next.argtypes = [ctypes.POINTER(u64)]
        lib.or_splitmix64_next.restype = u64
        lib.or_alloc_create.argtypes = [i32, i32, u64, i32]
        lib.or_alloc_create.restype = P
        lib.or_alloc_destroy.argtypes = [P]
        lib.or_alloc_num_free.argtypes = [P]
        lib.or_alloc_num_free.restype = i32
        lib.or_alloc_add_seq.argtypes = [P, i32, i32]
        lib.or_alloc_add_seq.restype = i32
        lib.or_alloc_append.argtypes = [P, i32, ctypes.POINTER(i32)]
        lib.or_alloc_append.restype = i32
        lib.or_alloc_reserve.argtypes = [P, i32, i32]
        lib.or_alloc_reserve.restype = i32
        lib.or_alloc_fork.argtypes = [P, i32, i32, i32]
        lib.or_alloc_fork.restype = i32
        lib.or_alloc_take_copies.argtypes = [P, P, i32]
        lib.or_alloc_take_copies.restype = i32
        lib.or_alloc_refcount.argtypes = [P, i32]
        lib.or_alloc_refcount.restype = i32
        lib.or_copy_blocks.argtypes = [P, P, P, i32, i32, i32, i32, i32]
        lib.or_copy_blocks.restype = i32
        lib.or_alloc_free_seq.argtypes = [P, i32]
        lib.or_alloc_free_seq.restype = i32
        lib.or_alloc_slots.argtypes = [P, i32, i32, i32, P]
        lib.or_alloc_slots.restype = i32
        lib.or_alloc_block_tables.argtypes = [P, P, i32, i32, P]
        lib.or_alloc_block_tables.restype = i32
        lib.or_alloc_context_lens.argtypes = [P, P, i32, P]
        lib.or_alloc_context_lens.restype = i32
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


# --------------------------------------------------------------------------- conversions
def widen(bits: np.ndarray, dtype) -> np.ndarray:
    """16-bit float bit patterns -> exact float64 values."""
    lib = _load()
    b = _c(bits, np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    lib.or_widen_array(_ptr(b), _ptr(out), b.size, dtype_code(dtype))
    return out


def round_to(x: np.ndarray, dtype) -> np.ndarray:
    """float64 values -> 16-bit bit patterns, round to nearest, ties to even."""
    lib = _load()
    v = _c(x, np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    lib.or_round_array(_ptr(v), _ptr(out), v.size, dtype_code(dtype))
    return out


def decode_mq(q_bits, k_cache_bits, v_cache_bits, block_tables, context_lens, scale, dtype):
    """fp64 multi-query decode: q [S, q_len, Hq, D] -> [S, q_len, Hq, D]; new token j of a
    sequence of length L attends to tokens t < L - q_len + j + 1."""
    lib = _load()
    q = _c(q_bits, np.uint16)
    kc = _c(k_cache_bits, np.uint16)
    vc = _c(v_cache_bits, np.uint16)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    S, QL, Hq, D = q.shape
    NB, Hkv, bs, _ = kc.shape
    out = np.zeros((S, QL, Hq, D), dtype=np.float64)
    rc = lib.or_paged_decode_mq(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1],
                                _ptr(cl), S, QL, Hq, Hkv, D, bs, NB, float(scale),
                                dtype_code(dtype))
    if rc == -2:
        raise ValueError("oracle: unsupported shapes")
    if rc == -1:
        raise IndexError("oracle: block table entry outside the pool")
    return out


def e4m3_widen(bits: np.ndarray) -> np.ndarray:
    """fp8 E4M3 bit patterns (uint8) -> exact float64 values."""
    lib = _load()
    b = _c(bits, np.uint8)
    out = np.empty(b.shape, dtype=np.float64)
    lib.or_e4m3_widen_array(_ptr(b), _ptr(out), b.size)
    return out


def e4m3_round(x: np.ndarray) -> np.ndarray:
    """float64 -> E4M3 bit patterns, nearest-even, saturating at +-448."""
    lib = _load()
    v = _c(x, np.float64)
    out = np.empty(v.shape, dtype=np.uint8)
    lib.or_e4m3_round_array(_ptr(v), _ptr(out), v.size)
    return out


def reshape_and_cache_fp8(key_bits, value_bits, key_cache8, value_cache8, slot_mapping,
                          block_size: int, dtype, k_scale: float, v_scale: float) -> int:
    """Quantising scatter of 16-bit rows [T, Hkv, D] into uint8 E4M3 pools, in place."""
    lib = _load()
    k = _c(key_bits, np.uint16)
    v = _c(value_bits, np.uint16)
    sm = _c(slot_mapping, np.int32)
    assert key_cache8.dtype == np.uint8 and key_cache8.flags.c_contiguous
    assert value_cache8.dtype == np.uint8 and value_cache8.flags.c_contiguous
    T, Hkv, D = k.shape
    NB = key_cache8.shape[0]
    return int(lib.or_reshape_and_cache_fp8(_ptr(k), _ptr(v), _ptr(key_cache8), _ptr(value_cache8),
                                            _ptr(sm), T, Hkv, D, block_size, NB, dtype_code(dtype),
                                            float(k_scale), float(v_scale)))


def decode_fp8(q_bits, k_cache8, v_cache8, block_tables, context_lens, scale, k_scale, v_scale,
               dtype, only=None, strict: bool = True):
    """Exact fp64 decode over fp8 E4M3 pools (dequantised by the per-tensor scales).

    A token whose block the table does not give (its logical block past the table row,
    or an entry outside the pool) reads as zeros.  strict=True raises IndexError when
    that happened; strict=False returns (out, flagged) instead."""
    lib = _load()
    q = _c(q_bits, np.uint16)
    kc = _c(k_cache8, np.uint8)
    vc = _c(v_cache8, np.uint8)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    S, Hq, D = q.shape
    NB, Hkv, bs, _ = kc.shape
    out = np.zeros((S, Hq, D), dtype=np.float64)
    only_arr = None if only is None else _c(only, np.uint8).reshape(S * Hq)
    rc = lib.or_paged_decode_fp8(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1],
                                 _ptr(cl), S, Hq, Hkv, D, bs, NB, float(scale), float(k_scale),
                                 float(v_scale), dtype_code(dtype),
                                 _ptr(only_arr) if only_arr is not None else None)
    if rc == -2:
        raise ValueError("oracle: unsupported shapes")
    if not strict:
        return out, rc == -1
    if rc == -1:
        raise IndexError("oracle: block table entry outside the pool")
    return out


def splitmix64_stream(seed: int, n: int) -> list[int]:
    lib = _load()
    st = ctypes.c_uint64(seed)
    return [int(lib.or_splitmix64_next(ctypes.byref(st))) for _ in range(n)]


# --------------------------------------------------------------------------- reshape_and_cache
def reshape_and_cache(key_bits, value_bits, key_cache_bits, value_cache_bits, slot_mapping,
                      block_size: int) -> int:
    """Scatter rows [T, Hkv, D] into pools [NB, Hkv, bs, D] in place.

    Returns the count of out-of-range slots that were skipped."""
    lib = _load()
    k = _c(key_bits, np.uint16)
    v = _c(value_bits, np.uint16)
    sm = _c(slot_mapping, np.int32)
    assert key_cache_bits.flags.c_contiguous and key_cache_bits.dtype == np.uint16
    assert value_cache_bits.flags.c_contiguous and value_cache_bits.dtype == np.uint16
    T, Hkv, D = k.shape
    NB = key_cache_bits.shape[0]
    assert key_cache_bits.shape == (NB, Hkv, block_size, D)
    return int(lib.or_reshape_and_cache(_ptr(k), _ptr(v), _ptr(key_cache_bits),
                                        _ptr(value_cache_bits), _ptr(sm), T, Hkv, D,
                                        block_size, NB))


def copy_blocks(key_cache_bits, value_cache_bits, pairs) -> int:
    """Copy whole blocks old -> new for each (old, new) row of pairs, in place."""
    lib = _load()
    pr = _c(pairs, np.int32).reshape(-1, 2)
    NB, Hkv, bs, D = key_cache_bits.shape
    return int(lib.or_copy_blocks(_ptr(key_cache_bits), _ptr(value_cache_bits), _ptr(pr),
                                  pr.shape[0], Hkv, D, bs, NB))


# --------------------------------------------------------------------------- decode
def _decode(fn, q_bits, k_cache_bits, v_cache_bits, block_tables, context_lens, scale, dtype,
            only=None, extra=()):
    lib = _load()
    q = _c(q_bits, np.uint16)
    kc = _c(k_cache_bits, np.uint16)
    vc = _c(v_cache_bits, np.uint16)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    S, Hq, D = q.shape
    NB, Hkv, bs, D2 = kc.shape
    assert D2 == D and vc.shape == kc.shape and bt.shape[0] == S and cl.shape == (S,)
    out = np.zeros((S, Hq, D), dtype=np.float64)
    only_arr = None
    if only is not None:
        only_arr = _c(only, np.uint8).reshape(S * Hq)
    rc = fn(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], _ptr(cl), S, Hq,
            Hkv, D, bs, NB, float(scale), dtype_code(dtype),
            _ptr(only_arr) if only_arr is not None else None, *extra)
    if rc == -2:
        raise ValueError("oracle: unsupported shapes")
    if rc == -1:
        raise IndexError("oracle: block table entry outside the pool")
    return out


def decode_v1(q_bits, k_cache_bits, v_cache_bits, block_tables, context_lens, scale, dtype,
              only=None) -> np.ndarray:
    """Exact fp64 paged decode over each sequence's whole context -> [S, Hq, D] float64."""
    return _decode(_load().or_paged_decode_v1, q_bits, k_cache_bits, v_cache_bits,
                   block_tables, context_lens, scale, dtype, only)


def decode_v2(q_bits, k_cache_bits, v_cache_bits, block_tables, context_lens, scale, dtype,
              partition_size: int, only=None) -> np.ndarray:
    """fp64 partitioned decode with log-sum-exp merge -> [S, Hq, D] float64."""
    return _decode(_load().or_paged_decode_v2, q_bits, k_cache_bits, v_cache_bits,
                   block_tables, context_lens, scale, dtype, only,
                   extra=(int(partition_size),))


# --------------------------------------------------------------------------- allocator
class OracleAllocError(RuntimeError):
    pass


class Alloc:
    """The oracle's block allocator (same written spec as the product's)."""

    def __init__(self, num_blocks: int, block_size: int, seed: int, max_seqs: int = 1 << 16):
        self._lib = _load()
        self.block_size = block_size
        self._h = self._lib.or_alloc_create(num_blocks, block_size, seed & (2**64 - 1), max_seqs)
        if not self._h:
            raise ValueError("oracle alloc: bad arguments")

    def close(self):
        if self._h:
            self._lib.or_alloc_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _chk(self, rc):
        if rc == -3:
            raise OracleAllocError("no free blocks")
        if rc != 0:
            raise OracleAllocError(f"bad request ({rc})")

    @property
    def num_free(self) -> int:
        return int(self._lib.or_alloc_num_free(self._h))

    def add_seq(self, seq_id: int, num_tokens: int):
        self._chk(self._lib.or_alloc_add_seq(self._h, seq_id, num_tokens))

    def append(self, seq_id: int) -> int:
        slot = ctypes.c_int32(0)
        self._chk(self._lib.or_alloc_append(self._h, seq_id, ctypes.byref(slot)))
        return int(slot.value)

    def reserve(self, seq_id: int, extra_tokens: int):
        self._chk(self._lib.or_alloc_reserve(self._h, seq_id, extra_tokens))

    def fork(self, src: int, dst: int, num_tokens: int):
        self._chk(self._lib.or_alloc_fork(self._h, src, dst, num_tokens))

    def take_copies(self) -> np.ndarray:
        """Pending copy-on-write pairs [n, 2] (old, new), cleared."""
        n = self._lib.or_alloc_take_copies(self._h, None, 0)
        out = np.zeros((max(n, 1), 2), dtype=np.int32)
        got = self._lib.or_alloc_take_copies(self._h, _ptr(out), n)
        assert got == n
        return out[:n]

    def refcount(self, block: int) -> int:
        return int(self._lib.or_alloc_refcount(self._h, block))

    def free_seq(self, seq_id: int):
        self._chk(self._lib.or_alloc_free_seq(self._h, seq_id))

    def slots(self, seq_id: int, start: int, n: int) -> np.ndarray:
        out = np.empty(n, dtype=np.int32)
        self._chk(self._lib.or_alloc_slots(self._h, seq_id, start, n, _ptr(out)))
        return out

    def block_tables(self, seq_ids, max_blocks_per_seq: int) -> np.ndarray:
        ids = _c(seq_ids, np.int32)
        out = np.empty((ids.size, max_blocks_per_seq), dtype=np.int32)
        self._chk(self._lib.or_alloc_block_tables(self._h, _ptr(ids), ids.size,
                                                  max_blocks_per_seq, _ptr(out)))
        return out

    def context_lens(self, seq_ids) -> np.ndarray:
        ids = _c(seq_ids, np.int32)
        out = np.empty(ids.size, dtype=np.int32)
        self._chk(self._lib.or_alloc_context_lens(self._h, _ptr(ids), ids.size, _ptr(out)))
        return out
