"""GB300-native paged-attention decode: reshape_and_cache, PagedAttention V1 / V2 decode,
an auto dispatcher, a device-side advance_step for multi-step loops and a host block
allocator, behind the C ABI of include/pa.h.

The CUDA library (libpa.so, sm_103a) is loaded on first use of any ``pa_*`` / ``PA_*``
name; there is no CPU fallback.  ``workloads`` (seeded synthetic inputs) imports
without it.
"""
import importlib

_OTHER_BINDING_NAMES = {"PagedAllocator", "PAError", "PANoBlocks", "library_path", "raw"}


def __getattr__(name):
    if name.startswith(("pa_", "PA_")) or name in _OTHER_BINDING_NAMES:
        return getattr(importlib.import_module("._binding", __name__), name)
    if name == "DecodeRunner":
        return getattr(importlib.import_module(".runner", __name__), name)
    raise AttributeError(name)
