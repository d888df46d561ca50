"""GB300-native paged-attention decode: reshape_and_cache, PagedAttention V1 / V2 decode,
an auto dispatcher and a host block allocator, behind the C ABI of include/pa.h.

The CUDA library (libpa.so, sm_103a) is loaded on first use of any pa_* name; there
is no CPU fallback.  ``workloads`` (seeded synthetic inputs) imports without it.
"""
import importlib

_BINDING_NAMES = {
    "pa_reshape_and_cache", "pa_decode_v1", "pa_decode_v2", "pa_decode_v2_noalloc", "PA_NOALLOC_SCRATCH_BYTES", "pa_decode_v2_workspace_size",
    "pa_decode_auto", "pa_decode_auto_plan", "pa_decode_auto_workspace_size", "pa_decode_step",
    "pa_set_gqa_tensor_cores", "pa_set_kernel_events", "PagedAllocator", "PAError", "PANoBlocks", "library_path", "raw",
    "PA_DEVERR_BAD_SLOT", "PA_DEVERR_BAD_BLOCK", "PA_DEVERR_BAD_LEN", "PA_DEVERR_TIMEOUT",
}


def __getattr__(name):
    if name in _BINDING_NAMES:
        return getattr(importlib.import_module("._binding", __name__), name)
    if name in ("DecodeRunner",):
        return getattr(importlib.import_module(".runner", __name__), name)
    raise AttributeError(name)
