"""Grouped-query attention with learned per-head sinks for GB300 (sm_103a).

The computation lives in libsinkattn.so (C ABI: include/sinkattn.h); this
package holds its ctypes binding, its build script and the seeded synthetic
input generators. Importing the package does not load the library; the first
call does, and raises if the library is missing.
"""
from .sinkattn import (  # noqa: F401
    SinkAttnError,
    load,
    sinkattn_decode,
    sinkattn_decode_fp8,
    sinkattn_debug_stall_waits,
    sinkattn_decode_workspace_size,
    sinkattn_get_device_error,
    sinkattn_merge,
    sinkattn_decode_noalloc,
    sinkattn_prefill,
    sinkattn_prefill_backward,
    sinkattn_prefill_backward_workspace_size,
    sinkattn_prefill_paged,
    sinkattn_prefill_paged_fp8,
    sinkattn_prefill_paged_workspace_size,
    sinkattn_prefill_workspace_size,
)
