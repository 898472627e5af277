"""fa512: head-dim-512 FlashAttention forward for GB300 (sm_103a).

The compute lives in hand-written CUDA kernels behind the C ABI declared in
``include/fa512.h``; :mod:`._binding` marshals torch tensors into that ABI.
Importing this package does not load the shared library; the first call does,
and it raises if the library has not been built.
"""
from ._binding import (  # noqa: F401
    Fa512Error,
    fa512_decode_auto_splits,
    fa512_decode_auto_splits_fp8,
    fa512_decode_paged,
    fa512_decode_paged_noalloc,
    fa512_decode_paged_fp8,
    fa512_decode_paged_q,
    fa512_decode_workspace_bytes,
    fa512_decode_workspace_bytes_fp8,
    fa512_device_status,
    fa512_prefill,
    fa512_prefill_d256,
    fa512_prefill_paged,
    fa512_status_string,
    library_path,
    load_library,
)
