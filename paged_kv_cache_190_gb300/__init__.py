"""GB300-native paged-KV-cache decode.

A thin Python binding of ``libpagedattn.so`` (CUDA C++ for sm_103a, C ABI in
``include/pa.h``).  Each function here has the C entry point's name and only
marshals arguments: torch tensors become raw device pointers, the current CUDA
stream becomes a ``cudaStream_t``.  Every step of the path runs in the library's
kernels; there is no fallback -- if the library is missing or was not built,
the first call raises.

PyTorch provides device memory and streams; nothing else.
"""
from ._lib import (  # noqa: F401
    PA_BF16, PA_F32, PA_ERR_SWAPPED, PA_DEVERR_BAD_BLOCK, PA_DEVERR_BAD_LENGTH, PA_DEVERR_BAD_SLOT,
    PA_DEVERR_TIMEOUT, PA_NOALLOC_SCRATCH_BYTES, EXPORTED_SYMBOLS, BlockManager, OutOfBlocks,
    PaError, PreparedCall, Swapped, library, library_path, pa_copy_blocks, pa_debug_set_wait_limit,
    pa_decode, pa_cascade_groups, pa_decode_cascade, pa_decode_cascade_workspace_size,
    pa_decode_chunk_tokens, pa_decode_fp8, pa_decode_multi, pa_decode_noalloc,
    pa_decode_workspace_size,
    pa_get_error_string, pa_read_device_errors, pa_reshape_and_cache, pa_reshape_and_cache_fp8,
    pa_swap_blocks,
)
