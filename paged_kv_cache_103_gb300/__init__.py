"""GB300-native paged KV-cache decode attention (sm_103a).

The compute path is ``libpa.so`` (C ABI, ``include/pa.h``); ``binding``
exposes it under the same names.  Importing the package loads nothing; the
library is loaded on first use and its absence is an error, never a fallback.
"""
from .binding import (Allocator, PaError, Step, load, pa_check_device_errors,  # noqa: F401
                      pa_copy_blocks,
                      pa_decode, pa_decode_fp8, pa_decode_grid_size, pa_decode_int8,
                      pa_multi_query,
                      pa_multi_query_workspace_size, pa_decode_workspace_init,
                      pa_decode_workspace_size, pa_reshape_and_cache, pa_reshape_and_cache_fp8,
                      pa_reshape_and_cache_int8,
                      pa_swap_blocks)
