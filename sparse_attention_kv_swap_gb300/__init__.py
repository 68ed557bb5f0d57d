"""GB300-native decode KV swap-in for HiSparse-style sparse attention.

The compute path is the CUDA library built from ``csrc/`` (C ABI in
``include/hisparse_swap.h``); ``binding`` marshals arguments to it and
``cache`` allocates the caller-owned buffers with PyTorch.
"""
from . import binding  # noqa: F401
from .binding import (HsConfig, HsError, make_config, load_library,  # noqa: F401
                      hs_config_check, hs_state_bytes, hs_workspace_bytes, hs_device_kv_bytes,
                      hs_host_pool_bytes, hs_hash_size, hs_create_state, hs_destroy_state,
                      hs_swap_in, hs_page_table, hs_reset_requests, hs_get_status,
                      hs_export_request_state, hs_status_string, hs_version,
                      hs_set_timeline, hs_set_copy_ctas, hs_set_defer_copy,
                      hs_copy_planned, hs_append_rows, hs_get_stats)


def __getattr__(name):
    if name == "SwapInCache":
        from .cache import SwapInCache
        return SwapInCache
    raise AttributeError(name)
