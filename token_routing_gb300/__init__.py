"""GB300 (sm_103a) MoE layer: token routing and expert compute behind a C ABI (libmoe.so).

The compute runs only in the CUDA kernels of libmoe.so; this package marshals torch
tensors to its entry points. Build the library with `python -m token_routing_gb300.build`.
"""
from ._lib import (MoeConfig, MoeError, LIB_PATH, HEADER_PATH, load, header_symbols,  # noqa: F401
                   MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA,
                   MOE_ERR_DEVICE_TIMEOUT, MOE_ERR_DEVICE_BOUNDS, MOE_F32, MOE_BF16,
                   MOE_ROW_ALIGN, MOE_MAX_WINDOW)
from .layer import (make_config, config_from, workspace_bytes, alloc_buffers, route,  # noqa: F401
                    dispatch, expert_ffn, combine, backward, forward, forward_backward, coselect,
                    soft_balance, soft_balance_backward, soft_balance_window,
                    soft_balance_window_backward,
                    get_error, kernel_launches, selftest_wait_timeout, StepGraph, KernelTrace)

__version__ = "0.1"
