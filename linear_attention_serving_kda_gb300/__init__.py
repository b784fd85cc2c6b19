"""GB300 (sm_103a) implementation of the Kimi Delta Attention (KDA) layer.

The compute lives in the CUDA library ``_build/libkda.so`` behind the C ABI
of ``include/kda.h``; ``kda`` is its ctypes binding (same function names),
``workloads`` the seeded input generator, ``runtime`` device-buffer helpers.
"""
from .kda import (  # noqa: F401
    KDA_DEV_BAD_ACCEPTED, KDA_DEV_BAD_SEQLENS, KDA_DEV_BAD_SLOT, KDA_DTYPE_BF16,
    KDA_ACT_EXP, KDA_ACT_RCP, KDA_ACT_SIGMOID, KDA_ACT_SILU,
    KDA_DTYPE_F32, KDA_ERR_DEVICE, KDA_ERR_INVALID_ARGUMENT, KDA_ERR_INVALID_BOUND,
    KDA_ERR_LAUNCH, KDA_ERR_UNSUPPORTED_GEOMETRY, KDA_ERR_WORKSPACE, KDA_GATE_SAFE,
    KDA_GATE_SOFTPLUS, KDA_OK, KdaError, Params, Prepared, check, kda_commit, kda_commit_verify, kda_debug_activations, kda_decode,
    kda_prefill_scan, kda_prefill_scan_workspace_bytes, kda_prefill_static_workspace_capacity,
    kda_prefill_varlen, kda_prefill_varlen_static_ws,
    kda_prefill_workspace_bytes, kda_verify_log_bytes, kda_verify_window,
    load, status_string,
)
