"""Python binding of the C ABI in include/kda.h (ctypes; marshalling only).

Each function has the name of its C entry point and passes device pointers
of torch tensors straight through; every step of the layer runs in the CUDA
library.  Loading fails loudly when the library has not been built: there is
no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_build", "libkda.so")

KDA_OK = 0
KDA_ERR_INVALID_ARGUMENT = 1
KDA_ERR_UNSUPPORTED_GEOMETRY = 2
KDA_ERR_INVALID_BOUND = 3
KDA_ERR_WORKSPACE = 4
KDA_ERR_LAUNCH = 5
KDA_ERR_DEVICE = 6
KDA_DEV_BAD_SEQLENS = 1
KDA_DEV_BAD_SLOT = 2
KDA_DEV_BAD_ACCEPTED = 4
KDA_DEV_TIMEOUT = 8
KDA_ACT_EXP = 0
KDA_ACT_RCP = 1
KDA_ACT_SIGMOID = 2
KDA_ACT_SILU = 3
KDA_DTYPE_F32 = 0
KDA_DTYPE_BF16 = 1
KDA_GATE_SOFTPLUS = 0
KDA_GATE_SAFE = 1


class kda_params(ctypes.Structure):
    _fields_ = [
        ("num_heads", ctypes.c_int32), ("head_dim_k", ctypes.c_int32),
        ("head_dim_v", ctypes.c_int32), ("conv_kernel", ctypes.c_int32),
        ("gate_mode", ctypes.c_int32), ("gate_lower_bound", ctypes.c_float),
        ("l2_eps", ctypes.c_float), ("norm_eps", ctypes.c_float),
        ("scale", ctypes.c_float), ("io_dtype", ctypes.c_int32),
        ("out_dtype", ctypes.c_int32), ("num_slots", ctypes.c_int32),
        ("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
        ("conv_weight", ctypes.c_void_p), ("norm_weight", ctypes.c_void_p),
    ]


_VP = ctypes.c_void_p
_I32 = ctypes.c_int32
_SIG = {
    "kda_prefill_varlen": (ctypes.c_int, [ctypes.POINTER(kda_params), _VP, _I32, _I32, _VP, _VP, _VP, _VP,
                                          _VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_size_t, _VP, _VP]),
    "kda_prefill_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(kda_params), _I32, _I32]),
    "kda_prefill_varlen_static_ws": (ctypes.c_int, [ctypes.POINTER(kda_params), _VP, _I32, _I32, _VP, _VP, _VP,
                                                    _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "kda_prefill_static_workspace_capacity": (ctypes.c_size_t, []),
    "kda_prefill_scan": (ctypes.c_int, [ctypes.POINTER(kda_params), _VP, _I32, _I32, _VP, _VP, _VP, _VP, _VP,
                                        _VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_size_t, _I32, _VP, _VP]),
    "kda_prefill_scan_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(kda_params), _I32, _I32, _I32]),
    "kda_debug_split_chains_only": (ctypes.c_int, [ctypes.POINTER(kda_params), _VP, _I32, _I32, _VP, _VP, _VP,
                                                   _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_size_t,
                                                   _VP, ctypes.c_uint32, _VP]),
    "kda_debug_activations": (ctypes.c_int, [_I32, _VP, _VP, _I32, _VP]),
    "kda_decode": (ctypes.c_int, [ctypes.POINTER(kda_params), _I32, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                  _VP, _VP, _VP, _VP, _VP]),
    "kda_verify_window": (ctypes.c_int, [ctypes.POINTER(kda_params), _I32, _I32, _VP, _VP, _VP, _VP, _VP,
                                         _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "kda_verify_log_bytes": (ctypes.c_size_t, [ctypes.POINTER(kda_params), _I32, _I32]),
    "kda_commit_verify": (ctypes.c_int, [ctypes.POINTER(kda_params), _I32, _I32] + [_VP] * 14 + [_VP]),
    "kda_commit": (ctypes.c_int, [ctypes.POINTER(kda_params), _I32, _I32, _VP, _VP, _VP, _VP, _VP,
                                  _VP, _VP]),
    "kda_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "kda_abi_version": (ctypes.c_int, []),
}

_lib = None


def load(path: Optional[str] = None):
    """Load libkda.so (raises if it is missing)."""
    global _lib
    if _lib is None:
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"KDA CUDA library not built: {p} is missing "
                               "(run linear_attention_serving_kda_gb300.build.build())")
        lib = ctypes.CDLL(p)
        for name, (res, args) in _SIG.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


class KdaError(RuntimeError):
    def __init__(self, rc: int):
        super().__init__(f"{status_string(rc)} ({rc})")
        self.rc = rc


def status_string(rc: int) -> str:
    return load().kda_status_string(rc).decode()


def check(rc: int) -> None:
    if rc != KDA_OK:
        raise KdaError(rc)


@dataclass
class Params:
    """Layer configuration; the four parameter tensors live on the device."""

    num_heads: int
    head_dim: int
    conv_kernel: int
    gate_mode: int
    A_log: object
    dt_bias: object
    conv_weight: object
    norm_weight: object = None
    gate_lower_bound: float = -5.0
    l2_eps: float = 1e-6
    norm_eps: float = 1e-6
    scale: float = 1.0
    io_dtype: int = KDA_DTYPE_BF16
    out_dtype: int = KDA_DTYPE_BF16
    num_slots: int = 1
    head_dim_v: Optional[int] = None

    def c_struct(self) -> kda_params:
        return kda_params(
            num_heads=self.num_heads, head_dim_k=self.head_dim,
            head_dim_v=self.head_dim if self.head_dim_v is None else self.head_dim_v,
            conv_kernel=self.conv_kernel, gate_mode=self.gate_mode,
            gate_lower_bound=self.gate_lower_bound, l2_eps=self.l2_eps,
            norm_eps=self.norm_eps, scale=self.scale, io_dtype=self.io_dtype,
            out_dtype=self.out_dtype, num_slots=self.num_slots,
            A_log=_ptr(self.A_log), dt_bias=_ptr(self.dt_bias),
            conv_weight=_ptr(self.conv_weight), norm_weight=_ptr(self.norm_weight))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def kda_prefill_workspace_bytes(params: Params, N: int, T: int) -> int:
    return load().kda_prefill_workspace_bytes(ctypes.byref(params.c_struct()), N, T)


def kda_verify_log_bytes(params: Params, B: int, W: int) -> int:
    return load().kda_verify_log_bytes(ctypes.byref(params.c_struct()), B, W)


def kda_prefill_varlen(params: Params, cu_seqlens, N: int, T: int, q, k, v, gate, beta, out_gate,
                       slots, conv_state, rec_state, out, workspace=None, ws_bytes: int = 0,
                       dev_status=None, stream=None) -> int:
    return load().kda_prefill_varlen(
        ctypes.byref(params.c_struct()), _ptr(cu_seqlens), N, T, _ptr(q), _ptr(k), _ptr(v), _ptr(gate),
        _ptr(beta), _ptr(out_gate), _ptr(slots), _ptr(conv_state), _ptr(rec_state), _ptr(out),
        _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream))


def kda_prefill_varlen_static_ws(params: Params, cu_seqlens, N: int, T: int, q, k, v, gate, beta, out_gate,
                                 slots, conv_state, rec_state, out, dev_status=None, stream=None) -> int:
    """kda_prefill_varlen with the library's built-in scratch instead of a
    caller workspace (for callers that cannot allocate device memory)."""
    return load().kda_prefill_varlen_static_ws(
        ctypes.byref(params.c_struct()), _ptr(cu_seqlens), N, T, _ptr(q), _ptr(k), _ptr(v), _ptr(gate),
        _ptr(beta), _ptr(out_gate), _ptr(slots), _ptr(conv_state), _ptr(rec_state), _ptr(out),
        _ptr(dev_status), _stream(stream))


def kda_prefill_scan(params: Params, cu_seqlens, N: int, T: int, q, k, v, gate, beta, out_gate, slots,
                     conv_state, rec_state, out, workspace, ws_bytes: int, segments: int, dev_status=None,
                     stream=None) -> int:
    return load().kda_prefill_scan(
        ctypes.byref(params.c_struct()), _ptr(cu_seqlens), N, T, _ptr(q), _ptr(k), _ptr(v), _ptr(gate),
        _ptr(beta), _ptr(out_gate), _ptr(slots), _ptr(conv_state), _ptr(rec_state), _ptr(out),
        _ptr(workspace), ws_bytes, segments, _ptr(dev_status), _stream(stream))


def kda_prefill_scan_workspace_bytes(params: Params, N: int, T: int, segments: int) -> int:
    return load().kda_prefill_scan_workspace_bytes(ctypes.byref(params.c_struct()), N, T, segments)


def kda_debug_split_chains_only(params: Params, cu_seqlens, N: int, T: int, q, k, v, gate, beta, out_gate,
                                slots, conv_state, rec_state, out, workspace, ws_bytes: int, dev_status,
                                poll_limit: int, stream=None) -> int:
    """Test hook: the split path's chains without producers, flag waits
    limited to poll_limit polls (they run out and report KDA_DEV_TIMEOUT)."""
    return load().kda_debug_split_chains_only(
        ctypes.byref(params.c_struct()), _ptr(cu_seqlens), N, T, _ptr(q), _ptr(k), _ptr(v), _ptr(gate),
        _ptr(beta), _ptr(out_gate), _ptr(slots), _ptr(conv_state), _ptr(rec_state), _ptr(out),
        _ptr(workspace), ws_bytes, _ptr(dev_status), poll_limit, _stream(stream))


def kda_debug_activations(which: int, x, y, n: int, stream=None) -> int:
    """Test hook: y[i] = f(x[i]) with the kernels' shared activation f
    (KDA_ACT_EXP, KDA_ACT_RCP, KDA_ACT_SIGMOID, KDA_ACT_SILU)."""
    return load().kda_debug_activations(which, _ptr(x), _ptr(y), n, _stream(stream))


def kda_prefill_static_workspace_capacity() -> int:
    return load().kda_prefill_static_workspace_capacity()


def kda_decode(params: Params, B: int, q, k, v, gate, beta, out_gate, slots, conv_state, rec_state,
               out, dev_status=None, stream=None) -> int:
    return load().kda_decode(
        ctypes.byref(params.c_struct()), B, _ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(beta),
        _ptr(out_gate), _ptr(slots), _ptr(conv_state), _ptr(rec_state), _ptr(out), _ptr(dev_status),
        _stream(stream))


def kda_verify_window(params: Params, B: int, W: int, q, k, v, gate, beta, out_gate, slots,
                      conv_state, rec_state, log, out, dev_status=None, stream=None) -> int:
    return load().kda_verify_window(
        ctypes.byref(params.c_struct()), B, W, _ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(beta),
        _ptr(out_gate), _ptr(slots), _ptr(conv_state), _ptr(rec_state), _ptr(log), _ptr(out),
        _ptr(dev_status), _stream(stream))


def kda_commit(params: Params, B: int, W: int, accepted, slots, log, conv_state, rec_state,
               dev_status=None, stream=None) -> int:
    return load().kda_commit(
        ctypes.byref(params.c_struct()), B, W, _ptr(accepted), _ptr(slots), _ptr(log),
        _ptr(conv_state), _ptr(rec_state), _ptr(dev_status), _stream(stream))


def kda_commit_verify(params: Params, B: int, W: int, accepted, log_prev, q, k, v, gate, beta, out_gate,
                      slots, conv_state, rec_state, log, out, dev_status=None, stream=None) -> int:
    """Commit the previous window's accepted rows, then verify a new window."""
    return load().kda_commit_verify(
        ctypes.byref(params.c_struct()), B, W, _ptr(accepted), _ptr(log_prev), _ptr(q), _ptr(k), _ptr(v),
        _ptr(gate), _ptr(beta), _ptr(out_gate), _ptr(slots), _ptr(conv_state), _ptr(rec_state), _ptr(log),
        _ptr(out), _ptr(dev_status), _stream(stream))


class Prepared:
    """A call of one entry point with its arguments marshalled once.

    ``Prepared("kda_decode", params, B, q, ...)()`` calls the C function with
    the same pointers every time (the tensors must stay alive and in place).
    """

    def __init__(self, name: str, params: Params, *args, stream=None):
        self.fn = getattr(load(), name)
        self.pstruct = params.c_struct()
        conv = []
        for a in args:
            if a is None or isinstance(a, int):
                conv.append(a)
            else:
                conv.append(a.data_ptr())
        self.args = (ctypes.byref(self.pstruct), *conv, _stream(stream))

    def __call__(self) -> int:
        return self.fn(*self.args)
