"""fp64 CPU oracle for the KDA layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library and its Python
binding never do.  The arithmetic lives in ``kda_oracle.c`` (plain C, fp64,
no fast-math); this module compiles it with gcc, loads it with ctypes and runs
independent (sequence, head) units on a thread pool (ctypes drops the GIL
during the call).

Parity status: pinned by the CPU tests, except the two gate formulas, whose
choice the pages leave open ("parity unpinned", see the header of
``kda_oracle.c``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_OUT = os.path.join(_HERE, "_build", "libkda_oracle.so")
_lock = threading.Lock()
_lib = None


class Cfg(ctypes.Structure):
    _fields_ = [
        ("H", ctypes.c_int32), ("dk", ctypes.c_int32), ("dv", ctypes.c_int32),
        ("K", ctypes.c_int32), ("gate_mode", ctypes.c_int32),
        ("has_out_gate", ctypes.c_int32), ("chunk", ctypes.c_int32),
        ("reserved", ctypes.c_int32), ("lower_bound", ctypes.c_double),
        ("l2_eps", ctypes.c_double), ("norm_eps", ctypes.c_double),
        ("scale", ctypes.c_double),
    ]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math); returns the .so path."""
    if force or not os.path.exists(_OUT) or os.path.getmtime(_OUT) < os.path.getmtime(_SRC):
        os.makedirs(os.path.dirname(_OUT), exist_ok=True)
        tmp = _OUT + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c11",
                               "-fno-fast-math", "-ffp-contract=off",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _OUT)
    return _OUT


_D = ctypes.POINTER(ctypes.c_double)
_I = ctypes.POINTER(ctypes.c_int32)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            L.kda_ref_sigmoid.restype = ctypes.c_double
            L.kda_ref_sigmoid.argtypes = [ctypes.c_double]
            L.kda_ref_silu.restype = ctypes.c_double
            L.kda_ref_silu.argtypes = [ctypes.c_double]
            L.kda_ref_softplus.restype = ctypes.c_double
            L.kda_ref_softplus.argtypes = [ctypes.c_double]
            L.kda_ref_log_alpha.restype = ctypes.c_double
            L.kda_ref_log_alpha.argtypes = [ctypes.c_int32, ctypes.c_double, ctypes.c_double,
                                            ctypes.c_double, ctypes.c_double]
            L.kda_ref_l2norm.restype = None
            L.kda_ref_l2norm.argtypes = [ctypes.c_int32, _D, ctypes.c_double, _D]
            L.kda_ref_gated_rmsnorm.restype = None
            L.kda_ref_gated_rmsnorm.argtypes = [ctypes.c_int32, _D, _D, _D, ctypes.c_double, _D]
            L.kda_ref_conv1d.restype = None
            L.kda_ref_conv1d.argtypes = [ctypes.c_int32] * 3 + [_D] * 4
            L.kda_ref_conv_history.restype = None
            L.kda_ref_conv_history.argtypes = [ctypes.c_int32] * 3 + [_D] * 3
            L.kda_ref_delta_step.restype = None
            L.kda_ref_delta_step.argtypes = [ctypes.c_int32, ctypes.c_int32, _D, _D, ctypes.c_double,
                                             _D, _D, _D, ctypes.c_double, _D, _D]
            L.kda_ref_forward.restype = ctypes.c_int
            L.kda_ref_forward.argtypes = ([ctypes.POINTER(Cfg), ctypes.c_int32, _I] + [_D] * 13
                                          + [ctypes.c_int32, ctypes.c_int32])
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(_D)


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


# ----------------------------------------------------------- step functions

def sigmoid(x): return lib().kda_ref_sigmoid(float(x))
def silu(x): return lib().kda_ref_silu(float(x))
def softplus(x): return lib().kda_ref_softplus(float(x))


def log_alpha(gate_mode, lower_bound, A_log_h, f, dt_bias):
    return lib().kda_ref_log_alpha(int(gate_mode), float(lower_bound), float(A_log_h),
                                   float(f), float(dt_bias))


def l2norm(x, eps):
    x = _f64(x)
    y = np.empty_like(x)
    lib().kda_ref_l2norm(x.size, _p(x), float(eps), _p(y))
    return y


def gated_rmsnorm(o, g, w, eps):
    o, g, w = _f64(o), _f64(g), _f64(w)
    y = np.empty_like(o)
    lib().kda_ref_gated_rmsnorm(o.size, _p(o), _p(g), _p(w), float(eps), _p(y))
    return y


def conv1d(x, hist, w):
    """x [T, C], hist [K-1, C], w [C, K] -> pre-activation [T, C]."""
    x, hist, w = _f64(x), _f64(hist), _f64(w)
    T, C = x.shape
    K = w.shape[1]
    y = np.empty((T, C))
    if hist.size == 0:
        hist = np.zeros((1, C))
    lib().kda_ref_conv1d(T, C, K, _p(x), _p(hist), _p(w), _p(y))
    return y


def conv_history(x, hist, K):
    x, hist = _f64(x), _f64(hist)
    T, C = x.shape
    out = np.empty((max(K - 1, 1), C))
    lib().kda_ref_conv_history(T, C, K, _p(x), _p(hist), _p(out))
    return out[:K - 1]


def delta_step(S, alpha, beta, k, v, q, scale=1.0):
    """One token; returns (new S, o, u).  S is [dk, dv]."""
    S = _f64(S).copy()
    alpha, k, v, q = _f64(alpha), _f64(k), _f64(v), _f64(q)
    dk, dv = S.shape
    o = np.empty(dv)
    u = np.empty(dv)
    lib().kda_ref_delta_step(dk, dv, _p(S), _p(alpha), float(beta), _p(k), _p(v), _p(q),
                             float(scale), _p(o), _p(u))
    return S, o, u


# ----------------------------------------------------------- full layer

def forward(wl, chunk: int = 0, threads: int = 0, units=None, arrays=None):
    """Run the layer on a workload (see ``workloads.Workload``).

    Returns dict(out [T,H,dv], conv_state [N,K-1,conv_dim], rec_state
    [N,H,dk,dv]) in float64.  chunk=0: serial recurrence; chunk=C: the
    chunked form.  units: optional iterable of (seq, head) to compute (others
    are left as zeros in ``out`` and untouched in the states).
    """
    a = arrays if arrays is not None else wl.arrays
    cfg = Cfg(H=wl.H, dk=wl.dk, dv=wl.dv, K=wl.K, gate_mode=int(wl.gate_mode),
              has_out_gate=int(wl.has_out_gate), chunk=int(chunk), reserved=0,
              lower_bound=float(wl.lower_bound), l2_eps=float(wl.l2_eps),
              norm_eps=float(wl.norm_eps), scale=float(wl.scale))
    cu = np.ascontiguousarray(wl.cu_seqlens, dtype=np.int32)
    ins = {nm: _f64(a[nm]) for nm in ("q", "k", "v", "f", "b", "A_log", "dt_bias", "conv_w")}
    g = _f64(a["g"]) if wl.has_out_gate else None
    norm_w = _f64(a.get("norm_w"))
    conv_state = _f64(a["conv_state"]).copy()
    S = _f64(a["rec_state"]).copy()
    out = np.zeros((wl.T, wl.H, wl.dv))
    N, H = wl.N, wl.H
    if units is None:
        ulist = list(range(N * H))
    else:
        ulist = sorted(s * H + h for s, h in units)
    L = lib()

    def run(u):
        rc = L.kda_ref_forward(ctypes.byref(cfg), N, cu.ctypes.data_as(_I),
                               _p(ins["q"]), _p(ins["k"]), _p(ins["v"]), _p(ins["f"]),
                               _p(ins["b"]), _p(g), _p(ins["A_log"]), _p(ins["dt_bias"]),
                               _p(ins["conv_w"]), _p(norm_w), _p(conv_state), _p(S), _p(out),
                               u, u + 1)
        if rc != 0:
            raise ValueError("oracle rejected its arguments")

    nthreads = threads or (os.cpu_count() or 1)
    if nthreads <= 1 or len(ulist) <= 1:
        for u in ulist:
            run(u)
    else:
        with ThreadPoolExecutor(max_workers=nthreads) as ex:
            list(ex.map(run, ulist))
    return {"out": out, "conv_state": conv_state, "rec_state": S}
