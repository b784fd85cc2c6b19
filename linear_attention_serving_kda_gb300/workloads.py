"""Seeded synthetic inputs for the KDA layer.

This module only draws random numbers and encodes them in the storage type
(fp32, or bfloat16 by round-to-nearest-even, the rounding rule of ONNX Runtime
GenAI PR #2898 "Add Ling-3.0-flash-VL export and Engine image inputs",
"Behavioral scope").  It holds none of the layer's arithmetic, so the CUDA
path and the CPU oracle can both take their inputs from it.

Every array is returned twice over: ``a.f32`` holds the stored values as
float32 (exact for both storage types) and the workload remembers the storage
type, so a caller can build a bf16 device tensor with identical bits
(``to_torch``) or widen to float64 for the oracle with no rounding.

Recipe (one ``numpy.random.default_rng(seed)`` per workload, draws in this
order): sequence lengths (varlen workloads only), q, k, v, gate f, beta
logit b, output gate g (when present), A_log ~ U(-1, 1), dt_bias ~ N(0, 0.1),
conv weight ~ N(0, 1/sqrt(K)), conv state ~ N(0, 1), recurrent state
~ N(0, 0.02), accepted lengths ~ U{0..W} (verify only).  Rows are ~ N(0, 1).
"N(0, s)" means standard deviation s throughout.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, Optional

import numpy as np

F32 = "f32"
BF16 = "bf16"
SOFTPLUS = 0
SAFE = 1


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest, ties to even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _encode(x: np.ndarray, dtype: str) -> np.ndarray:
    """Values exactly representable in the storage type, held as float32."""
    x = np.asarray(x, dtype=np.float32)
    if dtype == BF16:
        return bf16_bits_to_f32(round_to_bf16_bits(x))
    return x


@dataclass
class Workload:
    """One seeded problem.  Row tensors are token-major [T, H, d]."""

    name: str
    H: int
    dk: int
    dv: int
    K: int
    io_dtype: str
    gate_mode: int
    lower_bound: float
    has_out_gate: bool
    cu_seqlens: np.ndarray            # int32 [N+1]
    arrays: Dict[str, np.ndarray] = field(default_factory=dict)
    W: int = 1                        # window rows per sequence (verify)
    l2_eps: float = 1e-6
    norm_eps: float = 1e-6
    scale: float = 1.0
    chunk: int = 64

    @property
    def N(self) -> int:
        return int(self.cu_seqlens.shape[0] - 1)

    @property
    def T(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def conv_dim(self) -> int:
        return self.H * (2 * self.dk + self.dv)

    def storage(self, name: str) -> str:
        """Storage type of an array: rows and conv state use the io type."""
        if name in ("q", "k", "v", "f", "b", "g", "conv_state"):
            return self.io_dtype
        return F32

    def to_torch(self, name: str, device="cpu"):
        import torch

        a = self.arrays[name]
        if a.dtype.kind in "iu":
            return torch.from_numpy(np.ascontiguousarray(a)).to(device)
        if self.storage(name) == BF16:
            bits = round_to_bf16_bits(a)  # exact: a already holds bf16 values
            t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
        else:
            t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
        return t.to(device)


def _normal(rng, shape, std=1.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def make_workload(name: str, seed: int, lens, H: int, d: int, K: int = 4,
                  io_dtype: str = BF16, gate_mode: int = SAFE,
                  lower_bound: float = -5.0, out_gate: bool = False,
                  init_state: str = "random", W: int = 1,
                  accepted: bool = False, draw_lens: Optional[tuple] = None,
                  chunk: int = 64) -> Workload:
    """Generic seeded case.

    lens: per-sequence row counts (ignored when ``draw_lens=(n, lo, hi)``
    asks for n lengths drawn from U{lo..hi} with this seed first).
    init_state: "random" (conv ~ N(0,1), recurrent ~ N(0,0.02)) or "zero".
    """
    rng = np.random.default_rng(seed)
    if draw_lens is not None:
        n, lo, hi = draw_lens
        lens = rng.integers(lo, hi + 1, size=n)
    lens = np.asarray(lens, dtype=np.int64)
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    T = int(cu[-1])
    N = len(lens)
    dk = dv = d
    wl = Workload(name=name, H=H, dk=dk, dv=dv, K=K, io_dtype=io_dtype,
                  gate_mode=gate_mode, lower_bound=lower_bound,
                  has_out_gate=out_gate, cu_seqlens=cu, W=W, chunk=chunk)
    a = wl.arrays
    a["q"] = _encode(_normal(rng, (T, H, dk)), io_dtype)
    a["k"] = _encode(_normal(rng, (T, H, dk)), io_dtype)
    a["v"] = _encode(_normal(rng, (T, H, dv)), io_dtype)
    a["f"] = _encode(_normal(rng, (T, H, dk)), io_dtype)
    a["b"] = _encode(_normal(rng, (T, H)), io_dtype)
    if out_gate:
        a["g"] = _encode(_normal(rng, (T, H, dv)), io_dtype)
    a["A_log"] = rng.uniform(-1.0, 1.0, size=(H,)).astype(np.float32)
    a["dt_bias"] = _normal(rng, (H, dk), 0.1)
    a["conv_w"] = _normal(rng, (wl.conv_dim, K), 1.0 / np.sqrt(K))
    a["norm_w"] = np.ones((dv,), dtype=np.float32)
    if init_state == "random":
        a["conv_state"] = _encode(_normal(rng, (N, K - 1, wl.conv_dim)), io_dtype)
        a["rec_state"] = _normal(rng, (N, H, dk, dv), 0.02)
    else:
        a["conv_state"] = np.zeros((N, K - 1, wl.conv_dim), dtype=np.float32)
        a["rec_state"] = np.zeros((N, H, dk, dv), dtype=np.float32)
    if accepted:
        a["accepted"] = rng.integers(0, W + 1, size=(N,)).astype(np.int32)
    return wl


# ---------------------------------------------------------------- the five
# named workloads (sizes and distributions of the serving scenarios).

def tiny_oracle_case() -> Workload:
    """1 sequence, T=64, H=2, dk=dv=32, conv 4, fp32, safe gate lb=-5,
    zero initial states.  Seed 0."""
    return make_workload("tiny_t64_h2_d32_f32", 0, [64], H=2, d=32, K=4,
                         io_dtype=F32, gate_mode=SAFE, lower_bound=-5.0,
                         init_state="zero")


def decode_case(B: int = 64) -> Workload:
    """B sequences x 1 token, H=32, dk=dv=128, conv 4, bf16 rows, softplus
    gate, output gate, carried fp32 state ~N(0,0.02), bf16 conv state.
    Seed 1."""
    return make_workload(f"decode_b{B}_h32_d128_bf16", 1, [1] * B, H=32, d=128,
                         K=4, io_dtype=BF16, gate_mode=SOFTPLUS, out_gate=True,
                         init_state="random")


def varlen_prefill_case() -> Workload:
    """8 sequences, lengths ~U{512..8192}, H=32, dk=dv=128, chunk 64, bf16,
    safe gate lb=-5, random nonzero initial states.  Seed 2."""
    return make_workload("prefill_varlen_n8_h32_d128_bf16", 2, None, H=32,
                         d=128, K=4, io_dtype=BF16, gate_mode=SAFE,
                         lower_bound=-5.0, init_state="random",
                         draw_lens=(8, 512, 8192))


def verify_case() -> Workload:
    """32 sequences x 8 draft rows, H=32, dk=dv=128, bf16, carried random
    state, accepted prefix lengths ~U{0..8}.  Seed 3."""
    return make_workload("verify_b32_w8_h32_d128_bf16", 3, [8] * 32, H=32,
                         d=128, K=4, io_dtype=BF16, gate_mode=SOFTPLUS,
                         init_state="random", W=8, accepted=True)


def long_prefill_case(T: int = 32768) -> Workload:
    """1 sequence of T rows, H=32, dk=dv=128, bf16, output gate, gated
    RMSNorm (eps 1e-6, unit weight), safe gate lb=-5, zero states.  Seed 4."""
    return make_workload(f"prefill_long_t{T}_h32_d128_bf16", 4, [T], H=32,
                         d=128, K=4, io_dtype=BF16, gate_mode=SAFE,
                         lower_bound=-5.0, out_gate=True, init_state="zero")


NAMED = {
    "tiny": tiny_oracle_case,
    "decode": decode_case,
    "prefill_varlen": varlen_prefill_case,
    "verify": verify_case,
    "prefill_long": long_prefill_case,
}


def head_slice(wl: Workload, seq: int, head: int) -> Workload:
    """The sub-problem of one (sequence, head) unit as an H=1, N=1 workload.

    Pure data movement: rows of that sequence and head, that head's conv
    channels (q, k and v parts) of the conv state and conv weight, and that
    head's parameters.  Used to check sampled units of large workloads.
    """
    t0, t1 = int(wl.cu_seqlens[seq]), int(wl.cu_seqlens[seq + 1])
    H, dk, dv = wl.H, wl.dk, wl.dv
    chans = np.concatenate([
        np.arange(head * dk, (head + 1) * dk),
        H * dk + np.arange(head * dk, (head + 1) * dk),
        2 * H * dk + np.arange(head * dv, (head + 1) * dv),
    ])
    sub = Workload(name=f"{wl.name}[s{seq},h{head}]", H=1, dk=dk, dv=dv, K=wl.K,
                   io_dtype=wl.io_dtype, gate_mode=wl.gate_mode,
                   lower_bound=wl.lower_bound, has_out_gate=wl.has_out_gate,
                   cu_seqlens=np.array([0, t1 - t0], dtype=np.int32), W=wl.W,
                   l2_eps=wl.l2_eps, norm_eps=wl.norm_eps, scale=wl.scale,
                   chunk=wl.chunk)
    a, s = wl.arrays, sub.arrays
    for nm in ("q", "k", "v", "f", "g"):
        if nm in a:
            s[nm] = np.ascontiguousarray(a[nm][t0:t1, head:head + 1, :])
    s["b"] = np.ascontiguousarray(a["b"][t0:t1, head:head + 1])
    s["A_log"] = a["A_log"][head:head + 1].copy()
    s["dt_bias"] = a["dt_bias"][head:head + 1].copy()
    s["conv_w"] = np.ascontiguousarray(a["conv_w"][chans])
    s["norm_w"] = a["norm_w"].copy()
    s["conv_state"] = np.ascontiguousarray(a["conv_state"][seq:seq + 1][:, :, chans])
    s["rec_state"] = np.ascontiguousarray(a["rec_state"][seq:seq + 1, head:head + 1])
    if "accepted" in a:
        s["accepted"] = a["accepted"][seq:seq + 1].copy()
    return sub
