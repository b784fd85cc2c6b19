"""Device buffers for one workload, and calls of the four entry points on them.

A thin convenience over the binding: torch allocates device memory, the
binding passes pointers to the CUDA library.  Used by the tests, the
benchmark and the smoke check.

Every buffer the library writes (outputs, conv and recurrent states, the
verify log, the prefill workspace) sits inside a larger allocation between
two guard regions of GUARD_BYTES filled with the byte SENTINEL; a write past
either end shows up as a changed guard byte (``DeviceCase.guards_intact``).
"""
from __future__ import annotations

import weakref

import torch

from . import kda as K
from . import workloads as W


GUARD_BYTES = 4096
SENTINEL = 0xA5

# every live DeviceCase, so a test harness can check all guards after a test
LIVE = weakref.WeakSet()


class Guarded:
    """A device tensor of `shape` and `dtype` with GUARD_BYTES of SENTINEL
    bytes before and after it (the tensor starts 4 KiB into the allocation,
    so it keeps the allocation's alignment)."""

    def __init__(self, shape, dtype, device):
        n = 1
        for x in shape:
            n *= int(x)
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        self.nbytes = nbytes
        self.raw = torch.full((2 * GUARD_BYTES + (nbytes + 15) // 16 * 16,), SENTINEL, dtype=torch.uint8,
                              device=device)
        self.tensor = self.raw[GUARD_BYTES:GUARD_BYTES + nbytes].view(dtype).view(tuple(shape))

    def intact(self) -> bool:
        head = self.raw[:GUARD_BYTES]
        tail = self.raw[GUARD_BYTES + self.nbytes:]
        return bool((head == SENTINEL).all().item()) and bool((tail == SENTINEL).all().item())


def io_code(dtype: str) -> int:
    return K.KDA_DTYPE_BF16 if dtype == W.BF16 else K.KDA_DTYPE_F32


class DeviceCase:
    """All tensors of a workload on one device.

    out_dtype: "f32" or "bf16" (the layer's output storage type).
    num_slots: state-pool size (defaults to one slot per sequence).
    """

    def __init__(self, wl: W.Workload, device="cuda", out_dtype: str = W.F32,
                 num_slots: int | None = None, slots=None):
        self.wl = wl
        self.device = torch.device(device)
        self.out_dtype = out_dtype
        t = lambda nm: wl.to_torch(nm, self.device)  # noqa: E731
        self.q, self.k, self.v, self.f, self.b = t("q"), t("k"), t("v"), t("f"), t("b")
        self.g = t("g") if wl.has_out_gate else None
        self.A_log, self.dt_bias, self.conv_w = t("A_log"), t("dt_bias"), t("conv_w")
        self.norm_w = t("norm_w")
        self.conv_state0 = t("conv_state")
        self.rec_state0 = t("rec_state")
        self.num_slots = num_slots or wl.N
        self.slots = None if slots is None else torch.as_tensor(slots, dtype=torch.int32, device=self.device)
        if slots is not None:
            # a state pool: sequence b lives in slot slots[b] (negative: skipped)
            cs = torch.zeros((self.num_slots,) + tuple(self.conv_state0.shape[1:]),
                             dtype=self.conv_state0.dtype, device=self.device)
            rs = torch.zeros((self.num_slots,) + tuple(self.rec_state0.shape[1:]),
                             dtype=torch.float32, device=self.device)
            for bi, sl in enumerate(list(slots)):
                if 0 <= sl < self.num_slots:
                    cs[sl] = self.conv_state0[bi]
                    rs[sl] = self.rec_state0[bi]
            self.conv_state0, self.rec_state0 = cs, rs
        self.cu_seqlens = torch.from_numpy(wl.cu_seqlens).to(self.device)
        self.accepted = t("accepted") if "accepted" in wl.arrays else None
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self._guards = []
        self.conv_state = self._guarded(self.conv_state0.shape, self.conv_state0.dtype)
        self.rec_state = self._guarded(self.rec_state0.shape, self.rec_state0.dtype)
        self.reset_states()
        odt = torch.bfloat16 if out_dtype == W.BF16 else torch.float32
        self.out = self._guarded((max(wl.T, 1), wl.H, wl.dv), odt)
        LIVE.add(self)

    def _guarded(self, shape, dtype):
        g = Guarded(shape, dtype, self.device)
        self._guards.append(g)
        return g.tensor

    def guards_intact(self) -> bool:
        """True when no guard byte around any library-written buffer changed."""
        return all(g.intact() for g in self._guards)

    def params(self) -> K.Params:
        wl = self.wl
        return K.Params(num_heads=wl.H, head_dim=wl.dk, conv_kernel=wl.K, gate_mode=wl.gate_mode,
                        A_log=self.A_log, dt_bias=self.dt_bias, conv_weight=self.conv_w,
                        norm_weight=self.norm_w, gate_lower_bound=wl.lower_bound,
                        l2_eps=wl.l2_eps, norm_eps=wl.norm_eps, scale=wl.scale,
                        io_dtype=io_code(wl.io_dtype), out_dtype=io_code(self.out_dtype),
                        num_slots=self.num_slots)

    def reset_states(self):
        self.conv_state.copy_(self.conv_state0)
        self.rec_state.copy_(self.rec_state0)

    # -------------------------------------------------------- entry points
    def prefill(self, stream=None) -> int:
        wl = self.wl
        p = self.params()
        need = K.kda_prefill_workspace_bytes(p, wl.N, wl.T)
        if need and (getattr(self, "workspace", None) is None or self.workspace.numel() < need):
            self.workspace = self._guarded((need,), torch.uint8)
        ws = self.workspace if need else None
        return K.kda_prefill_varlen(p, self.cu_seqlens, wl.N, wl.T, self.q, self.k, self.v, self.f,
                                    self.b, self.g, self.slots, self.conv_state, self.rec_state,
                                    self.out, ws, need, self.dev_status, stream)

    def decode(self, rows=None, stream=None) -> int:
        """One decode row per sequence; rows selects the row tensors'
        slice (default: the workload's own B rows)."""
        sl = slice(None) if rows is None else rows
        q, k, v, f, b = self.q[sl], self.k[sl], self.v[sl], self.f[sl], self.b[sl]
        g = None if self.g is None else self.g[sl]
        B = q.shape[0]
        out = self.out[:B] if rows is None else self._guarded(self.out[:B].shape, self.out.dtype)
        rc = K.kda_decode(self.params(), B, q.contiguous(), k.contiguous(), v.contiguous(), f.contiguous(),
                          b.contiguous(), None if g is None else g.contiguous(), self.slots,
                          self.conv_state, self.rec_state, out, self.dev_status, stream)
        self.last_out = out
        return rc

    def alloc_log(self):
        wl = self.wl
        n = K.kda_verify_log_bytes(self.params(), wl.N, wl.W)
        self.log = self._guarded((max(n, 16),), torch.uint8)
        return self.log

    def verify(self, stream=None) -> int:
        wl = self.wl
        if getattr(self, "log", None) is None:
            self.alloc_log()
        return K.kda_verify_window(self.params(), wl.N, wl.W, self.q, self.k, self.v, self.f, self.b,
                                   self.g, self.slots, self.conv_state, self.rec_state, self.log,
                                   self.out, self.dev_status, stream)

    def commit(self, accepted=None, stream=None) -> int:
        wl = self.wl
        acc = self.accepted if accepted is None else accepted
        return K.kda_commit(self.params(), wl.N, wl.W, acc, self.slots, self.log, self.conv_state,
                            self.rec_state, self.dev_status, stream)
