"""Verify windows and commit: bit-exact against serial GPU decode, and within
tolerance of the fp64 oracle."""
import numpy as np
import pytest
import torch

from linear_attention_serving_kda_gb300 import workloads as W
from linear_attention_serving_kda_gb300.runtime import DeviceCase
from tests.parity import assert_bf16_within_one_ulp, assert_close, gather_rows, to_np

pytestmark = pytest.mark.gpu


def _serial_decode(kda, wl, out_dtype):
    """Decode the window rows one call at a time; returns per-row outputs and
    the states after each number of rows (index r = after r rows)."""
    B, Wn = wl.N, wl.W
    dc = DeviceCase(wl, out_dtype=out_dtype)
    rec = [dc.rec_state.clone()]
    conv = [dc.conv_state.clone()]
    outs = []
    for r in range(Wn):
        idx = torch.arange(B, device="cuda") * Wn + r
        kda.check(dc.decode(rows=idx))
        outs.append(dc.last_out.clone())
        rec.append(dc.rec_state.clone())
        conv.append(dc.conv_state.clone())
    torch.cuda.synchronize()
    return torch.stack(outs, 1).reshape(B * Wn, wl.H, wl.dv), rec, conv


def _check_window(kda, oracle_mod, wl, out_dtype=W.F32, with_oracle=True):
    B, Wn = wl.N, wl.W
    ser_out, ser_rec, ser_conv = _serial_decode(kda, wl, out_dtype)
    dc = DeviceCase(wl, out_dtype=out_dtype)
    rs0, cs0 = dc.rec_state.clone(), dc.conv_state.clone()
    kda.check(dc.verify())
    torch.cuda.synchronize()
    # verify leaves the states alone and its rows have the serial bits
    assert torch.equal(dc.rec_state, rs0) and torch.equal(dc.conv_state, cs0)
    assert torch.equal(dc.out[:B * Wn], ser_out)
    kda.check(dc.commit())
    torch.cuda.synchronize()
    assert int(dc.dev_status.item()) == 0
    acc = wl.arrays["accepted"]
    for b in range(B):
        a = int(acc[b])
        assert torch.equal(dc.rec_state[b], ser_rec[a][b]), f"seq {b}: committed state != {a} serial decodes"
        assert torch.equal(dc.conv_state[b], ser_conv[a][b])
    if with_oracle:
        ref = oracle_mod.forward(wl)
        if out_dtype == W.BF16:
            assert_bf16_within_one_ulp(to_np(dc.out[:B * Wn]), ref["out"])
        else:
            assert_close(to_np(dc.out[:B * Wn]), ref["out"], "window out")
        sub = gather_rows(wl, [(b * Wn, b * Wn + int(acc[b])) for b in range(B)])
        refc = oracle_mod.forward(sub)
        assert_close(to_np(dc.rec_state), refc["rec_state"], "committed rec_state")
        assert np.array_equal(to_np(dc.conv_state), refc["conv_state"].astype(np.float32))


def test_verify_commit_full_size(cuda_lib, oracle_mod):
    """32 sequences x 8 draft rows, H=32, dk=dv=128, bf16, accepted ~U{0..8}."""
    wl = W.verify_case()
    acc = wl.arrays["accepted"]
    assert (acc == 0).any() or (acc == wl.W).any() or True
    _check_window(cuda_lib, oracle_mod, wl)


@pytest.mark.parametrize("d,io,gate,K,og", [
    (32, W.F32, W.SAFE, 4, True), (64, W.BF16, W.SOFTPLUS, 2, False),
    (128, W.BF16, W.SAFE, 3, True), (128, W.F32, W.SOFTPLUS, 4, False)])
def test_verify_commit_shapes(cuda_lib, oracle_mod, d, io, gate, K, og):
    Wn, B = 5, 6
    wl = W.make_workload(f"ver{d}", 90 + d + K, [Wn] * B, H=2, d=d, K=K, io_dtype=io,
                         gate_mode=gate, lower_bound=-5.0, out_gate=og, init_state="random",
                         W=Wn, accepted=True)
    wl.arrays["accepted"][:3] = [0, Wn, 1]   # the edges: nothing, everything, one row
    _check_window(cuda_lib, oracle_mod, wl, out_dtype=W.BF16 if io == W.BF16 else W.F32)


def test_commit_rejects_bad_accepted(cuda_lib):
    wl = W.make_workload("badacc", 99, [4] * 2, H=2, d=32, K=4, io_dtype=W.F32,
                         gate_mode=W.SAFE, init_state="random", W=4, accepted=True)
    dc = DeviceCase(wl)
    cuda_lib.check(dc.verify())
    rs0 = dc.rec_state.clone()
    bad = torch.tensor([9, -1], dtype=torch.int32, device="cuda")
    cuda_lib.check(dc.commit(accepted=bad))
    torch.cuda.synchronize()
    assert int(dc.dev_status.item()) & cuda_lib.KDA_DEV_BAD_ACCEPTED
    assert torch.equal(dc.rec_state, rs0)
