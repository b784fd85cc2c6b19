"""Decode rows on the GPU against the fp64 oracle."""
import numpy as np
import pytest
import torch

from linear_attention_serving_kda_gb300 import workloads as W
from linear_attention_serving_kda_gb300.runtime import DeviceCase
from tests.parity import assert_bf16_within_one_ulp, assert_close, to_np

pytestmark = pytest.mark.gpu


def _run_decode(kda, wl, out_dtype=W.F32, **kw):
    dc = DeviceCase(wl, out_dtype=out_dtype, **kw)
    kda.check(dc.decode())
    torch.cuda.synchronize()
    return dc


def test_decode_full_size_matches_oracle(cuda_lib, oracle_mod):
    """64 sequences x 1 row, H=32, dk=dv=128, bf16 rows, softplus gate, gated
    RMSNorm epilogue; every output, state and conv state checked."""
    wl = W.decode_case()
    ref = oracle_mod.forward(wl)
    dc = _run_decode(cuda_lib, wl)
    assert int(dc.dev_status.item()) == 0
    assert_close(to_np(dc.out), ref["out"], "out")
    assert_close(to_np(dc.rec_state), ref["rec_state"], "rec_state")
    assert np.array_equal(to_np(dc.conv_state), ref["conv_state"].astype(np.float32))
    dcb = _run_decode(cuda_lib, wl, out_dtype=W.BF16)
    assert_bf16_within_one_ulp(to_np(dcb.out), ref["out"])


CASES = [
    # d, io, gate, K, out_gate, B
    (32, W.F32, W.SAFE, 4, False, 3),
    (32, W.BF16, W.SOFTPLUS, 2, True, 5),
    (64, W.F32, W.SOFTPLUS, 3, True, 2),
    (64, W.BF16, W.SAFE, 4, False, 7),
    (128, W.F32, W.SAFE, 2, True, 1),
    (128, W.BF16, W.SOFTPLUS, 3, False, 9),
]


@pytest.mark.parametrize("d,io,gate,K,og,B", CASES)
def test_decode_shapes(cuda_lib, oracle_mod, d, io, gate, K, og, B):
    wl = W.make_workload(f"dec{d}", 40 + d + B, [1] * B, H=3, d=d, K=K, io_dtype=io,
                         gate_mode=gate, lower_bound=-4.0, out_gate=og, init_state="random")
    ref = oracle_mod.forward(wl)
    dc = _run_decode(cuda_lib, wl)
    assert_close(to_np(dc.out), ref["out"], "out")
    assert_close(to_np(dc.rec_state), ref["rec_state"], "rec_state")
    assert np.array_equal(to_np(dc.conv_state), ref["conv_state"].astype(np.float32))


def test_decode_repeated_steps_carry_state(cuda_lib, oracle_mod):
    """Eight decode calls in a row equal the oracle over the eight rows."""
    B, steps = 4, 8
    wl = W.make_workload("multi", 77, [steps] * B, H=2, d=64, K=4, io_dtype=W.BF16,
                         gate_mode=W.SAFE, out_gate=True, init_state="random")
    ref = oracle_mod.forward(wl)
    dc = DeviceCase(wl)
    outs = []
    for r in range(steps):
        idx = torch.arange(B, device="cuda") * steps + r
        cuda_lib.check(dc.decode(rows=idx))
        outs.append(dc.last_out.clone())
    torch.cuda.synchronize()
    got = torch.stack(outs, 1).reshape(B * steps, 2, 64)
    assert_close(to_np(got), ref["out"], "out")
    assert_close(to_np(dc.rec_state), ref["rec_state"], "rec_state")
    assert np.array_equal(to_np(dc.conv_state), ref["conv_state"].astype(np.float32))


def test_decode_slots_and_negative_skip(cuda_lib, oracle_mod):
    """slots map sequences into a larger pool; a negative slot skips its
    sequence (no output written, no state touched)."""
    wl = W.make_workload("slots", 78, [1] * 3, H=2, d=32, K=4, io_dtype=W.F32,
                         gate_mode=W.SOFTPLUS, out_gate=False, init_state="random")
    ref = oracle_mod.forward(wl)
    dc = DeviceCase(wl, num_slots=6, slots=[4, -1, 1])
    rs0, cs0 = dc.rec_state.clone(), dc.conv_state.clone()
    dc.out.fill_(float("nan"))
    cuda_lib.check(dc.decode())
    torch.cuda.synchronize()
    out = to_np(dc.out)
    assert np.all(np.isnan(out[1]))
    for b, sl in ((0, 4), (2, 1)):
        assert_close(out[b], ref["out"][b], "out")
        assert_close(to_np(dc.rec_state[sl]), ref["rec_state"][b], "rec_state")
        assert np.array_equal(to_np(dc.conv_state[sl]), ref["conv_state"][b].astype(np.float32))
    for sl in (0, 2, 3, 5):
        assert torch.equal(dc.rec_state[sl], rs0[sl]) and torch.equal(dc.conv_state[sl], cs0[sl])


def test_decode_bad_slot_sets_status(cuda_lib):
    wl = W.make_workload("bad", 79, [1] * 2, H=2, d=32, K=4, io_dtype=W.F32,
                         gate_mode=W.SOFTPLUS, init_state="random")
    dc = DeviceCase(wl, num_slots=2, slots=[0, 7])
    rs0 = dc.rec_state.clone()
    cuda_lib.check(dc.decode())
    torch.cuda.synchronize()
    assert int(dc.dev_status.item()) & cuda_lib.KDA_DEV_BAD_SLOT
    assert torch.equal(dc.rec_state[1], rs0[1])
