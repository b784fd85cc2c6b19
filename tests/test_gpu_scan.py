"""The chunk-parallel prefill by an affine state scan (kda_prefill_scan).

Each sequence is cut into segments whose zero-state and transfer runs go in
one launch; a scan gives each segment's start state and a fix-up corrects its
outputs.  The results must match the fp64 oracle's serial recurrence within
the parity tolerance (they are not bit-identical to kda_prefill_varlen: the
summation order differs)."""
import numpy as np
import pytest
import torch

from linear_attention_serving_kda_gb300 import kda as K
from linear_attention_serving_kda_gb300 import workloads as W
from linear_attention_serving_kda_gb300.runtime import DeviceCase
from tests.parity import assert_close, to_np

pytestmark = pytest.mark.gpu


def _scan(dc, segments, out_fill=None):
    wl = dc.wl
    p = dc.params()
    need = K.kda_prefill_scan_workspace_bytes(p, wl.N, wl.T, segments)
    assert need > 0
    ws = dc._guarded((need,), torch.uint8)
    if out_fill is not None:
        dc.out.fill_(out_fill)
    rc = K.kda_prefill_scan(p, dc.cu_seqlens, wl.N, wl.T, dc.q, dc.k, dc.v, dc.f, dc.b, dc.g, dc.slots,
                            dc.conv_state, dc.rec_state, dc.out, ws, need, segments, dc.dev_status)
    K.check(rc)
    torch.cuda.synchronize()
    return dc


def _check(dc, ref, rows=None):
    T = dc.wl.T
    assert int(dc.dev_status.item()) == 0
    assert_close(to_np(dc.out[:T]), ref["out"], "scan out")
    assert_close(to_np(dc.rec_state), ref["rec_state"], "scan rec_state")
    assert np.array_equal(to_np(dc.conv_state), ref["conv_state"].astype(np.float32))


CASES = [
    # lens, segments, gate, lb, K, out_gate, init
    ([1000], 4, W.SAFE, -5.0, 4, True, "random"),
    ([640, 65, 0, 3, 700], 3, W.SAFE, -5.0, 3, False, "random"),
    ([513], 8, W.SAFE, -5.0, 2, True, "zero"),        # more segments than whole chunks: empty pieces
    ([300, 129], 2, W.SOFTPLUS, -5.0, 4, True, "random"),  # data-dependent chunks inside the pieces
    ([256], 1, W.SAFE, -5.0, 4, False, "random"),     # one segment: no transfer runs
    ([2, 1], 5, W.SAFE, -8.0, 4, True, "random"),     # rows shorter than the conv history
]


@pytest.mark.parametrize("lens,segments,gate,lb,K_,og,init", CASES)
def test_scan_matches_oracle(cuda_lib, oracle_mod, lens, segments, gate, lb, K_, og, init):
    wl = W.make_workload("scan", 1200 + sum(lens) + segments, lens, H=3, d=128, K=K_, io_dtype=W.BF16,
                         gate_mode=gate, lower_bound=lb, out_gate=og, init_state=init)
    _check(_scan(DeviceCase(wl), segments), oracle_mod.forward(wl))


def test_scan_agrees_with_the_chunk_path_and_skips_slots(cuda_lib, oracle_mod):
    """Against kda_prefill_varlen on the same rows (to rounding), with a state
    pool: a negative slot skips its sequence (no output rows, no state)."""
    wl = W.make_workload("scanslot", 1300, [700, 90, 400], H=2, d=128, K=4, io_dtype=W.BF16, gate_mode=W.SAFE,
                         lower_bound=-5.0, out_gate=True, init_state="random")
    ref = oracle_mod.forward(wl)
    dc = DeviceCase(wl, num_slots=5, slots=[4, -1, 1])
    rs0 = dc.rec_state.clone()
    _scan(dc, 3, out_fill=float("nan"))
    out = to_np(dc.out)
    assert np.all(np.isnan(out[700:790]))
    assert_close(out[:700], ref["out"][:700], "scan out s0")
    assert_close(out[790:], ref["out"][790:], "scan out s2")
    assert_close(to_np(dc.rec_state[4]), ref["rec_state"][0], "scan state s0")
    assert_close(to_np(dc.rec_state[1]), ref["rec_state"][2], "scan state s2")
    for sl in (0, 2, 3):
        assert torch.equal(dc.rec_state[sl], rs0[sl])
    plain = DeviceCase(wl, num_slots=5, slots=[4, -1, 1])
    K.check(plain.prefill())
    torch.cuda.synchronize()
    assert_close(to_np(dc.out[:700]), to_np(plain.out[:700]), "scan vs chunk path s0")
    assert_close(to_np(dc.rec_state), to_np(plain.rec_state), "scan vs chunk path states")


def test_scan_rejects_before_launch(cuda_lib):
    wl = W.make_workload("scanbad", 5, [64], H=1, d=128, K=4, io_dtype=W.BF16, gate_mode=W.SAFE,
                         lower_bound=-5.0, init_state="zero")
    dc = DeviceCase(wl)
    p = dc.params()
    for seg in (0, 65):
        assert K.kda_prefill_scan(p, dc.cu_seqlens, wl.N, wl.T, dc.q, dc.k, dc.v, dc.f, dc.b, None, None,
                                  dc.conv_state, dc.rec_state, dc.out, dc.out, 1 << 30, seg,
                                  dc.dev_status) == K.KDA_ERR_INVALID_ARGUMENT
    need = K.kda_prefill_scan_workspace_bytes(p, wl.N, wl.T, 2)
    assert K.kda_prefill_scan(p, dc.cu_seqlens, wl.N, wl.T, dc.q, dc.k, dc.v, dc.f, dc.b, None, None,
                              dc.conv_state, dc.rec_state, dc.out, dc.out, need - 16, 2,
                              dc.dev_status) == K.KDA_ERR_WORKSPACE


@pytest.mark.slow
def test_scan_long_prefill_full_size(cuda_lib, oracle_mod):
    """1 sequence of 32768 rows, H=32, dk=dv=128, bf16, gated RMSNorm: four
    segments of 8192 rows, every head against the oracle (whole tensors)."""
    wl = W.long_prefill_case()
    dc = _scan(DeviceCase(wl), 4)
    _check(dc, oracle_mod.forward(wl))


def test_scan_flags_bad_inputs_without_faulting(cuda_lib, oracle_mod):
    """An out-of-range slot and a non-monotone cu_seqlens are flagged in the
    status word and their sequences skipped (no output rows, no state
    written); the other sequences still match the oracle."""
    wl = W.make_workload("scanbad2", 1400, [200, 90, 150], H=2, d=128, K=4, io_dtype=W.BF16, gate_mode=W.SAFE,
                         lower_bound=-5.0, out_gate=False, init_state="random")
    ref = oracle_mod.forward(wl)
    dc = DeviceCase(wl, num_slots=3, slots=[0, 7, 2])  # sequence 1's slot is out of range
    rs0 = dc.rec_state.clone()
    dc.out.fill_(float("nan"))
    p = dc.params()
    need = K.kda_prefill_scan_workspace_bytes(p, wl.N, wl.T, 2)
    ws = dc._guarded((need,), torch.uint8)
    K.check(K.kda_prefill_scan(p, dc.cu_seqlens, wl.N, wl.T, dc.q, dc.k, dc.v, dc.f, dc.b, None, dc.slots,
                               dc.conv_state, dc.rec_state, dc.out, ws, need, 2, dc.dev_status))
    torch.cuda.synchronize()
    assert int(dc.dev_status.item()) & K.KDA_DEV_BAD_SLOT
    out = to_np(dc.out)
    assert np.all(np.isnan(out[200:290]))
    assert torch.equal(dc.rec_state[1], rs0[1])  # no sequence's slot
    assert_close(out[:200], ref["out"][:200], "scan out s0")
    assert_close(out[290:], ref["out"][290:], "scan out s2")
    assert_close(to_np(dc.rec_state[0]), ref["rec_state"][0], "scan state s0")
    assert_close(to_np(dc.rec_state[2]), ref["rec_state"][2], "scan state s2")
    # a non-monotone cu_seqlens: flagged, no fault
    dc2 = DeviceCase(wl)
    dc2.cu_seqlens.copy_(torch.tensor([0, 210, 190, 440], dtype=torch.int32))
    K.check(K.kda_prefill_scan(p, dc2.cu_seqlens, wl.N, wl.T, dc2.q, dc2.k, dc2.v, dc2.f, dc2.b, None, None,
                               dc2.conv_state, dc2.rec_state, dc2.out, ws, need, 2, dc2.dev_status))
    torch.cuda.synchronize()
    assert int(dc2.dev_status.item()) & K.KDA_DEV_BAD_SEQLENS
