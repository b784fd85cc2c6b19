"""The split (producer / chain) prefill path for few long chains.

With N * H <= 64 and T >= 1024 rows, kda_prefill_varlen runs one persistent
grid in which producer CTAs compute each chunk's state-independent operands
and chain CTAs apply them in order.  Both run the fused kernel's steps on
the same values (the producers publish the bf16 tiles the fused kernel builds,
and the chain runs its bf16 products), so the results must have the fused
kernel's bits -- the allocation-free entry point always takes the fused
kernel, which gives the reference here -- and stay within the parity
tolerance of the oracle.
"""
import numpy as np
import pytest
import torch

from linear_attention_serving_kda_gb300 import kda as K
from linear_attention_serving_kda_gb300 import workloads as W
from linear_attention_serving_kda_gb300.runtime import DeviceCase
from tests.parity import assert_close, to_np

pytestmark = pytest.mark.gpu


def _fused(dc):
    wl = dc.wl
    return K.kda_prefill_varlen_static_ws(dc.params(), dc.cu_seqlens, wl.N, wl.T, dc.q, dc.k, dc.v, dc.f, dc.b,
                                          dc.g, dc.slots, dc.conv_state, dc.rec_state, dc.out, dc.dev_status)


def _both(wl, out_dtype=W.BF16, **kw):
    p = DeviceCase(wl, out_dtype=out_dtype, **kw)
    assert K.kda_prefill_workspace_bytes(p.params(), wl.N, wl.T) > 2**20, "not the split path"
    p.out.fill_(float("nan"))
    K.check(p.prefill())
    f = DeviceCase(wl, out_dtype=out_dtype, **kw)
    f.out.fill_(float("nan"))
    K.check(_fused(f))
    torch.cuda.synchronize()
    assert int(p.dev_status.item()) == 0 and int(f.dev_status.item()) == 0
    return p, f


CASES = [
    # lens, H, out_gate, init
    ([1500, 700, 0, 1100], 8, True, "random"),
    ([4096], 16, False, "zero"),
    ([1, 63, 1025, 130], 4, True, "random"),
]


def _units_close(oracle_mod, wl, dc, units, what):
    """The oracle on the given (sequence, head) units: all their rows and their
    final states, compared together."""
    ref = oracle_mod.forward(wl, units=units)
    cu = wl.cu_seqlens
    xo, ro, xs, rs = [], [], [], []
    for s_, h in units:
        xo.append(to_np(dc.out[cu[s_]:cu[s_ + 1], h]))
        ro.append(ref["out"][cu[s_]:cu[s_ + 1], h])
        xs.append(to_np(dc.rec_state[s_, h]))
        rs.append(ref["rec_state"][s_, h])
    assert_close(np.concatenate([x.ravel() for x in xo]), np.concatenate([r.ravel() for r in ro]), what + " out")
    assert_close(np.concatenate([x.ravel() for x in xs]), np.concatenate([r.ravel() for r in rs]), what + " state")


@pytest.mark.parametrize("lens,H,og,init", CASES)
def test_split_has_fused_bits_and_oracle_parity(cuda_lib, oracle_mod, lens, H, og, init):
    wl = W.make_workload("split", 800 + sum(lens) + H, lens, H=H, d=128, K=4, io_dtype=W.BF16,
                         gate_mode=W.SAFE, lower_bound=-5.0, out_gate=og, init_state=init)
    p, f = _both(wl, out_dtype=W.F32)
    assert torch.equal(p.out[:wl.T], f.out[:wl.T])
    assert torch.equal(p.rec_state, f.rec_state)
    assert torch.equal(p.conv_state, f.conv_state)
    units = [(s_, h) for s_ in range(wl.N) if lens[s_] > 0 for h in sorted({0, H - 1})]
    _units_close(oracle_mod, wl, p, units, "split vs oracle")


@pytest.mark.parametrize("og", [True, False])
def test_split_bf16_outputs_have_fused_bits(cuda_lib, og):
    """bf16 outputs (the serving case) through the split path's output
    epilogue: the same bits as the fused kernel's output steps, with a short
    last chunk in every sequence."""
    lens, H = [1031, 90, 1700], 4
    wl = W.make_workload("split_b", 812 + int(og), lens, H=H, d=128, K=4, io_dtype=W.BF16, gate_mode=W.SAFE,
                         lower_bound=-5.0, out_gate=og, init_state="random")
    p, f = _both(wl, out_dtype=W.BF16)
    assert torch.equal(p.out[:wl.T], f.out[:wl.T])
    assert torch.equal(p.rec_state, f.rec_state)


def test_split_against_oracle(cuda_lib, oracle_mod):
    """Every (sequence, head) of a small split-path case against the oracle."""
    lens, H = [1100, 200, 77], 2
    wl = W.make_workload("split_o", 811, lens, H=H, d=128, K=3, io_dtype=W.BF16, gate_mode=W.SAFE,
                         lower_bound=-5.0, out_gate=True, init_state="random")
    dc = DeviceCase(wl, out_dtype=W.F32)
    assert K.kda_prefill_workspace_bytes(dc.params(), wl.N, wl.T) > 2**20
    K.check(dc.prefill())
    torch.cuda.synchronize()
    assert int(dc.dev_status.item()) == 0
    ref = oracle_mod.forward(wl)
    assert_close(to_np(dc.out[:wl.T]), ref["out"], "out")
    assert_close(to_np(dc.rec_state), ref["rec_state"], "rec_state")
    assert np.array_equal(to_np(dc.conv_state), ref["conv_state"].astype(np.float32))


def test_split_slots(cuda_lib):
    """A state pool with a skipped sequence: split and fused agree bit for
    bit, and the skipped sequence's slot and rows are untouched."""
    lens = [900, 500, 800]
    wl = W.make_workload("split_s", 812, lens, H=4, d=128, K=4, io_dtype=W.BF16, gate_mode=W.SAFE,
                         lower_bound=-5.0, out_gate=True, init_state="random")
    slots = [2, -1, 0]
    p, f = _both(wl, out_dtype=W.F32, num_slots=4, slots=slots)
    rs0 = DeviceCase(wl, num_slots=4, slots=slots).rec_state
    assert torch.equal(p.rec_state, f.rec_state) and torch.equal(p.conv_state, f.conv_state)
    assert torch.equal(p.rec_state[1], rs0[1]) and torch.equal(p.rec_state[3], rs0[3])
    t0, t1 = 900, 1400
    assert torch.all(torch.isnan(p.out[t0:t1]))
    assert torch.equal(p.out[:t0], f.out[:t0]) and torch.equal(p.out[t1:wl.T], f.out[t1:wl.T])


UNBOUNDED = [
    # lens, H, gate, lower bound, A_log (all heads or None), out_gate
    ([1500, 0, 1100], 4, W.SOFTPLUS, -5.0, None, True),     # mostly whole chunks
    ([1200, 3], 2, W.SOFTPLUS, -5.0, 3.0, False),           # chunks of a few rows, first chunks < 3 rows
    ([1030], 4, W.SAFE, -12.0, 2.0, True),                  # safe gate below -5
]


@pytest.mark.parametrize("lens,H,gate,lb,alog,og", UNBOUNDED)
def test_split_unbounded_gates(cuda_lib, oracle_mod, lens, H, gate, lb, alog, og):
    """Gates with unbounded log-decay on the split path: a pass fixes each
    chain's chunk boundaries by the fused kernel's rule on the same decays,
    so split and fused agree bit for bit, and both match the oracle."""
    wl = W.make_workload("split_u", 820 + sum(lens) + H, lens, H=H, d=128, K=4, io_dtype=W.BF16,
                         gate_mode=gate, lower_bound=lb, out_gate=og, init_state="random")
    if alog is not None:
        wl.arrays["A_log"] = np.full_like(wl.arrays["A_log"], alog)
    p, f = _both(wl, out_dtype=W.F32)
    assert torch.equal(p.out[:wl.T], f.out[:wl.T])
    assert torch.equal(p.rec_state, f.rec_state)
    assert torch.equal(p.conv_state, f.conv_state)
    units = [(s_, h) for s_ in range(wl.N) if lens[s_] > 0 for h in sorted({0, H - 1})]
    _units_close(oracle_mod, wl, p, units, "split vs oracle")


def test_chain_flag_wait_runs_out_and_reports(cuda_lib):
    """A bounded wait that runs out: the split path's chains launched without
    the producers that would publish their operands (a host-side fault: the
    flag is never set), each flag wait limited to 1024 polls.  Every chain
    gives up, reports KDA_DEV_TIMEOUT and returns with nothing in flight: the
    states are untouched and the same context then runs the normal call with
    the fused kernel's bits."""
    wl = W.make_workload("tmo", 818, [2048], H=4, d=128, K=4, io_dtype=W.BF16, gate_mode=W.SAFE,
                         lower_bound=-5.0, out_gate=True, init_state="random")
    dc = DeviceCase(wl, out_dtype=W.BF16)
    p = dc.params()
    need = K.kda_prefill_workspace_bytes(p, wl.N, wl.T)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    rs0, cs0 = dc.rec_state.clone(), dc.conv_state.clone()
    rc = K.kda_debug_split_chains_only(p, dc.cu_seqlens, wl.N, wl.T, dc.q, dc.k, dc.v, dc.f, dc.b, dc.g, None,
                                       dc.conv_state, dc.rec_state, dc.out, ws, need, dc.dev_status, 1024)
    assert rc == K.KDA_OK
    torch.cuda.synchronize()
    assert int(dc.dev_status.item()) & K.KDA_DEV_TIMEOUT
    assert torch.equal(dc.rec_state, rs0) and torch.equal(dc.conv_state, cs0)
    # other shapes are refused before any launch
    assert K.kda_debug_split_chains_only(p, dc.cu_seqlens, wl.N, wl.T, dc.q, dc.k, dc.v, dc.f, dc.b, dc.g, None,
                                         dc.conv_state, dc.rec_state, dc.out, ws, need, dc.dev_status,
                                         0) == K.KDA_ERR_INVALID_ARGUMENT
    # the context is still usable: the normal call gives the fused kernel's bits
    pp, ff = _both(wl)
    assert torch.equal(pp.out[:wl.T], ff.out[:wl.T]) and torch.equal(pp.rec_state, ff.rec_state)
