"""Serving-loop use of the entry points: CUDA-graph capture with slot
indirection, paused (negative-slot) sequences over many steps, and the
prefill -> decode hand-off of the carried states.

The library enqueues only kernels on the caller's stream and allocates
nothing, so a captured call replays with whatever the captured buffers hold
(rows, slot map, accepted counts) at replay time.
"""
import numpy as np
import pytest
import torch

from linear_attention_serving_kda_gb300 import kda as K
from linear_attention_serving_kda_gb300 import workloads as W
from linear_attention_serving_kda_gb300.runtime import DeviceCase
from tests.parity import assert_close, to_np

pytestmark = pytest.mark.gpu

ROWS = ("q", "k", "v", "f", "b", "g")


def _step_rows(seed, B, H, d, gate, W_rows=1):
    """Seeded rows for one step (B sequences x W_rows rows)."""
    return make_rows(seed, [W_rows] * B, H, d, gate)


def make_rows(seed, lens, H, d, gate):
    return W.make_workload("rows", seed, lens, H=H, d=d, K=4, io_dtype=W.BF16, gate_mode=gate,
                           out_gate=True, init_state="zero")


def _load_rows(dc, rows_wl):
    for nm in ROWS:
        getattr(dc, nm).copy_(rows_wl.to_torch(nm, "cuda"))


def _pair(wl, **kw):
    """Two device cases with identical contents (eager and captured)."""
    return DeviceCase(wl, out_dtype=W.BF16, **kw), DeviceCase(wl, out_dtype=W.BF16, **kw)


def test_graph_decode_with_slot_map(cuda_lib):
    """A captured decode replayed over changing rows and slot maps gives the
    bits of eager calls; paused sequences leave their slots untouched."""
    B, H, d, NS = 8, 4, 128, 12
    wl = W.make_workload("gdec", 601, [1] * B, H=H, d=d, K=4, io_dtype=W.BF16,
                         gate_mode=W.SOFTPLUS, out_gate=True, init_state="random")
    slots = [5, 1, 0, 11, 3, 9, 7, 2]
    ea, gr = _pair(wl, num_slots=NS, slots=slots)
    for dc in (ea, gr):  # first calls outside capture (one-time function set-up)
        K.check(dc.decode())
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        K.check(gr.decode())
    torch.cuda.synchronize()
    for step in range(4):
        rows = _step_rows(700 + step, B, H, d, W.SOFTPLUS)
        cur = [s if (b + step) % 3 else -1 for b, s in enumerate(slots)]  # some sequences paused
        for dc in (ea, gr):
            _load_rows(dc, rows)
            dc.slots.copy_(torch.tensor(cur, dtype=torch.int32))
        rs0 = gr.rec_state.clone()
        K.check(ea.decode())
        graph.replay()
        torch.cuda.synchronize()
        assert int(gr.dev_status.item()) == 0 and int(ea.dev_status.item()) == 0
        assert torch.equal(gr.rec_state, ea.rec_state)
        assert torch.equal(gr.conv_state, ea.conv_state)
        live = [b for b in range(B) if cur[b] >= 0]
        assert torch.equal(gr.out[live], ea.out[live])
        for b in range(B):
            if cur[b] < 0:
                assert torch.equal(gr.rec_state[slots[b]], rs0[slots[b]])


def test_graph_verify_commit(cuda_lib):
    """Verify and commit captured in one graph, replayed with new drafts and
    new accepted counts, match eager calls bit for bit."""
    B, Wn, H, d = 6, 8, 4, 128
    wl = W.make_workload("gver", 602, [Wn] * B, H=H, d=d, K=4, io_dtype=W.BF16,
                         gate_mode=W.SOFTPLUS, out_gate=True, init_state="random", W=Wn,
                         accepted=True)
    ea, gr = _pair(wl)
    for dc in (ea, gr):
        dc.alloc_log()
        K.check(dc.verify())
        K.check(dc.commit())
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        K.check(gr.verify())
        K.check(gr.commit())
    torch.cuda.synchronize()
    rng = np.random.default_rng(603)
    for step in range(3):
        rows = _step_rows(710 + step, B, H, d, W.SOFTPLUS, W_rows=Wn)
        acc = torch.tensor(rng.integers(0, Wn + 1, size=B), dtype=torch.int32)
        for dc in (ea, gr):
            _load_rows(dc, rows)
            dc.accepted.copy_(acc)
        K.check(ea.verify())
        K.check(ea.commit())
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(gr.out[:B * Wn], ea.out[:B * Wn])
        assert torch.equal(gr.rec_state, ea.rec_state)
        assert torch.equal(gr.conv_state, ea.conv_state)


PREFILL_GRAPH = [
    # lens, H, gate, A_log (all heads or None): fused / split path, bounded / unbounded gates
    ([130, 70, 1], 2, W.SAFE, None),
    ([200, 9], 2, W.SOFTPLUS, 3.0),
    ([1100, 300], 2, W.SAFE, None),
    ([1100, 300], 2, W.SOFTPLUS, 3.0),
]


@pytest.mark.parametrize("lens,H,gate,alog", PREFILL_GRAPH)
def test_graph_prefill(cuda_lib, lens, H, gate, alog):
    """A captured prefill (fused or split path; for unbounded gates with the
    chunk-boundary kernels in the graph) replayed over new rows and reset
    states gives the bits of eager calls."""
    d = 128
    wl = W.make_workload("gpre", 604, lens, H=H, d=d, K=4, io_dtype=W.BF16, gate_mode=gate,
                         lower_bound=-5.0, out_gate=True, init_state="random")
    if alog is not None:
        wl.arrays["A_log"] = np.full_like(wl.arrays["A_log"], alog)
    ea, gr = _pair(wl)
    for dc in (ea, gr):  # first calls outside capture (one-time set-up, workspace)
        K.check(dc.prefill())
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        K.check(gr.prefill())
    torch.cuda.synchronize()
    for step in range(2):
        rows = make_rows(720 + step, lens, H, d, gate)
        for dc in (ea, gr):  # new rows, initial states back in place (the graph holds the buffers)
            _load_rows(dc, rows)
            dc.conv_state.copy_(dc.conv_state0)
            dc.rec_state.copy_(dc.rec_state0)
        K.check(ea.prefill())
        graph.replay()
        torch.cuda.synchronize()
        assert int(gr.dev_status.item()) == 0 and int(ea.dev_status.item()) == 0
        assert torch.equal(gr.out[:wl.T], ea.out[:wl.T])
        assert torch.equal(gr.rec_state, ea.rec_state)
        assert torch.equal(gr.conv_state, ea.conv_state)


def test_serving_loop_against_oracle(cuda_lib, oracle_mod):
    """Six decode steps with sequences paused and resumed (negative slots):
    every slot ends where the oracle puts its sequence after the rows it
    actually took, and every live output matches the oracle's row."""
    B, H, d, NS, steps = 6, 3, 128, 9, 6
    base = W.make_workload("loop", 604, [1] * B, H=H, d=d, K=4, io_dtype=W.BF16,
                           gate_mode=W.SOFTPLUS, out_gate=True, init_state="random")
    slots = [4, 0, 8, 2, 6, 1]
    dc = DeviceCase(base, out_dtype=W.F32, num_slots=NS, slots=slots)
    live = np.array([[(b * 7 + t * 3) % 4 != 0 for t in range(steps)] for b in range(B)])
    step_rows, outs = [], []
    for t in range(steps):
        rows = _step_rows(720 + t, B, H, d, W.SOFTPLUS)
        step_rows.append(rows)
        _load_rows(dc, rows)
        dc.slots.copy_(torch.tensor([slots[b] if live[b, t] else -1 for b in range(B)], dtype=torch.int32))
        K.check(dc.decode())
        outs.append(dc.out[:B].clone())
    torch.cuda.synchronize()
    assert int(dc.dev_status.item()) == 0
    # the oracle's view: sequence b took the rows of the steps where it was live
    lens = live.sum(1)
    ref_wl = W.Workload(**{**base.__dict__, "arrays": dict(base.arrays)})
    ref_wl.cu_seqlens = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    for nm in ROWS:
        ref_wl.arrays[nm] = np.concatenate(
            [np.stack([step_rows[t].arrays[nm][b] for t in range(steps) if live[b, t]]) for b in range(B)
             if lens[b] > 0])
    ref = oracle_mod.forward(ref_wl)
    rec, conv = to_np(dc.rec_state), to_np(dc.conv_state)
    for b in range(B):
        assert_close(rec[slots[b]], ref["rec_state"][b], f"slot of seq {b}")
        assert np.array_equal(conv[slots[b]], ref["conv_state"][b].astype(np.float32))
        r = int(ref_wl.cu_seqlens[b])
        for t in range(steps):
            if live[b, t]:
                assert_close(to_np(outs[t][b]), ref["out"][r], f"seq {b} step {t}")
                r += 1
    for sl in set(range(NS)) - set(slots):  # slots no sequence owns
        assert torch.equal(dc.rec_state[sl], dc.rec_state0[sl])


@pytest.mark.parametrize("T", [64, 200])
def test_prefill_then_decode(cuda_lib, oracle_mod, T):
    """A prompt prefilled on the chunk path, then two rows decoded: the
    decoded rows and the final states match the oracle over all T + 2 rows."""
    H, d = 2, 128
    full = W.make_workload("pd", 605 + T, [T + 2], H=H, d=d, K=4, io_dtype=W.BF16,
                           gate_mode=W.SAFE, lower_bound=-5.0, out_gate=True, init_state="random")
    ref = oracle_mod.forward(full)
    from tests.parity import gather_rows

    pre = DeviceCase(gather_rows(full, [(0, T)]))
    K.check(pre.prefill())
    outs = []
    for r in (T, T + 1):
        step = gather_rows(full, [(r, r + 1)])
        dec = DeviceCase(step)
        dec.conv_state.copy_(pre.conv_state)
        dec.rec_state.copy_(pre.rec_state)
        K.check(dec.decode())
        outs.append(dec.out[:1].clone())
        pre.conv_state.copy_(dec.conv_state)
        pre.rec_state.copy_(dec.rec_state)
    torch.cuda.synchronize()
    assert_close(to_np(pre.out[:T]), ref["out"][:T], "prefill rows")
    assert_close(np.concatenate([to_np(o) for o in outs]), ref["out"][T:], "decoded rows")
    assert_close(to_np(pre.rec_state), ref["rec_state"], "final state")
    assert np.array_equal(to_np(pre.conv_state), ref["conv_state"].astype(np.float32))
