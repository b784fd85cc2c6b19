"""Verify windows and commit: bit-exact against serial GPU decode, and within
tolerance of the fp64 oracle."""
import numpy as np
import pytest
import torch

from linear_attention_serving_kda_gb300 import kda as K
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
    # the seeded counts reach both edges: a sequence that keeps nothing and one that keeps the whole window
    assert acc.min() == 0 and acc.max() == wl.W and np.all((acc >= 0) & (acc <= wl.W))
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


@pytest.mark.parametrize("Wn,io,gate,og", [(1, W.BF16, W.SAFE, True), (13, W.BF16, W.SOFTPLUS, True),
                                         (16, W.BF16, W.SAFE, False), (17, W.F32, W.SAFE, False)])
def test_verify_commit_window_lengths(cuda_lib, oracle_mod, Wn, io, gate, og):
    """dk = dv = 128 windows of one row and of several staged 8-row blocks with
    a ragged last block, and the longest window the streaming commit stages
    (16 rows; 17 commits through the per-unit kernel): serial-decode bits and
    oracle tolerance."""
    B = 4
    wl = W.make_workload(f"verw{Wn}", 300 + Wn, [Wn] * B, H=3, d=128, K=4, io_dtype=io,
                         gate_mode=gate, lower_bound=-5.0, out_gate=og, init_state="random",
                         W=Wn, accepted=True)
    wl.arrays["accepted"][:2] = [Wn, Wn - 1]
    _check_window(cuda_lib, oracle_mod, wl, out_dtype=W.BF16 if io == W.BF16 else W.F32)


@pytest.mark.parametrize("d,io", [(32, W.F32), (128, W.BF16)])
def test_commit_rejects_bad_accepted(cuda_lib, d, io):
    wl = W.make_workload("badacc", 99, [4] * 3, H=2, d=d, K=4, io_dtype=io,
                         gate_mode=W.SAFE, init_state="random", W=4, accepted=True)
    dc = DeviceCase(wl)
    cuda_lib.check(dc.verify())
    rs0, cs0 = dc.rec_state.clone(), dc.conv_state.clone()
    bad = torch.tensor([9, -1, 2], dtype=torch.int32, device="cuda")
    cuda_lib.check(dc.commit(accepted=bad))
    torch.cuda.synchronize()
    assert int(dc.dev_status.item()) & cuda_lib.KDA_DEV_BAD_ACCEPTED
    # the bad sequences keep their states; the good one commits its two rows
    assert torch.equal(dc.rec_state[:2], rs0[:2]) and torch.equal(dc.conv_state[:2], cs0[:2])
    assert not torch.equal(dc.rec_state[2], rs0[2])


def _commit_verify(dc, accepted, log_prev, log_new):
    wl = dc.wl
    return K.kda_commit_verify(dc.params(), wl.N, wl.W, accepted, log_prev, dc.q, dc.k, dc.v, dc.f, dc.b, dc.g,
                               dc.slots, dc.conv_state, dc.rec_state, log_new, dc.out, dc.dev_status)


def _load_rows(dc, wl):
    for nm in ("q", "k", "v", "f", "b", "g"):
        t = getattr(dc, nm)
        if t is not None:
            t.copy_(wl.to_torch(nm, "cuda"))


@pytest.mark.parametrize("d,io,gate,alias", [(128, W.BF16, W.SOFTPLUS, False), (128, W.BF16, W.SAFE, True),
                                             (64, W.F32, W.SAFE, False), (32, W.BF16, W.SOFTPLUS, True)])
def test_commit_verify_equals_separate_calls(cuda_lib, d, io, gate, alias):
    """kda_commit_verify = kda_commit then kda_verify_window, bit for bit
    (outputs, both states, the new log), also with the new log written over
    the previous one."""
    B, Wn, H = 5, 8, 3
    kw = dict(H=H, d=d, K=4, io_dtype=io, gate_mode=gate, lower_bound=-5.0, out_gate=True,
              init_state="random", W=Wn, accepted=True)
    win1 = W.make_workload("cv1", 901 + d, [Wn] * B, **kw)
    win2 = W.make_workload("cv2", 902 + d, [Wn] * B, **kw)
    acc = torch.tensor([0, 3, 8, 1, 5], dtype=torch.int32, device="cuda")
    sep = DeviceCase(win1, out_dtype=W.F32, num_slots=6, slots=[4, 0, 2, 5, 1])
    fus = DeviceCase(win1, out_dtype=W.F32, num_slots=6, slots=[4, 0, 2, 5, 1])
    for dc in (sep, fus):
        dc.alloc_log()
        K.check(dc.verify())
    # separate calls: commit window 1, verify window 2
    K.check(sep.commit(accepted=acc))
    _load_rows(sep, win2)
    K.check(sep.verify())
    # one call
    _load_rows(fus, win2)
    log2 = fus.log if alias else fus._guarded(fus.log.shape, torch.uint8)  # sentinel-filled like the others
    K.check(_commit_verify(fus, acc, fus.log, log2))
    torch.cuda.synchronize()
    assert int(sep.dev_status.item()) == 0 and int(fus.dev_status.item()) == 0
    assert torch.equal(fus.out[:B * Wn], sep.out[:B * Wn])
    assert torch.equal(fus.rec_state, sep.rec_state)
    assert torch.equal(fus.conv_state, sep.conv_state)
    assert torch.equal(log2, sep.log)


@pytest.mark.parametrize("Wn,alias", [(12, True), (9, False)])
def test_commit_verify_long_windows(cuda_lib, Wn, alias):
    """Commit of more than one staged block of log rows fused into the next
    verify (dk = dv = 128) = the separate calls, bit for bit."""
    B, H, d = 4, 2, 128
    kw = dict(H=H, d=d, K=4, io_dtype=W.BF16, gate_mode=W.SAFE, lower_bound=-5.0, out_gate=True,
              init_state="random", W=Wn, accepted=True)
    win1 = W.make_workload("cvl1", 921 + Wn, [Wn] * B, **kw)
    win2 = W.make_workload("cvl2", 922 + Wn, [Wn] * B, **kw)
    acc = torch.tensor([Wn, 9, 0, 3], dtype=torch.int32, device="cuda")
    sep = DeviceCase(win1, out_dtype=W.F32)
    fus = DeviceCase(win1, out_dtype=W.F32)
    for dc in (sep, fus):
        dc.alloc_log()
        K.check(dc.verify())
    K.check(sep.commit(accepted=acc))
    _load_rows(sep, win2)
    K.check(sep.verify())
    _load_rows(fus, win2)
    log2 = fus.log if alias else fus._guarded(fus.log.shape, torch.uint8)  # sentinel-filled like the others
    K.check(_commit_verify(fus, acc, fus.log, log2))
    torch.cuda.synchronize()
    assert int(sep.dev_status.item()) == 0 and int(fus.dev_status.item()) == 0
    assert torch.equal(fus.out[:B * Wn], sep.out[:B * Wn])
    assert torch.equal(fus.rec_state, sep.rec_state)
    assert torch.equal(fus.conv_state, sep.conv_state)
    assert torch.equal(log2, sep.log)


def test_commit_verify_bad_accepted(cuda_lib):
    """An out-of-range accepted count is flagged and its sequence skipped; the
    other sequences match the separate calls."""
    B, Wn, H, d = 3, 4, 2, 64
    kw = dict(H=H, d=d, K=4, io_dtype=W.F32, gate_mode=W.SAFE, lower_bound=-5.0, init_state="random", W=Wn,
              accepted=True)
    win1 = W.make_workload("cvb1", 911, [Wn] * B, **kw)
    win2 = W.make_workload("cvb2", 912, [Wn] * B, **kw)
    fus = DeviceCase(win1, out_dtype=W.F32)
    sep = DeviceCase(win1, out_dtype=W.F32)
    for dc in (fus, sep):
        dc.alloc_log()
        K.check(dc.verify())
    rs0, cs0 = fus.rec_state.clone(), fus.conv_state.clone()
    bad = torch.tensor([2, Wn + 1, 1], dtype=torch.int32, device="cuda")
    good = torch.tensor([2, 0, 1], dtype=torch.int32, device="cuda")
    _load_rows(fus, win2)
    fus.out.fill_(float("nan"))
    log2 = fus._guarded(fus.log.shape, torch.uint8)
    K.check(_commit_verify(fus, bad, fus.log, log2))
    K.check(sep.commit(accepted=good))
    _load_rows(sep, win2)
    K.check(sep.verify())
    torch.cuda.synchronize()
    assert int(fus.dev_status.item()) & K.KDA_DEV_BAD_ACCEPTED
    assert torch.equal(fus.rec_state[1], rs0[1]) and torch.equal(fus.conv_state[1], cs0[1])
    assert torch.all(torch.isnan(fus.out[Wn:2 * Wn]))
    for b in (0, 2):
        assert torch.equal(fus.rec_state[b], sep.rec_state[b])
        assert torch.equal(fus.out[b * Wn:(b + 1) * Wn], sep.out[b * Wn:(b + 1) * Wn])


def test_verify_slot_map_negative_and_bad(cuda_lib):
    """dk = dv = 128 verify, commit and commit+verify with a slot map: a
    negative slot skips its sequence (outputs and state untouched), a slot past
    the pool is flagged and skipped, and the other sequences equal the same
    window run with valid slots."""
    B, Wn, H = 4, 6, 2
    wl = W.make_workload("vslot", 77, [Wn] * B, H=H, d=128, K=4, io_dtype=W.BF16, gate_mode=W.SOFTPLUS,
                         lower_bound=-5.0, out_gate=True, init_state="random", W=Wn, accepted=True)
    ref = DeviceCase(wl, out_dtype=W.F32, num_slots=5, slots=[3, 0, 1, 2])
    dc = DeviceCase(wl, out_dtype=W.F32, num_slots=5, slots=[3, -1, 1, 9])
    for c in (ref, dc):
        c.alloc_log()
    dc.out.fill_(float("nan"))
    rs0, cs0 = dc.rec_state.clone(), dc.conv_state.clone()
    K.check(ref.verify())
    K.check(dc.verify())
    torch.cuda.synchronize()
    assert int(dc.dev_status.item()) & K.KDA_DEV_BAD_SLOT
    for b in (1, 3):
        assert torch.all(torch.isnan(dc.out[b * Wn:(b + 1) * Wn]))
    for b in (0, 2):
        assert torch.equal(dc.out[b * Wn:(b + 1) * Wn], ref.out[b * Wn:(b + 1) * Wn])
    # commit, then commit fused into a second verify of the same rows
    acc = torch.tensor([3, 5, Wn, 2], dtype=torch.int32, device="cuda")
    K.check(ref.commit(accepted=acc))
    K.check(dc.commit(accepted=acc))
    torch.cuda.synchronize()
    assert torch.equal(dc.rec_state[0], rs0[0]) and torch.equal(dc.conv_state[0], cs0[0])  # slot 0: unused
    for sl in (3, 1):
        assert torch.equal(dc.rec_state[sl], ref.rec_state[sl])
        assert torch.equal(dc.conv_state[sl], ref.conv_state[sl])
    dc.out.fill_(float("nan"))
    log2r, log2d = ref._guarded(ref.log.shape, torch.uint8), dc._guarded(dc.log.shape, torch.uint8)
    K.check(_commit_verify(ref, acc, ref.log, log2r))
    K.check(_commit_verify(dc, acc, dc.log, log2d))
    torch.cuda.synchronize()
    for b, sl in ((0, 3), (2, 1)):
        assert torch.equal(dc.out[b * Wn:(b + 1) * Wn], ref.out[b * Wn:(b + 1) * Wn])
        assert torch.equal(dc.rec_state[sl], ref.rec_state[sl])
    for b in (1, 3):
        assert torch.all(torch.isnan(dc.out[b * Wn:(b + 1) * Wn]))


def _sweep_cases(n=12, seed=2024):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        d = 128 if i < 8 else int(rng.choice([32, 64]))
        cases.append(dict(d=d, Wn=int(rng.integers(1, 21)), B=int(rng.integers(1, 4)), H=int(rng.integers(1, 3)),
                          K=int(rng.integers(2, 5)), gate=[W.SAFE, W.SOFTPLUS][i % 2],
                          io=[W.BF16, W.F32][(i // 2) % 2], og=bool(rng.integers(0, 2)), seed=5000 + i))
    return cases


@pytest.mark.parametrize("case", _sweep_cases(), ids=lambda c: f"d{c['d']}w{c['Wn']}b{c['B']}h{c['H']}k{c['K']}")
def test_verify_commit_sweep(cuda_lib, oracle_mod, case):
    """Seeded sweep of window lengths, batch sizes, head counts, conv taps,
    gates, row types and output gates: verify and commit against serial
    decode (bits) and the oracle."""
    c = case
    wl = W.make_workload(f"vsweep{c['seed']}", c["seed"], [c["Wn"]] * c["B"], H=c["H"], d=c["d"], K=c["K"],
                         io_dtype=c["io"], gate_mode=c["gate"], lower_bound=-5.0, out_gate=c["og"],
                         init_state="random", W=c["Wn"], accepted=True)
    _check_window(cuda_lib, oracle_mod, wl, out_dtype=W.BF16 if c["io"] == W.BF16 else W.F32)
