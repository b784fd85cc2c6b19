"""Variable-length prefill on the GPU against the fp64 oracle."""
import numpy as np
import pytest
import torch

from linear_attention_serving_kda_gb300 import workloads as W
from linear_attention_serving_kda_gb300.runtime import DeviceCase
from tests.parity import assert_bf16_within_one_ulp, assert_close, to_np

pytestmark = pytest.mark.gpu


def _prefill(kda, wl, out_dtype=W.F32, **kw):
    dc = DeviceCase(wl, out_dtype=out_dtype, **kw)
    kda.check(dc.prefill())
    torch.cuda.synchronize()
    assert int(dc.dev_status.item()) == 0
    return dc


def _check_all(dc, ref):
    T = dc.wl.T
    assert_close(to_np(dc.out[:T]), ref["out"], "out")
    assert_close(to_np(dc.rec_state), ref["rec_state"], "rec_state")
    assert np.array_equal(to_np(dc.conv_state), ref["conv_state"].astype(np.float32))


def test_tiny_case(cuda_lib, oracle_mod):
    """1 sequence, T=64, H=2, dk=dv=32, conv 4, fp32, safe gate, zero states."""
    wl = W.tiny_oracle_case()
    _check_all(_prefill(cuda_lib, wl), oracle_mod.forward(wl))


VARLEN = [
    # lens, d, io, gate, K, out_gate, init
    ([1, 15, 16, 17], 32, W.F32, W.SAFE, 4, False, "random"),
    ([63, 64, 65], 64, W.BF16, W.SAFE, 4, True, "random"),
    ([130, 0, 2, 1], 128, W.BF16, W.SAFE, 3, False, "random"),
    ([129, 64, 200], 128, W.BF16, W.SOFTPLUS, 4, True, "zero"),
    ([257, 3], 128, W.F32, W.SAFE, 2, True, "random"),
    ([1, 0, 2, 9, 3], 128, W.BF16, W.SOFTPLUS, 4, True, "random"),
    ([8, 16, 7, 24], 128, W.F32, W.SOFTPLUS, 3, False, "random"),
    ([0, 0], 64, W.F32, W.SAFE, 4, False, "random"),
]


@pytest.mark.parametrize("lens,d,io,gate,K,og,init", VARLEN)
def test_varlen_cases(cuda_lib, oracle_mod, lens, d, io, gate, K, og, init):
    wl = W.make_workload("vl", 300 + sum(lens) + d, lens, H=3, d=d, K=K, io_dtype=io,
                         gate_mode=gate, lower_bound=-5.0, out_gate=og, init_state=init)
    _check_all(_prefill(cuda_lib, wl), oracle_mod.forward(wl))


CHUNK = [
    # lens, K, out_gate, init -- dk = dv = 128, bf16 rows, safe gate: the tensor-core path
    ([1, 63, 64, 65], 4, True, "random"),
    ([128, 200, 17], 2, False, "zero"),
    ([333], 3, True, "random"),
]


@pytest.mark.parametrize("io,gate,K,og", [(W.F32, W.SOFTPLUS, 4, True), (W.F32, W.SAFE, 3, False),
                                           (W.F32, W.SOFTPLUS, 2, False)])
def test_row_path_prefill_is_decode_bits(cuda_lib, io, gate, K, og):
    """dk = dv = 128 shapes the chunk kernel does not take (fp32 rows) run the
    delta rule row by row: a prefilled sequence has the bits of the same rows
    decoded one at a time (outputs, final state, conv state)."""
    from tests.parity import gather_rows

    T = 21
    wl = W.make_workload("rowbits", 640 + K, [T], H=3, d=128, K=K, io_dtype=io,
                         gate_mode=gate, lower_bound=-5.0, out_gate=og, init_state="random")
    full = _prefill(cuda_lib, wl)
    dec = DeviceCase(gather_rows(wl, [(0, 1)]))
    outs = []
    for r in range(T):
        step = DeviceCase(gather_rows(wl, [(r, r + 1)]))
        step.conv_state.copy_(dec.conv_state)
        step.rec_state.copy_(dec.rec_state)
        cuda_lib.check(step.decode())
        outs.append(step.out[:1].clone())
        dec = step
    torch.cuda.synchronize()
    assert int(dec.dev_status.item()) == 0
    assert torch.equal(torch.cat(outs), full.out[:T])
    assert torch.equal(dec.rec_state, full.rec_state)
    assert torch.equal(dec.conv_state, full.conv_state)


@pytest.mark.parametrize("lens,K,og,init", CHUNK)
def test_chunk_path_cases(cuda_lib, oracle_mod, lens, K, og, init):
    wl = W.make_workload("ck", 400 + sum(lens) + K, lens, H=2, d=128, K=K, io_dtype=W.BF16,
                         gate_mode=W.SAFE, lower_bound=-5.0, out_gate=og, init_state=init)
    _check_all(_prefill(cuda_lib, wl), oracle_mod.forward(wl))


@pytest.mark.parametrize("fval", [-30.0, 30.0])
def test_chunk_gate_extremes(cuda_lib, oracle_mod, fval):
    """Every row at the gate's ends: alpha ~ 1 (long memory, f -> -inf) and
    log alpha ~ -5 (the lower bound, the widest factor range in a chunk)."""
    wl = W.make_workload("gx", 420, [150, 64], H=2, d=128, K=4, io_dtype=W.BF16,
                         gate_mode=W.SAFE, lower_bound=-5.0, out_gate=False, init_state="random")
    wl.arrays["f"][:] = fval
    wl.arrays["A_log"][:] = 0.0
    _check_all(_prefill(cuda_lib, wl), oracle_mod.forward(wl))


def test_bf16_output(cuda_lib, oracle_mod):
    wl = W.make_workload("vlb", 311, [100, 37], H=2, d=128, K=4, io_dtype=W.BF16,
                         gate_mode=W.SAFE, lower_bound=-5.0, out_gate=True, init_state="random")
    ref = oracle_mod.forward(wl)
    dc = _prefill(cuda_lib, wl, out_dtype=W.BF16)
    assert_bf16_within_one_ulp(to_np(dc.out[:wl.T]), ref["out"])


def test_prompt_cut_bits(cuda_lib):
    """A prompt cut at a multiple of 64 rows gives the bits of one uncut call."""
    T, cut = 320, 128
    wl = W.make_workload("cut", 312, [T], H=2, d=128, K=4, io_dtype=W.BF16,
                         gate_mode=W.SAFE, lower_bound=-5.0, out_gate=True, init_state="random")
    full = _prefill(cuda_lib, wl)
    from tests.parity import gather_rows

    a = gather_rows(wl, [(0, cut)])
    b = gather_rows(wl, [(cut, T)])
    da = _prefill(cuda_lib, a)
    db = DeviceCase(b)
    db.conv_state.copy_(da.conv_state)
    db.rec_state.copy_(da.rec_state)
    cuda_lib.check(db.prefill())
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([da.out[:cut], db.out[:T - cut]]), full.out[:T])
    assert torch.equal(db.rec_state, full.rec_state)
    assert torch.equal(db.conv_state, full.conv_state)


@pytest.mark.parametrize("T,pieces", [(2304, 3), (3072, 2), (1000, 4)])
def test_prompt_cuts_in_order_share_states(cuda_lib, T, pieces):
    """A prompt cut by ``shard.prompt_cuts`` and run in order on one stream,
    every cut bound to the same state tensors, gives the uncut call's bits --
    whichever path (split or fused) the whole prompt and each cut take."""
    from linear_attention_serving_kda_gb300 import shard

    wl = W.make_workload("cuts", 314 + T, [T], H=2, d=128, K=4, io_dtype=W.BF16,
                         gate_mode=W.SAFE, lower_bound=-5.0, out_gate=True, init_state="random")
    full = _prefill(cuda_lib, wl, out_dtype=W.BF16)
    cuts = shard.prompt_cuts(T, pieces)
    cases = [DeviceCase(shard.cut_prompt(wl, a, b), out_dtype=W.BF16) for a, b in cuts]
    for dc in cases[1:]:
        dc.conv_state, dc.rec_state = cases[0].conv_state, cases[0].rec_state
    for dc in cases:
        cuda_lib.check(dc.prefill())
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([dc.out[:dc.wl.T] for dc in cases]), full.out[:T])
    assert torch.equal(cases[0].rec_state, full.rec_state)
    assert torch.equal(cases[0].conv_state, full.conv_state)


def test_slots_and_bad_seqlens(cuda_lib, oracle_mod):
    wl = W.make_workload("pslot", 313, [70, 5, 33], H=2, d=64, K=4, io_dtype=W.F32,
                         gate_mode=W.SAFE, lower_bound=-5.0, init_state="random")
    ref = oracle_mod.forward(wl)
    dc = DeviceCase(wl, num_slots=5, slots=[3, -1, 0])
    rs0 = dc.rec_state.clone()
    dc.out.fill_(float("nan"))
    cuda_lib.check(dc.prefill())
    torch.cuda.synchronize()
    out = to_np(dc.out)
    assert np.all(np.isnan(out[70:75]))
    assert_close(out[:70], ref["out"][:70], "out s0")
    assert_close(out[75:], ref["out"][75:], "out s2")
    assert_close(to_np(dc.rec_state[3]), ref["rec_state"][0], "state s0")
    assert_close(to_np(dc.rec_state[0]), ref["rec_state"][2], "state s2")
    for sl in (1, 2, 4):
        assert torch.equal(dc.rec_state[sl], rs0[sl])
    # a non-monotone cu_seqlens is flagged, not trapped
    dc2 = DeviceCase(wl)
    dc2.cu_seqlens.copy_(torch.tensor([0, 80, 75, 108], dtype=torch.int32))
    cuda_lib.check(dc2.prefill())
    torch.cuda.synchronize()
    assert int(dc2.dev_status.item()) & cuda_lib.KDA_DEV_BAD_SEQLENS


def _check_conv_rows(wl, dc):
    """The new conv state of each sequence: its last K-1 raw rows, exactly."""
    cs = to_np(dc.conv_state)
    K1 = wl.K - 1
    for s in range(wl.N):
        t1 = wl.cu_seqlens[s + 1]
        raw = np.concatenate([wl.arrays[nm][t1 - K1:t1].reshape(K1, -1) for nm in ("q", "k", "v")], axis=1)
        assert np.array_equal(cs[s], raw)


@pytest.mark.slow
def test_varlen_full_size(cuda_lib, oracle_mod):
    """8 sequences, lengths ~U{512..8192} (29 273 rows), H=32, dk=dv=128, bf16,
    safe gate lb=-5, random initial states: every (sequence, head) unit
    against the oracle -- relative L2 and max-abs/RMS over the whole output
    and final-state tensors, conv states exact."""
    wl = W.varlen_prefill_case()
    dc = _prefill(cuda_lib, wl)
    ref = oracle_mod.forward(wl)
    _check_all(dc, ref)
    _check_conv_rows(wl, dc)


@pytest.mark.slow
def test_long_prefill_full_size(cuda_lib, oracle_mod):
    """1 sequence of 32768 rows, H=32, dk=dv=128, bf16, sigmoid-gated RMSNorm
    (eps 1e-6, unit weight), zero states: all 32 heads against the oracle,
    whole tensors."""
    wl = W.long_prefill_case()
    dc = _prefill(cuda_lib, wl)
    ref = oracle_mod.forward(wl)
    _check_all(dc, ref)
    _check_conv_rows(wl, dc)


def _prefill_sweep_cases(n=16, seed=4242):
    """Seeded shapes over both prefill paths: the tensor-core chunk kernel
    (dk = dv = 128, bf16 rows, safe gate with lb >= -5) and the row kernels
    (everything else), with empty, one-row, chunk-edge and ragged lengths."""
    rng = np.random.default_rng(seed)
    edge = [0, 1, 2, 3, 63, 64, 65, 127, 128, 129]
    cases = []
    for i in range(n):
        chunk = i < 6  # the first six take the chunk kernel's shapes
        d = 128 if chunk or i % 3 == 0 else int(rng.choice([32, 64]))
        io = W.BF16 if chunk or i == n - 1 else [W.BF16, W.F32][i % 2]
        gate = W.SAFE if chunk else [W.SOFTPLUS, W.SAFE][(i // 2) % 2]
        lb = -5.0 if chunk else float(rng.choice([-5.0, -8.0, -1.5]))
        N = int(rng.integers(1, 5))
        lens = [int(rng.choice(edge)) if rng.random() < 0.5 else int(rng.integers(4, 300)) for _ in range(N)]
        cases.append(dict(lens=lens, d=d, io=io, gate=gate, lb=lb, K=int(rng.integers(2, 5)),
                          H=int(rng.integers(1, 4)), og=bool(rng.integers(0, 2)),
                          init=["random", "zero"][int(rng.integers(0, 2))], seed=7000 + i))
    return cases


@pytest.mark.parametrize("case", _prefill_sweep_cases(),
                         ids=lambda c: f"d{c['d']}{c['io']}g{c['gate']}k{c['K']}h{c['H']}n{len(c['lens'])}")
def test_prefill_sweep(cuda_lib, oracle_mod, case):
    """Seeded sweep of prefill shapes against the oracle: outputs, final
    recurrent state and conv state (bit-equal: it holds raw rows)."""
    c = case
    wl = W.make_workload(f"psweep{c['seed']}", c["seed"], c["lens"], H=c["H"], d=c["d"], K=c["K"],
                         io_dtype=c["io"], gate_mode=c["gate"], lower_bound=c["lb"], out_gate=c["og"],
                         init_state=c["init"])
    _check_all(_prefill(cuda_lib, wl), oracle_mod.forward(wl))


UNBOUNDED = [
    # lens, gate, lower bound, A_log (all heads), K, out_gate -- bf16 rows, dk = dv = 128
    ([200, 7, 130], W.SOFTPLUS, -5.0, 3.0, 4, True),    # ~-16 per row: chunks of a few rows
    ([150, 64], W.SAFE, -12.0, 2.0, 3, False),          # safe gate below -5: cut near 13-16 rows
    ([40, 3], W.SOFTPLUS, -5.0, 5.0, 2, True),          # ~-100 per row: one-row chunks
    ([333, 1, 65], W.SOFTPLUS, -5.0, None, 4, False),   # A_log ~ U(-1, 1): mostly whole chunks
    ([2048], W.SOFTPLUS, -5.0, 2.0, 4, True),           # hundreds of cut chunks in one chain
]


@pytest.mark.parametrize("lens,gate,lb,alog,K,og", UNBOUNDED)
def test_chunk_path_unbounded_gates(cuda_lib, oracle_mod, lens, gate, lb, alog, K, og):
    """Gates whose per-row log-decay is not bounded by -5 take the chunk
    kernel with data-dependent chunk boundaries (a chunk ends before the first
    row whose decay would take a factor out of range): against the oracle,
    including decays strong enough for chunks of a single row."""
    wl = W.make_workload("unb", 900 + sum(lens) + K, lens, H=2, d=128, K=K, io_dtype=W.BF16,
                         gate_mode=gate, lower_bound=lb, out_gate=og, init_state="random")
    if alog is not None:
        wl.arrays["A_log"] = np.full_like(wl.arrays["A_log"], alog)
    _check_all(_prefill(cuda_lib, wl), oracle_mod.forward(wl))


@pytest.mark.slow
def test_varlen_full_size_softplus(cuda_lib, oracle_mod):
    """The varlen workload's lengths and rows (29 273 rows, H=32, bf16) with the
    softplus gate: the chunk kernel with data-dependent chunk boundaries,
    every unit against the oracle (whole tensors)."""
    wl = W.make_workload("prefill_varlen_softplus_n8_h32_d128_bf16", 2, None, H=32, d=128, K=4, io_dtype=W.BF16,
                         gate_mode=W.SOFTPLUS, lower_bound=-5.0, init_state="random", draw_lens=(8, 512, 8192))
    dc = _prefill(cuda_lib, wl)
    _check_all(dc, oracle_mod.forward(wl))


@pytest.mark.slow
def test_long_prefill_full_size_softplus(cuda_lib, oracle_mod):
    """A 32 768-row prompt, H=32, bf16, gated RMSNorm, softplus gate: the split
    path with each chain's chunk list fixed by the boundary pass, all heads
    against the oracle (whole tensors)."""
    wl = W.make_workload("prefill_long_softplus_t32768_h32_d128_bf16", 4, [32768], H=32, d=128, K=4,
                         io_dtype=W.BF16, gate_mode=W.SOFTPLUS, lower_bound=-5.0, out_gate=True,
                         init_state="zero")
    dc = _prefill(cuda_lib, wl)
    assert cuda_lib.kda_prefill_workspace_bytes(dc.params(), wl.N, wl.T) > 2**25  # the split path's ring
    _check_all(dc, oracle_mod.forward(wl))
