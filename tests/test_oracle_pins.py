"""Pins for the fp64 oracle: closed forms, invariants, special cases and brute
force, none of which re-types the oracle's own formulas.

Each test names the mistake it is there to catch.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

from linear_attention_serving_kda_gb300 import workloads as W

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ------------------------------------------------------------------ scalars

def test_scalar_special_values(oracle_mod):
    o = oracle_mod
    assert o.sigmoid(0.0) == 0.5
    assert o.silu(0.0) == 0.0
    assert abs(o.softplus(0.0) - math.log(2.0)) < 1e-16
    for x in (-30.0, -3.0, -0.5, 0.5, 3.0, 30.0):
        # sigmoid symmetry and the softplus identity softplus(x) - softplus(-x) = x
        assert abs(o.sigmoid(x) + o.sigmoid(-x) - 1.0) < 1e-15
        assert abs(o.softplus(x) - o.softplus(-x) - x) < 1e-13
        # silu(x) - silu(-x) = x  (x s(x) + x s(-x) = x)
        assert abs(o.silu(x) - o.silu(-x) - x) < 1e-13
    # the small tail of softplus survives for very negative x (no log(1+tiny) loss)
    assert abs(o.softplus(-50.0) / math.exp(-50.0) - 1.0) < 1e-12
    assert abs(o.softplus(800.0) - 800.0) < 1e-12  # no overflow


def test_gate_special_values(oracle_mod):
    """f + dt_bias = 0 and A_log = 0: softplus gate gives alpha = 1/2, safe gate
    gives log alpha = lb / 2.  Catches a dropped sign, a missing exp(A_log) or
    a sigmoid/softplus mix-up."""
    o = oracle_mod
    la = o.log_alpha(W.SOFTPLUS, -5.0, 0.0, 0.0, 0.0)
    assert abs(la + math.log(2.0)) < 1e-16
    assert abs(math.exp(la) - 0.5) < 1e-16
    assert o.log_alpha(W.SAFE, -5.0, 0.0, 0.0, 0.0) == -2.5
    assert o.log_alpha(W.SAFE, -3.0, 0.0, 0.0, 0.0) == -1.5
    # saturation: the safe gate tends to lb for large argument and to 0 for small
    assert abs(o.log_alpha(W.SAFE, -5.0, 0.0, 1e3, 0.0) + 5.0) < 1e-15
    assert o.log_alpha(W.SAFE, -5.0, 0.0, -1e3, 0.0) == 0.0
    # exp(A_log) -> 0 switches the decay off in both modes (alpha = 1)
    assert o.log_alpha(W.SOFTPLUS, -5.0, -1000.0, 3.0, 0.2) == 0.0
    assert o.log_alpha(W.SAFE, -5.0, -1000.0, 3.0, 0.2) == -2.5  # sigmoid(0) * lb


def test_gate_structure(oracle_mod):
    """Where the parameters enter: dt_bias adds to f; exp(A_log) scales the
    softplus gate outside and the safe gate's sigmoid argument inside."""
    o = oracle_mod
    rng = np.random.default_rng(7)
    for _ in range(50):
        a, f, dt = rng.uniform(-1, 1), rng.normal(), rng.normal(0, 0.3)
        for mode in (W.SOFTPLUS, W.SAFE):
            assert abs(o.log_alpha(mode, -5.0, a, f, dt) - o.log_alpha(mode, -5.0, a, f + dt, 0.0)) < 1e-14
        # softplus: log alpha(A_log = a) = e^a * log alpha(A_log = 0)
        assert abs(o.log_alpha(W.SOFTPLUS, -5, a, f, dt)
                   - math.exp(a) * o.log_alpha(W.SOFTPLUS, -5, 0.0, f, dt)) < 1e-13
        # safe: the factor exp(A_log) multiplies the sigmoid's argument
        assert abs(o.log_alpha(W.SAFE, -5, a, f, dt)
                   - o.log_alpha(W.SAFE, -5, 0.0, math.exp(a) * (f + dt), 0.0)) < 1e-13
        # ranges: safe in (lb, 0), softplus < 0; more f means more decay
        s = o.log_alpha(W.SAFE, -5.0, a, f, dt)
        assert -5.0 < s < 0.0
        assert o.log_alpha(W.SOFTPLUS, -5.0, a, f, dt) < 0.0
        assert o.log_alpha(W.SAFE, -5.0, a, f + 0.5, dt) < s
        assert o.log_alpha(W.SOFTPLUS, -5.0, a, f + 0.5, dt) < o.log_alpha(W.SOFTPLUS, -5.0, a, f, dt)


# ------------------------------------------------------------- vector ops

def test_l2norm(oracle_mod):
    rng = np.random.default_rng(1)
    x = rng.normal(size=128)
    y = oracle_mod.l2norm(x, 0.0)
    assert abs(np.linalg.norm(y) - 1.0) < 1e-14
    assert np.allclose(y / np.linalg.norm(y), x / np.linalg.norm(x), atol=1e-15)
    # eps only matters for tiny vectors: |y| = |x| / sqrt(|x|^2 + eps)
    z = 1e-4 * x / np.linalg.norm(x)
    yz = oracle_mod.l2norm(z, 1e-6)
    assert abs(np.linalg.norm(yz) - 1e-4 / math.sqrt(1e-8 + 1e-6)) < 1e-12
    assert np.all(oracle_mod.l2norm(np.zeros(16), 1e-6) == 0.0)


def test_gated_rmsnorm(oracle_mod):
    rng = np.random.default_rng(2)
    o = rng.normal(size=64) * 3.0
    big = np.full(64, 800.0)            # sigmoid -> 1
    y = oracle_mod.gated_rmsnorm(o, big, np.ones(64), 0.0)
    assert abs(np.sqrt(np.mean(y * y)) - 1.0) < 1e-14
    assert np.allclose(y, o / np.sqrt(np.mean(o * o)), rtol=1e-14)
    y0 = oracle_mod.gated_rmsnorm(o, np.zeros(64), np.ones(64), 0.0)   # sigmoid(0) = 1/2
    assert np.allclose(y0, 0.5 * y, rtol=1e-14)
    # scale invariance of the norm and per-channel weight
    w = rng.uniform(0.5, 2.0, size=64)
    g = rng.normal(size=64)
    ya = oracle_mod.gated_rmsnorm(o, g, w, 0.0)
    yb = oracle_mod.gated_rmsnorm(7.0 * o, g, np.ones(64), 0.0)
    assert np.allclose(ya, yb * w, rtol=1e-13)
    # eps: output RMS with sigmoid -> 1 is sqrt(ms / (ms + eps))
    ye = oracle_mod.gated_rmsnorm(o, big, np.ones(64), 1e-6)
    ms = np.mean(o * o)
    assert abs(np.sqrt(np.mean(ye * ye)) - math.sqrt(ms / (ms + 1e-6))) < 1e-14


# --------------------------------------------------------------------- conv

def test_conv_impulse_response(oracle_mod):
    """One nonzero raw row gives the weights back in reversed tap order;
    catches a reversed or shifted tap index."""
    K, C, T = 4, 3, 10
    rng = np.random.default_rng(3)
    w = rng.normal(size=(C, K))
    x = np.zeros((T, C))
    x[4, 1] = 1.0
    y = oracle_mod.conv1d(x, np.zeros((K - 1, C)), w)
    for m in range(K):
        assert y[4 + m, 1] == w[1, K - 1 - m]
    assert np.count_nonzero(y) == K
    # an impulse in history row r (oldest first) reaches output row t with tap r - t
    for r in range(K - 1):
        hist = np.zeros((K - 1, C))
        hist[r, 2] = 1.0
        y = oracle_mod.conv1d(np.zeros((T, C)), hist, w)
        for t in range(T):
            expect = w[2, r - t] if t <= r else 0.0
            assert y[t, 2] == expect


@pytest.mark.parametrize("K", [2, 3, 4])
def test_conv_matches_numpy_convolve(oracle_mod, K):
    """A causal depthwise conv is np.convolve with the taps reversed, run over
    the history rows followed by the new rows."""
    rng = np.random.default_rng(K)
    T, C = 13, 5
    x, hist, w = rng.normal(size=(T, C)), rng.normal(size=(K - 1, C)), rng.normal(size=(C, K))
    y = oracle_mod.conv1d(x, hist, w)
    for c in range(C):
        full = np.convolve(np.concatenate([hist[:, c], x[:, c]]), w[c, ::-1])
        assert np.allclose(y[:, c], full[K - 1:K - 1 + T], rtol=1e-13, atol=1e-13)


def test_conv_history_shift(oracle_mod):
    K, C = 4, 2
    hist = np.arange(6, dtype=float).reshape(3, 2)
    x = 100 + np.arange(4, dtype=float).reshape(2, 2)
    nh = oracle_mod.conv_history(x, hist, K)      # T=2 < K-1: old tail then new rows
    assert np.array_equal(nh, np.stack([hist[2], x[0], x[1]]))
    x5 = 200 + np.arange(10, dtype=float).reshape(5, 2)
    assert np.array_equal(oracle_mod.conv_history(x5, hist, K), x5[2:])
    assert np.array_equal(oracle_mod.conv_history(np.zeros((0, C)), hist, K), hist)


# --------------------------------------------------------------- delta step

def test_delta_overwrite_row(oracle_mod):
    """alpha = 1, beta = 1, k = e_i writes v into row i (up to the one rounding
    of s + (v - s)) and leaves the other rows bit-for-bit alone."""
    rng = np.random.default_rng(4)
    dk, dv = 6, 5
    S = rng.normal(size=(dk, dv))
    v, q = rng.normal(size=dv), rng.normal(size=dk)
    for i in range(dk):
        k = np.zeros(dk)
        k[i] = 1.0
        S2, o, u = oracle_mod.delta_step(S, np.ones(dk), 1.0, k, v, q)
        bound = 2 * np.finfo(float).eps * np.maximum(np.abs(S[i]), np.abs(v))
        assert np.all(np.abs(S2[i] - v) <= bound)
        assert np.array_equal(np.delete(S2, i, 0), np.delete(S, i, 0))
        assert np.allclose(o, S2.T @ q, rtol=1e-14)     # output reads the new state


def test_delta_write_invariant(oracle_mod):
    """For any decay, any state and a unit key, beta = 1 makes k^T S_new = v^T."""
    rng = np.random.default_rng(5)
    for dk, dv in ((8, 8), (7, 3), (3, 9)):
        for _ in range(20):
            S = rng.normal(size=(dk, dv))
            alpha = np.exp(-rng.uniform(0, 5, size=dk))
            k = rng.normal(size=dk)
            k /= np.linalg.norm(k)
            v = rng.normal(size=dv)
            S2, _, _ = oracle_mod.delta_step(S, alpha, 1.0, k, v, rng.normal(size=dk))
            assert np.allclose(k @ S2, v, atol=1e-12)


def test_delta_decay_only(oracle_mod):
    """beta = 0 only decays: S_new = Diag(alpha) S, u = 0."""
    rng = np.random.default_rng(6)
    S = rng.normal(size=(4, 3))
    alpha = rng.uniform(0.1, 1.0, size=4)
    q = rng.normal(size=4)
    S2, o, u = oracle_mod.delta_step(S, alpha, 0.0, rng.normal(size=4), rng.normal(size=3), q, 2.0)
    assert np.allclose(S2, alpha[:, None] * S, rtol=1e-15)
    assert np.all(u == 0.0)
    assert np.allclose(o, 2.0 * (alpha[:, None] * S).T @ q, rtol=1e-14)


def _frac(x):
    return Fraction(float(x))


def test_delta_matches_exact_matrix_form(oracle_mod):
    """Brute force in exact rational arithmetic of the matrix form
    S_new = (I - beta k k^T) Diag(alpha) S + beta k v^T and o = S_new^T q, on
    non-square states (catches a transposed operand or a dropped term)."""
    rng = np.random.default_rng(8)
    for dk, dv in ((3, 2), (2, 4), (4, 4)):
        for _ in range(5):
            S = rng.normal(size=(dk, dv))
            alpha = rng.uniform(0.2, 1.0, size=dk)
            beta = rng.uniform(0, 1)
            k, v, q = rng.normal(size=dk), rng.normal(size=dv), rng.normal(size=dk)
            Sf = [[_frac(S[i, j]) for j in range(dv)] for i in range(dk)]
            af, kf, vf, qf, bf = ([_frac(t) for t in alpha], [_frac(t) for t in k],
                                  [_frac(t) for t in v], [_frac(t) for t in q], _frac(beta))
            DS = [[af[i] * Sf[i][j] for j in range(dv)] for i in range(dk)]
            M = [[(1 if i == m else 0) - bf * kf[i] * kf[m] for m in range(dk)] for i in range(dk)]
            Snew = [[sum(M[i][m] * DS[m][j] for m in range(dk)) + bf * kf[i] * vf[j]
                     for j in range(dv)] for i in range(dk)]
            onew = [sum(Snew[i][j] * qf[i] for i in range(dk)) for j in range(dv)]
            S2, o, _ = oracle_mod.delta_step(S, alpha, beta, k, v, q)
            exact = np.array([[float(x) for x in row] for row in Snew])
            assert np.allclose(S2, exact, rtol=1e-13, atol=1e-14)
            assert np.allclose(o, [float(x) for x in onew], rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------- full layer

def _identity_conv(wl):
    w = np.zeros_like(wl.arrays["conv_w"])
    w[:, wl.K - 1] = 1.0
    wl.arrays["conv_w"] = w


def test_layer_reduces_to_linear_attention(oracle_mod):
    """alpha = 1, zero initial state, mutually orthogonal unit keys: the delta
    rule never erases anything, so o_t = sum_{s<=t} beta_s v'_s (k_s . q_t),
    plain (beta-weighted) linear attention."""
    T, d = 8, 8
    wl = W.make_workload("la", 11, [T], H=1, d=d, K=4, io_dtype=W.F32,
                         gate_mode=W.SOFTPLUS, init_state="zero")
    wl.l2_eps = 0.0
    _identity_conv(wl)
    a = wl.arrays
    a["A_log"][:] = -1000.0                      # exp(A_log) = 0: alpha = 1
    perm = np.random.default_rng(0).permutation(d)
    a["k"][:] = 0.0
    for t in range(T):
        a["k"][t, 0, perm[t]] = 3.0              # silu(3) e_perm -> unit basis key
    res = oracle_mod.forward(wl)
    qh = np.stack([oracle_mod.l2norm([oracle_mod.silu(x) for x in a["q"][t, 0]], 0.0) for t in range(T)])
    vv = np.array([[oracle_mod.silu(x) for x in a["v"][t, 0]] for t in range(T)])
    beta = np.array([oracle_mod.sigmoid(a["b"][t, 0]) for t in range(T)])
    keys = np.eye(d)[perm[:T]]
    for t in range(T):
        expect = sum(beta[s] * vv[s] * (keys[s] @ qh[t]) for s in range(t + 1))
        assert np.allclose(res["out"][t, 0], expect, rtol=1e-12, atol=1e-14)


def test_layer_beta_zero_freezes_writes(oracle_mod):
    """beta = 0: the state only decays, S_T = Diag(prod_t alpha_t) S_0, and each
    output reads the decayed initial state."""
    T, d = 9, 8
    wl = W.make_workload("b0", 12, [T], H=2, d=d, K=3, io_dtype=W.F32,
                         gate_mode=W.SAFE, lower_bound=-2.0, init_state="random")
    a = wl.arrays
    a["b"][:] = -1000.0                          # sigmoid = 0 exactly
    res = oracle_mod.forward(wl)
    for h in range(2):
        la = np.array([[oracle_mod.log_alpha(W.SAFE, -2.0, a["A_log"][h], a["f"][t, h, i], a["dt_bias"][h, i])
                        for i in range(d)] for t in range(T)])
        S0 = a["rec_state"][0, h].astype(np.float64)
        assert np.allclose(res["rec_state"][0, h], np.exp(la.sum(0))[:, None] * S0, rtol=1e-12)
        cw = a["conv_w"].astype(np.float64)
        hist = a["conv_state"][0].astype(np.float64)
        x = np.concatenate([a["q"][:, h, :], a["k"][:, h, :], a["v"][:, h, :]], axis=1).astype(np.float64)
        chans = np.concatenate([np.arange(h * d, h * d + d)])
        pre = oracle_mod.conv1d(x[:, :d], hist[:, chans], cw[chans])
        for t in range(T):
            qh = oracle_mod.l2norm([oracle_mod.silu(z) for z in pre[t]], wl.l2_eps)
            St = np.exp(la[:t + 1].sum(0))[:, None] * S0
            assert np.allclose(res["out"][t, h], St.T @ qh, rtol=1e-11, atol=1e-14)


def test_layer_unit_key_overwrite(oracle_mod):
    """alpha = 1, beta = 1 and a unit basis key on the last row: after the row,
    row i of the state holds that row's activated value exactly."""
    d = 8
    wl = W.make_workload("ow", 13, [5], H=1, d=d, K=4, io_dtype=W.F32,
                         gate_mode=W.SOFTPLUS, init_state="random")
    wl.l2_eps = 0.0
    _identity_conv(wl)
    a = wl.arrays
    a["A_log"][:] = -1000.0
    a["b"][:] = 1000.0
    a["k"][4, 0, :] = 0.0
    a["k"][4, 0, 5] = 2.0
    res = oracle_mod.forward(wl)
    vv = np.array([oracle_mod.silu(x) for x in a["v"][4, 0]])
    assert np.allclose(res["rec_state"][0, 0, 5], vv, rtol=1e-14, atol=1e-15)


CHUNK_CASES = [(T, d, mode, init) for T in (1, 15, 16, 17, 63, 64, 65, 130)
               for d in (8, 32) for mode in (W.SOFTPLUS, W.SAFE) for init in ("zero", "random")]


@pytest.mark.parametrize("T,d,mode,init", CHUNK_CASES)
def test_chunked_equals_serial(oracle_mod, T, d, mode, init):
    """The chunked WY/UT form (chunks restart at each segment's first row)
    reaches the serial recurrence's result."""
    wl = W.make_workload("ch", 100 + T + d, [T, max(T // 3, 1)], H=2, d=d, K=4,
                         io_dtype=W.F32, gate_mode=mode, lower_bound=-5.0,
                         out_gate=True, init_state=init)
    ser = oracle_mod.forward(wl)
    for C in (16, 64):
        ch = oracle_mod.forward(wl, chunk=C)
        for key in ("out", "rec_state"):
            ref = ser[key]
            err = np.linalg.norm(ch[key] - ref) / max(np.linalg.norm(ref), 1e-300)
            assert err < 1e-11, (key, C, err)
        assert np.array_equal(ch["conv_state"], ser["conv_state"])


def test_zero_length_sequences_leave_state(oracle_mod):
    wl = W.make_workload("z", 21, [0, 5, 0], H=2, d=8, K=4, io_dtype=W.F32,
                         gate_mode=W.SAFE, init_state="random")
    res = oracle_mod.forward(wl)
    for s in (0, 2):
        assert np.array_equal(res["rec_state"][s], wl.arrays["rec_state"][s])
        assert np.array_equal(res["conv_state"][s], wl.arrays["conv_state"][s])
    assert not np.array_equal(res["rec_state"][1], wl.arrays["rec_state"][1])


def test_prompt_cut_invariance(oracle_mod):
    """Running rows [0, a) then [a, T) with the carried states gives the same
    bits as one call over [0, T)."""
    T, cut = 40, 17
    wl = W.make_workload("cut", 22, [T], H=2, d=8, K=4, io_dtype=W.F32,
                         gate_mode=W.SAFE, out_gate=True, init_state="random")
    full = oracle_mod.forward(wl)
    first = W.make_workload("cut", 22, [T], H=2, d=8, K=4, io_dtype=W.F32,
                            gate_mode=W.SAFE, out_gate=True, init_state="random")
    for part, (t0, t1) in enumerate(((0, cut), (cut, T))):
        sub = W.Workload(**{**first.__dict__, "arrays": {}})
        sub.cu_seqlens = np.array([0, t1 - t0], dtype=np.int32)
        for nm in ("q", "k", "v", "f", "b", "g"):
            sub.arrays[nm] = wl.arrays[nm][t0:t1]
        for nm in ("A_log", "dt_bias", "conv_w", "norm_w"):
            sub.arrays[nm] = wl.arrays[nm]
        if part == 0:
            sub.arrays["conv_state"], sub.arrays["rec_state"] = wl.arrays["conv_state"], wl.arrays["rec_state"]
            r0 = oracle_mod.forward(sub)
        else:
            sub.arrays["conv_state"], sub.arrays["rec_state"] = r0["conv_state"], r0["rec_state"]
            r1 = oracle_mod.forward(sub)
    assert np.array_equal(np.concatenate([r0["out"], r1["out"]]), full["out"])
    assert np.array_equal(r1["rec_state"], full["rec_state"])
    assert np.array_equal(r1["conv_state"], full["conv_state"])


def test_heads_and_sequences_are_independent(oracle_mod):
    """Each (sequence, head) unit equals the same unit run alone: catches a
    wrong channel offset in the q|k|v conv layout or a state index mix-up."""
    wl = W.make_workload("ind", 23, [7, 3, 11], H=3, d=8, K=4, io_dtype=W.F32,
                         gate_mode=W.SOFTPLUS, out_gate=True, init_state="random")
    full = oracle_mod.forward(wl)
    cd = wl.conv_dim
    for s in range(3):
        for h in range(3):
            sub = W.head_slice(wl, s, h)
            r = oracle_mod.forward(sub)
            t0, t1 = wl.cu_seqlens[s], wl.cu_seqlens[s + 1]
            assert np.array_equal(r["out"][:, 0], full["out"][t0:t1, h])
            assert np.array_equal(r["rec_state"][0, 0], full["rec_state"][s, h])
            chans = np.concatenate([np.arange(h * 8, h * 8 + 8), 24 + np.arange(h * 8, h * 8 + 8),
                                    48 + np.arange(h * 8, h * 8 + 8)])
            assert cd == 72
            assert np.array_equal(r["conv_state"][0], full["conv_state"][s][:, chans])


def test_epilogue_composes(oracle_mod):
    """The gated output norm applied to the raw outputs equals the layer run
    with the output gate."""
    wl = W.make_workload("ep", 24, [12], H=2, d=16, K=4, io_dtype=W.F32,
                         gate_mode=W.SAFE, out_gate=True, init_state="random")
    gated = oracle_mod.forward(wl)
    wl.has_out_gate = False
    raw = oracle_mod.forward(wl)
    for t in range(12):
        for h in range(2):
            y = oracle_mod.gated_rmsnorm(raw["out"][t, h], wl.arrays["g"][t, h], wl.arrays["norm_w"], wl.norm_eps)
            assert np.allclose(gated["out"][t, h], y, rtol=1e-14, atol=1e-15)


def test_state_transfer_decomposition(oracle_mod):
    """What the affine state scan relies on, pinned on the oracle alone: the
    rows of a segment map any start state S linearly, S_out = M S + N and
    o = obar + psi S, where (N, obar) come from S = 0 and (M, psi) from the
    identity with the values v set to zero; outputs before the gated norm."""
    from linear_attention_serving_kda_gb300 import workloads as W

    wl = W.make_workload("xfer", 77, [23], H=1, d=8, K=3, io_dtype=W.F32, gate_mode=W.SOFTPLUS,
                         lower_bound=-5.0, out_gate=False, init_state="random")
    S = wl.arrays["rec_state"][0, 0].astype(np.float64)
    full = oracle_mod.forward(wl)
    zero = dict(wl.arrays)
    zero["rec_state"] = np.zeros_like(wl.arrays["rec_state"])
    r0 = oracle_mod.forward(wl, arrays=zero)
    ident = dict(zero)
    ident["rec_state"] = np.eye(8)[None, None].astype(np.float64)
    ident["v"] = np.zeros_like(wl.arrays["v"])
    # v = 0 must not change the conv taps of the other channels: v's own
    # channels see zero rows, and its carried history is zeroed too
    cs = wl.arrays["conv_state"].copy()
    cs[:, :, 2 * 8:] = 0.0
    ident["conv_state"] = cs
    rm = oracle_mod.forward(wl, arrays=ident)
    M, N = rm["rec_state"][0, 0], r0["rec_state"][0, 0]
    np.testing.assert_allclose(full["rec_state"][0, 0], M @ S + N, rtol=0, atol=1e-12)
    np.testing.assert_allclose(full["out"][:, 0], r0["out"][:, 0] + rm["out"][:, 0] @ S, rtol=0, atol=1e-12)
