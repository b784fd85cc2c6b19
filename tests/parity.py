"""Comparison helpers for GPU-vs-oracle parity.

Tolerances for floating-point results (fp32 state, bf16 or fp32 rows):
relative L2 over the whole tensor <= 2e-3, and max-abs error <= 5e-3 times
the RMS of the oracle tensor.  Conv states are pure copies and must match
exactly.
"""
import numpy as np

from linear_attention_serving_kda_gb300 import workloads as W

REL_L2 = 2e-3
MAX_ABS_RMS = 5e-3
BF16_SLACK_RMS = 1e-3

# (what, rel L2, max-abs / RMS) of every comparison, printed at the end of the run
RECORD = []
# the running test's name (set by a fixture), prefixed to each record
CURRENT = [""]


def to_np(t):
    import torch

    if t.dtype == torch.bfloat16:
        return t.detach().float().cpu().numpy()
    return t.detach().cpu().numpy()


def rel_l2(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return np.linalg.norm(x - ref) / (den if den > 0 else 1.0)


def assert_close(x, ref, what="", rel=REL_L2, maxabs_rms=MAX_ABS_RMS):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert x.shape == ref.shape, (what, x.shape, ref.shape)
    assert np.all(np.isfinite(x)), f"{what}: non-finite values"
    e = rel_l2(x, ref)
    rms = np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    m = np.max(np.abs(x - ref)) if ref.size else 0.0
    RECORD.append((f"{CURRENT[0]}: {what}", e, m / max(rms, 1e-30)))
    assert e <= rel, f"{what}: rel L2 {e:.3e} > {rel:.1e}"
    assert m <= maxabs_rms * max(rms, 1e-30), f"{what}: max abs {m:.3e} > {maxabs_rms:.0e} * RMS {rms:.3e}"
    return e, m / max(rms, 1e-30)


def assert_bf16_within_one_ulp(x_bf16, ref):
    """bf16 outputs: within one bf16 ulp of the oracle rounded to nearest even,
    plus 1e-3 x RMS(oracle) for the fp32 path's own error (which, for outputs
    near zero, spans many ulps at their own magnitude)."""
    x = np.asarray(x_bf16, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    r = W.bf16_bits_to_f32(W.round_to_bf16_bits(ref.astype(np.float32))).astype(np.float64)
    mag = np.maximum(np.maximum(np.abs(x), np.abs(r)), 1e-30)
    ulp = np.exp2(np.floor(np.log2(mag)) - 7)
    rms = np.sqrt(np.mean(ref * ref))
    bad = np.abs(x - r) > ulp + BF16_SLACK_RMS * rms
    RECORD.append((f"{CURRENT[0]}: bf16 out: max |x - RNE(ref)| / ulp", float(np.max(np.abs(x - r) / ulp)), 0.0))
    assert not bad.any(), f"{bad.sum()} bf16 outputs more than one ulp (+1e-3 RMS) from RNE(oracle)"


def gather_rows(wl, ranges, name=None):
    """A workload whose sequence s holds rows ranges[s] = (start, stop) of wl
    (pure data movement; parameters and initial states unchanged)."""
    idx = np.concatenate([np.arange(a, b) for a, b in ranges]) if ranges else np.zeros(0, int)
    lens = [b - a for a, b in ranges]
    sub = W.Workload(**{**wl.__dict__, "arrays": {}})
    sub.name = name or wl.name + "[gathered]"
    sub.cu_seqlens = np.zeros(len(lens) + 1, dtype=np.int32)
    sub.cu_seqlens[1:] = np.cumsum(lens)
    for nm, a in wl.arrays.items():
        if nm in ("q", "k", "v", "f", "b", "g"):
            sub.arrays[nm] = np.ascontiguousarray(a[idx])
        else:
            sub.arrays[nm] = a
    return sub
