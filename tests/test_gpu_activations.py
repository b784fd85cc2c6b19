"""The device activations every kernel shares, against their error bounds.

e^x is 2^(x log2 e) on the special-function unit: the product x log2 e is
rounded to fp32 (relative error 2^-24, and log2 e itself to 2^-24), which
moves the result by up to |x| 2^-23 relatively; the base-2 exponential adds
a few ulp.  1/x is the SFU's reciprocal (about an ulp).  Sigmoid and SiLU
compose them with one rounded add (and, for SiLU, one rounded multiply).
Bounds below allow 2^-21 for each SFU result, generous against those
figures and far below what a wrong constant, sign or operand would give.
"""
import numpy as np
import pytest
import torch

from linear_attention_serving_kda_gb300 import kda as K

pytestmark = pytest.mark.gpu

SFU = 2.0 ** -21


def _run(which, x):
    xd = torch.from_numpy(x.astype(np.float32)).cuda()
    yd = torch.empty_like(xd)
    assert K.kda_debug_activations(which, xd, yd, xd.numel()) == K.KDA_OK
    torch.cuda.synchronize()
    return yd.cpu().numpy().astype(np.float64), xd.cpu().numpy().astype(np.float64)


def _rel(y, ref):
    return np.abs(y - ref) / np.abs(ref)


def test_exp(cuda_lib):
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.uniform(-80, 80, 200_000), np.linspace(-1, 1, 4097), [0.0, 1.0, -1.0, 80.0, -80.0]])
    y, x = _run(K.KDA_ACT_EXP, x)
    ref = np.exp(x)
    assert np.all(_rel(y, ref) <= SFU + np.abs(x) * 2.0 ** -23)
    assert y[x == 0.0][0] == 1.0
    # far below the fp32 normal range the result is 0 (subnormals flushed), never negative
    yt, _ = _run(K.KDA_ACT_EXP, np.array([-90.0, -200.0, -1e30]))
    assert np.all(yt == 0.0)


def test_reciprocal(cuda_lib):
    rng = np.random.default_rng(8)
    x = np.concatenate([rng.uniform(1e-3, 1e3, 100_000), -rng.uniform(1e-3, 1e3, 100_000), [1.0, 2.0, 0.5]])
    y, x = _run(K.KDA_ACT_RCP, x)
    assert np.all(_rel(y, 1.0 / x) <= SFU)
    assert np.array_equal(y[-3:], [1.0, 0.5, 2.0])


def test_sigmoid_and_silu(cuda_lib):
    rng = np.random.default_rng(9)
    x = np.concatenate([rng.normal(0, 4, 200_000), np.linspace(-30, 30, 6001)])
    s, xs = _run(K.KDA_ACT_SIGMOID, x)
    ref = 1.0 / (1.0 + np.exp(-xs))
    bound = 2 * SFU + 2.0 ** -23 + np.abs(xs) * 2.0 ** -23
    assert np.all(_rel(s, ref) <= bound)
    assert np.all((s >= 0) & (s <= 1))
    u, xu = _run(K.KDA_ACT_SILU, x)
    nz = xu != 0
    assert np.all(_rel(u[nz], xu[nz] * ref[nz]) <= bound[nz] + 2.0 ** -24)
    assert np.all(u[~nz] == 0)
    # saturation: sigmoid -> 0 and 1 without NaN; SiLU of a large negative input -> -0
    sat, _ = _run(K.KDA_ACT_SIGMOID, np.array([-200.0, 200.0]))
    assert sat[0] == 0.0 and sat[1] == 1.0
    neg, _ = _run(K.KDA_ACT_SILU, np.array([-200.0]))
    assert neg[0] == 0.0


def test_activations_reject_before_launch(cuda_lib):
    x = torch.zeros(8, device="cuda")
    assert K.kda_debug_activations(4, x, x, 8) == K.KDA_ERR_INVALID_ARGUMENT
    assert K.kda_debug_activations(K.KDA_ACT_EXP, x, x, -1) == K.KDA_ERR_INVALID_ARGUMENT
    assert K.kda_debug_activations(K.KDA_ACT_EXP, None, x, 8) == K.KDA_ERR_INVALID_ARGUMENT
    assert K.kda_debug_activations(K.KDA_ACT_EXP, None, None, 0) == K.KDA_OK
