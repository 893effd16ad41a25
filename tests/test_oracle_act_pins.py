"""Pins of the oracle's activation-backward epilogues for GELU (erf form) and
SiLU: out = dX * f'(x), x the activation's saved input.

* f'(x) (oracle.act_grad) against central finite differences of f itself,
  written here from the definitions f(x) = x * (1 + erf(x / sqrt 2)) / 2 and
  f(x) = x / (1 + exp(-x)) with Python's math module;
* known values: f'(0) = 1/2 for both; f'(x) -> 1 for large x, -> 0 for very
  negative x; both derivatives are negative below a crossing near x = -0.75
  (GELU) and x = -1.28 (SiLU);
* the gated dgrad equals the ungated one times f'(x) element by element.
"""
import math

import numpy as np
import pytest

import oracle
from implicit_gemm_dgrad_gb300 import synth


def gelu(x):
    return x * 0.5 * (1.0 + math.erf(x / math.sqrt(2.0)))


def silu(x):
    return x / (1.0 + math.exp(-x))


F = {"gelu": gelu, "silu": silu}


@pytest.mark.parametrize("act", ["gelu", "silu"])
def test_derivative_matches_finite_differences(act):
    f = F[act]
    h = 1e-5
    for x in np.linspace(-8.0, 8.0, 321):
        fd = (f(x + h) - f(x - h)) / (2 * h)
        assert abs(oracle.act_grad(x, act) - fd) <= 1e-8, (act, x)


def test_known_values():
    assert oracle.act_grad(0.0, "gelu") == 0.5 and oracle.act_grad(0.0, "silu") == 0.5
    assert abs(oracle.act_grad(12.0, "gelu") - 1.0) < 1e-12 and abs(oracle.act_grad(-12.0, "gelu")) < 1e-12
    assert abs(oracle.act_grad(40.0, "silu") - 1.0) < 1e-12 and abs(oracle.act_grad(-40.0, "silu")) < 1e-12
    assert oracle.act_grad(-1.0, "gelu") < 0 < oracle.act_grad(-0.5, "gelu")
    assert oracle.act_grad(-1.5, "silu") < 0 < oracle.act_grad(-1.0, "silu")


@pytest.mark.parametrize("act", ["gelu", "silu"])
def test_gated_dgrad_is_dgrad_times_derivative(act):
    rng = np.random.default_rng(5)
    N, H, W, C, K = 2, 7, 6, 8, 16
    dY = synth.to_bits(rng.standard_normal((N, H, W, K)).astype(np.float32), "bf16")
    Wt = synth.to_bits((0.2 * rng.standard_normal((K, 3, 3, C))).astype(np.float32), "bf16")
    x = synth.to_bits((2.0 * rng.standard_normal((N, H, W, C))).astype(np.float32), "bf16")
    plain = oracle.dgrad(dY, Wt, H, W, 1, 1, 1, dtype="bf16")
    gated = oracle.dgrad(dY, Wt, H, W, 1, 1, 1, x=x, dtype="bf16", act=act)
    xd = synth.bits_to_f32(x, "bf16").astype(np.float64)
    d = np.vectorize(lambda v: oracle.act_grad(v, act))(xd)
    np.testing.assert_allclose(gated, plain * d, rtol=1e-15, atol=0)
    pix = np.array([[0, 0, 0], [1, 6, 5], [1, 3, 2]], np.int32)
    sel = oracle.dgrad_pixels(dY, Wt, H, W, pix, 1, 1, 1, x=x, dtype="bf16", act=act)
    np.testing.assert_array_equal(sel, gated[pix[:, 0], pix[:, 1], pix[:, 2]])
