"""Pins of the oracle's back-to-back dgrad (oracle.dgrad_fused) and of the
rounding it applies to the intermediate g (oracle.round_to):

* round_to for fp16 equals numpy's float64 -> float16 conversion on values
  across the whole range (subnormals, overflow, exact ties); for bf16 every
  result is the nearest bf16 value, ties going to the even one, checked
  against the neighbours of the result and on exact midpoints;
* in double precision the two dgrads compose to one: dgrad_1x1(dgrad(dY, W2),
  W1) = dgrad(dY, W2') with W2'[k,r,s,c1] = sum over c2 of W2[k,r,s,c2] *
  W1[c2,0,0,c1] (the chain rule), to 1e-12;
* with an identity 1x1 filter dX1 is g itself, bit for bit after rounding.
"""
import numpy as np
import pytest

import oracle
from implicit_gemm_dgrad_gb300 import synth


def test_fp16_rounding_matches_numpy():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-9, 6, 4000),
                        [0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 2 ** -24, 2 ** -25, 3 * 2 ** -26,
                         2 ** -26, 1 + 2 ** -11, 1 + 3 * 2 ** -11, np.inf, -np.inf]])
    got = oracle.round_to(x, "f16")
    with np.errstate(over="ignore"):
        np.testing.assert_array_equal(got, x.astype(np.float16).view(np.uint16))
    assert (oracle.round_to(np.array([np.nan]), "f16")[0] & 0x7C00) == 0x7C00


def test_bf16_rounding_is_nearest_ties_to_even():
    rng = np.random.default_rng(2)
    x = rng.standard_normal(3000) * 10.0 ** rng.integers(-30, 30, 3000)
    b = oracle.round_to(x, "bf16").astype(np.int64)
    dec = lambda bits: np.array([oracle.bf16_to_double(int(v) & 0xFFFF) for v in bits])  # noqa: E731
    here, up, down = dec(b), dec(b + 1), dec(b - 1)
    err = np.abs(x - here)
    assert np.all(err <= np.abs(x - up)) and np.all(err <= np.abs(x - down))
    # exact midpoints between neighbours go to the even pattern; a hair above goes up
    lo = rng.integers(0x0080, 0x7F00, 500)
    mid = (dec(lo) + dec(lo + 1)) / 2
    r = oracle.round_to(mid, "bf16").astype(np.int64)
    assert np.all(r == np.where(lo % 2 == 0, lo, lo + 1))
    r2 = oracle.round_to(np.nextafter(mid, np.inf), "bf16").astype(np.int64)
    assert np.all(r2 == lo + 1)
    # the double rounding trap: just above a bf16 tie, but a tie in float32
    assert oracle.round_to(np.array([1 + 2 ** -8 + 2 ** -40]), "bf16")[0] == 0x3F81
    assert oracle.round_to(np.array([1e-40, 3.4e38, -0.0]), "bf16").tolist() == [0x0001, 0x7F80, 0x8000]


@pytest.mark.parametrize("geom", [(2, 7, 6, 5, 8, 6, 3, 3, 1, 1), (1, 9, 8, 3, 4, 7, 3, 2, 2, 2),
                                  (2, 5, 5, 4, 6, 2, 1, 1, 0, 1)])
def test_fused_is_the_composed_dgrad_in_double(geom):
    N, H, W, C1, C2, K2, R2, S2, pad2, dil2 = geom
    P, Q = oracle.out_extent(H, R2, 1, pad2, dil2), oracle.out_extent(W, S2, 1, pad2, dil2)
    rng = np.random.default_rng(3)
    dY = rng.standard_normal((N, P, Q, K2))
    W2 = rng.standard_normal((K2, R2, S2, C2))
    W1 = rng.standard_normal((C2, 1, 1, C1))
    dX1, g = oracle.dgrad_fused(dY, W2, None, W1, H, W, pad2, dil2, act=None)
    W2c = np.einsum("krsm,mc->krsc", W2, W1[:, 0, 0, :])
    ref = oracle.dgrad(dY, W2c, H, W, 1, pad2, dil2)
    np.testing.assert_allclose(dX1, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    np.testing.assert_array_equal(g, oracle.dgrad(dY, W2, H, W, 1, pad2, dil2))


@pytest.mark.parametrize("act", ["relu", "gelu", None])
def test_identity_1x1_returns_the_rounded_gated_intermediate(act):
    rng = np.random.default_rng(4)
    N, H, W, C2, K2 = 2, 6, 7, 8, 16
    dY = synth.to_bits(rng.standard_normal((N, H, W, K2)).astype(np.float32), "bf16")
    W2 = synth.to_bits((0.2 * rng.standard_normal((K2, 3, 3, C2))).astype(np.float32), "bf16")
    x2 = synth.to_bits(rng.standard_normal((N, H, W, C2)).astype(np.float32), "bf16") if act else None
    eye = synth.to_bits(np.eye(C2, dtype=np.float32).reshape(C2, 1, 1, C2), "bf16")
    dX1, g = oracle.dgrad_fused(dY, W2, x2, eye, H, W, 1, 1, dtype="bf16", act=act or "relu")
    assert g.dtype == np.uint16
    np.testing.assert_array_equal(dX1, synth.bits_to_f32(g, "bf16").astype(np.float64))
    ref = oracle.dgrad(dY, W2, H, W, 1, 1, 1, x=x2, dtype="bf16", act=act or "relu")
    np.testing.assert_array_equal(g, oracle.round_to(ref, "bf16"))
