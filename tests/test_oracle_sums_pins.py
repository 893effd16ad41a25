"""Pins of the oracle's per-channel output sums (oracle.channel_sums), the
reductions the fused epilogue produces:
    s1[c] = sum over n,h,w of out[n,h,w,c]
    s2[c] = sum over n,h,w with x > 0 of out[n,h,w,c] * x[n,h,w,c]
with out the (ReLU-backward gated) dgrad output.  They are pinned by
  * the adjoint identity through the oracle's forward convolution, which is
    separate code: the sum of channel c of dgrad(dY, W) over all pixels is
    <dY, conv_fwd(E_c, W)> for E_c the image that is 1 in channel c and 0
    elsewhere; gated by x, E_c becomes (x > 0) E_c for s1 and relu(x) E_c for
    s2;
  * a case worked by hand (tests/golden/channel_sums_1x1.json);
  * the rule that masked positions add nothing to s2, NaN in x included.
"""
import json
import os

import numpy as np
import pytest

import oracle
from implicit_gemm_dgrad_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "channel_sums_1x1.json")

GEOMS = [  # N, H, W, C, K, R, S, stride, pad, dil
    (2, 7, 6, 5, 3, 3, 3, 1, 1, 1),
    (1, 9, 8, 4, 6, 3, 3, 2, 1, 1),
    (2, 8, 9, 3, 4, 1, 1, 2, 0, 1),
    (1, 10, 7, 4, 3, 3, 2, 2, 2, 2),
    (2, 6, 6, 6, 5, 2, 2, 3, 0, 1),
]


def _inputs(g, seed):
    N, H, W, C, K, R, S, st, pad, dil = g
    P, Q = oracle.out_extent(H, R, st, pad, dil), oracle.out_extent(W, S, st, pad, dil)
    rng = np.random.default_rng(seed)
    dY = rng.standard_normal((N, P, Q, K))
    Wt = rng.standard_normal((K, R, S, C))
    x = rng.standard_normal((N, H, W, C))
    return dY, Wt, x


@pytest.mark.parametrize("g", GEOMS)
def test_s1_is_the_adjoint_of_a_channel_of_ones(g):
    N, H, W, C, K, R, S, st, pad, dil = g
    dY, Wt, _ = _inputs(g, 1)
    out = oracle.dgrad(dY, Wt, H, W, st, pad, dil)
    s1, s2, a1, _ = oracle.channel_sums(out)
    assert s2 is None
    for c in range(C):
        E = np.zeros((N, H, W, C))
        E[..., c] = 1.0
        expect = float(np.sum(dY * oracle.conv_fwd(E, Wt, st, pad, dil)))
        assert abs(s1[c] - expect) <= 1e-10 * max(1.0, a1[c])


@pytest.mark.parametrize("g", GEOMS)
def test_gated_sums_are_adjoints_of_masked_and_relu_images(g):
    N, H, W, C, K, R, S, st, pad, dil = g
    dY, Wt, x = _inputs(g, 2)
    out = oracle.dgrad(dY, Wt, H, W, st, pad, dil, x=x)
    s1, s2, a1, a2 = oracle.channel_sums(out, x)
    for c in range(C):
        E = np.zeros((N, H, W, C))
        E[..., c] = (x[..., c] > 0).astype(np.float64)
        assert abs(s1[c] - float(np.sum(dY * oracle.conv_fwd(E, Wt, st, pad, dil)))) <= 1e-10 * max(1.0, a1[c])
        E[..., c] = np.maximum(x[..., c], 0.0)
        assert abs(s2[c] - float(np.sum(dY * oracle.conv_fwd(E, Wt, st, pad, dil)))) <= 1e-10 * max(1.0, a2[c])


def test_hand_worked_case():
    d = json.load(open(GOLDEN))
    g = d["geometry"]
    dY = synth.to_bits(np.array(d["dY_nhwk"], np.float32).reshape(g["N"], g["H"], g["W"], g["K"]), "bf16")
    Wt = synth.to_bits(np.array(d["W_krsc"], np.float32).reshape(g["K"], g["R"], g["S"], g["C"]), "bf16")
    x = synth.to_bits(np.array(d["x_nhwc"], np.float32).reshape(g["N"], g["H"], g["W"], g["C"]), "bf16")
    out = oracle.dgrad(dY, Wt, g["H"], g["W"], g["stride"], g["pad"], g["dil"], x=x, dtype="bf16")
    assert out.reshape(-1).tolist() == d["out_nhwc"]
    s1, s2, a1, a2 = oracle.channel_sums(out, x, dtype="bf16")
    assert s1.tolist() == d["s1"] and s2.tolist() == d["s2"]
    assert a1.tolist() == [25.0, 14.0] and a2.tolist() == [32.0, 42.0]


def test_masked_positions_add_nothing_to_s2_even_nan():
    out = np.array([[1.0, 2.0], [0.0, 0.0], [3.0, 4.0]])
    # pixel 1 is masked in both channels: x = NaN and -0.0 (its out is +0.0, as the gate leaves it)
    x = synth.to_bits(np.array([[1.0, 0.5], [0.0, 0.0], [2.0, 1.0]], np.float32), "bf16")
    x[1, 0], x[1, 1] = 0x7FC0, 0x8000
    s1, s2, _, _ = oracle.channel_sums(out, x, dtype="bf16")
    assert s1.tolist() == [4.0, 6.0] and s2.tolist() == [7.0, 5.0]
