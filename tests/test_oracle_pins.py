"""Pins for the CPU oracle: each checks it against something other than itself.

* brute force: the dense forward-convolution matrix, built here from the
  forward definition, transposed and applied to dY;
* the adjoint identity <conv_fwd(x, W), dY> = <x, dgrad(dY, W)>;
* closed forms: 1x1 stride-1 = matrix product, impulse response, identity filter;
* hand-worked fixtures under tests/golden/;
* integer inputs, where the result is exact;
* an independent library routine (torch.nn.grad.conv2d_input in float64, CPU);
* the fp16/bf16 decoders against numpy's conversions, bit pattern by bit pattern.

A plausible mistake in the oracle -- a sign in the pad, a swapped r/s, a stride
applied on the wrong side, a dropped tap -- fails several of these.
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle
from implicit_gemm_dgrad_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def out_ext(n, f, s, p, d):
    return (n + 2 * p - d * (f - 1) - 1) // s + 1


def forward_matrix(N, H, W, C, K, R, S, stride, pad, dil):
    """Dense matrix A with vec(y) = A vec(x) for the forward cross-correlation
    y[n,p,q,k] = sum_{r,s,c} x[n, p*stride-pad+r*dil, q*stride-pad+s*dil, c] W[k,r,s,c].
    Returned as a function of W: entries are (row, col, weight index)."""
    P, Q = out_ext(H, R, stride, pad, dil), out_ext(W, S, stride, pad, dil)
    rows, cols, widx = [], [], []
    for n, p, q, k in itertools.product(range(N), range(P), range(Q), range(K)):
        row = ((n * P + p) * Q + q) * K + k
        for r, s in itertools.product(range(R), range(S)):
            h = p * stride - pad + r * dil
            w = q * stride - pad + s * dil
            if 0 <= h < H and 0 <= w < W:
                for c in range(C):
                    rows.append(row)
                    cols.append(((n * H + h) * W + w) * C + c)
                    widx.append(((k * R + r) * S + s) * C + c)
    return P, Q, np.array(rows), np.array(cols), np.array(widx)


def brute_force_dgrad(dY, Wt, H, W, stride, pad, dil, dtype=object):
    N, P, Q, K = dY.shape
    _, R, S, C = Wt.shape
    P2, Q2, rows, cols, widx = forward_matrix(N, H, W, C, K, R, S, stride, pad, dil)
    assert (P2, Q2) == (P, Q)
    A = np.zeros((N * P * Q * K, N * H * W * C), dtype=dtype)
    np.add.at(A, (rows, cols), Wt.reshape(-1)[widx])
    return (A.T @ dY.reshape(-1)).reshape(N, H, W, C)


SWEEP = []
_rng = np.random.default_rng(7)
for stride, pad, dil, R, S in itertools.product((1, 2, 3), (0, 1, 2), (1, 2), (1, 2, 3), (1, 2, 3)):
    H, W = int(_rng.integers(3, 10)), int(_rng.integers(3, 10))
    if out_ext(H, R, stride, pad, dil) <= 0 or out_ext(W, S, stride, pad, dil) <= 0:
        continue
    SWEEP.append((int(_rng.integers(1, 3)), H, W, int(_rng.integers(1, 6)),
                  int(_rng.integers(1, 6)), R, S, stride, pad, dil))
# keep the brute-force sweep quick but spread over every (stride, pad, dil)
SWEEP_BF = [c for i, c in enumerate(SWEEP) if i % 3 == 0]


@pytest.mark.parametrize("case", SWEEP_BF, ids=lambda c: "N{}H{}W{}C{}K{}R{}S{}s{}p{}d{}".format(*c))
def test_brute_force_matrix(case):
    N, H, W, C, K, R, S, stride, pad, dil = case
    P, Q = out_ext(H, R, stride, pad, dil), out_ext(W, S, stride, pad, dil)
    rng = np.random.default_rng(hash(case) & 0xFFFF)
    dY = rng.standard_normal((N, P, Q, K))
    Wt = rng.standard_normal((K, R, S, C))
    ref = brute_force_dgrad(dY, Wt, H, W, stride, pad, dil, dtype=np.float64)
    got = oracle.dgrad(dY, Wt, H, W, stride, pad, dil)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("case", SWEEP, ids=lambda c: "N{}H{}W{}C{}K{}R{}S{}s{}p{}d{}".format(*c))
def test_adjoint_identity(case):
    N, H, W, C, K, R, S, stride, pad, dil = case
    P, Q = out_ext(H, R, stride, pad, dil), out_ext(W, S, stride, pad, dil)
    rng = np.random.default_rng(1000 + (hash(case) & 0xFFFF))
    x = rng.standard_normal((N, H, W, C))
    dY = rng.standard_normal((N, P, Q, K))
    Wt = rng.standard_normal((K, R, S, C))
    lhs = float(np.sum(oracle.conv_fwd(x, Wt, stride, pad, dil) * dY))
    rhs = float(np.sum(x * oracle.dgrad(dY, Wt, H, W, stride, pad, dil)))
    scale = float(np.sum(np.abs(x))) * float(np.sum(np.abs(dY))) * float(np.max(np.abs(Wt)))
    assert abs(lhs - rhs) <= 1e-10 * max(abs(lhs), 1e-3 * scale, 1.0)


def test_adjoint_identity_workload_shapes():
    """The identity at every benchmarked layer geometry (batch 1, channels cut to 8)."""
    from implicit_gemm_dgrad_gb300.workloads import ALL
    seen = set()
    rng = np.random.default_rng(3)
    for L in ALL:
        key = (L.H, L.W, L.R, L.S, L.stride, L.pad, L.dil)
        if key in seen:
            continue
        seen.add(key)
        C, K = 8, 8
        x = rng.standard_normal((1, L.H, L.W, C))
        dY = rng.standard_normal((1, L.P, L.Q, K))
        Wt = rng.standard_normal((K, L.R, L.S, C))
        lhs = float(np.sum(oracle.conv_fwd(x, Wt, L.stride, L.pad, L.dil) * dY))
        rhs = float(np.sum(x * oracle.dgrad(dY, Wt, L.H, L.W, L.stride, L.pad, L.dil)))
        assert abs(lhs - rhs) <= 1e-10 * max(abs(lhs), 1.0), L.name


def test_out_extent_matches_workloads():
    # 56, 3x3, stride 2, pad 1 -> 28; 56, 1x1, stride 2, pad 0 -> 28; same-padded 3x3 keeps size
    assert oracle.out_extent(56, 3, 2, 1, 1) == 28
    assert oracle.out_extent(56, 1, 2, 0, 1) == 28
    assert oracle.out_extent(14, 3, 1, 1, 1) == 14
    assert oracle.out_extent(7, 3, 2, 1, 1) == 4
    assert oracle.out_extent(2, 5, 1, 0, 1) == -1


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.mark.parametrize("name", ["gemm_1x1.json", "strided_3x3_s2_p1.json"])
def test_golden_hand_worked(name):
    g = _golden(name)
    geo = g["geometry"]
    N, H, W, C, K, R, S = (geo[k] for k in ("N", "H", "W", "C", "K", "R", "S"))
    P, Q = out_ext(H, R, geo["stride"], geo["pad"], geo["dil"]), out_ext(W, S, geo["stride"], geo["pad"], geo["dil"])
    dY = np.array(g["dY_nhwk"], np.float64).reshape(N, P, Q, K)
    Wt = np.array(g["W_krsc"], np.float64).reshape(K, R, S, C)
    got = oracle.dgrad(dY, Wt, H, W, geo["stride"], geo["pad"], geo["dil"])
    np.testing.assert_array_equal(got.reshape(-1), np.array(g["dX_nhwc"], np.float64))


def test_golden_relu_gate_special_values():
    g = _golden("relu_gate_special.json")
    geo = g["geometry"]
    dY = np.array([int(b, 16) for b in g["dY_f16_bits"]], np.uint16).reshape(1, 1, 8, 1)
    Wt = np.array([int(b, 16) for b in g["W_f16_bits"]], np.uint16).reshape(1, 1, 1, 1)
    x = np.array([int(b, 16) for b in g["x_f16_bits"]], np.uint16).reshape(1, 1, 8, 1)
    got = oracle.dgrad(dY, Wt, geo["H"], geo["W"], 1, 0, 1, x=x, dtype="f16").reshape(-1)
    np.testing.assert_array_equal(got, np.array(g["dX"]))
    is_pos_zero = (got == 0) & ~np.signbit(got)
    assert list(is_pos_zero) == g["dX_is_positive_zero"]


def test_1x1_stride1_is_gemm():
    rng = np.random.default_rng(11)
    N, H, W, C, K = 2, 5, 7, 24, 40
    dY = rng.standard_normal((N, H, W, K))
    Wt = rng.standard_normal((K, 1, 1, C))
    ref = dY.reshape(-1, K) @ Wt.reshape(K, C)
    got = oracle.dgrad(dY, Wt, H, W, 1, 0, 1)
    np.testing.assert_allclose(got.reshape(-1, C), ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("stride,pad,dil,R,S", [(1, 1, 1, 3, 3), (2, 1, 1, 3, 3), (2, 0, 1, 1, 1),
                                                (3, 2, 2, 3, 2), (2, 2, 1, 5, 3)])
def test_impulse_response(stride, pad, dil, R, S):
    """One-hot dY at (n,p,q,k): dX = W[k,r,s,:] at (p*stride-pad+r*dil, q*stride-pad+s*dil), else 0."""
    rng = np.random.default_rng(5)
    N, H, W, C, K = 2, 9, 8, 3, 4
    P, Q = out_ext(H, R, stride, pad, dil), out_ext(W, S, stride, pad, dil)
    Wt = rng.standard_normal((K, R, S, C))
    for (n, p, q, k) in [(0, 0, 0, 0), (1, P - 1, Q - 1, K - 1), (1, P // 2, 0, 2), (0, 0, Q // 2, 1)]:
        dY = np.zeros((N, P, Q, K))
        dY[n, p, q, k] = 1.0
        expect = np.zeros((N, H, W, C))
        for r in range(R):
            for s in range(S):
                h, w = p * stride - pad + r * dil, q * stride - pad + s * dil
                if 0 <= h < H and 0 <= w < W:
                    expect[n, h, w, :] += Wt[k, r, s, :]
        got = oracle.dgrad(dY, Wt, H, W, stride, pad, dil)
        np.testing.assert_array_equal(got, expect)


def test_identity_filter():
    """3x3, pad 1, stride 1, W[k,1,1,c] = delta_kc: dX = dY exactly."""
    rng = np.random.default_rng(9)
    N, H, W, C = 2, 6, 5, 7
    dY = rng.standard_normal((N, H, W, C))
    Wt = np.zeros((C, 3, 3, C))
    Wt[np.arange(C), 1, 1, np.arange(C)] = 1.0
    np.testing.assert_array_equal(oracle.dgrad(dY, Wt, H, W, 1, 1, 1), dY)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_integer_exact(dtype):
    """Integer inputs in {-2..2}: the oracle equals exact integer arithmetic."""
    rng = np.random.default_rng(21)
    for (H, W, R, S, stride, pad, dil) in [(7, 6, 3, 3, 1, 1, 1), (8, 9, 3, 3, 2, 1, 1), (9, 7, 2, 3, 3, 1, 2)]:
        N, C, K = 2, 5, 6
        P, Q = out_ext(H, R, stride, pad, dil), out_ext(W, S, stride, pad, dil)
        dYi = rng.integers(-2, 3, (N, P, Q, K))
        Wi = rng.integers(-2, 3, (K, R, S, C))
        exact = brute_force_dgrad(dYi.astype(object), Wi.astype(object), H, W, stride, pad, dil)
        got = oracle.dgrad(synth.to_bits(dYi.astype(np.float32), dtype),
                           synth.to_bits(Wi.astype(np.float32), dtype),
                           H, W, stride, pad, dil, dtype=dtype)
        np.testing.assert_array_equal(got, exact.astype(np.float64))


def test_against_torch_conv2d_input():
    """torch.nn.grad.conv2d_input (float64, CPU, NCHW) is the same operation."""
    torch = pytest.importorskip("torch")
    for case in SWEEP[::4]:
        N, H, W, C, K, R, S, stride, pad, dil = case
        P, Q = out_ext(H, R, stride, pad, dil), out_ext(W, S, stride, pad, dil)
        rng = np.random.default_rng(77 + len(case))
        dY = rng.standard_normal((N, P, Q, K))
        Wt = rng.standard_normal((K, R, S, C))
        ref = torch.nn.grad.conv2d_input(
            (N, C, H, W), torch.from_numpy(Wt.transpose(0, 3, 1, 2).copy()),
            torch.from_numpy(dY.transpose(0, 3, 1, 2).copy()),
            stride=stride, padding=pad, dilation=dil).numpy().transpose(0, 2, 3, 1)
        got = oracle.dgrad(dY, Wt, H, W, stride, pad, dil)
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_linearity_and_empty_phases():
    rng = np.random.default_rng(31)
    N, H, W, C, K = 1, 8, 8, 4, 3
    dY1, dY2 = rng.standard_normal((2, N, 4, 4, K))
    Wt = rng.standard_normal((K, 1, 1, C))
    a, b = 0.75, -1.5
    lhs = oracle.dgrad(a * dY1 + b * dY2, Wt, H, W, 2, 0, 1)
    rhs = a * oracle.dgrad(dY1, Wt, H, W, 2, 0, 1) + b * oracle.dgrad(dY2, Wt, H, W, 2, 0, 1)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-12)
    # 1x1 stride 2: only even (h, w) receive a tap; the other three phases are exactly zero
    out = oracle.dgrad(dY1, Wt, H, W, 2, 0, 1)
    assert np.all(out[:, 1::2, :, :] == 0) and np.all(out[:, :, 1::2, :] == 0)
    assert np.all(out[:, ::2, ::2, :] != 0)


def test_pixels_match_full():
    rng = np.random.default_rng(41)
    N, H, W, C, K, R, S = 2, 9, 7, 8, 16, 3, 3
    for stride, pad in [(1, 1), (2, 1), (3, 0)]:
        P, Q = out_ext(H, R, stride, pad, 1), out_ext(W, S, stride, pad, 1)
        dY = synth.to_bits(rng.standard_normal((N, P, Q, K)).astype(np.float32), "bf16")
        Wt = synth.to_bits(rng.standard_normal((K, R, S, C)).astype(np.float32), "bf16")
        x = synth.to_bits(rng.standard_normal((N, H, W, C)).astype(np.float32), "bf16")
        full = oracle.dgrad(dY, Wt, H, W, stride, pad, 1, x=x, dtype="bf16")
        pix = np.array([(n, h, w) for n in range(N) for h in range(H) for w in range(W)])[::5]
        got = oracle.dgrad_pixels(dY, Wt, H, W, pix, stride, pad, 1, x=x, dtype="bf16")
        np.testing.assert_array_equal(got, full[pix[:, 0], pix[:, 1], pix[:, 2]])


def test_f16_decoder_all_bit_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits[::1]])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()
    assert np.array_equal(np.signbit(got[~np.isnan(got)]), np.signbit(ref[~np.isnan(ref)]))


def test_bf16_decoder_all_bit_patterns():
    bits = np.arange(65536, dtype=np.uint32)
    ref = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_synth_rounding_and_prefix():
    # bf16 RNE: 1 + 2^-8 is a tie between 1 and 1 + 2^-7 -> even (1.0); 1 + 3*2^-8 -> 1 + 2^-6
    a = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -2.5, 0.0], np.float32)
    b = synth.f32_to_bf16_bits(a)
    assert list(b) == [0x3F80, 0x3F82, 0xC020, 0x0000]
    from implicit_gemm_dgrad_gb300.workloads import BATCH8
    L = BATCH8[0]
    full = synth.make_inputs(L.shape(), L.dtype, L.dist, L.workload, L.index, batch=3)[0]
    part = synth.make_inputs(L.shape(), L.dtype, L.dist, L.workload, L.index, batch=2)[0]
    np.testing.assert_array_equal(full[:2], part)
