"""Pins for the CPU oracle's weight gradient (wgrad), each against something
other than the oracle itself:

* brute force: the forward convolution's sparse structure (every (output,
  input, filter) triple of the forward definition), summed here in numpy;
* an independent library routine: torch.nn.grad.conv2d_weight in float64 (CPU);
* the closed form for 1x1 stride-1 filters: dW = dY^T X, a matrix product;
* the adjoint identity <dY, conv_fwd(x, W)> = <W, wgrad(dY, x)>;
* a hand-worked case;
* integer inputs in bf16 and fp16, where the result is exact.

A swapped r/s, a pad sign, a stride on the wrong side or a dropped edge term
fails several of these.
"""
import itertools

import numpy as np
import pytest

import oracle
from test_oracle_pins import forward_matrix

SHAPES = [  # N, H, W, C, K, R, S, stride, pad, dil
    (2, 7, 6, 3, 4, 3, 3, 1, 1, 1),
    (1, 9, 9, 2, 3, 3, 3, 2, 1, 1),
    (2, 8, 7, 3, 2, 1, 1, 2, 0, 1),
    (1, 11, 10, 2, 2, 3, 2, 3, 2, 2),
    (1, 13, 13, 4, 3, 2, 2, 2, 0, 1),   # the last row and column reach no tap
    (3, 5, 5, 5, 2, 5, 5, 1, 2, 1),
]


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _case(shape, seed=0):
    N, H, W, C, K, R, S, st, pd, dl = shape
    P, Q = oracle.out_extent(H, R, st, pd, dl), oracle.out_extent(W, S, st, pd, dl)
    return _rand((N, P, Q, K), seed), _rand((N, H, W, C), seed + 1)


@pytest.mark.parametrize("shape", SHAPES)
def test_wgrad_matches_forward_structure_brute_force(shape):
    N, H, W, C, K, R, S, st, pd, dl = shape
    dY, x = _case(shape, 3)
    _, _, rows, cols, widx = forward_matrix(N, H, W, C, K, R, S, st, pd, dl)
    ref = np.zeros(K * R * S * C)
    np.add.at(ref, widx, dY.reshape(-1)[rows] * x.reshape(-1)[cols])
    got = oracle.wgrad(dY, x, R, S, st, pd, dl)
    np.testing.assert_allclose(got.reshape(-1), ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("shape", SHAPES)
def test_wgrad_matches_torch_conv2d_weight(shape):
    torch = pytest.importorskip("torch")
    N, H, W, C, K, R, S, st, pd, dl = shape
    dY, x = _case(shape, 7)
    ref = torch.nn.grad.conv2d_weight(torch.from_numpy(x).permute(0, 3, 1, 2), (K, C, R, S),
                                      torch.from_numpy(dY).permute(0, 3, 1, 2), stride=st, padding=pd, dilation=dl)
    got = oracle.wgrad(dY, x, R, S, st, pd, dl)
    np.testing.assert_allclose(got, ref.permute(0, 2, 3, 1).numpy(), rtol=1e-11, atol=1e-11)


def test_wgrad_1x1_is_a_matrix_product():
    N, H, W, C, K = 3, 5, 4, 6, 7
    dY, x = _rand((N, H, W, K), 11), _rand((N, H, W, C), 12)
    got = oracle.wgrad(dY, x, 1, 1)
    np.testing.assert_allclose(got[:, 0, 0, :], dY.reshape(-1, K).T @ x.reshape(-1, C), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("shape", SHAPES)
def test_wgrad_adjoint_of_the_forward_convolution(shape):
    N, H, W, C, K, R, S, st, pd, dl = shape
    dY, x = _case(shape, 21)
    Wt = _rand((K, R, S, C), 23)
    lhs = float(np.sum(dY * oracle.conv_fwd(x, Wt, st, pd, dl)))
    rhs = float(np.sum(Wt * oracle.wgrad(dY, x, R, S, st, pd, dl)))
    assert abs(lhs - rhs) <= 1e-10 * max(1.0, abs(lhs))


def test_wgrad_hand_worked():
    # x = 1..9 on a 3x3 image, dY = [[1, 0], [0, 1]] (2x2 filter, stride 1,
    # no pad, so P = Q = 2): dW[r, s] = x[r, s] * 1 + x[1 + r, 1 + s] * 1,
    #   dW[0,0] = 1 + 5 = 6,  dW[0,1] = 2 + 6 = 8,
    #   dW[1,0] = 4 + 8 = 12, dW[1,1] = 5 + 9 = 14.
    x = np.arange(1, 10, dtype=np.float64).reshape(1, 3, 3, 1)
    dY = np.array([[1.0, 0.0], [0.0, 1.0]]).reshape(1, 2, 2, 1)
    got = oracle.wgrad(dY, x, 2, 2)
    assert got.reshape(2, 2).tolist() == [[6.0, 8.0], [12.0, 14.0]]
    # stride 2 with pad 1 on the same image (P = Q = 2): p = 0 reads row -1 + r,
    # p = 1 reads row 1 + r; with dY = 1 everywhere, dW[r, s] sums x over the
    # rows {r - 1, r + 1} and columns {s - 1, s + 1} that fall inside the image:
    #   dW[0,0] = x[1,1] = 5,          dW[0,1] = x[1,0] + x[1,2] = 4 + 6,
    #   dW[1,0] = x[0,1] + x[2,1] = 2 + 8,  dW[1,1] = 1 + 3 + 7 + 9.
    ones = np.ones((1, 2, 2, 1))
    g2 = oracle.wgrad(ones, x, 2, 2, 2, 1).reshape(2, 2)
    img = x.reshape(3, 3)
    expect = [[sum(img[h, w] for h in (r - 1, r + 1) if 0 <= h < 3 for w in (s - 1, s + 1) if 0 <= w < 3)
               for s in range(2)] for r in range(2)]
    assert g2.tolist() == expect == [[5.0, 10.0], [10.0, 20.0]]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_wgrad_integer_inputs_exact(dtype):
    from implicit_gemm_dgrad_gb300 import synth
    N, H, W, C, K, R, S, st, pd, dl = 2, 9, 8, 5, 4, 3, 3, 2, 1, 1
    P, Q = oracle.out_extent(H, R, st, pd, dl), oracle.out_extent(W, S, st, pd, dl)
    rng = np.random.default_rng(31)
    dYi = rng.integers(-3, 4, size=(N, P, Q, K)).astype(np.float64)
    xi = rng.integers(-3, 4, size=(N, H, W, C)).astype(np.float64)
    got = oracle.wgrad(synth.to_bits(dYi.astype(np.float32), dtype), synth.to_bits(xi.astype(np.float32), dtype),
                       R, S, st, pd, dl, dtype=dtype)
    exact = np.zeros((K, R, S, C))
    for n, p, q, k, r, s in itertools.product(range(N), range(P), range(Q), range(K), range(R), range(S)):
        h, w = p * st - pd + r * dl, q * st - pd + s * dl
        if 0 <= h < H and 0 <= w < W:
            exact[k, r, s] += dYi[n, p, q, k] * xi[n, h, w]
    assert np.array_equal(got, exact)


@pytest.mark.parametrize("shape", SHAPES)
def test_wgrad_elements_agree_with_the_full_oracle(shape):
    """The spot-check form (each element summed on its own) equals the pinned
    full wgrad at every element."""
    N, H, W, C, K, R, S, st, pd, dl = shape
    dY, x = _case(shape, 41)
    full = oracle.wgrad(dY, x, R, S, st, pd, dl)
    idx = np.array(list(itertools.product(range(K), range(R), range(S), range(C))), np.int32)
    got = oracle.wgrad_elements(dY, x, R, S, idx, st, pd, dl)
    np.testing.assert_allclose(got, full.reshape(-1), rtol=1e-12, atol=1e-12)
