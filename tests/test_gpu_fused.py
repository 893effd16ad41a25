"""Back-to-back dgrads in one persistent kernel (cdg_dgrad_fused) against the
oracle's composition (oracle.dgrad_fused): g = act_bwd(dgrad(dY2, W2), x2),
rounded once to the storage type, then dX1 = dgrad_1x1(g, W1).

The comparison follows the two rounding steps:
  * g (written on request) against the oracle's g under the usual 16-bit
    element tolerance;
  * dX1 against the oracle's 1x1 dgrad of the GPU's own g (the same input
    to the second layer) under the usual tolerance;
  * dX1 against the oracle's end-to-end dX1 under the usual tolerance plus
    the sum over the 1x1 filter of ulp(g) * |W1|: g is rounded once to
    bf16 from an fp32 sum, so an element whose exact value lies within the
    fp32 error of a rounding boundary may take the neighbouring bf16 value,
    one unit in the last place away from the oracle's, and that difference
    passes through the 1x1 layer.
Integer inputs make both GEMMs exact, so dX1 and g must equal the oracle's
bit for bit.  The batch-256 ResNet-50 stage-1 pair (3x3 64 -> 64 at 56x56,
gated by ReLU, then 1x1 64 -> 256) runs at full size, every element of dX1
checked."""
import numpy as np
import pytest

import implicit_gemm_dgrad_gb300 as cdg
import oracle
from implicit_gemm_dgrad_gb300 import synth

from gpu_util import GuardedOutput, assert_close, decode_out, to_dev, torch_cuda

pytestmark = pytest.mark.gpu


def _inputs(N, H, W, C1, C2, K2, R2, S2, pad2, dil2, dtype, dist, seed, act):
    P = H + 2 * pad2 - dil2 * (R2 - 1)
    Q = W + 2 * pad2 - dil2 * (S2 - 1)
    rng = np.random.default_rng(seed)
    if dist == "int":
        draw = lambda shape, std: rng.integers(-2, 3, shape).astype(np.float32)  # noqa: E731
    else:
        draw = lambda shape, std: (std * rng.standard_normal(shape)).astype(np.float32)  # noqa: E731
    dY2 = synth.to_bits(draw((N, P, Q, K2), 1.0), dtype)
    W2 = synth.to_bits(draw((K2, R2, S2, C2), np.sqrt(2.0 / (C2 * R2 * S2))), dtype)
    W1 = synth.to_bits(draw((C2, 1, 1, C1), np.sqrt(2.0 / C1)), dtype)
    x2 = None
    if act == "relu":
        x2 = synth.to_bits(np.maximum(draw((N, H, W, C2), 1.0), 0.0), dtype)
    elif act:
        x2 = synth.to_bits(draw((N, H, W, C2), 2.0), dtype)
    return dY2, W2, W1, x2


def bf16_ulp(bits: np.ndarray) -> np.ndarray:
    """One unit in the last place of each bf16 value (bit patterns), as float64."""
    e = (bits.astype(np.int64) >> 7) & 0xFF
    return np.ldexp(1.0, np.maximum(e, 1) - 127 - 7)


def end_to_end_bound(g_bits, W1, H, W):
    """sum over the 1x1 filter of ulp(g) * |W1|, per dX1 element (oracle dgrad)."""
    absW1 = np.abs(synth.bits_to_f32(W1, "bf16").astype(np.float64))
    return oracle.dgrad(bf16_ulp(g_bits), absW1, H, W, 1, 0, 1)


def assert_fused_close(got, ref, g_bits, W1, H, W, what):
    extra = end_to_end_bound(g_bits, W1, H, W)
    err = np.abs(got - ref)
    bad = ~(err <= 1e-2 * np.maximum(1.0, np.abs(ref)) + extra)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} out of the bound, "
                           f"first at {np.argwhere(bad)[:3].tolist()}")


def run_fused(geom, dtype="bf16", dist="normal", act="relu", write_g=True, seed=0):
    torch = torch_cuda()
    N, H, W, C1, C2, K2, R2, S2, pad2, dil2 = geom
    dY2, W2, W1, x2 = _inputs(*geom, dtype, dist, seed, act)
    f = cdg.FusedPlan(N, H, W, C1, C2, K2, R2, S2, pad2, dil2, dtype, act=act, write_g=write_g)
    b2, b1 = f.packed_weight_bytes
    d_W2p = torch.empty(b2 // 2, dtype=torch.int16, device="cuda")
    d_W1p = torch.empty(b1 // 2, dtype=torch.int16, device="cuda")
    f.prepack_weights(to_dev(W2, dtype), to_dev(W1, dtype), d_W2p, d_W1p)
    out = GuardedOutput(N * H * W * C1, 2)
    gout = GuardedOutput(N * H * W * C2, 2) if write_g else None
    d_x2 = to_dev(x2, dtype) if x2 is not None else None
    f.dgrad(to_dev(dY2, dtype), d_W2p, d_x2, d_W1p, out.ptr, gout.ptr if gout else None)
    torch.cuda.synchronize()
    assert f.device_status() == 0
    assert out.guards_intact() and (gout is None or gout.guards_intact())
    return f, (dY2, W2, W1, x2), out, gout


CASES = [  # N, H, W, C1, C2, K2, R2, S2, pad2, dil2
    (2, 12, 12, 256, 64, 64, 3, 3, 1, 1),
    (3, 9, 7, 96, 64, 40, 3, 3, 1, 1),       # C1 not a multiple of 64, K2 not of 64
    (2, 20, 19, 64, 64, 128, 2, 2, 0, 1),    # two K blocks in GEMM 1, a 2x2 filter
    (1, 14, 30, 200, 64, 64, 3, 3, 2, 2),    # dilation, wider than one tile row
    (4, 5, 6, 16, 64, 16, 3, 3, 1, 1),       # small C1: GEMM 2 with N = 16
    (2, 8, 8, 128, 64, 64, 1, 3, 0, 1),      # 1x3: P = H, Q = W - 2
]


@pytest.mark.parametrize("act", ["relu", "gelu", "silu", None])
@pytest.mark.parametrize("geom", CASES, ids=lambda g: "x".join(map(str, g)))
def test_fused_matches_oracle(geom, act):
    N, H, W, C1, C2, K2, R2, S2, pad2, dil2 = geom
    f, (dY2, W2, W1, x2), out, gout = run_fused(geom, act=act, seed=hash((geom, act)) % 1000)
    ref, g_ref = oracle.dgrad_fused(dY2, W2, x2, W1, H, W, pad2, dil2, dtype="bf16", act=act or "relu")
    got = decode_out(out.body().cpu().numpy(), "bf16").reshape(ref.shape)
    g_bits = gout.body().cpu().numpy().view(np.uint16).reshape(N, H, W, C2)
    g_got = synth.bits_to_f32(g_bits, "bf16").astype(np.float64)
    assert_close(g_got, synth.bits_to_f32(g_ref, "bf16").astype(np.float64), "bf16", f"g {geom} {act}")
    second = oracle.dgrad(np.ascontiguousarray(g_bits), W1, H, W, 1, 0, 1, dtype="bf16")
    assert_close(got, second, "bf16", f"dX1 against the 1x1 dgrad of the GPU's g {geom} {act}")
    assert_fused_close(got, ref, g_ref, W1, H, W, f"dX1 end to end {geom} {act}")


@pytest.mark.parametrize("geom", CASES[:4], ids=lambda g: "x".join(map(str, g)))
def test_fused_integer_inputs_bit_exact(geom):
    """Integer inputs: both GEMMs are exact in fp32, g is an integer (exact in
    bf16 below 256), so dX1 and g equal the oracle's bit for bit."""
    N, H, W, C1, C2, K2, R2, S2, pad2, dil2 = geom
    f, (dY2, W2, W1, x2), out, gout = run_fused(geom, dist="int", act="relu")
    ref, g_ref = oracle.dgrad_fused(dY2, W2, x2, W1, H, W, pad2, dil2, dtype="bf16")
    assert np.abs(synth.bits_to_f32(g_ref, "bf16")).max() <= 256
    np.testing.assert_array_equal(gout.body().cpu().numpy().view(np.uint16), g_ref.reshape(-1))
    np.testing.assert_array_equal(out.body().cpu().numpy().view(np.uint16),
                                  oracle.round_to(ref, "bf16").reshape(-1))


def test_fused_without_writing_g():
    geom = CASES[0]
    N, H, W, C1, C2, K2, R2, S2, pad2, dil2 = geom
    f, (dY2, W2, W1, x2), out, _ = run_fused(geom, write_g=False)
    ref, g_ref = oracle.dgrad_fused(dY2, W2, x2, W1, H, W, pad2, dil2, dtype="bf16")
    assert_fused_close(decode_out(out.body().cpu().numpy(), "bf16").reshape(ref.shape), ref, g_ref, W1, H, W,
                       "dX1 without g")


def test_fused_resnet50_stage1_pair_full_size():
    """Batch 256: the 3x3 64 -> 64 layer at 56x56 gated by ReLU, then the 1x1
    64 -> 256 layer; every element of dX1 against the oracle."""
    torch = torch_cuda()
    geom = (256, 56, 56, 256, 64, 64, 3, 3, 1, 1)
    N, H, W, C1, C2, K2, R2, S2, pad2, dil2 = geom
    f, (dY2, W2, W1, x2), out, _ = run_fused(geom, write_g=False)
    bits = out.body().view(torch.int16).view(N, -1)
    chunk = 16
    for n0 in range(0, N, chunk):
        ref, g_ref = oracle.dgrad_fused(dY2[n0:n0 + chunk], W2, x2[n0:n0 + chunk], W1, H, W, pad2, dil2,
                                        dtype="bf16")
        got = decode_out(bits[n0:n0 + chunk].cpu().numpy().view(np.uint8), "bf16").reshape(ref.shape)
        assert_fused_close(got, ref, g_ref, W1, H, W, f"dX1 images {n0}..{n0 + chunk - 1}")


def test_fused_plan_limits():
    """What does not fit on chip is refused at plan time: C2 other than 64,
    C1 above 256, filters whose weights do not fit beside W1."""
    for args in [(2, 12, 12, 64, 128, 64, 3, 3, 1, 1), (2, 12, 12, 512, 64, 64, 3, 3, 1, 1),
                 (2, 12, 12, 64, 64, 64, 5, 5, 2, 1), (2, 12, 12, 64, 64, 128, 3, 3, 1, 1)]:
        with pytest.raises(cdg.CdgError) as e:
            cdg.FusedPlan(*args, "bf16", host_sms=152)
        assert e.value.status == 2
