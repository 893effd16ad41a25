"""Per-channel output sums fused into the dgrad epilogue (cdg_dgrad_sums)
against the oracle (oracle.channel_sums of the oracle's dgrad):
    s1[c] = sum over n,h,w of out[n,h,w,c]
    s2[c] = sum over n,h,w with x > 0 of out[n,h,w,c] * x[n,h,w,c]

* Integer inputs in {-2..2} (x in {0,1,2}): every product, every dX value and
  every partial sum is an integer below 2^24, so fp32 arithmetic is exact in
  any order and the GPU's sums must equal the oracle's bit for bit.  This runs
  in every operand, tile and issue mode, so a dropped row, tile, phase or
  channel shows as a wrong integer.
* Normal inputs: within the worst-case rounding bound of the GPU's order of
  operations.  Each dX value is an fp32 sum of m = K*R*S products, off by at
  most gamma_m times the sum of their magnitudes (gamma_n = n*u/(1 - n*u),
  u = 2^-24); the sums then add at most D = 8 + work items + CTAs values in a
  row (5 lane levels, 3 across warps, one per item in a CTA, one per CTA), off
  by at most gamma_D times the sum of magnitudes.  So
      |gpu - oracle| <= gamma_m * P + gamma_D * A
  with P the same sums of dgrad(|dY|, |W|) (gated alike; for s2 times x, and
  m + 1 for the extra product) and A the sum of |terms|, both from the oracle.
* The dX written alongside passes the usual element tolerance, and two calls
  give the same bits.
"""
import numpy as np
import pytest

import implicit_gemm_dgrad_gb300 as cdg
import oracle
from implicit_gemm_dgrad_gb300 import synth
from implicit_gemm_dgrad_gb300.workloads import FUSED_RELU, RESNET50_B256, Layer

from gpu_util import GuardedOutput, assert_close, decode_out, to_dev, torch_cuda

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


def gamma(n):
    return n * U / (1 - n * U)


def _case(N, H, W, C, K, R, S, stride, pad, dil, dtype="bf16", out="same", relu=False, idx=0):
    return Layer(f"sum_N{N}H{H}W{W}C{C}K{K}R{R}S{S}s{stride}p{pad}d{dil}{dtype}{out}{'relu' if relu else ''}",
                 N, H, W, C, K, R, S, stride, pad, dil, dtype=dtype, out=out, relu=relu, workload=13, index=idx)


class SumRun:
    """Plan (with sums), prepack and cdg_dgrad_sums for one layer."""

    def __init__(self, L, inputs, nsum, gate="x", env=None):
        torch = torch_cuda()
        self.L, self.nsum = L, nsum
        self.dY, self.W, self.x = inputs
        self.odt = "f32" if L.out == "f32" else L.dtype
        self.plan = cdg.plan(L.N, L.H, L.W, L.C, L.K, L.R, L.S, L.stride, L.pad, L.dil, L.dtype,
                             relu=(L.relu and gate == "x"), relu_bits=(L.relu and gate == "bits"),
                             out_f32=(L.out == "f32"), sums=nsum)
        self.d_dY, d_W = to_dev(self.dY, L.dtype), to_dev(self.W, L.dtype)
        self.d_Wp = torch.empty(self.plan.packed_weight_bytes // 2, dtype=torch.int16, device="cuda")
        self.plan.prepack_weights(d_W, self.d_Wp)
        self.gate = None
        if L.relu:
            d_x = to_dev(self.x, L.dtype)
            if gate == "x":
                self.gate = d_x
            else:
                px = L.N * L.H * L.W
                self.gate = torch.empty(cdg.relu_mask_bytes(px, L.C), dtype=torch.uint8, device="cuda")
                cdg.pack_relu_mask(d_x, self.gate, px, L.C, L.dtype)
        self.out = GuardedOutput(L.N * L.H * L.W * L.C, 4 if self.odt == "f32" else 2)
        self.sums = torch.full((nsum * L.C,), float("nan"), dtype=torch.float32, device="cuda")
        self.ws = torch.full((self.plan.sums_workspace_bytes // 4,), float("nan"), dtype=torch.float32,
                             device="cuda")

    def run(self):
        torch = torch_cuda()
        self.plan.dgrad_sums(self.d_dY, self.d_Wp, self.out.ptr, self.sums, self.ws, self.gate)
        torch.cuda.synchronize()
        assert self.plan.device_status() == 0
        assert self.out.guards_intact()
        s = self.sums.cpu().numpy().astype(np.float64)
        return s[:self.L.C], (s[self.L.C:] if self.nsum == 2 else None)

    def dX(self):
        L = self.L
        return decode_out(self.out.body().cpu().numpy(), self.odt).reshape(L.N, L.H, L.W, L.C)


def _oracle(run, x_for_sums):
    L = run.L
    ref = oracle.dgrad(run.dY, run.W, L.H, L.W, L.stride, L.pad, L.dil, x=run.x, dtype=L.dtype)
    return ref, oracle.channel_sums(ref, x_for_sums, dtype=L.dtype)


# (layer, sums, gate, planner overrides, what the plan must reach)
EXACT = [
    (_case(3, 13, 11, 200, 72, 1, 1, 1, 0, 1, idx=0), 1, "x", "", {"a_mode": 1}),            # rows, C tail
    (_case(2, 14, 14, 64, 128, 1, 1, 2, 0, 1, idx=1), 1, "x", "", {"a_mode": 1}),            # whole rows, zero phases
    (_case(2, 13, 13, 64, 64, 1, 1, 2, 0, 1, "f16", idx=2), 1, "x", "", {"a_mode": 0}),      # boxes, zero phases
    (_case(2, 20, 20, 64, 64, 3, 3, 1, 1, 1, relu=True, idx=3), 2, "x", "CDG_HALO=1", {"a_mode": 3}),  # halo, resident
    (_case(2, 12, 12, 128, 128, 3, 3, 1, 1, 1, relu=True, idx=4), 2, "x", "CDG_HALO=1", {"a_mode": 2}),
    (_case(2, 14, 14, 256, 256, 3, 3, 1, 1, 1, relu=True, idx=5), 2, "x", "", {"cta_pair": 1}),
    (_case(4, 16, 16, 128, 256, 3, 3, 2, 1, 1, relu=True, idx=6), 2, "x", "", {"mma_warps": 2}),
    (_case(2, 10, 10, 96, 48, 3, 3, 1, 1, 1, "f16", out="f32", relu=True, idx=7), 2, "x", "", {}),
    (_case(2, 9, 9, 64, 64, 1, 1, 1, 0, 1, out="f32", relu=True, idx=8), 2, "x", "", {"a_mode": 1}),
    (_case(2, 11, 13, 72, 136, 3, 3, 2, 1, 1, "f16", relu=True, idx=9), 1, "bits", "", {}),
    (_case(1, 30, 30, 520, 64, 3, 3, 1, 1, 1, idx=10), 1, "x", "", {}),                      # several N tiles
    (_case(2, 13, 11, 32, 16, 3, 3, 4, 1, 1, idx=11), 1, "x", "", {"num_phases": 16}),
]


@pytest.mark.parametrize("L,nsum,gate,env,reach", EXACT, ids=lambda v: v.name if isinstance(v, Layer) else None)
def test_integer_inputs_sums_exact(L, nsum, gate, env, reach, monkeypatch):
    for kv in env.split():
        k, v = kv.split("=")
        monkeypatch.setenv(k, v)
    inputs = synth.make_inputs(L.shape(), L.dtype, "int", L.workload, L.index, with_x=L.relu)
    run = SumRun(L, inputs, nsum, gate)
    info = run.plan.info()
    for k, v in reach.items():
        assert info[k] == v, (k, info)
    s1, s2 = run.run()
    ref, (r1, r2, a1, a2) = _oracle(run, run.x if nsum == 2 else None)
    assert np.max(a1) < 2 ** 24 and (a2 is None or np.max(a2) < 2 ** 24)
    np.testing.assert_array_equal(s1, r1)
    if nsum == 2:
        np.testing.assert_array_equal(s2, r2)
    assert_close(run.dX(), ref, run.odt, L.name)


def _bound_check(run, s1, s2, ref, sums):
    """|gpu - oracle| <= gamma_m * P + gamma_D * A, P from dgrad(|dY|, |W|)."""
    L = run.L
    r1, r2, a1, a2 = sums
    absdY = synth.to_bits(np.abs(synth.bits_to_f32(run.dY, L.dtype)), L.dtype)
    absW = synth.to_bits(np.abs(synth.bits_to_f32(run.W, L.dtype)), L.dtype)
    info = run.plan.info()
    D = 8 + info["work_items"] + info["grid"]
    m = L.K * L.R * L.S
    P1 = np.zeros(L.C)
    P2 = np.zeros(L.C)
    chunk = max(1, (1 << 23) // (L.H * L.W * L.C))
    for n0 in range(0, L.N, chunk):
        x = None if run.x is None else run.x[n0:n0 + chunk]
        pa = oracle.dgrad(absdY[n0:n0 + chunk], absW, L.H, L.W, L.stride, L.pad, L.dil, x=x, dtype=L.dtype)
        q1, q2, _, _ = oracle.channel_sums(pa, x if run.nsum == 2 else None, dtype=L.dtype)
        P1 += q1
        if run.nsum == 2:
            P2 += q2
    tol1 = gamma(m) * P1 + gamma(D) * a1
    assert np.all(np.abs(s1 - r1) <= tol1), np.max(np.abs(s1 - r1) / tol1)
    if run.nsum == 2:
        tol2 = gamma(m + 1) * P2 + gamma(D) * a2
        assert np.all(np.abs(s2 - r2) <= tol2), np.max(np.abs(s2 - r2) / tol2)


@pytest.mark.parametrize("L,nsum,gate,env,reach", EXACT[:9], ids=lambda v: v.name if isinstance(v, Layer) else None)
def test_normal_inputs_sums_within_rounding_bound(L, nsum, gate, env, reach, monkeypatch):
    for kv in env.split():
        k, v = kv.split("=")
        monkeypatch.setenv(k, v)
    inputs = synth.make_inputs(L.shape(), L.dtype, "normal", L.workload, L.index, with_x=L.relu)
    run = SumRun(L, inputs, nsum, gate)
    s1, s2 = run.run()
    ref, sums = _oracle(run, run.x if nsum == 2 else None)
    assert_close(run.dX(), ref, run.odt, L.name)
    _bound_check(run, s1, s2, ref, sums)
    b1, b2 = run.run()  # deterministic: the same bits again
    assert np.array_equal(b1, s1) and (s2 is None or np.array_equal(b2, s2))


FULL = [(FUSED_RELU[0], 2), (FUSED_RELU[1], 2)] + [(L, 1) for L in RESNET50_B256
                                                   if L.name[:3] in ("L03", "L10", "L21")]


@pytest.mark.parametrize("L,nsum", FULL, ids=lambda v: v.name if isinstance(v, Layer) else str(v))
def test_full_size_sums(L, nsum):
    """Batch-256 layers: the x-gated layers of the fused ReLU-backward config
    with both sums, and three ungated layers (row matrix, tap-less phases,
    CTA pairs) with s1; every element of dX against the oracle as well."""
    run = SumRun(L, synth.make_inputs(L.shape(), L.dtype, L.dist, L.workload, L.index, with_x=L.relu), nsum)
    s1, s2 = run.run()
    torch = torch_cuda()
    bits = run.out.body().view(torch.int16).view(L.N, -1)
    per_image = L.H * L.W * L.C
    chunk = max(1, (1 << 24) // per_image)
    r1 = np.zeros(L.C)
    r2 = np.zeros(L.C)
    a1 = np.zeros(L.C)
    a2 = np.zeros(L.C)
    for n0 in range(0, L.N, chunk):
        n1 = min(L.N, n0 + chunk)
        x = None if run.x is None else run.x[n0:n1]
        ref = oracle.dgrad(run.dY[n0:n1], run.W, L.H, L.W, L.stride, L.pad, L.dil, x=x, dtype=L.dtype)
        got = decode_out(bits[n0:n1].cpu().numpy().view(np.uint8), run.odt).reshape(ref.shape)
        assert_close(got, ref, run.odt, f"{L.name} images {n0}..{n1 - 1}")
        q1, q2, b1, b2 = oracle.channel_sums(ref, x if nsum == 2 else None, dtype=L.dtype)
        r1 += q1
        a1 += b1
        if nsum == 2:
            r2 += q2
            a2 += b2
    _bound_check(run, s1, s2, None, (r1, r2 if nsum == 2 else None, a1, a2 if nsum == 2 else None))
