"""GPU parity: the sm_103a library against the CPU oracle, element by element.

Bar (per element): |gpu - oracle| <= 2e-3*max(1,|oracle|) for fp32 dX and
1e-2*max(1,|oracle|) for fp16/bf16 dX; integer inputs must give the oracle's
value rounded once to the output type, bit for bit; the ReLU-backward gate
must leave +0.0 at every gated-off position and no zero at any other position
unless the oracle's value there rounds to zero in the output type (the zero
pattern is checked in both directions).  dX is pre-filled with NaN
(or garbage) and surrounded by sentinel guard bands for every call.
"""
import numpy as np
import pytest

import oracle
from implicit_gemm_dgrad_gb300 import synth
from implicit_gemm_dgrad_gb300.workloads import BATCH8, TINY, Layer

from gpu_util import GpuRun, assert_close, check_gate_zero_pattern, decode_out

pytestmark = pytest.mark.gpu


def oracle_full(run: GpuRun) -> np.ndarray:
    L = run.layer
    return oracle.dgrad(run.dY, run.W, L.H, L.W, L.stride, L.pad, L.dil, x=run.x, dtype=L.dtype)


def check_layer(L, prefill="nan", dist=None):
    run = GpuRun(L, dist=dist, prefill=prefill)
    run.run()
    got = run.result()
    assert run.out.guards_intact(), "write outside dX"
    assert run.status() == 0
    ref = oracle_full(run)
    assert_close(got, ref, run.odt, L.name)
    if L.relu:
        check_gate_zero_pattern(run.result_bytes(), run.x, ref, run.odt, L.dtype)
    return run, got, ref


def test_tiny_config():
    check_layer(TINY)


@pytest.mark.parametrize("L", BATCH8, ids=lambda L: L.name)
def test_batch8_configs(L):
    check_layer(L)


def _case(N, H, W, C, K, R, S, stride, pad, dil, dtype, out="same", relu=False, idx=0):
    return Layer(f"N{N}H{H}W{W}C{C}K{K}R{R}S{S}s{stride}p{pad}d{dil}{dtype}{out}{'relu' if relu else ''}",
                 N, H, W, C, K, R, S, stride, pad, dil, dtype=dtype, out=out, relu=relu,
                 dist="normal", workload=9, index=idx)


SWEEP = [
    _case(2, 9, 7, 24, 40, 3, 3, 1, 1, 1, "bf16"),
    _case(2, 11, 13, 72, 136, 3, 3, 2, 1, 1, "f16", relu=True),
    _case(3, 10, 9, 8, 8, 1, 1, 2, 0, 1, "bf16", out="f32"),
    _case(2, 7, 7, 136, 72, 1, 1, 1, 0, 1, "bf16"),
    _case(1, 12, 10, 16, 24, 5, 3, 3, 2, 2, "f16", out="f32"),
    _case(2, 9, 9, 40, 24, 2, 3, 2, 2, 1, "bf16", relu=True),
    _case(4, 6, 5, 264, 80, 3, 3, 1, 1, 2, "bf16"),
    _case(1, 1, 3, 8, 8, 1, 1, 2, 0, 1, "f16"),            # phase with no dX row (H < stride)
    _case(2, 13, 11, 32, 16, 3, 3, 4, 1, 1, "bf16"),       # 16 phases
    _case(3, 5, 17, 48, 200, 1, 1, 1, 1, 1, "f16", out="f32"),  # 1x1 with padding: box path
    _case(1, 30, 30, 520, 64, 3, 3, 1, 1, 1, "bf16"),       # C > 256: several N tiles
    _case(2, 14, 14, 64, 520, 3, 3, 2, 1, 1, "f16", relu=True),
    _case(5, 3, 4, 16, 8, 3, 3, 1, 2, 1, "bf16"),           # dX smaller than the halo
    _case(1, 57, 3, 16, 16, 3, 1, 1, 1, 1, "f16"),          # tall and narrow
    _case(2, 16, 16, 8, 8, 7, 7, 2, 3, 1, "bf16", out="f32"),
    _case(5, 14, 14, 64, 64, 1, 1, 2, 0, 1, "bf16"),  # three of four phases zero-filled, 7x7 sub-grids
    _case(1, 12, 20, 16, 16, 8, 16, 1, 4, 1, "bf16"),  # 128 taps, the most a filter may have
    _case(2, 16, 24, 24, 16, 8, 16, 2, 4, 1, "f16"),   # 128 taps over four phases of 32
]


@pytest.mark.parametrize("L", SWEEP, ids=lambda L: L.name)
def test_shape_sweep(L):
    check_layer(L)


@pytest.mark.parametrize("prefill", ["nan", "garbage"])
def test_prior_contents_do_not_matter(prefill):
    L = _case(2, 9, 9, 40, 24, 3, 3, 2, 1, 1, "bf16", relu=True)
    _, got, _ = check_layer(L, prefill=prefill)


@pytest.mark.parametrize("L", [
    _case(2, 9, 7, 24, 40, 3, 3, 1, 1, 1, "bf16"),
    _case(2, 11, 13, 72, 136, 3, 3, 2, 1, 1, "f16"),
    _case(2, 10, 12, 16, 32, 3, 3, 3, 1, 2, "f16", out="f32"),
    _case(3, 8, 8, 24, 16, 1, 1, 2, 0, 1, "bf16"),
    _case(2, 14, 14, 264, 72, 3, 3, 1, 1, 1, "bf16"),
], ids=lambda L: L.name)
def test_integer_inputs_bit_exact(L):
    """Inputs in {-2..2}: fp32 accumulation is exact, so dX = RNE(oracle) bit for bit."""
    inputs = synth.make_inputs(L.shape(), L.dtype, "int", L.workload, L.index, with_x=L.relu)
    run = GpuRun(L, inputs=inputs)
    run.run()
    raw = run.result_bytes()
    ref = oracle_full(run)
    if run.odt == "f32":
        expect = ref.astype(np.float32).view(np.uint32).reshape(-1)
        got = raw.view(np.uint32)
    elif run.odt == "f16":
        expect = ref.astype(np.float16).view(np.uint16).reshape(-1)
        got = raw.view(np.uint16)
    else:
        expect = synth.f32_to_bf16_bits(ref.astype(np.float32)).reshape(-1)
        got = raw.view(np.uint16)
    mism = np.flatnonzero(got != expect)
    assert mism.size == 0, f"{mism.size} mismatches, first at {mism[:5]}: {got[mism[:5]]} vs {expect[mism[:5]]}"


def test_deterministic():
    L = _case(2, 11, 13, 72, 136, 3, 3, 2, 1, 1, "bf16", relu=True)
    run = GpuRun(L)
    run.run()
    a = run.result_bytes().copy()
    run.run()
    b = run.result_bytes()
    assert np.array_equal(a, b)


def test_gate_special_values():
    """x = +0, -0, NaN, negative, subnormal, +Inf: only x > 0 passes the value through."""
    L = _case(1, 4, 4, 16, 16, 1, 1, 1, 0, 1, "f16", relu=True)
    dY, W, _ = synth.make_inputs(L.shape(), L.dtype, "uniform", L.workload, L.index)
    specials = np.array([0x3C00, 0x0000, 0x8000, 0x7E00, 0xBC00, 0x0001, 0x7C00, 0xFE00], np.uint16)
    x = np.resize(specials, (1, 4, 4, 16)).astype(np.uint16)
    run = GpuRun(L, inputs=(dY, W, x))
    run.run()
    raw = run.result_bytes()
    got = decode_out(raw, run.odt).reshape(1, 4, 4, 16)
    ref = oracle.dgrad(dY, W, 4, 4, 1, 0, 1, x=x, dtype="f16")
    counts = check_gate_zero_pattern(raw, x, ref, run.odt, "f16")
    # +0, -0, two NaNs and -1 are masked; 1.0, the subnormal and +Inf pass
    assert counts["masked"] == 5 * 4 * 4 * 16 // 8 and counts["unmasked_oracle_zero"] == 0
    assert_close(got, ref, run.odt, "specials")


def test_empty_phases_written_zero_and_linear_in_dY():
    """1x1 stride 2: odd rows/columns of dX are +0.0 exactly; dgrad(2*dY) = 2*dgrad(dY)."""
    L = _case(2, 12, 10, 32, 48, 1, 1, 2, 0, 1, "bf16", out="f32")
    run = GpuRun(L)
    run.run()
    got = run.result()
    bits = run.result_bytes().view(np.uint32).reshape(got.shape)
    assert np.all(bits[:, 1::2] == 0) and np.all(bits[:, :, 1::2] == 0)
    dY2 = synth.to_bits(2 * synth.bits_to_f32(run.dY, "bf16"), "bf16")
    run2 = GpuRun(L, inputs=(dY2, run.W, None))
    run2.run()
    np.testing.assert_array_equal(run2.result(), 2 * got)


def test_interleaved_plans():
    """Plans of different shapes (different shared-memory sizes, same kernel
    instantiation) stay valid when used after one another in any order."""
    cases = [_case(2, 9, 7, 256, 64, 3, 3, 1, 1, 1, "bf16"), _case(2, 9, 7, 16, 64, 3, 3, 1, 1, 1, "bf16"),
             _case(2, 8, 8, 64, 64, 1, 1, 2, 0, 1, "bf16")]
    runs = [GpuRun(L) for L in cases]
    for run in reversed(runs):
        run.run()
    for run in runs:
        got = run.result()
        assert run.status() == 0
        ref = oracle_full(run)
        assert_close(got, ref, run.odt, run.layer.name)


@pytest.mark.parametrize("nacc", ["2", "4"])
@pytest.mark.parametrize("L", [SWEEP[0], SWEEP[1], SWEEP[4], SWEEP[5], SWEEP[10], SWEEP[12], SWEEP[14], BATCH8[0]],
                         ids=lambda L: L.name)
def test_halo_operand_mode(L, nacc, monkeypatch):
    """The halo operand mode (one dY box per tile and K block serves every
    tap; weights streamed per tap, or resident when the whole filter of a
    single N tile fits) gives the same results, with two or four
    accumulators in flight (four only for N tiles up to 128 channels: wider
    ones would need more than the 512 TMEM columns, and keep two)."""
    monkeypatch.setenv("CDG_HALO", "1")
    monkeypatch.setenv("CDG_NACC", nacc)
    run, _, _ = check_layer(L)
    assert run.plan.info()["a_mode"] in (2, 3)


# halo boxes with CTA pairs (opt-in: CDG_HALO=1 CDG_PAIR=1): resident weight
# halves (a 3x3 128 -> 128 filter, twice what one CTA holds), streamed weight
# halves with an odd tile count (the partner tile lies out of range), four
# stride-2 phases under the ReLU gate, several N tiles, fp32 output
HALO_PAIR_CASES = [
    (_case(2, 28, 28, 128, 128, 3, 3, 1, 1, 1, "bf16", idx=30), {"a_mode": 3, "cta_pair": 1}),
    (_case(1, 9, 9, 256, 128, 3, 3, 1, 1, 1, "bf16", idx=31), {"a_mode": 2, "cta_pair": 1}),
    (_case(2, 14, 14, 128, 64, 3, 3, 2, 1, 1, "f16", relu=True, idx=32), {"cta_pair": 1}),
    (_case(1, 30, 30, 520, 64, 3, 3, 1, 1, 1, "bf16", idx=33), {"a_mode": 2, "cta_pair": 1}),
    (_case(2, 10, 10, 128, 48, 3, 3, 1, 1, 1, "f16", out="f32", idx=34), {"cta_pair": 1}),
]


@pytest.mark.parametrize("L,reach", HALO_PAIR_CASES, ids=lambda v: v.name if isinstance(v, Layer) else None)
def test_halo_operand_mode_with_cta_pairs(L, reach, monkeypatch):
    """Halo boxes with CTA pairs: each CTA of a pair loads its own tile's halo
    box and half of every weight tile, and the leader's 2-SM MMAs cover both
    tiles; the result is the oracle's."""
    monkeypatch.setenv("CDG_HALO", "1")
    monkeypatch.setenv("CDG_PAIR", "1")
    run, _, _ = check_layer(L)
    info = run.plan.info()
    assert info["a_mode"] in (2, 3)
    for k, v in reach.items():
        assert info[k] == v, (k, info)


# two MMA warps over the halo ring (the planner's choice for halo plans with
# resident weights; the test also sets CDG_DUAL=1).  The grid is capped
# (CDG_MAX_GRID) so that every CTA walks many items and the halo ring wraps
# around many times: three halo stages (odd, so a stage alternates between
# the warps) as in single CTAs of ResNet-50's 3x3 64-channel layer, six, CTA
# pairs at 64 and 128 channels, four stride-2 phases under the ReLU gate,
# fp32 output.
HALO_DUAL_CASES = [
    (_case(8, 56, 56, 64, 64, 3, 3, 1, 1, 1, "bf16", idx=40), "CDG_MAX_GRID=6 CDG_PAIR=0",
     {"a_mode": 3, "mma_warps": 2, "cta_pair": 0}),
    (_case(16, 12, 12, 64, 64, 3, 3, 1, 1, 1, "bf16", idx=41), "CDG_MAX_GRID=2 CDG_PAIR=0",
     {"a_mode": 3, "mma_warps": 2, "cta_pair": 0}),
    (_case(8, 56, 56, 64, 64, 3, 3, 1, 1, 1, "bf16", idx=45), "CDG_MAX_GRID=6", {"a_mode": 3, "mma_warps": 2, "cta_pair": 1}),
    (_case(8, 28, 28, 128, 128, 3, 3, 1, 1, 1, "bf16", idx=42), "CDG_MAX_GRID=6", {"a_mode": 3, "mma_warps": 2, "cta_pair": 1}),
    # gated by the activation: halo boxes only when asked
    (_case(8, 14, 14, 64, 64, 3, 3, 2, 1, 1, "bf16", relu=True, idx=43), "CDG_MAX_GRID=2 CDG_HALO=1", {"a_mode": 3, "mma_warps": 2}),
    (_case(40, 9, 7, 64, 64, 3, 3, 1, 1, 1, "f16", out="f32", relu=True, idx=44), "CDG_MAX_GRID=6 CDG_HALO=1",
     {"a_mode": 3, "mma_warps": 2}),
]


@pytest.mark.parametrize("L,env,reach", HALO_DUAL_CASES, ids=lambda v: v.name if isinstance(v, Layer) else None)
def test_halo_dual_issue(L, env, reach, monkeypatch):
    """Halo boxes with resident weights and two MMA warps taking alternate
    items from the one halo ring give the oracle's result."""
    monkeypatch.setenv("CDG_DUAL", "1")
    for kv in env.split():
        key, val = kv.split("=")
        monkeypatch.setenv(key, val)
    run, _, _ = check_layer(L)
    info = run.plan.info()
    for k, v in reach.items():
        assert info[k] == v, (k, info)
    grid = int(dict(kv.split("=") for kv in env.split())["CDG_MAX_GRID"])
    assert info["grid"] <= grid and info["work_items"] >= 4 * (info["grid"] // (2 if info["cta_pair"] else 1))


def test_chained_launches_keep_stream_order():
    """Launches on one stream start their set-up while the previous launch
    finishes (programmatic dependent launch), but must still see stream order:
    a dgrad that reads the previous dgrad's dX as its dY, then a dgrad that
    overwrites that dX while the reader may still be draining."""
    import torch
    A = _case(2, 20, 20, 64, 64, 3, 3, 1, 1, 1, "bf16", idx=3)
    B = _case(2, 40, 40, 32, 64, 3, 3, 2, 1, 1, "bf16", idx=4)  # B's dY has A's dX shape
    ra, rb = GpuRun(A), GpuRun(B)
    assert rb.plan.output_dims == (A.H, A.W)
    ra.run()
    first = ra.result_bytes().copy()  # A's dX, synchronised
    ra.out.body().view(torch.int16).fill_(0x7E01)  # NaN again
    neg_dY = -ra.d_dY  # exact in bf16: A's dX becomes its negation
    torch.cuda.synchronize()
    # the chain, with no synchronisation inside it
    ra.run()
    rb.plan.dgrad(ra.out.ptr, rb.d_Wp, rb.out.ptr, None)
    ra.plan.dgrad(neg_dY, ra.d_Wp, ra.out.ptr, None)
    got_b = rb.result()
    last_a = ra.result_bytes()
    assert ra.status() == 0 and rb.status() == 0
    assert_close(decode_out(last_a, ra.odt), -decode_out(first, ra.odt), ra.odt, "A rewritten after B")
    dY_b = first.view(np.uint16).reshape(A.N, A.H, A.W, A.C)
    ref_b = oracle.dgrad(dY_b, rb.W, B.H, B.W, B.stride, B.pad, B.dil, dtype=B.dtype)
    assert_close(got_b, ref_b, rb.odt, "B after A")


# Shapes that reach the planner's special paths by default: a CTA pair (256
# channels, 36 stages per tile), a pair whose partner M tile lies wholly out of
# range (one 9x9 tile), and four equal stride-2 phases with dual MMA issue and
# interleaved items.
MODE_CASES = [_case(2, 14, 14, 256, 256, 3, 3, 1, 1, 1, "bf16", idx=5),
              _case(1, 9, 9, 256, 128, 3, 3, 1, 1, 1, "bf16", idx=6),
              _case(4, 16, 16, 128, 256, 3, 3, 2, 1, 1, "bf16", relu=True, idx=7)]


def test_mode_cases_reach_their_paths():
    import implicit_gemm_dgrad_gb300 as cdg
    infos = [cdg.plan(L.N, L.H, L.W, L.C, L.K, L.R, L.S, L.stride, L.pad, L.dil, L.dtype, relu=L.relu).info()
             for L in MODE_CASES]
    assert infos[0]["cta_pair"] == 1 and infos[1]["cta_pair"] == 1
    assert infos[2]["mma_warps"] == 2 and infos[2]["num_phases"] == 4


@pytest.mark.parametrize("env", ["", "CDG_PAIR=0", "CDG_PAIR=1", "CDG_DUAL=0", "CDG_INTERLEAVE=0", "CDG_HALO=0",
                                 "CDG_PDL=0", "CDG_PREFETCH=1", "CDG_MAX_GRID=3"])
@pytest.mark.parametrize("L", MODE_CASES, ids=lambda L: L.name)
def test_planner_mode_overrides(L, env, monkeypatch):
    """Every planner mode and its override gives the oracle's result."""
    for kv in env.split():
        key, val = kv.split("=")
        monkeypatch.setenv(key, val)
    check_layer(L)


@pytest.mark.parametrize("L", [SWEEP[1], SWEEP[5], SWEEP[13], BATCH8[0]] + MODE_CASES, ids=lambda L: L.name)
def test_autotuned_plan_matches_oracle(L):
    """cdg_autotune times the planner's candidate configurations on the
    caller's tensors and keeps the fastest: the dX it leaves and every later
    call give the oracle's result."""
    run = GpuRun(L)
    best = run.plan.autotune(run.d_dY, run.d_Wp, run.out.ptr, run.d_x, reps=2)
    assert best > 0 and run.plan.info()["tuned"] == 1
    ref = oracle_full(run)
    assert_close(run.result(), ref, run.odt, L.name + " (autotune output)")
    assert run.out.guards_intact()
    run.out.body().fill_(0xA5)  # garbage, then the tuned plan again
    run.run()
    assert_close(run.result(), ref, run.odt, L.name + " (tuned plan)")
    assert run.status() == 0


def _packed_mask_numpy(x_bits: np.ndarray, dtype: str, C: int) -> np.ndarray:
    """The layout cdg_pack_relu_mask documents: per pixel, C bits (x > 0),
    channel c in bit c % 8 of byte c / 8, the row zero-padded to whole 16-byte
    units."""
    pos = synth.bits_to_f32(x_bits.reshape(-1, C), dtype) > 0  # NaN and -0 give False
    row = 16 * ((C + 127) // 128)
    padded = np.zeros((pos.shape[0], 8 * row), bool)
    padded[:, :C] = pos
    return np.packbits(padded, axis=1, bitorder="little").reshape(-1)


BITS_CASES = [_case(2, 11, 13, 72, 136, 3, 3, 2, 1, 1, "f16", relu=True, idx=10),
              _case(2, 9, 9, 40, 24, 2, 3, 2, 2, 1, "bf16", relu=True, idx=11),
              _case(2, 12, 12, 64, 64, 3, 3, 1, 1, 1, "bf16", relu=True, idx=12),
              _case(2, 10, 10, 32, 48, 3, 3, 2, 1, 1, "f16", out="f32", relu=True, idx=13)]


def _bits_gated(L, x_override=None):
    """Pack the saved activation with cdg_pack_relu_mask (checked against numpy)
    and run the bit-gated dgrad; returns (raw dX bytes, x bits, output dtype, plan)."""
    import torch
    import implicit_gemm_dgrad_gb300 as cdg
    from gpu_util import GuardedOutput, to_dev
    dY, W, x = synth.make_inputs(L.shape(), L.dtype, L.dist, L.workload, L.index, with_x=True)
    if x_override is not None:
        x = x_override(x)
    pixels = L.N * L.H * L.W
    d_x = to_dev(x, L.dtype)
    d_bits = torch.full((cdg.relu_mask_bytes(pixels, L.C),), 0xA5, dtype=torch.uint8, device="cuda")
    cdg.pack_relu_mask(d_x, d_bits, pixels, L.C, L.dtype)
    torch.cuda.synchronize()
    assert np.array_equal(d_bits.cpu().numpy(), _packed_mask_numpy(x, L.dtype, L.C))
    p = cdg.plan(L.N, L.H, L.W, L.C, L.K, L.R, L.S, L.stride, L.pad, L.dil, L.dtype, out_f32=(L.out == "f32"),
                 relu_bits=True)
    d_dY, d_W = to_dev(dY, L.dtype), to_dev(W, L.dtype)
    d_Wp = torch.empty(p.packed_weight_bytes // 2, dtype=torch.int16, device="cuda")
    p.prepack_weights(d_W, d_Wp)
    odt = "f32" if L.out == "f32" else L.dtype
    out = GuardedOutput(L.N * L.H * L.W * L.C, 4 if odt == "f32" else 2)
    p.dgrad(d_dY, d_Wp, out.ptr, d_bits)
    torch.cuda.synchronize()
    raw = out.body().cpu().numpy()
    assert out.guards_intact() and p.device_status() == 0
    ref = oracle.dgrad(dY, W, L.H, L.W, L.stride, L.pad, L.dil, x=x, dtype=L.dtype)
    check_gate_zero_pattern(raw, x, ref, odt, L.dtype)
    assert_close(decode_out(raw, odt).reshape(L.N, L.H, L.W, L.C), ref, odt, L.name)
    return raw, x, odt, p


@pytest.mark.parametrize("L", BITS_CASES, ids=lambda L: L.name)
def test_packed_relu_mask_gate(L):
    """CDG_EPI_RELU_BWD_BITS: the mask packed by cdg_pack_relu_mask equals the
    numpy packing of (x > 0), and the dgrad gated by it equals the oracle gated
    by x, with +0.0 exactly where x <= 0, -0.0 or NaN."""
    special = None
    if L.index == 12:  # special values in the saved activation
        specials = np.array([0x3F80, 0x0000, 0x8000, 0x7FC0, 0xBF80, 0x0001, 0x7F80, 0xFF80], np.uint16)
        special = lambda x: np.resize(specials, x.shape).astype(np.uint16)  # noqa: E731
    _bits_gated(L, special)


# (layer, planner override, what the plan must reach): the gate's inputs are
# copied ahead into the staging buffers in every kernel mode
GATE_CASES = [
    (_case(3, 13, 11, 200, 72, 1, 1, 1, 0, 1, "bf16", relu=True, idx=14), "", {"a_mode": 1}),  # rows, 8-ch tail chunk
    (_case(2, 14, 14, 64, 128, 1, 1, 2, 0, 1, "bf16", relu=True, idx=15), "", {"a_mode": 1}),  # rows, zero phases
    (_case(2, 13, 13, 64, 64, 1, 1, 2, 0, 1, "f16", relu=True, idx=16), "", {"a_mode": 0}),    # 4-D boxes, zero phases
    (_case(2, 20, 20, 64, 64, 3, 3, 1, 1, 1, "bf16", relu=True, idx=17), "CDG_HALO=1", {"a_mode": 3}),  # halo, resident weights
    # the activation's tiles issued by loader warp 3, many chunks per CTA
    (_case(4, 16, 16, 128, 64, 3, 3, 2, 1, 1, "bf16", relu=True, idx=24), "CDG_MAX_GRID=2", {"a_mode": 0, "mma_warps": 1}),
    (_case(2, 14, 14, 256, 128, 1, 1, 1, 0, 1, "bf16", relu=True, idx=25), "CDG_MAX_GRID=2", {"a_mode": 1, "mma_warps": 1}),
    (_case(2, 12, 12, 128, 128, 3, 3, 1, 1, 1, "bf16", relu=True, idx=18), "CDG_HALO=1", {"a_mode": 2}),
    (_case(2, 12, 12, 128, 128, 3, 3, 1, 1, 1, "bf16", relu=True, idx=23), "CDG_HALO=1 CDG_PAIR=1",
     {"cta_pair": 1}),
    (_case(2, 14, 14, 256, 256, 3, 3, 1, 1, 1, "bf16", relu=True, idx=19), "", {"cta_pair": 1}),
    (_case(4, 16, 16, 128, 256, 3, 3, 2, 1, 1, "bf16", relu=True, idx=20), "", {"mma_warps": 2}),
    (_case(2, 10, 10, 96, 48, 3, 3, 1, 1, 1, "f16", out="f32", relu=True, idx=21), "", {}),
    (_case(2, 9, 9, 64, 64, 1, 1, 1, 0, 1, "bf16", out="f32", relu=True, idx=22), "", {"a_mode": 1}),
    # 128-channel stride-1 tiles gated by x: halo pairs, streamed weight halves
    (_case(8, 14, 14, 128, 128, 3, 3, 1, 1, 1, "bf16", relu=True, idx=26), "CDG_MAX_GRID=4", {}),
]


@pytest.mark.parametrize("L", [
    GATE_CASES[-1][0],
    _case(8, 14, 14, 128, 128, 3, 3, 1, 1, 1, "f16", out="f32", relu=True, idx=27),
    _case(6, 15, 13, 128, 128, 3, 3, 1, 2, 2, "f16", relu=True, idx=28),  # dilation 2, ragged sub-grid
], ids=lambda L: L.name)
def test_gated_halo_pairs_by_default(L, monkeypatch):
    """Gated by the saved activation, a stride-1 layer with 128-channel N
    tiles runs halo boxes in CTA pairs with streamed weight halves (the
    activation's staging buffers leave no room for resident halves), and
    gives the oracle's result with several items per pair (fp16 and bf16,
    16-bit and fp32 output, dilation 2)."""
    monkeypatch.setenv("CDG_MAX_GRID", "4")
    run, _, _ = check_layer(L)
    info = run.plan.info()
    assert (info["a_mode"], info["cta_pair"], info["mma_warps"]) == (2, 1, 1), info
    assert info["work_items"] >= 4 * (info["grid"] // 2)


@pytest.mark.parametrize("gate", ["x", "bits"])
@pytest.mark.parametrize("L,env,reach", GATE_CASES, ids=lambda v: v.name if isinstance(v, Layer) else None)
def test_gate_in_every_mode(L, env, reach, gate, monkeypatch):
    """The fused ReLU-backward gate, from the saved activation or its packed
    mask, gives the oracle's result and +0.0 exactly where x <= 0 in every
    operand, tile and issue mode."""
    for kv in env.split():
        key, val = kv.split("=")
        monkeypatch.setenv(key, val)
    if gate == "x":
        run, _, _ = check_layer(L)
        info = run.plan.info()
    else:
        info = _bits_gated(L)[3].info()
    for k, v in reach.items():
        assert info[k] == v, (k, info)


@pytest.mark.parametrize("act", ["gelu", "silu"])
@pytest.mark.parametrize("L,env,reach", GATE_CASES, ids=lambda v: v.name if isinstance(v, Layer) else None)
def test_activation_backward_in_every_mode(L, env, reach, act, monkeypatch):
    """GELU (erf form) and SiLU backward fused into the epilogue: out = dX *
    f'(x) with x the activation's saved input (drawn N(0, 2^2), so both signs
    and the derivative's negative dip occur), against the oracle, in every
    operand, tile and issue mode."""
    import torch
    import implicit_gemm_dgrad_gb300 as cdg
    from gpu_util import GuardedOutput, to_dev
    for kv in env.split():
        key, val = kv.split("=")
        monkeypatch.setenv(key, val)
    dY, W, _ = synth.make_inputs(L.shape(), L.dtype, L.dist, L.workload, L.index)
    rng = np.random.default_rng(1000 + L.index)
    x = synth.to_bits((2.0 * rng.standard_normal((L.N, L.H, L.W, L.C))).astype(np.float32), L.dtype)
    p = cdg.plan(L.N, L.H, L.W, L.C, L.K, L.R, L.S, L.stride, L.pad, L.dil, L.dtype, relu=True, act=act,
                 out_f32=(L.out == "f32"))
    for k, v in reach.items():
        assert p.info()[k] == v, (k, p.info())
    d_W = to_dev(W, L.dtype)
    d_Wp = torch.empty(p.packed_weight_bytes // 2, dtype=torch.int16, device="cuda")
    p.prepack_weights(d_W, d_Wp)
    odt = "f32" if L.out == "f32" else L.dtype
    out = GuardedOutput(L.N * L.H * L.W * L.C, 4 if odt == "f32" else 2)
    p.dgrad(to_dev(dY, L.dtype), d_Wp, out.ptr, to_dev(x, L.dtype))
    torch.cuda.synchronize()
    assert out.guards_intact() and p.device_status() == 0
    ref = oracle.dgrad(dY, W, L.H, L.W, L.stride, L.pad, L.dil, x=x, dtype=L.dtype, act=act)
    assert_close(decode_out(out.body().cpu().numpy(), odt).reshape(ref.shape), ref, odt, f"{L.name} {act}")
