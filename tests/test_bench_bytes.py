"""The algorithmic byte counts bench.py divides by: the gated bytes count the
gate input only where some filter tap reaches dX (elsewhere dX is +0.0
whatever the gate holds), checked by brute force over the definition."""
import importlib.util
import itertools
import os

import pytest

from implicit_gemm_dgrad_gb300.workloads import RESNET50_B256, Layer

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod_bytes", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _reached_pixels(L) -> int:
    """dX pixels h = p*stride - pad + r*dil, w = q*stride - pad + s*dil that
    some (p, q, r, s) reaches, counted one image at a time."""
    hit = set()
    for p, q, r, s in itertools.product(range(L.P), range(L.Q), range(L.R), range(L.S)):
        h = p * L.stride - L.pad + r * L.dil
        w = q * L.stride - L.pad + s * L.dil
        if 0 <= h < L.H and 0 <= w < L.W:
            hit.add((h, w))
    return L.N * len(hit)


@pytest.mark.parametrize("shape", [
    (2, 9, 9, 8, 8, 1, 1, 2, 0, 1), (1, 10, 10, 8, 8, 3, 3, 2, 1, 1), (1, 12, 11, 8, 8, 1, 1, 3, 0, 1),
    (1, 13, 13, 8, 8, 2, 2, 2, 0, 1), (1, 16, 16, 8, 8, 3, 3, 4, 1, 2), (1, 7, 7, 8, 8, 3, 3, 1, 1, 1),
    (1, 14, 14, 8, 8, 1, 1, 2, 0, 1), (1, 11, 9, 8, 8, 5, 3, 3, 2, 1)])
def test_tap_pixels_match_the_definition(shape):
    L = Layer("t", *shape)
    assert _bench().tap_pixels(L) == _reached_pixels(L)


def test_gate_bytes_per_mode():
    b = _bench()
    for L in RESNET50_B256:
        px = b.tap_pixels(L)
        assert b.gate_bytes(L, "none") == L.bytes
        assert b.gate_bytes(L, "x") == L.bytes + 2 * px * L.C
        assert b.gate_bytes(L, "bits") == L.bytes + px * 16 * ((L.C + 127) // 128)
        if L.R == 1 and L.stride == 2:
            assert px * 4 == L.N * L.H * L.W  # three of four phases get no tap


def test_wgrad_bytes():
    """wgrad reads dY once, the forward input once where a tap reaches it,
    and writes dW once."""
    b = _bench()
    L = Layer("t", 2, 9, 7, 16, 24, 3, 3, 2, 1, 1)  # a 3x3 filter reaches every pixel
    assert b.wgrad_bytes(L) == 2 * (2 * L.P * L.Q * 24 + 2 * 9 * 7 * 16 + 24 * 9 * 16)
    from implicit_gemm_dgrad_gb300.workloads import by_name
    L01 = by_name("L01_1x1_64-64_56")  # 2 x 102.8 MB of activations, a 8 KB filter
    assert abs(b.wgrad_bytes(L01) / 1e6 - 205.5) < 0.1
    # 1x1 stride 2 (56 -> 28): x is read at the 28 x 28 pixels the filter reaches
    L10 = by_name("L10_1x1s2_256-512_56-28")
    assert b.wgrad_bytes(L10) == 2 * (256 * 28 * 28 * 512 + 256 * 28 * 28 * 256 + 512 * 256)


def test_peak_basis_follows_the_sampled_clock():
    """The tensor roofline uses the burst bf16 peak when the SM clock held its
    maximum during the timed region, else the sustained one; both fractions
    are printed."""
    b = _bench()
    assert b.peak_basis({"sm_mhz": 2070.0, "sm_max_mhz": 2070.0}) == "burst"
    assert b.peak_basis({"sm_mhz": 1440.0, "sm_max_mhz": 2070.0}) == "sustained"
    assert b.peak_basis({"sm_mhz": None, "sm_max_mhz": None}) == "sustained"
    peaks = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    L = [x for x in RESNET50_B256 if x.name.startswith("L21")][0]  # tensor-bound
    ms = L.flops / 950e12 * 1e3  # runs at 950 TFLOP/s
    burst = b.layer_record(L, ms, peaks, "burst")
    sus = b.layer_record(L, ms, peaks, "sustained")
    assert burst["bound"] == "tensor" and abs(burst["roofline_frac"] - 0.5) < 1e-3
    assert abs(sus["roofline_frac"] - 950 / 1700) < 1e-3 and abs(burst["roofline_frac_sustained"] - sus["roofline_frac"]) < 1e-9
    H = [x for x in RESNET50_B256 if x.name.startswith("L01")][0]  # HBM-bound: the basis does not matter
    ms = H.bytes / 3400e9 * 1e3
    assert abs(b.layer_record(H, ms, peaks, "burst")["roofline_frac"] - 0.5) < 1e-3
    assert b.layer_record(H, ms, peaks, "sustained")["roofline_frac"] == b.layer_record(H, ms, peaks, "burst")["roofline_frac"]
