"""Host-only checks of the C-ABI library: it loads, exports what include/cdg.h
declares, validates arguments without a device, and plans the phase
decomposition of strided dgrad as the definition requires."""
import ctypes
import os
import re

import pytest

import implicit_gemm_dgrad_gb300 as cdg
from implicit_gemm_dgrad_gb300.workloads import ALL

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cdg.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?(?:[a-z_0-9]+\s+)*[a-z_0-9]+\s*\*?\s*(cdg_[a-z_0-9]+)\s*\(", text,
                       flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol():
    lib = cdg.load_library()
    names = declared_functions()
    assert len(names) >= 10, names
    for name in names:
        assert hasattr(lib, name), f"{name} declared in cdg.h but not exported"
    assert set(names) == set(cdg.EXPORTS)


def test_status_strings():
    for code in range(0, 8):
        s = cdg.status_string(code)
        assert s and s != "unknown status"
    assert cdg.status_string(99) == "unknown status"


def _plan_rc(*args, host=True):
    lib = cdg.load_library()
    h = ctypes.c_void_p()
    if host:
        rc = lib.cdg_plan_host(*args, 148, ctypes.byref(h))
    else:
        rc = lib.cdg_plan(*args, ctypes.byref(h))
    if h.value:
        lib.cdg_destroy(h)
    return rc


GOOD = (2, 8, 8, 16, 16, 3, 3, 1, 1, 1, cdg.BF16, 0)


@pytest.mark.parametrize("host", [True, False])
@pytest.mark.parametrize("field,value,expect", [
    (0, 0, 1), (1, 0, 1), (3, 0, 1), (5, 0, 1), (7, 0, 1), (8, -1, 1), (9, 0, 1),
    (10, 2, 1), (11, 128, 1), (11, 5, 1),  # unknown epilogue flag; both ReLU gates at once
    (11, 16, 1), (11, 24, 1), (11, 28, 1),  # sums of out*x without the x gate (none, or the bit mask)
    (11, 33, 1), (11, 68, 1), (11, 96, 1), (11, 48, 1),  # two activations at once; GELU with sums of out*x
    (3, 12, 2), (4, 20, 2), (7, 5, 2),
])
def test_argument_validation_needs_no_device(host, field, value, expect):
    args = list(GOOD)
    args[field] = value
    assert _plan_rc(*args, host=host) == expect


def test_geometry_too_small_is_invalid():
    # H + 2*pad - dil*(R-1) - 1 < 0: empty forward output
    assert _plan_rc(1, 2, 2, 8, 8, 5, 5, 1, 0, 1, cdg.F16, 0) == 1


def test_filter_too_large_is_unsupported():
    assert _plan_rc(1, 40, 40, 8, 8, 12, 12, 1, 5, 1, cdg.F16, 0) == 2


def test_host_plan_refuses_device_work():
    p = cdg.plan_host(1, 8, 8, 16, 16, 3, 3, 1, 1, 1, "f16")
    with pytest.raises(cdg.CdgError) as e:
        p.dgrad(16, 16, 1024 * 1024)
    assert e.value.status == 7
    with pytest.raises(cdg.CdgError) as e:
        p.prepack_weights(16, 1024 * 1024)
    assert e.value.status == 7
    with pytest.raises(cdg.CdgError) as e:
        p.autotune(16, 16, 1024 * 1024)
    assert e.value.status == 7
    assert p.info()["tuned"] == 0


@pytest.mark.parametrize("reps", [0, -1, 1001])
def test_autotune_argument_errors(reps):
    p = cdg.plan_host(1, 8, 8, 16, 16, 3, 3, 1, 1, 1, "f16")
    with pytest.raises(cdg.CdgError) as e:
        p.autotune(16, 16, 1024 * 1024, reps=reps)
    assert e.value.status == 1
    with pytest.raises(cdg.CdgError) as e:  # a gated plan needs the mask, an ungated one refuses it
        p.autotune(16, 16, 1024 * 1024, relu_mask=4096)
    assert e.value.status == 1


def test_misaligned_and_aliased_pointers_rejected_before_launch():
    p = cdg.plan_host(1, 8, 8, 16, 16, 3, 3, 1, 1, 1, "f16")
    # host-only handles report NO_DEVICE after argument checks of NULLs
    with pytest.raises(cdg.CdgError) as e:
        p.dgrad(0, 16, 32)
    assert e.value.status == 1
    q = cdg.plan_host(1, 8, 8, 16, 16, 3, 3, 1, 1, 1, "f16", relu=True)
    with pytest.raises(cdg.CdgError) as e:  # gated plan without a gate tensor
        q.dgrad(16, 16, 4096, None)
    assert e.value.status == 1


@pytest.mark.parametrize("R,stride,pad,expect", [
    (3, 2, 1, [1, 2, 2, 4]),   # 3x3 stride 2, pad 1: even h = 2p-1+r needs r = 1; odd h takes r in {0, 2}
    (1, 2, 0, [1, 0, 0, 0]),   # 1x1 stride 2: three of four phases receive no tap
    (3, 1, 1, [9]),
    (3, 3, 1, [1, 1, 1, 1, 1, 1, 1, 1, 1]),
    (5, 2, 2, [9, 6, 6, 4]),
])
def test_phase_tap_counts(R, stride, pad, expect):
    p = cdg.plan_host(2, 16, 16, 32, 32, R, R, stride, pad, 1, "bf16")
    info = p.info()
    assert info["num_phases"] == stride * stride
    assert info["phase_taps"] == expect
    assert sum(info["phase_taps"]) == R * R


def test_phase_taps_match_definition_bruteforce():
    """Each tap lands in exactly the phase (h mod s, w mod s) the definition puts it in."""
    for R, S, stride, pad, dil in [(3, 3, 2, 1, 1), (3, 2, 3, 2, 2), (5, 5, 4, 2, 1), (2, 3, 2, 0, 3)]:
        H = W = 24
        p = cdg.plan_host(1, H, W, 8, 8, R, S, stride, pad, dil, "f16")
        counts = [0] * (stride * stride)
        for r in range(R):
            for s in range(S):
                # any p, q: h = p*stride - pad + r*dil -> residue of h
                ph = (-pad + r * dil) % stride
                pw = (-pad + s * dil) % stride
                counts[ph * stride + pw] += 1
        assert p.info()["phase_taps"] == counts


def test_workload_plans():
    for L in ALL:
        p = cdg.plan_host(L.N, L.H, L.W, L.C, L.K, L.R, L.S, L.stride, L.pad, L.dil, L.dtype,
                          relu=L.relu, out_f32=(L.out == "f32"), num_sms=148)
        info = p.info()
        assert (info["P"], info["Q"]) == (L.P, L.Q), L.name
        assert info["smem_bytes"] <= 232448
        assert info["stages"] >= 3
        assert info["tmem_cols"] <= 512 and info["tmem_cols"] >= 2 * info["tile_n"]
        assert info["grid"] <= 148
        if L.R == 1 and L.pad == 0:
            assert info["a_mode"] == 1
        else:
            assert info["box_w"] * info["box_h"] * info["box_n"] <= 128
        assert p.packed_weight_bytes == 2 * L.K * L.R * L.S * L.C
        if info["mma_warps"] == 2 and info["a_mode"] in (0, 1):
            # dual issue over per-tap or row boxes: two rings, two accumulators per MMA warp
            assert info["stages"] % 2 == 0 and info["stages"] >= 4
            assert info["tmem_cols"] >= 4 * info["tile_n"] and info["cta_pair"] == 0
        elif info["mma_warps"] == 2:
            # two MMA warps over the one halo ring with resident weights: at
            # most six halo stages and the weights' barrier
            assert info["a_mode"] == 3 and info["stages"] <= 7 and info["tmem_cols"] >= 4 * info["tile_n"]


def test_halo_resident_weights_when_the_filter_fits(monkeypatch):
    """A stride-1 filter whose packed weights fit resident as halves is kept
    resident by CTA pairs, half in each CTA (a_mode 3, cta_pair 1, the
    default); with pairs off, a filter that fits one CTA beside two halo
    stages is kept resident there.  Otherwise the default is per-tap boxes
    (a_mode 0), with streamed halo weights only when asked (a_mode 2).
    CDG_HALO=0 turns halo mode off, and CDG_PAIR=0 the pairs."""
    monkeypatch.delenv("CDG_HALO", raising=False)
    monkeypatch.delenv("CDG_PAIR", raising=False)
    small = cdg.plan_host(256, 56, 56, 64, 64, 3, 3, 1, 1, 1, "bf16", num_sms=148).info()
    assert small["a_mode"] == 3 and small["cta_pair"] == 1 and small["smem_bytes"] <= 232448
    monkeypatch.setenv("CDG_PAIR", "0")
    small = cdg.plan_host(256, 56, 56, 64, 64, 3, 3, 1, 1, 1, "bf16", num_sms=148).info()
    assert small["a_mode"] == 3 and small["cta_pair"] == 0
    monkeypatch.delenv("CDG_PAIR")
    halves = cdg.plan_host(256, 28, 28, 128, 128, 3, 3, 1, 1, 1, "bf16", num_sms=148).info()
    assert halves["a_mode"] == 3 and halves["cta_pair"] == 1 and halves["smem_bytes"] <= 232448
    # strided, or too large even as halves: per-tap boxes
    assert cdg.plan_host(256, 56, 56, 128, 128, 3, 3, 2, 1, 1, "bf16", num_sms=148).info()["a_mode"] == 0
    assert cdg.plan_host(256, 14, 14, 256, 256, 3, 3, 1, 1, 1, "bf16", num_sms=148).info()["a_mode"] == 0
    # gated by the saved activation: four staging buffers leave no room for the
    # halves, so 128-channel tiles take halo pairs with streamed weight halves
    # (one MMA warp); 64- and 256-channel tiles keep per-tap boxes
    gated = cdg.plan_host(256, 28, 28, 128, 128, 3, 3, 1, 1, 1, "bf16", relu=True, num_sms=148).info()
    assert (gated["a_mode"], gated["cta_pair"], gated["mma_warps"]) == (2, 1, 1)
    for shape in [(256, 56, 56, 64, 64), (256, 14, 14, 256, 256), (256, 7, 7, 512, 512)]:
        g = cdg.plan_host(*shape, 3, 3, 1, 1, 1, "bf16", relu=True, num_sms=148).info()
        assert g["a_mode"] == 0, (shape, g)
    g = cdg.plan_host(256, 28, 28, 128, 128, 3, 3, 1, 1, 1, "bf16", relu_bits=True, num_sms=148).info()
    assert g["a_mode"] != 2  # the packed mask keeps the ungated rules
    for kw in (dict(act="gelu"), dict(act="silu"), dict(sums=2)):  # heavier epilogues keep per-tap boxes
        g = cdg.plan_host(256, 28, 28, 128, 128, 3, 3, 1, 1, 1, "bf16", relu=True, num_sms=148, **kw).info()
        assert g["a_mode"] == 0, (kw, g)
    monkeypatch.setenv("CDG_PAIR", "0")
    assert cdg.plan_host(256, 28, 28, 128, 128, 3, 3, 1, 1, 1, "bf16", num_sms=148).info()["a_mode"] == 0
    monkeypatch.delenv("CDG_PAIR")
    monkeypatch.setenv("CDG_HALO", "1")
    info = cdg.plan_host(256, 28, 28, 128, 128, 3, 3, 1, 1, 1, "bf16", num_sms=148).info()
    assert info["a_mode"] == 2 and info["cta_pair"] == 0
    monkeypatch.setenv("CDG_HALO", "0")
    assert cdg.plan_host(256, 56, 56, 64, 64, 3, 3, 1, 1, 1, "bf16", num_sms=148).info()["a_mode"] == 0
    assert cdg.plan_host(256, 28, 28, 128, 128, 3, 3, 1, 1, 1, "bf16", num_sms=148).info()["a_mode"] == 0


def test_grid_cap_and_dual_halo_option(monkeypatch):
    """CDG_MAX_GRID caps the persistent grid (to an even count for CTA
    pairs); CDG_DUAL=1 gives halo plans with resident weights two MMA warps
    and at most six halo stages."""
    monkeypatch.setenv("CDG_MAX_GRID", "5")
    info = cdg.plan_host(256, 56, 56, 64, 64, 3, 3, 1, 1, 1, "bf16", num_sms=152).info()
    assert info["cta_pair"] == 1 and info["grid"] == 4
    info = cdg.plan_host(256, 56, 56, 64, 64, 1, 1, 1, 0, 1, "bf16", num_sms=152).info()
    assert info["cta_pair"] == 0 and info["grid"] == 5
    info = cdg.plan_host(256, 28, 28, 128, 128, 3, 3, 1, 1, 1, "bf16", num_sms=152).info()
    assert info["cta_pair"] == 1 and info["grid"] == 4
    monkeypatch.setenv("CDG_MAX_GRID", "1")
    assert cdg.plan_host(256, 28, 28, 128, 128, 3, 3, 1, 1, 1, "bf16", num_sms=152).info()["grid"] == 2
    monkeypatch.delenv("CDG_MAX_GRID")
    monkeypatch.setenv("CDG_DUAL", "1")
    for shape in ((256, 56, 56, 64, 64, 3, 3, 1, 1, 1), (256, 28, 28, 128, 128, 3, 3, 1, 1, 1),
                  (16, 12, 12, 64, 64, 3, 3, 1, 1, 1)):
        info = cdg.plan_host(*shape, "bf16", num_sms=152).info()
        assert info["a_mode"] == 3 and info["mma_warps"] == 2 and info["tmem_cols"] <= 512
        assert info["stages"] <= 7  # six halo stages and the resident weights' barrier


def test_four_accumulators_only_where_they_fit_tensor_memory(monkeypatch):
    """CDG_NACC=4 asks halo plans for four accumulators; N tiles over 128
    channels keep two, so no plan asks for more than the 512 TMEM columns."""
    monkeypatch.setenv("CDG_HALO", "1")
    monkeypatch.setenv("CDG_NACC", "4")
    for pair in ("0", "1"):
        monkeypatch.setenv("CDG_PAIR", pair)
        for C in (64, 128, 192, 256, 320, 520):
            for shape in ((256, 14, 14, C, C, 3, 3, 1, 1, 1), (8, 28, 28, C, 64, 3, 3, 2, 1, 1)):
                info = cdg.plan_host(*shape, "bf16", num_sms=152).info()
                assert info["tmem_cols"] <= 512, (shape, pair, info)
                assert info["tmem_cols"] in (32, 64, 128, 256, 512)


def test_halo_boxes_with_cta_pairs_when_asked(monkeypatch):
    """CDG_HALO=1 with CDG_PAIR=1 gives halo boxes with CTA pairs (N tiles of
    64 channels or more) wherever the geometry allows: resident halves where
    half of the filter fits, else streamed weight halves."""
    monkeypatch.setenv("CDG_HALO", "1")
    monkeypatch.setenv("CDG_PAIR", "1")
    info = cdg.plan_host(256, 28, 28, 128, 128, 3, 3, 1, 1, 1, "bf16", num_sms=152).info()
    assert info["a_mode"] == 3 and info["cta_pair"] == 1
    assert info["smem_bytes"] <= 232448 and info["grid"] % 2 == 0
    info = cdg.plan_host(256, 14, 14, 256, 256, 3, 3, 1, 1, 1, "bf16", num_sms=152).info()
    assert info["a_mode"] == 2 and info["cta_pair"] == 1
    info = cdg.plan_host(256, 28, 28, 256, 256, 3, 3, 2, 1, 1, "bf16", num_sms=152).info()
    assert info["a_mode"] == 2 and info["cta_pair"] == 1
    # 64-channel N tiles pair too (32 weight rows per CTA); narrower ones never
    info = cdg.plan_host(256, 56, 56, 64, 64, 3, 3, 1, 1, 1, "bf16", num_sms=152).info()
    assert info["a_mode"] == 3 and info["cta_pair"] == 1 and info["tile_n"] == 64
    info = cdg.plan_host(2, 10, 10, 48, 48, 3, 3, 1, 1, 1, "bf16", num_sms=152).info()
    assert info["tile_n"] < 64 and info["cta_pair"] == 0


@pytest.mark.parametrize("x,bits,pixels,C,dtype,expect", [
    (0, 4096, 4, 64, "bf16", 1),          # NULL activation
    (4096, 0, 4, 64, "bf16", 1),          # NULL mask
    (4096, 8192, -1, 64, "bf16", 1),      # negative pixel count
    (4096, 8192, 4, 0, "bf16", 1),        # no channels
    (4096, 8192, 4, 12, "bf16", 1),       # C not a multiple of 8
    (4096, 8192, 4, 64, 2, 1),            # f32 activations are not packed
    (4104, 8192, 4, 64, "f16", 3),        # x not 16-byte aligned
    (4096, 8200, 4, 64, "f16", 3),        # mask not 16-byte aligned
    (4096, 4352, 4, 64, "bf16", 4),       # mask overlaps x (x spans 512 bytes)
])
def test_pack_relu_mask_argument_errors(x, bits, pixels, C, dtype, expect):
    with pytest.raises(cdg.CdgError) as e:
        cdg.pack_relu_mask(x, bits, pixels, C, dtype)
    assert e.value.status == expect


def test_pack_relu_mask_empty_is_a_no_op():
    cdg.pack_relu_mask(4096, 8192, 0, 64, "bf16")  # no launch, so no device needed


@pytest.mark.parametrize("pixels,C,expect", [
    (1, 8, 16), (1, 128, 16), (1, 136, 32), (3, 256, 96), (10, 64, 160), (0, 64, 0), (7, 2048, 7 * 256)])
def test_relu_mask_bytes(pixels, C, expect):
    """A pixel's C bits fill whole 16-byte units: 16 * ceil(C / 128) bytes."""
    assert cdg.relu_mask_bytes(pixels, C) == expect


@pytest.mark.parametrize("pixels,C", [(-1, 64), (4, 0), (4, 12)])
def test_relu_mask_bytes_invalid(pixels, C):
    with pytest.raises(cdg.CdgError):
        cdg.relu_mask_bytes(pixels, C)


def test_bits_gate_tiles_start_on_mask_units():
    """With the packed mask, N tiles of a wide layer are multiples of 128
    channels, so each tile's mask bytes start on a 16-byte unit."""
    for C in (320, 384, 640, 1024, 2048):
        info = cdg.plan_host(8, 14, 14, C, 64, 1, 1, 1, 0, 1, "bf16", relu_bits=True, num_sms=148).info()
        assert info["tile_n"] % 128 == 0, (C, info["tile_n"])
    assert cdg.plan_host(8, 14, 14, 72, 64, 1, 1, 1, 0, 1, "bf16", relu_bits=True, num_sms=148).info()["tile_n"] == 80


def test_bits_gated_plan_needs_the_mask():
    q = cdg.plan_host(1, 8, 8, 16, 16, 3, 3, 1, 1, 1, "bf16", relu_bits=True)
    with pytest.raises(cdg.CdgError) as e:
        q.dgrad(16, 16, 4096, None)
    assert e.value.status == 1


@pytest.mark.parametrize("gate", ["x", "bits"])
@pytest.mark.parametrize("out_f32", [False, True])
def test_gated_plans_fit_shared_memory(gate, out_f32):
    """Gated plans carry four staging buffers (activation) or a mask-tile
    ring (packed mask) besides the operand ring: every ResNet-50 layer still
    plans within the 227 KB of shared memory with at least three stages, and
    bit-gated N tiles start on 16-byte mask units."""
    from implicit_gemm_dgrad_gb300.workloads import RESNET50_B256
    for L in RESNET50_B256:
        p = cdg.plan_host(L.N, L.H, L.W, L.C, L.K, L.R, L.S, L.stride, L.pad, L.dil, L.dtype,
                          relu=(gate == "x"), relu_bits=(gate == "bits"), out_f32=out_f32, num_sms=148)
        info = p.info()
        assert info["smem_bytes"] <= 232448, (L.name, info)
        assert info["stages"] >= 3, (L.name, info)
        if gate == "bits" and info["tile_n"] < L.C:
            assert info["tile_n"] % 128 == 0, (L.name, info)


WG_GOOD = (2, 8, 8, 16, 16, 3, 3, 1, 1, 1, cdg.BF16, 0, 0)


@pytest.mark.parametrize("field,value,expect", [
    (0, 0, 1), (3, 0, 1), (5, 0, 1), (8, -1, 1), (9, 0, 1), (10, 2, 1), (11, 2, 1), (12, -1, 1),
    (3, 12, 2), (4, 20, 2), (7, 5, 2),
    (1, 1, 0),  # H = 1 with a 3x3 pad-1 filter: P = 1, a valid geometry
])
def test_wgrad_argument_validation(field, value, expect):
    args = list(WG_GOOD)
    args[field] = value
    lib = cdg.load_library()
    h = ctypes.c_void_p()
    rc = lib.cdg_wgrad_plan_host(*args, 148, ctypes.byref(h))
    if h.value:
        lib.cdg_wgrad_destroy(h)
    assert rc == expect


def test_wgrad_input_smaller_than_stride_is_unsupported():
    with pytest.raises(cdg.CdgError) as e:
        cdg.wgrad_plan_host(1, 1, 5, 8, 8, 1, 1, 2, 0, 1, "bf16")
    assert e.value.status == 2


@pytest.mark.parametrize("shape", [
    (256, 56, 56, 64, 64, 1, 1, 1, 0, 1), (256, 56, 56, 64, 64, 3, 3, 1, 1, 1), (256, 28, 28, 128, 128, 3, 3, 1, 1, 1),
    (256, 14, 14, 256, 256, 3, 3, 1, 1, 1), (256, 7, 7, 512, 512, 3, 3, 1, 1, 1), (256, 56, 56, 128, 128, 3, 3, 2, 1, 1),
    (256, 14, 14, 1024, 2048, 1, 1, 2, 0, 1), (3, 9, 9, 8, 8, 3, 3, 2, 1, 1), (2, 7, 6, 320, 72, 3, 2, 1, 2, 2)])
def test_wgrad_plans(shape):
    """Position blocks hold exactly 64 positions; the splits divide the
    blocks without an empty range; the workspace holds every split's dW;
    shared memory and tensor memory stay within the SM's limits."""
    N, H, W, C, K, R, S, st, pd, dl = shape
    p = cdg.wgrad_plan_host(*shape, num_sms=148)
    i = p.info()
    qb, pb, nb = i["pos_box"]
    assert qb * pb * nb == 64
    P, Q = i["P"], i["Q"]
    assert i["blocks"] == -(-Q // qb) * -(-P // pb) * -(-N // nb)
    assert 1 <= i["splits"] <= i["blocks"]
    G = i["taps_per_item"]
    assert 1 <= G and G * i["tile_n"] <= 256
    if -(-C // i["tile_n"]) > 1:
        assert G == 1
    if i["x_major"]:  # M tiles of two (tap, 64-channel slice of x) units, N = the dY channels
        tiles = -(-(R * S * -(-C // 64)) // 2)
    else:
        tiles = -(-(R * S) // G) * -(-K // 128) * -(-C // i["tile_n"])
    assert i["work_items"] == i["splits"] * tiles
    assert i["work_items"] <= 148 or i["splits"] == 1
    assert p.workspace_bytes == i["splits"] * K * R * S * C * 4
    assert i["tile_n"] % 64 == 0 and i["tile_n"] <= 256
    assert i["smem_bytes"] <= 232448 and i["stages"] >= 3
    assert 2 * G * i["tile_n"] <= i["tmem_cols"] <= 512


def test_wgrad_explicit_splits_are_capped_by_the_blocks():
    p = cdg.wgrad_plan_host(1, 8, 8, 16, 16, 3, 3, 1, 1, 1, "bf16", splits=1000)
    assert p.info()["splits"] == p.info()["blocks"] == 1


def test_wgrad_host_plan_refuses_device_work():
    p = cdg.wgrad_plan_host(1, 8, 8, 16, 16, 3, 3, 1, 1, 1, "bf16")
    with pytest.raises(cdg.CdgError) as e:
        p.wgrad(4096, 8192, 1 << 20, 1 << 24)
    assert e.value.status == 7


def test_wait_limit_and_withheld_load_arguments():
    """The wait limit takes 0.1 ms .. 60 s; the test-only withheld load takes
    stage >= -1 and only plans whose loaders honour it (per-tap or row boxes,
    no CTA pairs, no halo boxes)."""
    p = cdg.plan_host(2, 12, 12, 64, 64, 3, 3, 1, 1, 1, "bf16", num_sms=148)
    assert p.info()["a_mode"] == 3  # halo boxes with resident weights
    for bad in (0, 99_999, 60_000_000_001):
        with pytest.raises(cdg.CdgError):
            p.set_wait_limit(bad)
    p.set_wait_limit(100_000)
    p.set_wait_limit(60_000_000_000)
    with pytest.raises(cdg.CdgError) as e:
        p.withhold_load_for_test(0)
    assert e.value.status == 2
    p.withhold_load_for_test(-1)  # restoring is always allowed
    with pytest.raises(cdg.CdgError):
        p.withhold_load_for_test(-2)
    pair = cdg.plan_host(2, 14, 14, 256, 256, 3, 3, 1, 1, 1, "bf16", num_sms=148)
    assert pair.info()["cta_pair"] == 1
    with pytest.raises(cdg.CdgError):
        pair.withhold_load_for_test(3)
    rows = cdg.plan_host(4, 14, 14, 256, 64, 1, 1, 1, 0, 1, "bf16", num_sms=148)
    rows.withhold_load_for_test(1)


def test_sum_plans_reserve_the_partials_and_size_the_workspace():
    """Plans with per-channel sums reserve 2 KB more shared memory for the
    epilogue warps' partials and need a workspace of one row per SM."""
    base = cdg.plan_host(4, 14, 14, 256, 64, 1, 1, 1, 0, 1, "bf16", num_sms=148)
    s1 = cdg.plan_host(4, 14, 14, 256, 64, 1, 1, 1, 0, 1, "bf16", num_sms=148, sums=1)
    s2 = cdg.plan_host(4, 14, 14, 256, 64, 1, 1, 1, 0, 1, "bf16", num_sms=148, relu=True, sums=2)
    assert base.sums_workspace_bytes == 0
    assert s1.sums_workspace_bytes == 148 * 256 * 4 and s2.sums_workspace_bytes == 148 * 2 * 256 * 4
    assert s1.info()["smem_bytes"] <= 232448 and s2.info()["smem_bytes"] <= 232448
    for p in (base, s1, s2):
        assert p.info()["stages"] >= 2
    with pytest.raises(cdg.CdgError) as e:  # plain cdg_dgrad refuses a plan with sums
        s1.dgrad(1 << 20, 2 << 20, 3 << 20)
    assert e.value.status == 1
    with pytest.raises(cdg.CdgError) as e:  # and a plan without them has no sums to give
        base.dgrad_sums(1 << 20, 2 << 20, 3 << 20, 4 << 20, 5 << 20)
    assert e.value.status == 1
    with pytest.raises(cdg.CdgError) as e:  # host-only plans refuse device work after the checks
        s1.dgrad_sums(1 << 20, 2 << 20, 3 << 20, 4 << 20, 5 << 20)
    assert e.value.status == 7
