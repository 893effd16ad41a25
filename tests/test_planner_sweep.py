"""Both planners over 300 seeded random shapes, every epilogue and output
mode: a shape is either rejected with a documented status (invalid argument
or unsupported) or planned within the SM's limits -- shared memory within the
227 KB opt-in, tensor memory within 512 columns, a grid of 1 to #SMs, tiles
within the MMA's N range.  No device is needed."""
import numpy as np
import pytest

import implicit_gemm_dgrad_gb300 as cdg

SMS = 148


def _shapes(n, seed=2026):
    rng = np.random.default_rng(seed)
    for _ in range(n):
        yield dict(N=int(rng.integers(1, 9)), H=int(rng.integers(1, 40)), W=int(rng.integers(1, 40)),
                   C=int(8 * rng.integers(1, 80)), K=int(8 * rng.integers(1, 80)), R=int(rng.integers(1, 8)),
                   S=int(rng.integers(1, 8)), stride=int(rng.integers(1, 5)), pad=int(rng.integers(0, 4)),
                   dil=int(rng.integers(1, 4)), dtype=["f16", "bf16"][int(rng.integers(0, 2))],
                   epi=int(rng.integers(0, 3)), out_f32=bool(rng.integers(0, 2)))


def _args(s):
    return (s["N"], s["H"], s["W"], s["C"], s["K"], s["R"], s["S"], s["stride"], s["pad"], s["dil"], s["dtype"])


def test_dgrad_planner_sweep():
    planned = 0
    for s in _shapes(300):
        try:
            p = cdg.plan_host(*_args(s), relu=s["epi"] == 1, relu_bits=s["epi"] == 2, out_f32=s["out_f32"],
                              num_sms=SMS)
        except cdg.CdgError as e:
            assert e.status in (1, 2), (s, e.status)
            continue
        i = p.info()
        assert i["smem_bytes"] <= 232448 and i["stages"] >= 2, (s, i)
        assert i["tmem_cols"] <= 512 and 1 <= i["grid"] <= SMS and i["work_items"] >= 1, (s, i)
        assert 16 <= i["tile_n"] <= 256 and i["tile_n"] % 16 == 0, (s, i)
        assert (i["P"], i["Q"]) == p.output_dims
        planned += 1
    assert planned > 150  # most random shapes are valid


def test_wgrad_planner_sweep():
    planned = 0
    for s in _shapes(300, seed=2027):
        try:
            w = cdg.wgrad_plan_host(*_args(s), out_f32=s["out_f32"], num_sms=SMS)
        except cdg.CdgError as e:
            assert e.status in (1, 2), (s, e.status)
            continue
        i = w.info()
        assert i["smem_bytes"] <= 232448 and i["stages"] >= 2, (s, i)
        assert i["tmem_cols"] <= 512 and 1 <= i["grid"] <= SMS, (s, i)
        assert i["taps_per_item"] * i["tile_n"] <= 256 and i["tile_n"] % 64 == 0, (s, i)
        assert 1 <= i["splits"] <= i["blocks"] and np.prod(i["pos_box"]) == 64, (s, i)
        assert w.workspace_bytes == i["splits"] * s["K"] * s["R"] * s["S"] * s["C"] * 4
        planned += 1
    assert planned > 150


def test_no_192_channel_tiles_unless_asked(monkeypatch):
    """For C > 256 the planner takes 256-channel N tiles (or the multiple of 64
    with the least padding); 192-channel tiles only when asked (CDG_BN=192),
    e.g. the 1x1 512 -> 2048 layer at 7x7 as 147 pair items instead of 98."""
    import implicit_gemm_dgrad_gb300 as cdg
    from implicit_gemm_dgrad_gb300.workloads import RESNET50_B256
    for L in RESNET50_B256:
        inf = cdg.plan_host(L.N, L.H, L.W, L.C, L.K, L.R, L.S, L.stride, L.pad, L.dil, L.dtype, num_sms=152).info()
        assert inf["tile_n"] in (64, 128, 256), (L.name, inf["tile_n"])
        if L.name.startswith("L19"):
            assert (inf["tile_n"], inf["cta_pair"], inf["work_items"]) == (256, 1, 98)
    monkeypatch.setenv("CDG_BN", "192")
    inf = cdg.plan_host(256, 7, 7, 512, 2048, 1, 1, 1, 0, 1, "bf16", num_sms=152).info()
    assert (inf["tile_n"], inf["cta_pair"], inf["work_items"]) == (192, 1, 147)


def test_wgrad_x_major_rule():
    """wgrad tiles are x-major exactly when the dY channels fill at most half
    of a 128-row M tile (K <= 64), the filter is 1x1 and x has at least two
    64-channel slices to pair; then N = 64 and M tiles = ceil(slices / 2)."""
    for s in _shapes(300, seed=2029):
        try:
            w = cdg.wgrad_plan_host(*_args(s), out_f32=s["out_f32"], num_sms=SMS)
        except cdg.CdgError:
            continue
        i = w.info()
        units = s["R"] * s["S"] * -(-s["C"] // 64)
        want = int(s["K"] <= 64 and s["R"] * s["S"] == 1 and units >= 2)
        assert i["x_major"] == want, (s, i)
        if want:
            assert i["tile_n"] == 64 and i["taps_per_item"] == 1, (s, i)
            assert i["work_items"] == i["splits"] * -(-units // 2), (s, i)
