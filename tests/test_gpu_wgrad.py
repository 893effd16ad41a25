"""GPU parity of wgrad (the weight gradient): the sm_103a split-K kernel and
its ordered reduction against the CPU oracle's definition, element by element,
with dW surrounded by sentinel guard bands and pre-filled with NaN.

Bar: |gpu - oracle| <= tol * max(1, |oracle|), tol 1e-2 for fp16/bf16 dW and
2e-3 for fp32 dW (fp32 accumulation of products of fp16/bf16 inputs)."""
import os

import numpy as np
import pytest

import oracle
from implicit_gemm_dgrad_gb300 import synth

from gpu_util import GuardedOutput, assert_close, decode_out, to_dev

pytestmark = pytest.mark.gpu

# N, H, W, C, K, R, S, stride, pad, dil, dtype, out, splits (0: planner)
CASES = [
    (2, 7, 6, 16, 24, 3, 3, 1, 1, 1, "bf16", "same", 0),
    (2, 9, 9, 40, 72, 3, 3, 2, 1, 1, "f16", "same", 2),
    (4, 8, 8, 64, 128, 1, 1, 1, 0, 1, "bf16", "same", 0),
    (2, 11, 10, 96, 200, 3, 2, 1, 2, 2, "bf16", "f32", 3),
    (3, 12, 12, 320, 64, 3, 3, 2, 1, 1, "bf16", "same", 5),
    (64, 7, 7, 256, 128, 3, 3, 1, 1, 1, "bf16", "same", 0),
    (2, 14, 14, 256, 256, 1, 1, 2, 0, 1, "bf16", "same", 1),
    (2, 10, 9, 64, 64, 5, 1, 1, 2, 1, "bf16", "same", 0),   # taps in groups of 3 and 2
    (2, 9, 8, 192, 40, 1, 1, 1, 0, 1, "bf16", "f32", 0),    # x-major: 3 slices of x, 40 dY channels
    (3, 10, 10, 72, 32, 1, 1, 2, 0, 1, "f16", "same", 2),   # x-major: 2 slices, stride 2
    (4, 12, 12, 256, 64, 1, 1, 1, 0, 1, "bf16", "same", 0), # x-major: the 1x1 256 -> 64 shape
]


def _name(c):
    return "N{}H{}W{}C{}K{}R{}S{}s{}p{}d{}{}{}sp{}".format(*c)


def _inputs(c, seed):
    N, H, W, C, K, R, S, st, pd, dl, dtype = c[:11]
    P, Q = oracle.out_extent(H, R, st, pd, dl), oracle.out_extent(W, S, st, pd, dl)
    rng = np.random.default_rng(seed)
    dY = synth.to_bits(rng.standard_normal((N, P, Q, K)).astype(np.float32), dtype)
    x = synth.to_bits(rng.standard_normal((N, H, W, C)).astype(np.float32), dtype)
    return dY, x


def _run(c, seed=5):
    import torch
    import implicit_gemm_dgrad_gb300 as cdg
    N, H, W, C, K, R, S, st, pd, dl, dtype, out, splits = c
    dY, x = _inputs(c, seed)
    p = cdg.wgrad_plan(N, H, W, C, K, R, S, st, pd, dl, dtype, out_f32=(out == "f32"), splits=splits)
    odt = "f32" if out == "f32" else dtype
    dW = GuardedOutput(K * R * S * C, 4 if odt == "f32" else 2)
    ws = torch.full((p.workspace_bytes // 4,), float("nan"), dtype=torch.float32, device="cuda")
    p.wgrad(to_dev(dY, dtype), to_dev(x, dtype), dW.ptr, ws)
    torch.cuda.synchronize()
    assert p.device_status() == 0
    assert dW.guards_intact(), "write outside dW"
    got = decode_out(dW.body().cpu().numpy(), odt).reshape(K, R, S, C)
    ref = oracle.wgrad(dY, x, R, S, st, pd, dl, dtype=dtype)
    return p, got, ref, odt


@pytest.mark.parametrize("c", CASES, ids=_name)
def test_wgrad_matches_oracle(c):
    p, got, ref, odt = _run(c)
    dump = os.environ.get("CDG_TEST_DUMP")
    try:
        assert_close(got, ref, odt, _name(c))
    except AssertionError:
        if dump:
            np.savez(os.path.join(dump, f"wgrad_{_name(c)}.npz"), got=got, ref=ref, info=str(p.info()))
        raise


def test_wgrad_is_deterministic():
    """The split partials are added in a fixed order: two runs give the same bits."""
    c = CASES[4]
    _, a, _, _ = _run(c)
    _, b, _, _ = _run(c)
    assert np.array_equal(a, b)


def test_wgrad_splits_agree():
    """One split and several splits compute the same sum (to rounding)."""
    c = list(CASES[1])
    c[12] = 1
    _, one, ref, odt = _run(tuple(c))
    c[12] = 3
    _, three, _, _ = _run(tuple(c))
    assert_close(one, ref, odt, "one split")
    assert_close(three, ref, odt, "three splits")


FULL = ["L01_1x1_64-64_56", "L03_1x1_256-64_56", "L04_3x3_64_56", "L06_3x3s2_128_56-28", "L20_1x1_2048-512_7",
        "L21_3x3_512_7"]


@pytest.mark.parametrize("name", FULL)
def test_wgrad_full_size_sampled(name):
    """Batch-256 ResNet-50 layers in the configuration bench.py --op wgrad
    times (planner defaults: up to 152 splits, tap groups, 1x1x64 position
    boxes), checked at 64 sampled filter elements (corners included) against
    the oracle's element-by-element definition."""
    import torch
    import implicit_gemm_dgrad_gb300 as cdg
    from implicit_gemm_dgrad_gb300.workloads import by_name
    L = by_name(name)
    dY, _, x = synth.make_inputs(L.shape(), L.dtype, L.dist, L.workload, L.index, with_x=True)
    p = cdg.wgrad_plan(L.N, L.H, L.W, L.C, L.K, L.R, L.S, L.stride, L.pad, L.dil, L.dtype)
    dW = GuardedOutput(L.K * L.R * L.S * L.C, 2)
    ws = torch.empty(p.workspace_bytes // 4, dtype=torch.float32, device="cuda")
    p.wgrad(to_dev(dY, L.dtype), to_dev(x.reshape(-1), L.dtype), dW.ptr, ws)
    torch.cuda.synchronize()
    assert p.device_status() == 0 and dW.guards_intact()
    got = decode_out(dW.body().cpu().numpy(), L.dtype).reshape(L.K, L.R, L.S, L.C)
    rng = np.random.default_rng(97)
    idx = np.stack([rng.integers(0, L.K, 62), rng.integers(0, L.R, 62), rng.integers(0, L.S, 62),
                    rng.integers(0, L.C, 62)], axis=1)
    idx = np.concatenate([idx, [[0, 0, 0, 0], [L.K - 1, L.R - 1, L.S - 1, L.C - 1]]]).astype(np.int32)
    ref = oracle.wgrad_elements(dY, x, L.R, L.S, idx, L.stride, L.pad, L.dil, dtype=L.dtype)
    assert_close(got[idx[:, 0], idx[:, 1], idx[:, 2], idx[:, 3]], ref, L.dtype, name)


def test_wgrad_rejects_misaligned_and_aliased_tensors_before_launch():
    """Pointer checks of cdg_wgrad on a device plan: 16-byte alignment of every
    tensor and no overlap of dW or the workspace with an input or each other;
    nothing is launched when they fail."""
    import torch
    import implicit_gemm_dgrad_gb300 as cdg
    p = cdg.wgrad_plan(1, 8, 8, 16, 16, 3, 3, 1, 1, 1, "bf16")
    dY = torch.zeros(8 * 8 * 16 + 64, dtype=torch.int16, device="cuda")
    x = torch.zeros(8 * 8 * 16 + 64, dtype=torch.int16, device="cuda")
    dW = torch.zeros(16 * 9 * 16 + 64, dtype=torch.int16, device="cuda")
    ws = torch.zeros(p.workspace_bytes // 4 + 64, dtype=torch.float32, device="cuda")
    base = (dY.data_ptr(), x.data_ptr(), dW.data_ptr(), ws.data_ptr())
    for i in range(4):  # one pointer 8 bytes off alignment at a time
        args = list(base)
        args[i] += 8
        with pytest.raises(cdg.CdgError) as e:
            p.wgrad(*args)
        assert e.value.status == 3
    with pytest.raises(cdg.CdgError) as e:  # dW inside the workspace
        p.wgrad(base[0], base[1], base[3], base[3])
    assert e.value.status == 4
    with pytest.raises(cdg.CdgError) as e:  # workspace over dY
        p.wgrad(base[0], base[1], base[2], base[0])
    assert e.value.status == 4
    torch.cuda.synchronize()
    assert p.device_status() == 0


def test_wgrad_plans_with_different_footprints_coexist():
    """A plan made after another, with less shared memory, leaves the earlier
    plan launchable (the kernel's shared-memory limit is not lowered)."""
    import torch
    import implicit_gemm_dgrad_gb300 as cdg
    big, small = CASES[5], CASES[1]  # 227 KB (256-channel tiles) and less (three 64-channel taps)
    N, H, W, C, K, R, S, st, pd, dl, dtype, _, splits = big
    a = cdg.wgrad_plan(N, H, W, C, K, R, S, st, pd, dl, dtype, splits=splits)
    b = cdg.wgrad_plan(*small[:11], splits=small[12])
    assert a.info()["smem_bytes"] > b.info()["smem_bytes"]
    dY, x = _inputs(big, 11)
    dW = GuardedOutput(K * R * S * C, 2)
    ws = torch.empty(a.workspace_bytes // 4, dtype=torch.float32, device="cuda")
    a.wgrad(to_dev(dY, dtype), to_dev(x, dtype), dW.ptr, ws)  # the earlier plan, launched last
    torch.cuda.synchronize()
    assert a.device_status() == 0 and dW.guards_intact()
    got = decode_out(dW.body().cpu().numpy(), dtype).reshape(K, R, S, C)
    assert_close(got, oracle.wgrad(dY, x, R, S, st, pd, dl, dtype=dtype), dtype, "earlier plan after a smaller one")
