"""The allocation-free entry point, cdg_dgrad_noalloc.

It serves callers that may not allocate device memory: it packs the filter
into a scratch array compiled into the library and runs the same dgrad kernel.
Its output must match the oracle (within the tolerance of every other parity
test, with the gate's zero pattern checked in both directions) and the regular
path (cdg_prepack_weights + cdg_dgrad into caller buffers) on two calls in a
row -- the second call finds the scratch holding the first call's packed
weights and must still be right.  After each call the scratch status word
(cdg_dgrad_noalloc_status) must read CDG_OK.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test; it passes run alone as well.
"""
import numpy as np
import pytest

import implicit_gemm_dgrad_gb300 as cdg
import oracle
from implicit_gemm_dgrad_gb300.workloads import Layer

from gpu_util import GpuRun, assert_close, check_gate_zero_pattern, decode_out

CASES = [
    Layer("noalloc_3x3_s1_f16_f32out", 2, 9, 7, 24, 40, 3, 3, 1, 1, 1, dtype="f16", out="f32", workload=7, index=0),
    Layer("noalloc_3x3_s2_bf16_relu", 2, 14, 14, 64, 96, 3, 3, 2, 1, 1, dtype="bf16", relu=True, workload=7, index=1),
    Layer("noalloc_1x1_s2_bf16", 4, 12, 10, 256, 512, 1, 1, 2, 0, 1, dtype="bf16", workload=7, index=2),
    # 256 channels and 36 pipeline stages per tile: the planner chooses CTA pairs
    Layer("noalloc_3x3_s1_bf16_pairs", 2, 14, 14, 256, 256, 3, 3, 1, 1, 1, dtype="bf16", workload=7, index=3),
]


def test_noalloc_rejects_oversized_filter_before_any_launch():
    # 3x3, 1024 -> 1024 channels: 18 MiB of packed weights, above the 8 MiB scratch.
    p = cdg.plan_host(1, 8, 8, 1024, 1024, 3, 3, 1, 1, 1, "bf16", num_sms=148)
    assert p.packed_weight_bytes > cdg.NOALLOC_MAX_WEIGHT_BYTES
    with pytest.raises(cdg.CdgError) as e:
        # the pointers are never touched: the size check comes first
        p.dgrad_noalloc(1 << 20, 2 << 20, 3 << 20)
    assert e.value.status == cdg.ERR_SCRATCH_TOO_SMALL
    assert "8 MiB" in cdg.status_string(cdg.ERR_SCRATCH_TOO_SMALL)


@pytest.mark.gpu
@pytest.mark.parametrize("host_planned", [True, False])
@pytest.mark.parametrize("L", CASES, ids=lambda L: L.name)
def test_noalloc_matches_oracle_and_regular_path_twice(L, host_planned):
    import torch
    run = GpuRun(L)                       # regular path: cdg_plan, prepack, cdg_dgrad
    run.run()
    regular = run.result()
    ref = oracle.dgrad(run.dY, run.W, L.H, L.W, L.stride, L.pad, L.dil, x=run.x, dtype=L.dtype)
    assert_close(regular, ref, run.odt, f"{L.name} regular path")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if host_planned:
        p = cdg.plan_host(L.N, L.H, L.W, L.C, L.K, L.R, L.S, L.stride, L.pad, L.dil, L.dtype,
                          relu=L.relu, out_f32=(L.out == "f32"), num_sms=sms)
    else:
        p = run.plan
    if L.name.endswith("pairs"):
        assert p.info()["cta_pair"] == 1
    esize = 4 if run.odt == "f32" else 2
    out = torch.empty(L.N * L.H * L.W * L.C * esize, dtype=torch.uint8, device="cuda")
    assert cdg.Plan.noalloc_status() == 0  # clears anything an earlier test left
    for call in range(2):
        out.fill_(0xA5)                   # stale contents must not leak through
        p.dgrad_noalloc(run.d_dY, run.d_W, out, run.d_x)
        assert cdg.Plan.noalloc_status() == 0, f"{L.name} call {call}: device status"
        raw = out.cpu().numpy()
        got = decode_out(raw, run.odt).reshape(ref.shape)
        assert_close(got, ref, run.odt, f"{L.name} call {call} against the oracle")
        assert_close(got, regular, run.odt, f"{L.name} call {call} against the regular path")
        if L.relu:
            check_gate_zero_pattern(raw, run.x, ref, run.odt, L.dtype)
    if host_planned and p.info()["cta_pair"]:
        # the first call sized the host plan's pair grid by what the device holds at once
        assert p.info()["grid"] <= run.plan.info()["grid"]
