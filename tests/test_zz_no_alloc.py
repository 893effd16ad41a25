"""The allocation-free entry point, cdg_dgrad_noalloc.

It serves callers that may not allocate device memory: it packs the filter
into a scratch array compiled into the library and runs the same dgrad kernel.
Its output must match the regular path (cdg_prepack_weights + cdg_dgrad into
caller buffers) on two calls in a row -- the second call finds the scratch
holding the first call's packed weights and must still be right.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test; it passes run alone as well.
"""
import numpy as np
import pytest

import implicit_gemm_dgrad_gb300 as cdg
from implicit_gemm_dgrad_gb300.workloads import Layer

from gpu_util import GpuRun, assert_close, decode_out

CASES = [
    Layer("noalloc_3x3_s1_f16_f32out", 2, 9, 7, 24, 40, 3, 3, 1, 1, 1, dtype="f16", out="f32", workload=7, index=0),
    Layer("noalloc_3x3_s2_bf16_relu", 2, 14, 14, 64, 96, 3, 3, 2, 1, 1, dtype="bf16", relu=True, workload=7, index=1),
    Layer("noalloc_1x1_s2_bf16", 4, 12, 10, 256, 512, 1, 1, 2, 0, 1, dtype="bf16", workload=7, index=2),
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
def test_noalloc_matches_regular_path_twice(L, host_planned):
    import torch
    run = GpuRun(L)                       # regular path: cdg_plan, prepack, cdg_dgrad
    run.run()
    ref = run.result()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if host_planned:
        p = cdg.plan_host(L.N, L.H, L.W, L.C, L.K, L.R, L.S, L.stride, L.pad, L.dil, L.dtype,
                          relu=L.relu, out_f32=(L.out == "f32"), num_sms=sms)
    else:
        p = run.plan
    esize = 4 if run.odt == "f32" else 2
    out = torch.empty(L.N * L.H * L.W * L.C * esize, dtype=torch.uint8, device="cuda")
    for call in range(2):
        out.fill_(0xA5)                   # stale contents must not leak through
        p.dgrad_noalloc(run.d_dY, run.d_W, out, run.d_x)
        torch.cuda.synchronize()
        got = decode_out(out.cpu().numpy(), run.odt).reshape(ref.shape)
        assert_close(got, ref, run.odt, f"{L.name} call {call}")
