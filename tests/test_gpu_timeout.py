"""The bounded-wait failure path on the GPU, exercised without any fault.

A test-only plan option withholds one operand load (in each CTA, the
pipeline stage with a given sequence number gets neither its tensor copies
nor their byte count), and the plan's wait limit is lowered to 2 ms.  The MMA
warp's wait for that stage then runs out: the launch must record
CDG_ERR_TIMEOUT in the plan's status word, stop every role, drain its own
copies and tensor-core work, release its tensor memory and return, writing
nothing outside dX.  Right after, a normal launch of the same plan must give
the oracle's result: the context and the plan stay usable.  Every wait in the
kernel is bounded, so nothing here can hang the GPU."""
import numpy as np
import pytest

import implicit_gemm_dgrad_gb300 as cdg
import oracle
from implicit_gemm_dgrad_gb300.workloads import Layer

from gpu_util import GpuRun, assert_close, torch_cuda

pytestmark = pytest.mark.gpu

ERR_TIMEOUT = 6

CASES = [
    # (layer, planner overrides, withheld stage, what the plan must be)
    # two MMA warps; the very first stage of each CTA is withheld
    (Layer("to_3x3_c64_dual", 2, 12, 12, 64, 64, 3, 3, 1, 1, 1, dtype="bf16", workload=12, index=0),
     "CDG_HALO=0", 0, {"a_mode": 0, "mma_warps": 2}),
    # one MMA warp, two tiles in most CTAs: the second tile's fourth stage is
    # withheld, after the first tile's epilogue has stored its output
    (Layer("to_3x3_c64_second_tile", 160, 12, 12, 64, 64, 3, 3, 1, 1, 1, dtype="bf16", workload=12, index=1),
     "CDG_HALO=0 CDG_DUAL=0", 12, {"a_mode": 0, "mma_warps": 1}),
    # dY rows as a matrix (1x1), four K blocks per tile
    (Layer("to_1x1_rows", 4, 14, 14, 64, 256, 1, 1, 1, 0, 1, dtype="bf16", workload=12, index=2),
     "", 1, {"a_mode": 1}),
    # strided phases and the gate from the saved activation, whose tiles loader
    # warp 3 loads ahead; those in flight must land before the CTA leaves
    (Layer("to_3x3s2_c256_relu", 2, 14, 14, 256, 128, 3, 3, 2, 1, 1, dtype="bf16", relu=True, workload=12,
           index=3), "CDG_PAIR=0", 3, {"a_mode": 0, "cta_pair": 0}),
]


@pytest.mark.parametrize("L,env,stage,reach", CASES, ids=lambda v: v.name if isinstance(v, Layer) else None)
def test_withheld_load_times_out_and_plan_stays_usable(L, env, stage, reach, monkeypatch):
    for kv in env.split():
        key, val = kv.split("=")
        monkeypatch.setenv(key, val)
    torch = torch_cuda()
    run = GpuRun(L)
    info = run.plan.info()
    for k, v in reach.items():
        assert info[k] == v, (k, info)
    run.plan.set_wait_limit(2_000_000)       # 2 ms
    run.plan.withhold_load_for_test(stage)
    run.run()
    torch.cuda.synchronize()
    assert run.plan.device_status() == ERR_TIMEOUT
    assert run.plan.device_status() == 0      # read and cleared
    assert run.out.guards_intact(), "aborted launch wrote outside dX"
    # the context is usable: a plain torch kernel and a normal launch of the same plan
    assert int(torch.arange(1000, device="cuda").sum().item()) == 499500
    run.plan.withhold_load_for_test(-1)
    run.plan.set_wait_limit(4_000_000_000)
    run.out.body().fill_(0xA5)
    run.run()
    got = run.result()
    assert run.plan.device_status() == 0
    assert run.out.guards_intact()
    ref = oracle.dgrad(run.dY, run.W, L.H, L.W, L.stride, L.pad, L.dil, x=run.x, dtype=L.dtype)
    assert_close(got, ref, run.odt, L.name)


def test_a_short_limit_alone_does_not_time_out(monkeypatch):
    """A 2 ms limit with every load issued: the launch completes normally."""
    monkeypatch.setenv("CDG_HALO", "0")
    L = CASES[1][0]
    run = GpuRun(L)
    run.plan.set_wait_limit(2_000_000)
    run.run()
    got = run.result()
    assert run.plan.device_status() == 0
    ref = oracle.dgrad(run.dY, run.W, L.H, L.W, L.stride, L.pad, L.dil, dtype=L.dtype)
    assert_close(got, ref, run.odt, L.name)
