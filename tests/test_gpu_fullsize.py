"""Parity at the full ResNet-50 batch-256 sizes, in the launch configuration the
benchmark times: EVERY element of dX against the oracle, which evaluates the
whole batch image chunk by image chunk (images are independent, so a chunk of
dY gives exactly that chunk of dX).  Also checked over the whole of dX: guard
bands intact, the tap-less phases of the 1x1 stride-2 layers +0.0 exactly, and
for the gated layers the two-sided zero pattern -- +0.0 at every position the
saved activation masks, and no zero at any other position unless the oracle's
value there rounds to zero in bf16."""
import numpy as np
import pytest

import oracle
from implicit_gemm_dgrad_gb300.workloads import FUSED_RELU, RESNET50_B256

from gpu_util import GpuRun, assert_close, check_gate_zero_pattern, decode_out, torch_cuda

pytestmark = pytest.mark.gpu

CHUNK_ELEMENTS = 1 << 24  # dX elements compared per chunk (bounds host memory)


@pytest.mark.parametrize("L", RESNET50_B256 + FUSED_RELU, ids=lambda L: L.name)
def test_full_size_layer(L):
    torch = torch_cuda()
    run = GpuRun(L)
    run.run()
    torch.cuda.synchronize()
    assert run.status() == 0
    assert run.out.guards_intact(), "write outside dX"
    per_image = L.H * L.W * L.C
    bits16 = run.out.body().view(torch.int16).view(L.N, per_image)
    chunk = max(1, CHUNK_ELEMENTS // per_image)
    masked = exact_zero = 0
    for n0 in range(0, L.N, chunk):
        n1 = min(L.N, n0 + chunk)
        x = None if run.x is None else run.x[n0:n1]
        ref = oracle.dgrad(run.dY[n0:n1], run.W, L.H, L.W, L.stride, L.pad, L.dil, x=x, dtype=L.dtype)
        raw = bits16[n0:n1].cpu().numpy()
        got = decode_out(raw.view(np.uint8), run.odt).reshape(ref.shape)
        assert_close(got, ref, run.odt, f"{L.name} images {n0}..{n1 - 1}")
        if L.R == 1 and L.stride == 2:  # phases no tap reaches: +0.0 bit-exactly
            b = raw.reshape(n1 - n0, L.H, L.W, L.C)
            assert not b[:, 1::2].any() and not b[:, :, 1::2].any()
        if L.relu:
            counts = check_gate_zero_pattern(raw.view(np.uint8), x, ref, run.odt, L.dtype)
            masked += counts["masked"]
            exact_zero += counts["unmasked_oracle_zero"]
    if L.relu:
        # about half of x = relu(N(0,1)) is zero; the oracle's unmasked values are never exactly zero here
        assert 0.45 < masked / (L.N * per_image) < 0.55
        assert exact_zero == 0
