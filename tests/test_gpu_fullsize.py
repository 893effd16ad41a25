"""Parity at the full ResNet-50 batch-256 sizes, in the launch configuration the
benchmark times: sampled output pixels against the oracle (evaluated pixel by
pixel), plus properties checked over the whole of dX on the device -- every
element written and finite, guard bands intact, empty phases exactly +0.0,
gated-off positions exactly +0.0."""
import numpy as np
import pytest

import oracle
from implicit_gemm_dgrad_gb300.workloads import FUSED_RELU, RESNET50_B256

from gpu_util import GpuRun, assert_close, decode_out, torch_cuda

pytestmark = pytest.mark.gpu


def sample_pixels(L, count=768, seed=0):
    rng = np.random.default_rng(seed)
    pix = [rng.integers(0, L.N, count), rng.integers(0, L.H, count), rng.integers(0, L.W, count)]
    pix = np.stack(pix, axis=1)
    corners = []
    for n in (0, L.N - 1):
        for h in (0, 1, L.H - 2, L.H - 1):
            for w in (0, 1, L.W - 2, L.W - 1):
                corners.append((n, h, w))
    return np.concatenate([pix, np.array(corners)], axis=0).astype(np.int32)


@pytest.mark.parametrize("L", RESNET50_B256 + FUSED_RELU, ids=lambda L: L.name)
def test_full_size_layer(L):
    torch = torch_cuda()
    run = GpuRun(L)
    run.run()
    torch.cuda.synchronize()
    assert run.status() == 0
    assert run.out.guards_intact(), "write outside dX"
    body = run.out.body()
    bits16 = body.view(torch.int16).view(L.N, L.H, L.W, L.C)
    vals = bits16.view(torch.bfloat16 if L.dtype == "bf16" else torch.float16)
    assert bool(torch.isfinite(vals).all().item()), "dX has unwritten (NaN-prefilled) or non-finite elements"
    if L.R == 1 and L.stride == 2:
        assert bool((bits16[:, 1::2] == 0).all().item()) and bool((bits16[:, :, 1::2] == 0).all().item())
    if L.relu:
        x = run.d_x.view(L.N, L.H, L.W, L.C).float()
        off = ~(x > 0)
        assert bool((bits16[off] == 0).all().item()), "gated-off positions must be +0.0"

    pix = sample_pixels(L)
    ref = oracle.dgrad_pixels(run.dY, run.W, L.H, L.W, pix, L.stride, L.pad, L.dil, x=run.x, dtype=L.dtype)
    idx = torch.from_numpy(pix.astype(np.int64)).cuda()
    got_bits = bits16[idx[:, 0], idx[:, 1], idx[:, 2]].cpu().numpy()
    got = decode_out(got_bits.view(np.uint8), run.odt).reshape(len(pix), L.C)
    assert_close(got, ref, run.odt, L.name)
