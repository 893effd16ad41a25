"""The Python binding checks tensor arguments before they become device
pointers: CUDA, contiguous, and at least the bytes the plan reads or writes
(the C ABI takes raw pointers and cannot).  Exact sizes pass through to the
library (whose host-only plans then answer NO_DEVICE); one byte less, a CPU
tensor or a non-contiguous tensor raises ValueError before any call.  Raw
integer pointers pass unchecked, as the C ABI defines them."""
import pytest

import implicit_gemm_dgrad_gb300 as cdg
from implicit_gemm_dgrad_gb300.workloads import RESNET50_B256


class FakeCuda:
    """Stands in for a CUDA tensor: size, contiguity and an aligned address."""
    is_cuda = True

    def __init__(self, nbytes, esize=2, contiguous=True):
        self.nbytes, self.esize, self.contig = nbytes, esize, contiguous

    def numel(self):
        return self.nbytes // self.esize

    def element_size(self):
        return self.esize

    def is_contiguous(self):
        return self.contig

    def data_ptr(self):
        return 1 << 24


def _dgrad_sizes(L, gate, out_f32):
    P, Q = L.P, L.Q
    px = L.N * L.H * L.W
    mask = {"none": 0, "x": 2 * px * L.C, "bits": cdg.relu_mask_bytes(px, L.C)}[gate]
    return 2 * L.N * P * Q * L.K, 2 * L.K * L.R * L.S * L.C, (4 if out_f32 else 2) * px * L.C, mask


def _plans():
    odd = [RESNET50_B256[0].__class__("odd", 2, 11, 13, 72, 136, 3, 3, 2, 1, 1),
           RESNET50_B256[0].__class__("odd2", 3, 10, 9, 8, 8, 1, 1, 2, 0, 1)]
    for L in list(RESNET50_B256) + odd:
        for gate in ("none", "x", "bits"):
            for out_f32 in (False, True):
                yield L, gate, out_f32


@pytest.mark.parametrize("L,gate,out_f32", list(_plans()), ids=lambda v: getattr(v, "name", str(v)))
def test_dgrad_exact_sizes_pass_and_short_ones_fail(L, gate, out_f32):
    p = cdg.plan_host(L.N, L.H, L.W, L.C, L.K, L.R, L.S, L.stride, L.pad, L.dil, "bf16",
                      relu=gate == "x", relu_bits=gate == "bits", out_f32=out_f32)
    ndy, nw, ndx, nmask = _dgrad_sizes(L, gate, out_f32)
    mask = FakeCuda(nmask) if gate != "none" else None
    full = dict(dY=FakeCuda(ndy), W_packed=FakeCuda(nw), dX=FakeCuda(ndx, 4 if out_f32 else 2), relu_mask=mask)
    with pytest.raises(cdg.CdgError) as e:  # the checks pass; the host-only plan refuses device work
        p.dgrad(**full)
    assert e.value.status == 7
    with pytest.raises(cdg.CdgError):
        p.dgrad_noalloc(full["dY"], FakeCuda(nw), full["dX"], mask)
    with pytest.raises(cdg.CdgError) as e:
        p.prepack_weights(FakeCuda(nw), FakeCuda(nw))
    assert e.value.status == 7
    for name in [k for k, v in full.items() if v is not None]:
        short = dict(full)
        short[name] = FakeCuda(full[name].nbytes - 1, 1)
        with pytest.raises(ValueError, match=name):
            p.dgrad(**short)


def test_wrong_device_and_layout_rejected():
    torch = pytest.importorskip("torch")
    p = cdg.plan_host(1, 8, 8, 16, 16, 3, 3, 1, 1, 1, "bf16")
    with pytest.raises(ValueError, match="CUDA"):
        p.dgrad(torch.zeros(1024, dtype=torch.int16), 16, 4096)
    with pytest.raises(ValueError, match="contiguous"):
        p.dgrad(FakeCuda(1 << 20, contiguous=False), 16, 4096)
    with pytest.raises(cdg.CdgError):  # raw pointers are the C ABI's business
        p.dgrad(16, 16, 4096)


@pytest.mark.parametrize("shape", [(2, 7, 6, 16, 24, 3, 3, 1, 1, 1), (3, 12, 12, 320, 64, 3, 3, 2, 1, 1),
                                   (64, 7, 7, 256, 128, 3, 3, 1, 1, 1), (256, 56, 56, 64, 64, 1, 1, 1, 0, 1)])
@pytest.mark.parametrize("out_f32", [False, True])
def test_wgrad_exact_sizes_pass_and_short_ones_fail(shape, out_f32):
    N, H, W, C, K, R, S, st, pd, dl = shape
    w = cdg.wgrad_plan_host(*shape, "bf16", out_f32=out_f32)
    i = w.info()
    full = dict(dY=FakeCuda(2 * N * i["P"] * i["Q"] * K), x=FakeCuda(2 * N * H * W * C),
                dW=FakeCuda((4 if out_f32 else 2) * K * R * S * C), workspace=FakeCuda(w.workspace_bytes, 4))
    with pytest.raises(cdg.CdgError) as e:
        w.wgrad(**full)
    assert e.value.status == 7
    for name in full:
        short = dict(full)
        short[name] = FakeCuda(full[name].nbytes - 1, 1)
        with pytest.raises(ValueError, match=name):
            w.wgrad(**short)


def test_pack_relu_mask_short_buffers():
    n = cdg.relu_mask_bytes(100, 64)
    with pytest.raises(ValueError, match="bits"):
        cdg.pack_relu_mask(FakeCuda(2 * 100 * 64), FakeCuda(n - 1, 1), 100, 64)
    with pytest.raises(ValueError, match="x"):
        cdg.pack_relu_mask(FakeCuda(2 * 100 * 64 - 2), FakeCuda(n, 1), 100, 64)


def test_tensor_on_another_device_is_rejected(monkeypatch):
    """A tensor on a GPU other than the current one raises ValueError before
    any call (the kernels launch on the current device)."""
    import types

    import torch
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    L = RESNET50_B256[0]
    p = cdg.plan_host(L.N, L.H, L.W, L.C, L.K, L.R, L.S, L.stride, L.pad, L.dil, L.dtype, num_sms=148)
    dy, w, dx, _ = _dgrad_sizes(L, "none", False)
    args = [FakeCuda(dy), FakeCuda(w), FakeCuda(dx)]
    for t in args:
        t.device = types.SimpleNamespace(index=0)
    args[2].device = types.SimpleNamespace(index=1)
    with pytest.raises(ValueError, match="cuda:1"):
        p.dgrad(*args)
    args[2].device = types.SimpleNamespace(index=0)
    with pytest.raises(cdg.CdgError) as e:  # same device: the host-only plan refuses device work
        p.dgrad(*args)
    assert e.value.status == 7
