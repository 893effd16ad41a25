"""Helpers for the GPU parity tests: upload seeded inputs, call the library
through its C-ABI binding, bring results back as float64, compare with the
oracle under the stated tolerance."""
from __future__ import annotations

import numpy as np

from implicit_gemm_dgrad_gb300 import synth

# per-element bound |gpu - oracle| <= TOL * max(1, |oracle|)
TOL = {"f32": 2e-3, "f16": 1e-2, "bf16": 1e-2}
GUARD_BYTES = 64 * 1024
SENTINEL = 0xA5


def torch_cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch


def to_dev(bits_or_f32: np.ndarray, dtype: str):
    torch = torch_cuda()
    if dtype in ("f16", "bf16"):
        t = torch.from_numpy(np.ascontiguousarray(bits_or_f32).view(np.int16))
        return t.cuda().view(torch.float16 if dtype == "f16" else torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(bits_or_f32, dtype=np.float32)).cuda()


class GuardedOutput:
    """dX inside a larger byte buffer with sentinel-filled guard bands on both sides."""

    def __init__(self, nelem: int, esize: int, prefill: str = "nan"):
        torch = torch_cuda()
        self.nbytes = nelem * esize
        self.esize = esize
        self.buf = torch.full((self.nbytes + 2 * GUARD_BYTES,), SENTINEL, dtype=torch.uint8, device="cuda")
        body = self.buf[GUARD_BYTES:GUARD_BYTES + self.nbytes]
        if prefill == "nan":
            if esize == 4:
                body.view(torch.int32).fill_(0x7FC00001)
            else:
                body.view(torch.int16).fill_(0x7E01)
        elif prefill == "garbage":
            body.copy_(torch.randint(0, 256, (self.nbytes,), dtype=torch.uint8, device="cuda"))
        self.ptr = self.buf.data_ptr() + GUARD_BYTES

    def guards_intact(self) -> bool:
        torch = torch_cuda()
        lo = self.buf[:GUARD_BYTES]
        hi = self.buf[GUARD_BYTES + self.nbytes:]
        return bool(torch.all(lo == SENTINEL).item() and torch.all(hi == SENTINEL).item())

    def body(self):
        return self.buf[GUARD_BYTES:GUARD_BYTES + self.nbytes]


def out_dtype(layer) -> str:
    return "f32" if layer.out == "f32" else layer.dtype


def decode_out(raw_bytes: np.ndarray, odt: str) -> np.ndarray:
    if odt == "f32":
        return raw_bytes.view(np.float32).astype(np.float64)
    return synth.bits_to_f32(raw_bytes.view(np.uint16), odt).astype(np.float64)


class GpuRun:
    """Plan + prepack + dgrad for one layer on seeded inputs."""

    def __init__(self, layer, dist=None, batch=None, inputs=None, prefill="nan"):
        import implicit_gemm_dgrad_gb300 as cdg
        torch = torch_cuda()
        self.layer = layer if batch is None else layer.with_batch(batch)
        L = self.layer
        if inputs is None:
            inputs = synth.make_inputs(L.shape(), L.dtype, dist or L.dist, L.workload, L.index, with_x=L.relu)
        self.dY, self.W, self.x = inputs
        self.odt = out_dtype(L)
        self.plan = cdg.plan(L.N, L.H, L.W, L.C, L.K, L.R, L.S, L.stride, L.pad, L.dil, L.dtype,
                             relu=L.relu, out_f32=(L.out == "f32"))
        self.d_dY = to_dev(self.dY, L.dtype)
        self.d_W = to_dev(self.W, L.dtype)
        self.d_x = to_dev(self.x, L.dtype) if L.relu else None
        self.d_Wp = torch.empty(self.plan.packed_weight_bytes // 2, dtype=torch.int16, device="cuda")
        self.plan.prepack_weights(self.d_W, self.d_Wp)
        esize = 4 if self.odt == "f32" else 2
        self.out = GuardedOutput(L.N * L.H * L.W * L.C, esize, prefill)

    def run(self):
        self.plan.dgrad(self.d_dY, self.d_Wp, self.out.ptr, self.d_x)

    def result_bytes(self) -> np.ndarray:
        torch = torch_cuda()
        torch.cuda.synchronize()
        return self.out.body().cpu().numpy()

    def result(self) -> np.ndarray:
        L = self.layer
        return decode_out(self.result_bytes(), self.odt).reshape(L.N, L.H, L.W, L.C)

    def status(self) -> int:
        return self.plan.device_status()


def assert_close(got: np.ndarray, ref: np.ndarray, odt: str, what: str = ""):
    tol = TOL[odt]
    err = np.abs(got - ref)
    bound = tol * np.maximum(1.0, np.abs(ref))
    bad = ~(err <= bound)  # NaN in got counts as bad
    if bad.any():
        idx = np.argwhere(bad)[:5]
        lines = [f"{tuple(i)} gpu={got[tuple(i)]!r} oracle={ref[tuple(i)]!r}" for i in idx]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance "
                             f"(tol {tol}, max err {np.nanmax(err):.3g}):\n" + "\n".join(lines))


# Half of the smallest subnormal of each output type: a value rounds (RNE) to
# +-0 in that type exactly when its magnitude is at most this (the tie rounds to
# the even neighbour, zero).
HALF_MIN_SUBNORMAL = {"f32": 2.0 ** -150, "f16": 2.0 ** -25, "bf16": 2.0 ** -134}


def check_gate_zero_pattern(raw_bits: np.ndarray, x_bits: np.ndarray, ref: np.ndarray, odt: str,
                            dtype: str) -> dict:
    """The ReLU-backward gate's zero pattern, checked in both directions.

    masked = positions where the saved activation x is <= 0, -0.0 or NaN.
      (1) every masked position holds +0.0 bit-exactly;
      (2) no unmasked position holds a zero (+0.0 or -0.0) unless the oracle's
          value there rounds (RNE) to zero in the output type.
    So the set of zero outputs equals the masked set, up to the unmasked
    positions whose exact value is itself zero in the output type; those are
    counted and returned separately (either result is accepted there, the
    tolerance governs their magnitude)."""
    x = synth.bits_to_f32(x_bits.reshape(-1), dtype)
    masked = ~(x > 0)
    if odt == "f32":
        out_bits = raw_bits.view(np.uint32).reshape(-1)
        mag = out_bits & np.uint32(0x7FFFFFFF)
    else:
        out_bits = raw_bits.view(np.uint16).reshape(-1)
        mag = out_bits & np.uint16(0x7FFF)
    ref = np.asarray(ref).reshape(-1)
    assert out_bits.size == masked.size == ref.size
    bad_masked = np.flatnonzero(masked & (out_bits != 0))
    assert bad_masked.size == 0, (f"{bad_masked.size} gated-off positions are not +0.0 bit-exactly, "
                                  f"first {bad_masked[:5]}: bits {out_bits[bad_masked[:5]]}")
    rounds_to_zero = np.abs(ref) <= HALF_MIN_SUBNORMAL[odt]
    spurious = np.flatnonzero(~masked & (mag == 0) & ~rounds_to_zero)
    assert spurious.size == 0, (f"{spurious.size} unmasked positions hold a zero the oracle does not round to, "
                                f"first {spurious[:5]}: oracle {ref[spurious[:5]]}")
    exact_zero = ~masked & rounds_to_zero
    return {"masked": int(masked.sum()), "unmasked": int((~masked).sum()),
            "unmasked_oracle_zero": int(exact_zero.sum()),
            "unmasked_oracle_zero_written_zero": int((exact_zero & (mag == 0)).sum())}
