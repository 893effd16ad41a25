"""GB300 (sm_103a) Conv2d backward-data engine: Python binding of libcdg.so.

Argument marshalling only: every step of dgrad runs in the library's CUDA
kernels.  Tensors may be torch CUDA tensors or raw device addresses (ints);
streams may be torch streams, raw ``cudaStream_t`` values (ints) or None (the
current torch stream when torch is loaded, else the legacy default stream).

The operation (apache/tvm PR #10110, "[CUTLASS] Conv2d dgrad"):
    dX[n,h,w,c] = sum_{k,r,s} dY[n,p,q,k] * W[k,r,s,c]
over every (p, q) with h = p*stride - pad + r*dil, w = q*stride - pad + s*dil.
NHWC dX/dY, KRSC W, fp16/bf16 inputs, fp32 accumulation.

There is no CPU fallback: if the library is missing, importing the functions
that need it raises.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libcdg.so")

OK = 0
STATUS_NAMES = {0: "CDG_OK", 1: "CDG_ERR_INVALID_ARG", 2: "CDG_ERR_UNSUPPORTED", 3: "CDG_ERR_ALIGNMENT",
                4: "CDG_ERR_ALIAS", 5: "CDG_ERR_CUDA", 6: "CDG_ERR_TIMEOUT", 7: "CDG_ERR_NO_DEVICE",
                8: "CDG_ERR_SCRATCH_TOO_SMALL"}
ERR_INVALID_ARG = 1
ERR_SCRATCH_TOO_SMALL = 8
NOALLOC_MAX_WEIGHT_BYTES = 8 << 20
F16, BF16 = 0, 1
EPI_RELU_BWD, EPI_OUT_F32, EPI_RELU_BWD_BITS, EPI_SUM, EPI_SUM_X = 1, 2, 4, 8, 16
EPI_GELU_BWD, EPI_SILU_BWD = 32, 64
FUSED_WRITE_G = 256
ACT_FLAGS = {"relu": EPI_RELU_BWD, "gelu": EPI_GELU_BWD, "silu": EPI_SILU_BWD}
DTYPES = {"f16": F16, "bf16": BF16}

EXPORTS = ("cdg_plan", "cdg_plan_host", "cdg_destroy", "cdg_get_output_dims", "cdg_packed_weight_bytes",
           "cdg_plan_get_info", "cdg_prepack_weights", "cdg_dgrad", "cdg_device_status", "cdg_status_string",
           "cdg_dgrad_noalloc", "cdg_dgrad_noalloc_status", "cdg_autotune", "cdg_plan_set_wait_limit",
           "cdg_plan_withhold_load_for_test", "cdg_dgrad_sums", "cdg_sums_workspace_bytes",
           "cdg_fused_plan", "cdg_fused_plan_host", "cdg_fused_destroy", "cdg_fused_packed_weight_bytes",
           "cdg_fused_prepack_weights", "cdg_dgrad_fused", "cdg_fused_get_info", "cdg_fused_device_status", "cdg_pack_relu_mask", "cdg_relu_mask_bytes",
           "cdg_wgrad_plan", "cdg_wgrad_plan_host", "cdg_wgrad_destroy", "cdg_wgrad_workspace_bytes",
           "cdg_wgrad_get_info", "cdg_wgrad", "cdg_wgrad_device_status")


class CdgError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} ({status_string(status)})")


class PlanInfo(ctypes.Structure):
    _fields_ = [("P", ctypes.c_int), ("Q", ctypes.c_int), ("num_phases", ctypes.c_int),
                ("phase_taps", ctypes.c_int * 16), ("tile_m", ctypes.c_int), ("tile_n", ctypes.c_int),
                ("tile_k", ctypes.c_int), ("a_mode", ctypes.c_int), ("box_w", ctypes.c_int),
                ("box_h", ctypes.c_int), ("box_n", ctypes.c_int), ("stages", ctypes.c_int),
                ("work_items", ctypes.c_int), ("grid", ctypes.c_int), ("smem_bytes", ctypes.c_int),
                ("tmem_cols", ctypes.c_int), ("cta_pair", ctypes.c_int),
                ("mma_warps", ctypes.c_int), ("tuned", ctypes.c_int)]

    def as_dict(self) -> dict:
        d = {name: getattr(self, name) for name, _ in self._fields_}
        d["phase_taps"] = list(self.phase_taps)[: self.num_phases]
        return d


_lib = None


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libcdg.so (building it first if the sources are newer)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or LIB_PATH
    if path == LIB_PATH:
        from . import build as _build
        if not _build.up_to_date():
            _build.build()
    if not os.path.exists(path):
        raise ImportError(f"libcdg.so not found at {path}; run `python -m implicit_gemm_dgrad_gb300.build`")
    lib = ctypes.CDLL(path)
    i, vp, hp = ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p
    lib.cdg_plan.argtypes = [i] * 12 + [ctypes.POINTER(hp)]
    lib.cdg_plan.restype = i
    lib.cdg_plan_host.argtypes = [i] * 13 + [ctypes.POINTER(hp)]
    lib.cdg_plan_host.restype = i
    lib.cdg_destroy.argtypes = [hp]
    lib.cdg_destroy.restype = None
    lib.cdg_get_output_dims.argtypes = [hp, ctypes.POINTER(i), ctypes.POINTER(i)]
    lib.cdg_get_output_dims.restype = i
    lib.cdg_packed_weight_bytes.argtypes = [hp]
    lib.cdg_packed_weight_bytes.restype = ctypes.c_size_t
    lib.cdg_plan_get_info.argtypes = [hp, ctypes.POINTER(PlanInfo)]
    lib.cdg_plan_get_info.restype = i
    lib.cdg_prepack_weights.argtypes = [hp, vp, vp, vp]
    lib.cdg_prepack_weights.restype = i
    lib.cdg_dgrad.argtypes = [hp, vp, vp, vp, vp, vp]
    lib.cdg_dgrad.restype = i
    lib.cdg_device_status.argtypes = [hp, vp]
    lib.cdg_device_status.restype = i
    lib.cdg_status_string.argtypes = [i]
    lib.cdg_status_string.restype = ctypes.c_char_p
    lib.cdg_dgrad_noalloc.argtypes = [hp, vp, vp, vp, vp, vp]
    lib.cdg_dgrad_noalloc.restype = i
    lib.cdg_dgrad_noalloc_status.argtypes = [vp]
    lib.cdg_dgrad_sums.argtypes = [hp, vp, vp, vp, vp, vp, vp, vp]
    lib.cdg_dgrad_sums.restype = i
    lib.cdg_sums_workspace_bytes.argtypes = [hp]
    lib.cdg_sums_workspace_bytes.restype = ctypes.c_size_t
    lib.cdg_fused_plan.argtypes = [i] * 12 + [ctypes.POINTER(hp)]
    lib.cdg_fused_plan.restype = i
    lib.cdg_fused_plan_host.argtypes = [i] * 13 + [ctypes.POINTER(hp)]
    lib.cdg_fused_plan_host.restype = i
    lib.cdg_fused_destroy.argtypes = [hp]
    lib.cdg_fused_destroy.restype = None
    lib.cdg_fused_packed_weight_bytes.argtypes = [hp, ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_size_t)]
    lib.cdg_fused_packed_weight_bytes.restype = i
    lib.cdg_fused_prepack_weights.argtypes = [hp, vp, vp, vp, vp, vp]
    lib.cdg_fused_prepack_weights.restype = i
    lib.cdg_dgrad_fused.argtypes = [hp, vp, vp, vp, vp, vp, vp, vp]
    lib.cdg_dgrad_fused.restype = i
    lib.cdg_fused_get_info.argtypes = [hp, ctypes.POINTER(PlanInfo)]
    lib.cdg_fused_get_info.restype = i
    lib.cdg_fused_device_status.argtypes = [hp, vp]
    lib.cdg_fused_device_status.restype = i
    lib.cdg_plan_set_wait_limit.argtypes = [hp, ctypes.c_ulonglong]
    lib.cdg_plan_set_wait_limit.restype = i
    lib.cdg_plan_withhold_load_for_test.argtypes = [hp, i]
    lib.cdg_plan_withhold_load_for_test.restype = i
    lib.cdg_dgrad_noalloc_status.restype = i
    lib.cdg_autotune.argtypes = [hp, vp, vp, vp, vp, vp, i, ctypes.POINTER(ctypes.c_float)]
    lib.cdg_autotune.restype = i
    lib.cdg_pack_relu_mask.argtypes = [vp, vp, ctypes.c_longlong, i, i, vp]
    lib.cdg_pack_relu_mask.restype = i
    lib.cdg_relu_mask_bytes.argtypes = [ctypes.c_longlong, i]
    lib.cdg_relu_mask_bytes.restype = ctypes.c_longlong
    lib.cdg_wgrad_plan.argtypes = [i] * 13 + [ctypes.POINTER(hp)]
    lib.cdg_wgrad_plan.restype = i
    lib.cdg_wgrad_plan_host.argtypes = [i] * 14 + [ctypes.POINTER(hp)]
    lib.cdg_wgrad_plan_host.restype = i
    lib.cdg_wgrad_destroy.argtypes = [hp]
    lib.cdg_wgrad_destroy.restype = None
    lib.cdg_wgrad_workspace_bytes.argtypes = [hp]
    lib.cdg_wgrad_workspace_bytes.restype = ctypes.c_size_t
    lib.cdg_wgrad_get_info.argtypes = [hp, ctypes.POINTER(WgradInfo)]
    lib.cdg_wgrad_get_info.restype = i
    lib.cdg_wgrad.argtypes = [hp, vp, vp, vp, vp, vp]
    lib.cdg_wgrad.restype = i
    lib.cdg_wgrad_device_status.argtypes = [hp, vp]
    lib.cdg_wgrad_device_status.restype = i
    if path == LIB_PATH:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load_library().cdg_status_string(status).decode()
    except Exception:  # noqa: BLE001 - message formatting must not raise
        return "?"


def _addr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _check_buffer(t, nbytes: int, what: str) -> None:
    """A tensor argument must be a contiguous CUDA tensor of at least nbytes
    (the kernels read and write exactly the planned extents, which the C ABI
    cannot check).  Raw integer pointers are passed through unchecked."""
    if t is None or isinstance(t, int):
        return
    if not getattr(t, "is_cuda", False):
        raise ValueError(f"{what} must be a CUDA tensor (or a device pointer)")
    idx = getattr(getattr(t, "device", None), "index", None)
    if idx is not None:
        import torch
        cur = torch.cuda.current_device()
        if idx != cur:
            # the library launches on the current device; a pointer into
            # another GPU's memory would be read by this one's kernels
            raise ValueError(f"{what} is on cuda:{idx}, but the current device is cuda:{cur}")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    have = t.numel() * t.element_size()
    if have < nbytes:
        raise ValueError(f"{what} holds {have} bytes; the plan needs {nbytes}")


def _stream(s) -> int | None:
    if s is None:
        try:
            import torch
            if torch.cuda.is_available() and torch.cuda.is_initialized():
                return torch.cuda.current_stream().cuda_stream
        except ImportError:
            pass
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


class Plan:
    """One planned dgrad shape (a ``cdg_handle_t``)."""

    def __init__(self, N, H, W, C, K, R, S, stride=1, pad=0, dil=1, dtype="bf16", relu=False,
                 out_f32=False, host_sms: int | None = None, relu_bits=False, sums: int = 0, act: str = "relu"):
        self.lib = load_library()
        self.shape = dict(N=N, H=H, W=W, C=C, K=K, R=R, S=S, stride=stride, pad=pad, dil=dil)
        self.dtype = dtype
        self.relu = relu          # the gate reads a saved tensor of dX's shape (ReLU's x, or act's input)
        self.relu_bits = relu_bits
        self.out_f32 = out_f32
        self.sums = int(sums)
        gate = ACT_FLAGS[act] if relu else 0
        epi = gate | (EPI_OUT_F32 if out_f32 else 0) | (EPI_RELU_BWD_BITS if relu_bits else 0)
        epi |= {0: 0, 1: EPI_SUM, 2: EPI_SUM | EPI_SUM_X}[self.sums]
        h = ctypes.c_void_p()
        dt = DTYPES[dtype] if isinstance(dtype, str) else int(dtype)
        if host_sms is None:
            rc = self.lib.cdg_plan(N, H, W, C, K, R, S, stride, pad, dil, dt, epi, ctypes.byref(h))
        else:
            rc = self.lib.cdg_plan_host(N, H, W, C, K, R, S, stride, pad, dil, dt, epi, host_sms, ctypes.byref(h))
        if rc != OK:
            raise CdgError(rc, "cdg_plan")
        self.handle = h

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            self.lib.cdg_destroy(self.handle)
        self.handle = None

    def __del__(self):
        self.close()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    @property
    def output_dims(self) -> tuple[int, int]:
        P, Q = ctypes.c_int(), ctypes.c_int()
        rc = self.lib.cdg_get_output_dims(self.handle, ctypes.byref(P), ctypes.byref(Q))
        if rc != OK:
            raise CdgError(rc, "cdg_get_output_dims")
        return P.value, Q.value

    @property
    def packed_weight_bytes(self) -> int:
        return int(self.lib.cdg_packed_weight_bytes(self.handle))

    def info(self) -> dict:
        inf = PlanInfo()
        rc = self.lib.cdg_plan_get_info(self.handle, ctypes.byref(inf))
        if rc != OK:
            raise CdgError(rc, "cdg_plan_get_info")
        return inf.as_dict()

    def _sizes(self) -> dict:
        """Bytes of each tensor of this plan's dgrad."""
        d = self.shape
        P, Q = self.output_dims
        pixels = d["N"] * d["H"] * d["W"]
        mask = 0
        if self.relu_bits:
            mask = relu_mask_bytes(pixels, d["C"])
        elif self.relu:
            mask = 2 * pixels * d["C"]
        return {"dY": 2 * d["N"] * P * Q * d["K"], "W": 2 * d["K"] * d["R"] * d["S"] * d["C"],
                "dX": (4 if self.out_f32 else 2) * pixels * d["C"], "mask": mask}

    def _check(self, dY=None, W=None, W_packed=None, dX=None, relu_mask=None) -> None:
        z = self._sizes()
        _check_buffer(dY, z["dY"], "dY")
        _check_buffer(W, z["W"], "W")
        _check_buffer(W_packed, z["W"], "W_packed")
        _check_buffer(dX, z["dX"], "dX")
        _check_buffer(relu_mask, z["mask"], "relu_mask")

    def prepack_weights(self, W_krsc, W_packed, stream=None) -> None:
        self._check(W=W_krsc, W_packed=W_packed)
        rc = self.lib.cdg_prepack_weights(self.handle, _addr(W_krsc), _addr(W_packed), _stream(stream))
        if rc != OK:
            raise CdgError(rc, "cdg_prepack_weights")

    def dgrad(self, dY, W_packed, dX, relu_mask=None, stream=None) -> None:
        self._check(dY=dY, W_packed=W_packed, dX=dX, relu_mask=relu_mask)
        rc = self.lib.cdg_dgrad(self.handle, _addr(dY), _addr(W_packed), _addr(dX), _addr(relu_mask),
                                _stream(stream))
        if rc != OK:
            raise CdgError(rc, "cdg_dgrad")

    @property
    def sums_workspace_bytes(self) -> int:
        return int(self.lib.cdg_sums_workspace_bytes(self.handle))

    def dgrad_sums(self, dY, W_packed, dX, sums, workspace, relu_mask=None, stream=None) -> None:
        """dgrad plus the per-channel sums of its output (cdg_dgrad_sums):
        sums (fp32, C values, or 2*C for sums=2) receives sum(out) per channel
        and, for sums=2, sum(out * x) where the gate passes."""
        self._check(dY=dY, W_packed=W_packed, dX=dX, relu_mask=relu_mask)
        _check_buffer(sums, 4 * self.sums * self.shape["C"], "sums")
        _check_buffer(workspace, self.sums_workspace_bytes, "workspace")
        rc = self.lib.cdg_dgrad_sums(self.handle, _addr(dY), _addr(W_packed), _addr(dX), _addr(relu_mask),
                                     _addr(sums), _addr(workspace), _stream(stream))
        if rc != OK:
            raise CdgError(rc, "cdg_dgrad_sums")

    def dgrad_noalloc(self, dY, W_krsc, dX, relu_mask=None, stream=None) -> None:
        """dgrad from the unpacked KRSC filter without any device allocation
        (the packed weights live in the library's own scratch array; see
        cdg_dgrad_noalloc in cdg.h for the size limit and the sharing rules)."""
        self._check(dY=dY, W=W_krsc, dX=dX, relu_mask=relu_mask)
        rc = self.lib.cdg_dgrad_noalloc(self.handle, _addr(dY), _addr(W_krsc), _addr(dX), _addr(relu_mask),
                                        _stream(stream))
        if rc != OK:
            raise CdgError(rc, "cdg_dgrad_noalloc")

    @staticmethod
    def noalloc_status(stream=None) -> int:
        """Read and clear the status word of cdg_dgrad_noalloc launches on the
        current device (cdg_dgrad_noalloc_status): 0, or the CDG_ERR_TIMEOUT
        code of a launch that gave up a bounded wait."""
        return int(load_library().cdg_dgrad_noalloc_status(_stream(stream)))

    def autotune(self, dY, W_packed, dX, relu_mask=None, stream=None, reps: int = 3) -> float:
        """Time every configuration the planner can produce for this shape on
        these tensors and keep the fastest (cdg_autotune); returns its mean
        launch time in ms.  dX receives the correct result."""
        self._check(dY=dY, W_packed=W_packed, dX=dX, relu_mask=relu_mask)
        best = ctypes.c_float()
        rc = self.lib.cdg_autotune(self.handle, _addr(dY), _addr(W_packed), _addr(dX), _addr(relu_mask),
                                   _stream(stream), int(reps), ctypes.byref(best))
        if rc != OK:
            raise CdgError(rc, "cdg_autotune")
        return float(best.value)

    def device_status(self, stream=None) -> int:
        return int(self.lib.cdg_device_status(self.handle, _stream(stream)))

    def set_wait_limit(self, ns: int) -> None:
        """Longest time any single pipeline wait of this plan's kernel may
        take before the launch aborts with CDG_ERR_TIMEOUT (cdg_plan_set_wait_limit)."""
        rc = self.lib.cdg_plan_set_wait_limit(self.handle, int(ns))
        if rc != OK:
            raise CdgError(rc, "cdg_plan_set_wait_limit")

    def withhold_load_for_test(self, stage: int) -> None:
        """Test only: make launches withhold the operand load of pipeline stage
        `stage` in every CTA, so they take the bounded-wait timeout path
        (cdg_plan_withhold_load_for_test); -1 restores normal launches."""
        rc = self.lib.cdg_plan_withhold_load_for_test(self.handle, int(stage))
        if rc != OK:
            raise CdgError(rc, "cdg_plan_withhold_load_for_test")


class FusedPlan:
    """Back-to-back dgrads in one kernel (a ``cdg_fused_t``):
    g = act_bwd(dgrad(dY2, W2), x2) for a stride-1 R2 x S2 layer with C2 = 64
    channels, then dX1 = dgrad_1x1(g, W1) with C1 channels; g stays on chip
    and is written only with write_g=True."""

    def __init__(self, N, H, W, C1, C2, K2, R2, S2, pad2=1, dil2=1, dtype="bf16", act: str | None = "relu",
                 write_g=False, host_sms: int | None = None):
        self.lib = load_library()
        self.shape = dict(N=N, H=H, W=W, C1=C1, C2=C2, K2=K2, R2=R2, S2=S2, pad2=pad2, dil2=dil2)
        self.act = act
        self.write_g = bool(write_g)
        flags = (ACT_FLAGS[act] if act else 0) | (FUSED_WRITE_G if write_g else 0)
        dt = DTYPES[dtype] if isinstance(dtype, str) else int(dtype)
        h = ctypes.c_void_p()
        args = (N, H, W, C1, C2, K2, R2, S2, pad2, dil2, dt, flags)
        if host_sms is None:
            rc = self.lib.cdg_fused_plan(*args, ctypes.byref(h))
        else:
            rc = self.lib.cdg_fused_plan_host(*args, host_sms, ctypes.byref(h))
        if rc != OK:
            raise CdgError(rc, "cdg_fused_plan")
        self.handle = h

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            self.lib.cdg_fused_destroy(self.handle)
        self.handle = None

    def __del__(self):
        self.close()

    @property
    def packed_weight_bytes(self) -> tuple[int, int]:
        b2, b1 = ctypes.c_size_t(), ctypes.c_size_t()
        rc = self.lib.cdg_fused_packed_weight_bytes(self.handle, ctypes.byref(b2), ctypes.byref(b1))
        if rc != OK:
            raise CdgError(rc, "cdg_fused_packed_weight_bytes")
        return int(b2.value), int(b1.value)

    def info(self) -> dict:
        inf = PlanInfo()
        rc = self.lib.cdg_fused_get_info(self.handle, ctypes.byref(inf))
        if rc != OK:
            raise CdgError(rc, "cdg_fused_get_info")
        return inf.as_dict()

    def prepack_weights(self, W2, W1, W2p, W1p, stream=None) -> None:
        b2, b1 = self.packed_weight_bytes
        for t, n, what in ((W2, b2, "W2"), (W1, b1, "W1"), (W2p, b2, "W2p"), (W1p, b1, "W1p")):
            _check_buffer(t, n, what)
        rc = self.lib.cdg_fused_prepack_weights(self.handle, _addr(W2), _addr(W1), _addr(W2p), _addr(W1p),
                                                _stream(stream))
        if rc != OK:
            raise CdgError(rc, "cdg_fused_prepack_weights")

    def dgrad(self, dY2, W2p, x2, W1p, dX1, g=None, stream=None) -> None:
        d = self.shape
        P = d["H"] + 2 * d["pad2"] - d["dil2"] * (d["R2"] - 1)
        Q = d["W"] + 2 * d["pad2"] - d["dil2"] * (d["S2"] - 1)
        px = d["N"] * d["H"] * d["W"]
        b2, b1 = self.packed_weight_bytes
        _check_buffer(dY2, 2 * d["N"] * P * Q * d["K2"], "dY2")
        _check_buffer(W2p, b2, "W2p")
        _check_buffer(W1p, b1, "W1p")
        _check_buffer(x2, 2 * px * d["C2"], "x2")
        _check_buffer(dX1, 2 * px * d["C1"], "dX1")
        _check_buffer(g, 2 * px * d["C2"], "g")
        rc = self.lib.cdg_dgrad_fused(self.handle, _addr(dY2), _addr(W2p), _addr(x2), _addr(W1p), _addr(g),
                                      _addr(dX1), _stream(stream))
        if rc != OK:
            raise CdgError(rc, "cdg_dgrad_fused")

    def device_status(self, stream=None) -> int:
        return int(self.lib.cdg_fused_device_status(self.handle, _stream(stream)))


class WgradInfo(ctypes.Structure):
    _fields_ = [("P", ctypes.c_int), ("Q", ctypes.c_int), ("tile_m", ctypes.c_int), ("tile_n", ctypes.c_int),
                ("taps_per_item", ctypes.c_int), ("splits", ctypes.c_int), ("pos_box", ctypes.c_int * 3), ("blocks", ctypes.c_int),
                ("stages", ctypes.c_int), ("work_items", ctypes.c_int), ("grid", ctypes.c_int),
                ("smem_bytes", ctypes.c_int), ("tmem_cols", ctypes.c_int), ("x_major", ctypes.c_int)]

    def as_dict(self) -> dict:
        d = {name: getattr(self, name) for name, _ in self._fields_}
        d["pos_box"] = list(self.pos_box)
        return d


class WgradPlan:
    """One planned wgrad shape (a ``cdg_wgrad_t``): dW = wgrad(dY, x)."""

    def __init__(self, N, H, W, C, K, R, S, stride=1, pad=0, dil=1, dtype="bf16", out_f32=False, splits=0,
                 host_sms: int | None = None):
        self.lib = load_library()
        self.shape = dict(N=N, H=H, W=W, C=C, K=K, R=R, S=S, stride=stride, pad=pad, dil=dil)
        self.out_f32 = bool(out_f32)
        h = ctypes.c_void_p()
        dt = DTYPES[dtype] if isinstance(dtype, str) else int(dtype)
        args = (N, H, W, C, K, R, S, stride, pad, dil, dt, int(bool(out_f32)), int(splits))
        if host_sms is None:
            rc = self.lib.cdg_wgrad_plan(*args, ctypes.byref(h))
        else:
            rc = self.lib.cdg_wgrad_plan_host(*args, host_sms, ctypes.byref(h))
        if rc != OK:
            raise CdgError(rc, "cdg_wgrad_plan")
        self.handle = h

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            self.lib.cdg_wgrad_destroy(self.handle)
        self.handle = None

    def __del__(self):
        self.close()

    @property
    def workspace_bytes(self) -> int:
        return int(self.lib.cdg_wgrad_workspace_bytes(self.handle))

    def info(self) -> dict:
        inf = WgradInfo()
        rc = self.lib.cdg_wgrad_get_info(self.handle, ctypes.byref(inf))
        if rc != OK:
            raise CdgError(rc, "cdg_wgrad_get_info")
        return inf.as_dict()

    def wgrad(self, dY, x, dW, workspace, stream=None) -> None:
        d = self.shape
        inf = self.info()
        _check_buffer(dY, 2 * d["N"] * inf["P"] * inf["Q"] * d["K"], "dY")
        _check_buffer(x, 2 * d["N"] * d["H"] * d["W"] * d["C"], "x")
        _check_buffer(dW, (4 if self.out_f32 else 2) * d["K"] * d["R"] * d["S"] * d["C"], "dW")
        _check_buffer(workspace, self.workspace_bytes, "workspace")
        rc = self.lib.cdg_wgrad(self.handle, _addr(dY), _addr(x), _addr(dW), _addr(workspace), _stream(stream))
        if rc != OK:
            raise CdgError(rc, "cdg_wgrad")

    def device_status(self, stream=None) -> int:
        return int(self.lib.cdg_wgrad_device_status(self.handle, _stream(stream)))


def wgrad_plan(N, H, W, C, K, R, S, stride=1, pad=0, dil=1, dtype="bf16", out_f32=False, splits=0) -> WgradPlan:
    return WgradPlan(N, H, W, C, K, R, S, stride, pad, dil, dtype, out_f32, splits)


def wgrad_plan_host(N, H, W, C, K, R, S, stride=1, pad=0, dil=1, dtype="bf16", out_f32=False, splits=0,
                    num_sms=148) -> WgradPlan:
    return WgradPlan(N, H, W, C, K, R, S, stride, pad, dil, dtype, out_f32, splits, host_sms=num_sms)


def plan(N, H, W, C, K, R, S, stride=1, pad=0, dil=1, dtype="bf16", relu=False, out_f32=False,
         relu_bits=False, sums: int = 0, act: str = "relu") -> Plan:
    """relu=True: the epilogue applies the backward of activation `act`
    ("relu" gate, "gelu", "silu") with the saved tensor passed to dgrad."""
    return Plan(N, H, W, C, K, R, S, stride, pad, dil, dtype, relu, out_f32, relu_bits=relu_bits, sums=sums,
                act=act)


def relu_mask_bytes(pixels: int, C: int) -> int:
    """Bytes of the packed ReLU mask of `pixels` pixels of C channels (cdg_relu_mask_bytes)."""
    n = load_library().cdg_relu_mask_bytes(int(pixels), int(C))
    if n < 0:
        raise CdgError(ERR_INVALID_ARG, "cdg_relu_mask_bytes")
    return n


def pack_relu_mask(x, bits, pixels: int, C: int, dtype="bf16", stream=None) -> None:
    """bits (relu_mask_bytes(pixels, C) bytes) = the packed mask (x > 0) of the
    NHWC activation x, one bit per element in 16-byte units per pixel
    (cdg_pack_relu_mask), for plans made with relu_bits=True."""
    lib = load_library()
    dt = DTYPES[dtype] if isinstance(dtype, str) else int(dtype)
    if int(pixels) >= 0 and int(C) > 0 and int(C) % 8 == 0:
        _check_buffer(x, 2 * int(pixels) * int(C), "x")
        _check_buffer(bits, relu_mask_bytes(pixels, C), "bits")
    rc = lib.cdg_pack_relu_mask(_addr(x), _addr(bits), int(pixels), int(C), dt, _stream(stream))
    if rc != OK:
        raise CdgError(rc, "cdg_pack_relu_mask")


def plan_host(N, H, W, C, K, R, S, stride=1, pad=0, dil=1, dtype="bf16", relu=False, out_f32=False,
              num_sms=148, relu_bits=False, sums: int = 0, act: str = "relu") -> Plan:
    return Plan(N, H, W, C, K, R, S, stride, pad, dil, dtype, relu, out_f32, host_sms=num_sms, relu_bits=relu_bits,
                sums=sums, act=act)
