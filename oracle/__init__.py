"""CPU oracle for Conv2d dgrad -- TEST INFRASTRUCTURE ONLY.

A ctypes wrapper around ``oracle.c``: the plain double-precision statement of
the operation the GPU library computes (the gradient of a cross-correlation
Conv2d with respect to its input, "Conv2d dgrad" in apache/tvm PR #10110),
and of the weight gradient (wgrad) that the page names as its follow-up.

It also states the per-channel sums of the output that a fused epilogue
produces (``channel_sums``).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The GPU library never touches it; the two share
no code.  Arrays are numpy: fp16/bf16 tensors are passed as ``uint16`` bit
patterns, fp32 as ``float32`` and fp64 as ``float64``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

F16, BF16, F32, F64 = 0, 1, 2, 3
ACTS = {"relu": 0, "gelu": 1, "silu": 2}
DTYPE_CODES = {"f16": F16, "bf16": BF16, "f32": F32, "f64": F64}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, OpenMP) if missing or stale."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(LIB)
            vp, ip, i = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32), ctypes.c_int
            lib.oracle_dgrad_act.argtypes = [vp, vp, vp, i, i, vp] + [i] * 10
            lib.oracle_dgrad_act.restype = i
            lib.oracle_dgrad_pixels_act.argtypes = [vp, vp, vp, i, i, vp, ctypes.c_int64, vp] + [i] * 10
            lib.oracle_dgrad_pixels_act.restype = i
            lib.oracle_act_grad.argtypes = [ctypes.c_double, i]
            lib.oracle_act_grad.restype = ctypes.c_double
            lib.oracle_conv_fwd.argtypes = [vp, vp, i, vp] + [i] * 10
            lib.oracle_conv_fwd.restype = i
            lib.oracle_wgrad.argtypes = [vp, vp, i, vp] + [i] * 10
            lib.oracle_wgrad.restype = i
            lib.oracle_wgrad_elements.argtypes = [vp, vp, i, vp, ctypes.c_int64, vp] + [i] * 10
            lib.oracle_wgrad_elements.restype = i
            lib.oracle_channel_sums.argtypes = [vp, vp, i, ctypes.c_int64, i, vp, vp, vp, vp]
            lib.oracle_channel_sums.restype = i
            lib.oracle_out_extent.argtypes = [i] * 5
            lib.oracle_out_extent.restype = i
            lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_half_to_double.restype = ctypes.c_double
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_double.restype = ctypes.c_double
            lib.oracle_double_to_half.argtypes = [ctypes.c_double]
            lib.oracle_double_to_half.restype = ctypes.c_uint16
            lib.oracle_double_to_bf16.argtypes = [ctypes.c_double]
            lib.oracle_double_to_bf16.restype = ctypes.c_uint16
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = i
            _lib = lib
    return _lib


def _dtype_of(a: np.ndarray, dtype: str | None) -> int:
    if dtype is not None:
        return DTYPE_CODES[dtype]
    if a.dtype == np.float64:
        return F64
    if a.dtype == np.float32:
        return F32
    raise ValueError("uint16 arrays need an explicit dtype ('f16' or 'bf16')")


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(a, code):
    want = {F16: np.uint16, BF16: np.uint16, F32: np.float32, F64: np.float64}[code]
    if a.dtype != want or not a.flags.c_contiguous:
        raise ValueError(f"expected contiguous {np.dtype(want)} array, got {a.dtype}")


def out_extent(size: int, filt: int, stride: int, pad: int, dil: int) -> int:
    return _load().oracle_out_extent(size, filt, stride, pad, dil)


def num_threads() -> int:
    return _load().oracle_num_threads()


def half_to_double(bits: int) -> float:
    return _load().oracle_half_to_double(bits)


def bf16_to_double(bits: int) -> float:
    return _load().oracle_bf16_to_double(bits)


def act_grad(x: float, act: str) -> float:
    """Derivative of the activation ``act`` ("gelu": erf form, "silu") at x."""
    return _load().oracle_act_grad(float(x), ACTS[act])


def dgrad(dY, W, H, Wd, stride=1, pad=0, dil=1, x=None, dtype=None, act="relu"):
    """dX (float64, NHWC [N][H][Wd][C]) from dY [N][P][Q][K] and W [K][R][S][C].

    H and Wd are dX's spatial sizes.  ``x`` (same shape as dX, same element
    type as dY) enables the activation-backward epilogue: for act "relu" the
    gate (x > 0) ? dX : +0.0, for "gelu" and "silu" dX * f'(x) with x the
    activation's saved input.
    """
    code = _dtype_of(dY, dtype)
    N, P, Q, K = dY.shape
    K2, R, S, C = W.shape
    if K2 != K:
        raise ValueError("K mismatch")
    if (out_extent(H, R, stride, pad, dil), out_extent(Wd, S, stride, pad, dil)) != (P, Q):
        raise ValueError("dY spatial shape does not match the geometry")
    for a in (dY, W) + ((x,) if x is not None else ()):
        _check(a, code)
    if x is not None and x.shape != (N, H, Wd, C):
        raise ValueError("x must have dX's shape")
    out = np.empty((N, H, Wd, C), np.float64)
    rc = _load().oracle_dgrad_act(_ptr(dY), _ptr(W), _ptr(x), ACTS[act], code, _ptr(out),
                                  N, H, Wd, C, K, R, S, stride, pad, dil)
    if rc:
        raise RuntimeError("oracle_dgrad failed")
    return out


def dgrad_pixels(dY, W, H, Wd, pix, stride=1, pad=0, dil=1, x=None, dtype=None, act="relu"):
    """dgrad at the pixels ``pix`` (int array [npix][3] of (n, h, w)) -> [npix][C]."""
    code = _dtype_of(dY, dtype)
    N, P, Q, K = dY.shape
    _, R, S, C = W.shape
    for a in (dY, W) + ((x,) if x is not None else ()):
        _check(a, code)
    pix = np.ascontiguousarray(pix, dtype=np.int32).reshape(-1, 3)
    out = np.empty((pix.shape[0], C), np.float64)
    rc = _load().oracle_dgrad_pixels_act(_ptr(dY), _ptr(W), _ptr(x), ACTS[act], code,
                                         pix.ctypes.data_as(ctypes.c_void_p),
                                     pix.shape[0], _ptr(out),
                                     N, H, Wd, C, K, R, S, stride, pad, dil)
    if rc:
        raise RuntimeError("oracle_dgrad_pixels failed")
    return out


def wgrad(dY, x, R, S, stride=1, pad=0, dil=1, dtype=None):
    """dW (float64, KRSC [K][R][S][C]) from dY [N][P][Q][K] and the forward
    input x [N][H][W][C]: the weight gradient of the same cross-correlation."""
    code = _dtype_of(dY, dtype)
    N, P, Q, K = dY.shape
    N2, H, Wd, C = x.shape
    if N2 != N:
        raise ValueError("N mismatch")
    if (out_extent(H, R, stride, pad, dil), out_extent(Wd, S, stride, pad, dil)) != (P, Q):
        raise ValueError("dY spatial shape does not match the geometry")
    _check(dY, code)
    _check(x, code)
    dW = np.empty((K, R, S, C), np.float64)
    rc = _load().oracle_wgrad(_ptr(dY), _ptr(x), code, _ptr(dW), N, H, Wd, C, K, R, S, stride, pad, dil)
    if rc:
        raise RuntimeError("oracle_wgrad failed")
    return dW


def wgrad_elements(dY, x, R, S, idx, stride=1, pad=0, dil=1, dtype=None):
    """dW at the filter elements ``idx`` (int array [n][4] of (k, r, s, c)) -> [n]."""
    code = _dtype_of(dY, dtype)
    N, P, Q, K = dY.shape
    _, H, Wd, C = x.shape
    _check(dY, code)
    _check(x, code)
    idx = np.ascontiguousarray(idx, dtype=np.int32).reshape(-1, 4)
    out = np.empty(idx.shape[0], np.float64)
    rc = _load().oracle_wgrad_elements(_ptr(dY), _ptr(x), code, idx.ctypes.data_as(ctypes.c_void_p), idx.shape[0],
                                       _ptr(out), N, H, Wd, C, K, R, S, stride, pad, dil)
    if rc:
        raise RuntimeError("oracle_wgrad_elements failed")
    return out


def conv_fwd(x, W, stride=1, pad=0, dil=1, dtype=None):
    """Forward cross-correlation y [N][P][Q][K] (float64) of x [N][H][W][C]."""
    code = _dtype_of(x, dtype)
    N, H, Wd, C = x.shape
    K, R, S, C2 = W.shape
    if C2 != C:
        raise ValueError("C mismatch")
    _check(x, code)
    _check(W, code)
    P, Q = out_extent(H, R, stride, pad, dil), out_extent(Wd, S, stride, pad, dil)
    if P <= 0 or Q <= 0:
        raise ValueError("empty output")
    y = np.empty((N, P, Q, K), np.float64)
    rc = _load().oracle_conv_fwd(_ptr(x), _ptr(W), code, _ptr(y),
                                 N, H, Wd, C, K, R, S, stride, pad, dil)
    if rc:
        raise RuntimeError("oracle_conv_fwd failed")
    return y


def channel_sums(out, x=None, dtype=None):
    """Per-channel sums of a dgrad output ``out`` (float64, [..., C], the
    gated dX as ``dgrad`` returns it): returns (s1, s2, a1, a2) with
    s1[c] = sum of out[..., c], s2[c] = sum of out*x over the positions where
    x > 0 (None without x), and a1, a2 the sums of the absolute values of the
    same terms.  ``x`` is the saved activation (uint16 bits of ``dtype``, same
    shape as out)."""
    out = np.ascontiguousarray(out, dtype=np.float64)
    C = out.shape[-1]
    pixels = out.size // C
    code = 0
    if x is not None:
        code = _dtype_of(x, dtype)
        _check(x, code)
        if x.size != out.size:
            raise ValueError("x must have out's shape")
    s1, a1 = np.empty(C), np.empty(C)
    s2, a2 = (np.empty(C), np.empty(C)) if x is not None else (None, None)
    rc = _load().oracle_channel_sums(_ptr(out), _ptr(x), code, pixels, C, _ptr(s1), _ptr(s2), _ptr(a1), _ptr(a2))
    if rc:
        raise RuntimeError("oracle_channel_sums failed")
    return s1, s2, a1, a2


def round_to(values, dtype: str) -> np.ndarray:
    """Round float64 values once (to nearest, ties to even) to fp16 or bf16,
    returned as uint16 bit patterns (the oracle's own encoder)."""
    lib = _load()
    fn = lib.oracle_double_to_half if dtype == "f16" else lib.oracle_double_to_bf16
    flat = np.asarray(values, dtype=np.float64).reshape(-1)
    out = np.fromiter((fn(float(v)) for v in flat), dtype=np.uint16, count=flat.size)
    return out.reshape(np.shape(values))


def dgrad_fused(dY2, W2, x2, W1, H, Wd, pad2=1, dil2=1, dtype=None, act="relu"):
    """The back-to-back dgrads of a bottleneck's 1x1 -> 3x3 forward pair:
    g = act_bwd(dgrad(dY2, W2), x2) (stride 1; x2 None: no activation),
    rounded once to the storage type as a tensor written to memory would be,
    then dX1 = dgrad_1x1(g, W1) with W1 [C2][1][1][C1].  Returns (dX1, g)
    with dX1 in float64 and g as uint16 bits of ``dtype`` (float64, unrounded,
    for float64 inputs)."""
    g = dgrad(dY2, W2, H, Wd, 1, pad2, dil2, x=x2, dtype=dtype, act=act or "relu")
    if dtype in ("f16", "bf16"):
        g = round_to(g, dtype)
    dX1 = dgrad(g, W1, H, Wd, 1, 0, 1, dtype=dtype)
    return dX1, g
