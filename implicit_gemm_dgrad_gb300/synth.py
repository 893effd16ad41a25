"""Seeded synthetic inputs for the dgrad workloads.

This module holds random-number generation and rounding to the storage type
only -- none of the convolution's arithmetic.  Both the GPU path (through the
benchmark and tests) and the CPU oracle receive exactly the arrays made here.

Recipe:
  * generator: numpy ``Generator(PCG64(seed))``, seed =
    20260000 + 1000*workload + 10*layer + {dY: 0, W: 1, x: 2};
  * values are drawn in float32 and rounded once, round-to-nearest-even, to
    the storage type (fp16 or bf16); fp16/bf16 arrays are returned as uint16
    bit patterns;
  * distributions: "uniform" draws U[-1, 1]; "normal" draws dY ~ N(0, 1) and
    W ~ N(0, 2 / (C*R*S)) (He fan-in of the forward convolution); the saved
    activation for the ReLU-backward gate is x = relu(z), z ~ N(0, 1);
    "int" draws integers uniformly from {-2, ..., 2} (exact in every type).
"""
from __future__ import annotations

import numpy as np

ROLE_OFFSET = {"dY": 0, "W": 1, "x": 2}


def seed_for(workload: int, layer: int, role: str) -> int:
    return 20260000 + 1000 * workload + 10 * layer + ROLE_OFFSET[role]


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest-even), returned as uint16 bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    if nan.any():
        r = np.where(nan, ((u >> 16) | 0x40).astype(np.uint16), r)
    return r


def f32_to_f16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to IEEE binary16 (nearest-even), returned as uint16 bits."""
    return np.ascontiguousarray(a, dtype=np.float32).astype(np.float16).view(np.uint16)


def to_bits(a: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return f32_to_bf16_bits(a)
    if dtype == "f16":
        return f32_to_f16_bits(a)
    raise ValueError(dtype)


def bits_to_f32(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Widen stored fp16/bf16 bit patterns to float32 (exact)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << 16).view(np.float32)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float32)
    raise ValueError(dtype)


def _draw(rng, shape, dist, std=1.0):
    if dist == "uniform":
        return rng.uniform(-1.0, 1.0, size=shape).astype(np.float32)
    if dist == "normal":
        return (rng.standard_normal(size=shape, dtype=np.float32) * np.float32(std))
    if dist == "int":
        return rng.integers(-2, 3, size=shape).astype(np.float32)
    raise ValueError(dist)


def make_inputs(shape: dict, dtype: str, dist: str, workload: int, layer: int = 0,
                with_x: bool = False, batch: int | None = None):
    """dY [N][P][Q][K], W [K][R][S][C] and optionally x [N][H][W][C].

    ``shape`` has keys N, H, W, C, K, R, S, P, Q.  ``batch`` overrides N (the
    images drawn are then the first ``batch`` of a stream seeded the same way,
    so a smaller batch is a prefix of the full one).
    """
    N = shape["N"] if batch is None else batch
    P, Q, K, R, S, C = (shape[k] for k in ("P", "Q", "K", "R", "S", "C"))
    H, Wd = shape["H"], shape["W"]
    rng = np.random.Generator(np.random.PCG64(seed_for(workload, layer, "dY")))
    dY = to_bits(_draw(rng, (N, P, Q, K), dist), dtype)
    rng = np.random.Generator(np.random.PCG64(seed_for(workload, layer, "W")))
    std = float(np.sqrt(2.0 / (C * R * S)))
    W = to_bits(_draw(rng, (K, R, S, C), dist, std), dtype)
    x = None
    if with_x:
        rng = np.random.Generator(np.random.PCG64(seed_for(workload, layer, "x")))
        z = _draw(rng, (N, H, Wd, C), "normal" if dist != "int" else "int")
        x = to_bits(np.maximum(z, np.float32(0.0)), dtype)
    return dY, W, x
