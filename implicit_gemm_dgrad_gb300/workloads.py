"""The dgrad problem shapes that the tests and the benchmark run.

Layer shapes follow the ResNet-50 (v1.5) bottleneck convolutions that the
apache/tvm PR #10110 page ("[CUTLASS] Conv2d dgrad", benchmark comment)
benchmarks dgrad on at batch 8 and 256.  For every layer, C is the forward
convolution's input channel count (= dX channels), K its output channel count
(= dY channels), H x W the forward input size (= dX spatial size).

P and Q (dY's spatial size) follow the floor convention
P = floor((H + 2*pad - dil*(R-1) - 1)/stride) + 1.
"""
from __future__ import annotations

from dataclasses import dataclass, asdict


@dataclass(frozen=True)
class Layer:
    name: str
    N: int
    H: int
    W: int
    C: int
    K: int
    R: int
    S: int
    stride: int = 1
    pad: int = 0
    dil: int = 1
    dtype: str = "bf16"      # dY, W and the saved activation
    out: str = "same"        # "same" (dX in dtype) or "f32"
    relu: bool = False       # fused ReLU-backward gate
    dist: str = "normal"     # synth.make_inputs distribution
    workload: int = 0        # seed family
    index: int = 0           # seed index within the family

    @property
    def P(self) -> int:
        return (self.H + 2 * self.pad - self.dil * (self.R - 1) - 1) // self.stride + 1

    @property
    def Q(self) -> int:
        return (self.W + 2 * self.pad - self.dil * (self.S - 1) - 1) // self.stride + 1

    def shape(self) -> dict:
        d = asdict(self)
        d.update(P=self.P, Q=self.Q)
        return d

    @property
    def flops(self) -> int:
        """Useful multiply-adds x 2: 2*N*P*Q*K*C*R*S (no zero-insertion)."""
        return 2 * self.N * self.P * self.Q * self.K * self.C * self.R * self.S

    @property
    def flops_literal(self) -> int:
        """2*N*H*W*C*K*R*S: counts the zero-inserted work of strided layers."""
        return 2 * self.N * self.H * self.W * self.C * self.K * self.R * self.S

    def out_bytes_per_el(self) -> int:
        return 4 if self.out == "f32" else 2

    @property
    def bytes(self) -> int:
        """Algorithmic HBM bytes: dY + W + dX (+ x when gated), each once."""
        b = 2 * (self.N * self.P * self.Q * self.K + self.K * self.R * self.S * self.C)
        b += self.out_bytes_per_el() * self.N * self.H * self.W * self.C
        if self.relu:
            b += 2 * self.N * self.H * self.W * self.C
        return b

    def with_batch(self, n: int) -> "Layer":
        d = asdict(self)
        d["N"] = n
        return Layer(**d)


TINY = Layer("tiny", 1, 8, 8, 16, 16, 3, 3, 1, 1, 1, dtype="f16", out="f32",
             dist="uniform", workload=0)

BATCH8 = [
    Layer("b8_s1_3x3", 8, 56, 56, 64, 64, 3, 3, 1, 1, 1, dtype="f16", workload=1),
    Layer("b8_s2_3x3", 8, 56, 56, 128, 128, 3, 3, 2, 1, 1, dtype="f16", workload=2, index=0),
    Layer("b8_s2_1x1", 8, 56, 56, 256, 512, 1, 1, 2, 0, 1, dtype="f16", workload=2, index=1),
]


def _rn50(N: int = 256):
    # (name, H, C, K, R, stride, pad); W = H, S = R
    rows = [
        ("L01_1x1_64-64_56", 56, 64, 64, 1, 1, 0),
        ("L02_1x1_64-256_56", 56, 64, 256, 1, 1, 0),
        ("L03_1x1_256-64_56", 56, 256, 64, 1, 1, 0),
        ("L04_3x3_64_56", 56, 64, 64, 3, 1, 1),
        ("L05_1x1_256-128_56", 56, 256, 128, 1, 1, 0),
        ("L06_3x3s2_128_56-28", 56, 128, 128, 3, 2, 1),
        ("L07_1x1_128-512_28", 28, 128, 512, 1, 1, 0),
        ("L08_1x1_512-128_28", 28, 512, 128, 1, 1, 0),
        ("L09_3x3_128_28", 28, 128, 128, 3, 1, 1),
        ("L10_1x1s2_256-512_56-28", 56, 256, 512, 1, 2, 0),
        ("L11_1x1_512-256_28", 28, 512, 256, 1, 1, 0),
        ("L12_3x3s2_256_28-14", 28, 256, 256, 3, 2, 1),
        ("L13_1x1_256-1024_14", 14, 256, 1024, 1, 1, 0),
        ("L14_1x1_1024-256_14", 14, 1024, 256, 1, 1, 0),
        ("L15_3x3_256_14", 14, 256, 256, 3, 1, 1),
        ("L16_1x1s2_512-1024_28-14", 28, 512, 1024, 1, 2, 0),
        ("L17_1x1_1024-512_14", 14, 1024, 512, 1, 1, 0),
        ("L18_3x3s2_512_14-7", 14, 512, 512, 3, 2, 1),
        ("L19_1x1_512-2048_7", 7, 512, 2048, 1, 1, 0),
        ("L20_1x1_2048-512_7", 7, 2048, 512, 1, 1, 0),
        ("L21_3x3_512_7", 7, 512, 512, 3, 1, 1),
        ("L22_1x1s2_1024-2048_14-7", 14, 1024, 2048, 1, 2, 0),
    ]
    return [Layer(name, N, H, H, C, K, R, R, s, p, 1, dtype="bf16", workload=3, index=i)
            for i, (name, H, C, K, R, s, p) in enumerate(rows)]


RESNET50_B256 = _rn50(256)

FUSED_RELU = [
    Layer("F1_3x3_128_28_relu", 256, 28, 28, 128, 128, 3, 3, 1, 1, 1, dtype="bf16",
          relu=True, workload=4, index=0),
    Layer("F2_3x3s2_256_28-14_relu", 256, 28, 28, 256, 256, 3, 3, 2, 1, 1, dtype="bf16",
          relu=True, workload=4, index=1),
]

ALL = [TINY] + BATCH8 + RESNET50_B256 + FUSED_RELU


def by_name(name: str) -> Layer:
    for layer in ALL:
        if layer.name == name:
            return layer
    raise KeyError(name)
