"""The two-sided zero-pattern check of the ReLU-backward gate (tests/gpu_util)
catches both kinds of mistake: a gated-off position that is not +0.0, and a
zero written where the gate passes a value that is not zero.  CPU only: the
outputs here are built by hand, no kernel runs."""
import numpy as np
import pytest

from implicit_gemm_dgrad_gb300 import synth

from gpu_util import check_gate_zero_pattern


def _case():
    x = synth.to_bits(np.array([1.0, 0.0, -1.0, 2.0, 3.0, -0.0], np.float32), "bf16")
    x[5] = 0x8000  # -0.0
    ref = np.array([0.5, 7.0, -3.0, 0.0, 1e-45, 4.0])  # 0.0 and 1e-45 round to zero in bf16
    out = synth.to_bits(np.array([0.5, 0.0, 0.0, 0.0, 0.0, 0.0], np.float32), "bf16")
    return x, ref, out


def test_correct_pattern_passes_and_counts_exact_zeros():
    x, ref, out = _case()
    counts = check_gate_zero_pattern(out.view(np.uint8), x, ref, "bf16", "bf16")
    assert counts == {"masked": 3, "unmasked": 3, "unmasked_oracle_zero": 2,
                      "unmasked_oracle_zero_written_zero": 2}


def test_gated_off_value_that_is_not_plus_zero_fails():
    x, ref, out = _case()
    out[2] = 0x8000  # -0.0 where x < 0
    with pytest.raises(AssertionError, match="gated-off"):
        check_gate_zero_pattern(out.view(np.uint8), x, ref, "bf16", "bf16")


def test_spurious_zero_where_the_gate_passes_fails():
    x, ref, out = _case()
    out[0] = 0x0000  # x > 0 and the oracle is 0.5
    with pytest.raises(AssertionError, match="unmasked"):
        check_gate_zero_pattern(out.view(np.uint8), x, ref, "bf16", "bf16")
    out[0] = 0x8000  # -0.0 counts as a zero too
    with pytest.raises(AssertionError, match="unmasked"):
        check_gate_zero_pattern(out.view(np.uint8), x, ref, "bf16", "bf16")


def test_fp32_and_fp16_outputs():
    x = synth.to_bits(np.array([1.0, -1.0, 1.0], np.float32), "f16")
    ref = np.array([2.0, 5.0, 2.0 ** -26])  # 2^-26 rounds to zero in fp16, not in fp32
    out16 = synth.to_bits(np.array([2.0, 0.0, 0.0], np.float32), "f16")
    assert check_gate_zero_pattern(out16.view(np.uint8), x, ref, "f16", "f16")["unmasked_oracle_zero"] == 1
    out32 = np.array([2.0, 0.0, 0.0], np.float32)
    with pytest.raises(AssertionError, match="unmasked"):
        check_gate_zero_pattern(out32.view(np.uint8), x, ref, "f32", "f16")
