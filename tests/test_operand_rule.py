"""The prefill GEMM's operand rule, checked by enumeration on the host.

With bf16 block scales and no zero points a dequantised weight s (q - 8)
is one exact fp16 operand; with zero points (q - zp up to 15) it is not,
and the kernel splits it hi + lo.  bf16 tokens convert to fp16 exactly in
fp16's normal range.  These facts decide which form the kernel takes."""
import numpy as np
import torch


def _bf16_values(lo_exp, hi_exp):
    """Every positive bf16 value with exponent in [lo_exp, hi_exp]."""
    bits = np.arange(0, 1 << 15, dtype=np.int32)
    v = torch.from_numpy((bits << 16).astype(np.int32)).view(torch.float32).numpy().astype(np.float64)
    e = np.floor(np.log2(np.where(v > 0, v, 1.0)))
    return v[(v > 0) & np.isfinite(v) & (e >= lo_exp) & (e <= hi_exp)]


def _exact_in_f16(w):
    return np.array_equal(w.astype(np.float16).astype(np.float64), w)


def test_bf16_scale_symmetric_weight_is_one_fp16_operand():
    s = _bf16_values(-14, 11)            # products stay in fp16's normal range
    for v in range(-8, 8):
        assert _exact_in_f16(s * v), v


def test_bf16_scale_with_zero_points_needs_a_split():
    s = _bf16_values(-10, 8)
    inexact = [v for v in range(-15, 16) if not _exact_in_f16(s * v)]
    assert inexact == [-15, -13, -11, -9, 9, 11, 13, 15]


def test_fp16_scale_weight_needs_a_split():
    s = np.arange(1024, 2048, dtype=np.float64) * 2.0 ** -14   # every fp16 significand in [2^-4, 2^-3)
    assert not _exact_in_f16(s * 3)


def test_bf16_tokens_convert_to_fp16_exactly_in_range():
    x = _bf16_values(-14, 15)
    x = x[x <= 65504]
    assert _exact_in_f16(x) and _exact_in_f16(-x)
