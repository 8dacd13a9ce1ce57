"""Exact float64 values of fp8 e4m3 codes, for the fp8-KV-cache oracle.

TEST INFRASTRUCTURE (same rules as the rest of oracle/).

The format (OCP 8-bit floating point, "E4M3"; the page "GPT-OSS on day 0"
serves the model in FP8): bit 7 sign, bits 6-3 exponent with bias 7,
bits 2-0 mantissa. Exponent 0 is subnormal (value m/8 * 2^-6); every other
exponent is normal ((1 + m/8) * 2^(e - 7)), including e = 15, whose only
special code is mantissa 7 (NaN). There are no infinities; the largest
finite value is 448.

Attention over an fp8 cache is attention over the decoded values times the
per-KV-head scale: `dequantize` turns the codes into float64 values and the
float64 forward in `oracle.backward` does the rest.
"""
import numpy as np


def e4m3_to_float64(codes):
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = sign * val
    return np.where((e == 15) & (c & 0x7 == 7), np.nan, val)


def dequantize(codes, scale, head_axis):
    """codes (uint8 array or tensor) -> float64 values times scale[head]."""
    if hasattr(codes, "detach"):
        codes = codes.detach().cpu().numpy()
    if hasattr(scale, "detach"):
        scale = scale.detach().cpu().double().numpy()
    x = e4m3_to_float64(codes)
    shape = [1] * x.ndim
    shape[head_axis] = x.shape[head_axis]
    return x * np.asarray(scale, dtype=np.float64).reshape(shape)
