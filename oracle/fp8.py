"""Per-tensor FP8 (E4M3, current scaling) — CPU oracle (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may use
this module.  It shares no code with the CUDA path.

Source: BioNeMo Uses Grouped Kernels and MXFP8 (toolai.io), "Reducing memory
pressure with MXFP8": the recipe runs FP8 as well as MXFP8 through Transformer
Engine, and the two differ in scaling granularity — MXFP8 scales every block of
32 consecutive values separately, FP8 does not.  The pages give no FP8 scale
rule beyond that difference.  Readings (the plainest ones the rest supports):
  * the only difference from MXFP8 is the granularity, so a tensor takes the
    MX scale rule with the whole tensor as its block: exponent e =
    floor(log2(amax)) - 8 from the tensor's largest magnitude, clamped to
    [-127, 127] (-127 for an all-zero tensor); codes are v * 2^-e rounded to
    the nearest E4M3 value (ties to even), saturating to +-448; the
    dequantised value is code * 2^e.  Scaling by a power of two is exact, so
    every step is exact in fp64;
  * a tensor is one GEMM operand of one expert: the expert's weight matrix
    (GroupedLinear keeps weight0, weight1, ... separate) and the expert's rows
    of x, h, dy and dGU.  A transposed operand is the same tensor, so it has
    the same scale and the same codes.
"""
from __future__ import annotations

import numpy as np

from . import mx


def tensor_exponent(amax) -> int:
    """e = floor(log2 amax) - 8 clamped to [-127, 127]; -127 for amax == 0."""
    return int(mx.block_scale_exponent(np.float64(amax)))


def quantize(v, amax=None):
    """Codes (uint8, same shape) and the exponent e of one tensor."""
    v = np.asarray(v, dtype=np.float64)
    a = np.max(np.abs(v)) if amax is None else float(amax)
    e = tensor_exponent(a)
    return mx.e4m3_encode(mx.e4m3_round(v * np.ldexp(1.0, -e))), e


def dequantize(codes, e) -> np.ndarray:
    return mx.e4m3_decode(codes) * np.ldexp(1.0, e)


def fake_quant(v) -> np.ndarray:
    """Quantise then dequantise one tensor (values returned in fp64)."""
    v = np.asarray(v)
    if v.size == 0:
        return np.asarray(v, dtype=np.float64)
    codes, e = quantize(v)
    return dequantize(codes, e)
