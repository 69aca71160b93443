"""Per-tensor FP8 (E4M3, current scaling) — CPU oracle (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may use
this module.  It shares no code with the CUDA path.

Source: BioNeMo Uses Grouped Kernels and MXFP8 (toolai.io), "Reducing memory
pressure with MXFP8": the recipe runs FP8 as well as MXFP8 through Transformer
Engine, and the two differ in scaling granularity — MXFP8 scales every block of
32 consecutive values separately, FP8 does not.  The pages give no FP8 scale
rule.  Readings (the plainest ones the rest supports):
  * one scale per tensor, chosen from the tensor being quantised ("current
    scaling"): s = 448 / amax, with amax the largest magnitude of the tensor and
    448 E4M3's largest finite value, both in fp32 and the division rounded to
    nearest (fp32); an all-zero tensor takes s = 1 and s is capped at the
    largest finite fp32 (a tensor of tiny values);
  * a code is the E4M3 value nearest (ties to even) to the fp32 product v * s,
    saturating to +-448; the decision is taken in fp32 because the kernels take
    it there (a bf16 input is exact in fp32; an fp64 input is first rounded to
    fp32);
  * the dequantised value is code / s (exact in fp64);
  * a tensor is one GEMM operand of one expert: the expert's weight matrix
    (GroupedLinear keeps weight0, weight1, ... separate) and the expert's rows
    of x, h, dy and dGU.  A transposed operand is the same tensor, so it has
    the same scale and the same codes.
"""
from __future__ import annotations

import numpy as np

from . import mx

F32_MAX = np.float32(np.finfo(np.float32).max)


def tensor_scale(amax) -> np.float32:
    """s = 448 / amax in fp32 (1 for amax == 0, capped at the largest fp32)."""
    a = np.float32(amax)
    if not a > 0:
        return np.float32(1.0)
    with np.errstate(over="ignore"):
        s = np.float32(mx.E4M3_MAX) / a
    return np.minimum(s, F32_MAX)


def quantize(v, amax=None):
    """Codes (uint8, same shape) and the fp32 scale of one tensor."""
    v32 = np.asarray(v, dtype=np.float32)
    a = np.max(np.abs(v32)) if amax is None else np.float32(amax)
    s = tensor_scale(a)
    p = v32 * s                                     # fp32 product, rounded to nearest
    return mx.e4m3_encode(mx.e4m3_round(p.astype(np.float64))), s


def dequantize(codes, s) -> np.ndarray:
    return mx.e4m3_decode(codes) / np.float64(s)


def fake_quant(v) -> np.ndarray:
    """Quantise then dequantise one tensor (values returned in fp64)."""
    v = np.asarray(v)
    if v.size == 0:
        return np.asarray(v, dtype=np.float64)
    codes, s = quantize(v)
    return dequantize(codes, s)
