"""MXFP8 format and block quantiser — CPU oracle (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may use
this package.  It shares no code with the CUDA path.

Source of the format:
  * BioNeMo Uses Grouped Kernels and MXFP8 (toolai.io), "Reducing memory
    pressure with MXFP8" and Fig. 3: MXFP8 stores 8-bit E4M3 values with one
    shared E8M0 scale per block of 32 consecutive values.
  * How BioNeMo cuts overhead in biological AI training (roboticlifestyle.com),
    "How MXFP8 reduces memory use": one scaling factor per block of 32
    consecutive values; master weights stay 16-bit and are converted before the
    low-precision GEMMs.
The pages do not give the scale-selection rule.  This oracle takes the OCP
Microscaling (MX) v1.0 rule: shared exponent = floor(log2(max|v|)) - 8 (8 is
E4M3's largest normal exponent), clamped to the E8M0 range, elements rounded to
nearest-even and saturated to +-448.  Readings where the rule is silent:
  * an all-zero block gets exponent -127 (scale byte 0x00) and zero codes;
  * a negative value that rounds to zero keeps its sign (code 0x80);
  * NaN inputs are out of scope.

Everything here is exact fp64 arithmetic: scaling by a power of two, frexp for
floor(log2), np.rint for round-half-even.
"""
from __future__ import annotations

import numpy as np

BLOCK = 32               # values per shared scale (Fig. 3)
E4M3_MAX = 448.0         # largest finite E4M3 magnitude, 1.75 * 2^8
E4M3_EMAX = 8            # exponent of the largest normal E4M3 binade
E4M3_EMIN = -6           # exponent of the smallest normal E4M3 binade
E4M3_MBITS = 3
E8M0_BIAS = 127
SCALE_EXP_MIN, SCALE_EXP_MAX = -127, 127


def e4m3_decode(codes) -> np.ndarray:
    """E4M3 bit pattern -> value: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
    bits; exponent field 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; no Inf."""
    c = np.asarray(codes, dtype=np.int64)
    s = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** E4M3_EMIN, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def e8m0_decode(scale_bytes) -> np.ndarray:
    """E8M0 scale byte b -> 2^(b-127) (0xFF would be NaN; never produced here)."""
    b = np.asarray(scale_bytes, dtype=np.int64)
    return np.ldexp(1.0, b - E8M0_BIAS)


def floor_log2(a: np.ndarray) -> np.ndarray:
    """Exact floor(log2(a)) for finite a > 0, from the fp64 exponent (frexp)."""
    _, ex = np.frexp(a)
    return ex.astype(np.int64) - 1


def e4m3_round(s: np.ndarray) -> np.ndarray:
    """Round fp64 values onto the E4M3 grid, nearest-even, saturating to +-448."""
    s = np.asarray(s, dtype=np.float64)
    a = np.abs(s)
    with np.errstate(divide="ignore"):
        fl = np.where(a > 0, floor_log2(np.where(a > 0, a, 1.0)), E4M3_EMIN)
    fl = np.maximum(fl, E4M3_EMIN)                 # subnormal spacing below 2^-6
    quantum = np.ldexp(1.0, fl - E4M3_MBITS)
    q = np.rint(a / quantum) * quantum             # a/quantum is exact (power of two)
    q = np.minimum(q, E4M3_MAX)
    return np.copysign(q, s)


def e4m3_encode(q: np.ndarray) -> np.ndarray:
    """Values already on the E4M3 grid (|q| <= 448) -> bit patterns."""
    q = np.asarray(q, dtype=np.float64)
    sign = np.signbit(q).astype(np.int64)
    a = np.abs(q)
    normal = a >= 2.0 ** E4M3_EMIN
    fl = floor_log2(np.where(normal, a, 1.0))
    exp_field = np.where(normal, fl + 7, 0)
    frac = np.where(normal, a / np.ldexp(1.0, fl) - 1.0, a / 2.0 ** E4M3_EMIN)
    mant = frac * 8.0
    assert np.all(mant == np.rint(mant)), "value not on the E4M3 grid"
    return ((sign << 7) | (exp_field << 3) | mant.astype(np.int64)).astype(np.uint8)


def block_scale_exponent(amax: np.ndarray) -> np.ndarray:
    """Shared exponent of a block from its max magnitude: floor(log2 amax) - 8,
    clamped to [-127, 127]; amax == 0 -> -127."""
    amax = np.asarray(amax, dtype=np.float64)
    pos = amax > 0
    e = np.where(pos, floor_log2(np.where(pos, amax, 1.0)) - E4M3_EMAX, SCALE_EXP_MIN)
    return np.clip(e, SCALE_EXP_MIN, SCALE_EXP_MAX)


def quantize_blocks(v: np.ndarray):
    """MX-quantise along the last axis, whose length is a multiple of 32.

    Returns (codes uint8 same shape, scale bytes uint8 [..., K/32]).
    """
    v = np.asarray(v, dtype=np.float64)
    K = v.shape[-1]
    assert K % BLOCK == 0
    b = v.reshape(v.shape[:-1] + (K // BLOCK, BLOCK))
    amax = np.max(np.abs(b), axis=-1)
    e = block_scale_exponent(amax)
    scaled = b * np.ldexp(1.0, -e)[..., None]      # exact: multiply by 2^-e
    codes = e4m3_encode(e4m3_round(scaled)).reshape(v.shape)
    return codes, (e + E8M0_BIAS).astype(np.uint8)


def dequantize_blocks(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Inverse of quantize_blocks in exact fp64: E4M3(code) * 2^(byte-127)."""
    K = codes.shape[-1]
    vals = e4m3_decode(codes).reshape(codes.shape[:-1] + (K // BLOCK, BLOCK))
    return (vals * e8m0_decode(scales)[..., None]).reshape(codes.shape)


def fake_quant(v: np.ndarray, chunk_rows: int | None = None) -> np.ndarray:
    """Quantise then dequantise along the last axis, without materialising the
    bit patterns: the dequantised value is the E4M3-rounded scaled value times
    2^e (encode followed by decode is the identity on the E4M3 grid).  Same
    steps as quantize_blocks: block max, shared exponent, exact scaling, RNE
    with saturation.  Processed in row chunks to bound memory."""
    v = np.asarray(v, dtype=np.float64)
    K = v.shape[-1]
    assert K % BLOCK == 0
    flat = v.reshape(-1, K)
    out = np.empty_like(flat)
    if chunk_rows is None:                      # ~64K elements: temporaries stay in cache
        chunk_rows = max(1, 65536 // K)
    for r0 in range(0, flat.shape[0], chunk_rows):
        b = flat[r0:r0 + chunk_rows].reshape(-1, K // BLOCK, BLOCK)
        e = block_scale_exponent(np.max(np.abs(b), axis=-1))
        scale = np.ldexp(1.0, e)[..., None]
        out[r0:r0 + chunk_rows] = (e4m3_round(b / scale) * scale).reshape(-1, K)
    return out.reshape(v.shape)


def quantize_group_columns(a: np.ndarray) -> tuple:
    """Column-wise MX over the token dimension of one expert group.

    ``a`` is [m, C] (the group's rows in permuted order).  Blocks are 32
    consecutive rows starting at the group's first row; a short last block is
    padded with zero rows.  Returns (codesT uint8 [C, mpad], scalesT uint8
    [C, mpad/32]) with mpad = m rounded up to a multiple of 32, i.e. the
    transposed matrix quantised along its last axis.
    """
    m, C = a.shape
    mpad = -(-m // BLOCK) * BLOCK
    t = np.zeros((C, mpad), dtype=np.float64)
    t[:, :m] = a.T
    return quantize_blocks(t)


def fake_quant_group_columns(a: np.ndarray) -> np.ndarray:
    """Column-wise quantise-dequantise of one group, returned as [m, C]."""
    m = a.shape[0]
    c, s = quantize_group_columns(a)
    return dequantize_blocks(c, s)[:, :m].T
