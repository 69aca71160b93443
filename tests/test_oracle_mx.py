"""Pins for the oracle's MXFP8 quantiser against facts fixed outside the oracle:
the pages' format facts (golden fixture), an independent enumeration of the
E4M3 code table, brute-force nearest-code search, exact round trips, the OCP MX
special cases and the format's error bound."""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from conftest import read_golden
from oracle import mx


def _e4m3_table_by_enumeration():
    """Every E4M3 code's exact value, written from the bit layout (1/4/3, bias 7,
    subnormals at exponent 0, S.1111.111 = NaN), as Fractions."""
    vals = {}
    for code in range(256):
        sign = -1 if code & 0x80 else 1
        ef = (code >> 3) & 0xF
        mf = code & 0x7
        if ef == 0xF and mf == 0x7:
            continue                                   # NaN
        if ef == 0:
            v = Fraction(mf, 8) * Fraction(1, 2 ** 6)
        else:
            v = (1 + Fraction(mf, 8)) * (Fraction(2) ** (ef - 7))
        vals[code] = sign * v
    return vals


TABLE = _e4m3_table_by_enumeration()


def test_golden_format_facts():
    g = read_golden("mxfp8_format.txt")
    assert mx.BLOCK == g["mx_block_values"]
    assert g["e4m3_sign_bits"] + g["e4m3_exponent_bits"] + g["e4m3_mantissa_bits"] == g["mx_element_bits"]
    assert mx.E4M3_MBITS == g["e4m3_mantissa_bits"]
    # 4 exponent bits with bias 7 -> largest normal binade 2^8, smallest 2^-6
    assert mx.E4M3_EMAX == (2 ** g["e4m3_exponent_bits"] - 1) - 7
    assert mx.E4M3_EMIN == 1 - 7
    # E8M0: 8 exponent bits, bias 127
    assert mx.E8M0_BIAS == 2 ** (g["e8m0_exponent_bits"] - 1) - 1
    # BF16 1/8/7: decode a few bit patterns by hand and compare with torch's bf16
    assert g["bf16_sign_bits"] + g["bf16_exponent_bits"] + g["bf16_mantissa_bits"] == 16
    for bits in [0x3F80, 0xC000, 0x0001, 0x7F7F, 0x3E20]:
        s = -1.0 if bits >> 15 else 1.0
        e = (bits >> 7) & 0xFF
        m = bits & 0x7F
        v = s * (m / 128.0) * 2.0 ** -126 if e == 0 else s * (1 + m / 128.0) * 2.0 ** (e - 127)
        t = torch.from_numpy(np.array([bits], dtype=np.uint16).view(np.int16)).view(torch.bfloat16).double().item()
        assert v == t


def test_decode_matches_enumeration():
    dec = mx.e4m3_decode(np.arange(256))
    for code in range(256):
        if code in TABLE:
            assert dec[code] == float(TABLE[code]), hex(code)
        else:
            assert np.isnan(dec[code])
    assert max(float(v) for v in TABLE.values()) == mx.E4M3_MAX == 448.0
    assert len(TABLE) == 254


def _brute_nearest(values):
    """Nearest finite E4M3 code value to each value, ties to the code with an even
    mantissa; beyond the largest finite magnitude the nearest is +-448."""
    pos = sorted({float(v) for v in TABLE.values() if v >= 0})
    grid = np.array(pos)
    codes_of = {float(TABLE[c]): c for c in TABLE if TABLE[c] >= 0 and not (c & 0x80)}
    a = np.abs(values)
    hi = np.clip(np.searchsorted(grid, a, side="left"), 1, grid.size - 1)
    lo = hi - 1
    dlo = a - grid[lo]
    dhi = grid[hi] - a
    pick_hi = dhi < dlo
    tie = dhi == dlo
    even_hi = np.array([codes_of[g] % 2 == 0 for g in grid])[hi]
    pick_hi = pick_hi | (tie & even_hi)
    out = np.where(pick_hi, grid[hi], grid[lo])
    out = np.where(a >= grid[-1], grid[-1], out)
    out = np.where(a <= grid[0], grid[0], out)
    return np.copysign(out, values)


def test_element_rounding_brute_force_all_bf16():
    """Every finite bf16 value, scaled by 2^-e for e in [-20, 20], rounds to the
    brute-force nearest E4M3 value (ties to even, saturating)."""
    bits = np.arange(65536, dtype=np.uint32)
    f32 = (bits << 16).view(np.float32)
    f32 = f32[np.isfinite(f32)].astype(np.float64)
    for e in range(-20, 21):
        s = f32 * 2.0 ** -e
        got = mx.e4m3_round(s)
        want = _brute_nearest(s)
        bad = got != want
        assert not bad.any(), (e, s[bad][:5], got[bad][:5], want[bad][:5])
        codes = mx.e4m3_encode(got)
        back = mx.e4m3_decode(codes)
        assert np.array_equal(back, got)


def test_exact_blocks_round_trip():
    """Blocks of codes * 2^e whose largest code lies in [256, 448] quantise back to
    the same codes and exponent."""
    rng = np.random.default_rng(7)
    finite = np.array([c for c in TABLE if not (c & 0x80)])
    big = np.array([c for c in finite if 256 <= float(TABLE[c]) <= 448])
    for trial in range(200):
        e = int(rng.integers(-120, 118))
        codes = rng.choice(finite, size=32)
        codes[rng.integers(32)] = rng.choice(big)
        signs = rng.integers(0, 2, size=32)
        codes = codes | (signs << 7)
        codes = np.where(codes == 0x80, 0, codes)     # +0 only: -0 cannot come back from +0
        vals = np.array([float(TABLE[int(c)]) for c in codes]) * 2.0 ** e
        q, s = mx.quantize_blocks(vals[None, :])
        assert int(s[0, 0]) == e + 127
        assert np.array_equal(q[0].astype(np.int64), codes.astype(np.int64))


@pytest.mark.parametrize("n", [-100, -7, 0, 3, 60, 110])
def test_special_blocks(n):
    z = np.zeros((1, 32))
    q, s = mx.quantize_blocks(z)
    assert s[0, 0] == 0 and not q.any()
    # a single non-zero value v: e = floor(log2|v|) - 8
    v = z.copy()
    v[0, 5] = -3.0 * 2.0 ** n
    q, s = mx.quantize_blocks(v)
    assert int(s[0, 0]) == (n + 1) - 8 + 127
    assert float(TABLE[int(q[0, 5])]) * 2.0 ** (n + 1 - 8) == -3.0 * 2.0 ** n
    for amax, code in [(256.0, 0x78), (448.0, 0x7E), (464.0, 0x7E), (480.0, 0x7E), (511.0, 0x7E)]:
        v = z.copy()
        v[0, 0] = amax * 2.0 ** n
        v[0, 1] = 2.0 ** n                          # 1.0 after scaling -> code 0x38
        q, s = mx.quantize_blocks(v)
        assert int(s[0, 0]) == n + 127, amax
        assert int(q[0, 0]) == code and int(q[0, 1]) == 0x38, amax


def test_scale_byte_pure_python():
    """Shared exponent from math.frexp on each block, one block at a time."""
    rng = np.random.default_rng(3)
    v = rng.standard_normal((64, 128)) * np.exp2(rng.integers(-60, 60, size=(64, 1)))
    _, s = mx.quantize_blocks(v)
    for r in range(64):
        for b in range(4):
            amax = max(abs(float(t)) for t in v[r, 32 * b:32 * b + 32])
            m, ex = math.frexp(amax)
            assert int(s[r, b]) == (ex - 1) - 8 + 127


def test_error_bound():
    """|deq - v| <= 2^-4 * 2^floor(log2|v|) inside the normal range (3 mantissa
    bits), and saturated values land on 448 * 2^e."""
    rng = np.random.default_rng(11)
    v = rng.standard_normal((256, 64)) * np.exp2(rng.integers(-30, 30, size=(256, 1)))
    q, s = mx.quantize_blocks(v)
    d = mx.dequantize_blocks(q, s)
    e = (s.astype(np.int64) - 127).repeat(32, axis=1)
    scaled = np.abs(v) * np.exp2(-e)
    normal = (scaled >= 2.0 ** -6) & (scaled <= 448.0)
    fl = np.floor(np.log2(np.abs(v[normal])))
    assert np.all(np.abs(d[normal] - v[normal]) <= 2.0 ** (fl - 4) * (1 + 1e-12))
    sat = scaled > 448.0
    assert np.all(np.abs(d[sat]) == 448.0 * np.exp2(e[sat]))


def test_group_columns_blocks_restart_at_group_start():
    rng = np.random.default_rng(5)
    a = rng.standard_normal((40, 64))
    a[32:] *= 1e-3                                    # second block much smaller
    c, s = mx.quantize_group_columns(a)
    assert c.shape == (64, 64) and s.shape == (64, 2)
    # block 0 = rows 0..31, block 1 = rows 32..39 + 24 zero rows
    for col in range(64):
        e0 = math.frexp(np.abs(a[:32, col]).max())[1] - 1 - 8
        e1 = math.frexp(np.abs(a[32:, col]).max())[1] - 1 - 8
        assert int(s[col, 0]) == e0 + 127 and int(s[col, 1]) == e1 + 127
    assert not c[:, 40:].any()
    back = mx.fake_quant_group_columns(a)
    assert back.shape == a.shape
    np.testing.assert_array_equal(back[:32], mx.fake_quant(a[:32].T).T)


def test_fake_quant_equals_quantize_then_dequantize():
    """The direct fake-quantiser is the quantise -> encode -> decode -> dequantise
    round trip, bit for bit."""
    rng = np.random.default_rng(21)
    v = rng.standard_normal((300, 256)) * np.exp2(rng.integers(-50, 50, size=(300, 1)))
    v[0] = 0.0
    v[1, :32] = 448.0 * 2.0 ** 5
    v[2, 7] = 464.0
    v[3, 40:64] = 1e-300
    c, s = mx.quantize_blocks(v)
    ref = mx.dequantize_blocks(c, s)
    got = mx.fake_quant(v, chunk_rows=37)
    assert np.array_equal(got, ref)
    assert np.array_equal(np.signbit(got), np.signbit(ref))
