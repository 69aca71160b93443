"""Pins of the per-tensor FP8 oracle (oracle/fp8.py) to facts outside itself:
brute-force nearest E4M3 code over all 256 bit patterns, the tensor maximum
landing on 448, exact round trips of values on a per-tensor grid, the all-zero
tensor, the error bound of round-to-nearest, and the MoE oracle's fp8 mode
reducing to the exact MLP on inputs that lie on every expert operand's grid."""
import numpy as np

from oracle import fp8, moe


def _all_finite_codes():
    vals = []
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            continue                                       # NaN patterns
        mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
        vals.append((c, -mag if s else mag))
    return vals


CODES = _all_finite_codes()


def _brute(p: float) -> int:
    """Nearest finite E4M3 value to p, ties to the even mantissa; the sign of
    zero follows p; beyond +-448 the nearest finite value is +-448."""
    best = min(abs(v - p) for _, v in CODES)
    cands = [(c, v) for c, v in CODES if abs(v - p) == best]
    if len(cands) > 1:
        even = [(c, v) for c, v in cands if (c & 1) == 0]
        cands = even if even else cands
    if all(v == 0.0 for _, v in cands):
        return 0x80 if np.signbit(p) else 0x00
    return cands[0][0]


def test_codes_are_nearest_e4m3_of_scaled_values():
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 1 << 16, 4000, dtype=np.uint32) << 16
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    v = f[np.abs(f) < 1e30].astype(np.float64)
    amax = np.max(np.abs(v))
    codes, e = fp8.quantize(v)
    assert e == int(np.floor(np.log2(amax))) - 8
    p = v * 2.0 ** -e
    for i in range(0, v.size, 7):
        assert codes[i] == _brute(float(p[i])), (v[i], p[i], codes[i])


def test_tensor_scale_rule_and_saturation():
    codes, e = fp8.quantize(np.array([0.5, -3.0, 1.25, 2.0]))
    assert e == -7 and codes[1] == 0xFC                      # -3 * 2^7 = -384
    codes, e = fp8.quantize(np.array([1.9 * 2.0 ** 5, 1.0]))
    assert e == -3 and codes[0] == 0x7E                      # 486.4 saturates to 448
    assert fp8.tensor_exponent(0.0) == -127
    assert fp8.tensor_exponent(1e-45) == -127                # clamped


def test_zero_tensor():
    codes, e = fp8.quantize(np.zeros(64))
    assert e == -127 and not codes.any()


def test_grid_values_round_trip_exactly():
    rng = np.random.default_rng(5)
    grid = np.array([v for _, v in CODES if v >= 0])
    for j in (-6, 0, 5):
        vals = np.concatenate([[448.0], rng.choice(grid, 500)]) * 2.0 ** j * rng.choice([-1, 1], 501)
        codes, e = fp8.quantize(vals)
        assert e == j
        assert np.array_equal(fp8.dequantize(codes, e), vals)


def test_round_to_nearest_error_bound():
    rng = np.random.default_rng(7)
    v = rng.standard_normal(20000) * 3
    codes, e = fp8.quantize(v)
    d = fp8.dequantize(codes, e)
    # half an E4M3 quantum: 2^-4 relative for normals, 2^(e-10) absolute for subnormals;
    # the tensor maximum is at most 2^(e+9), so no value saturates by more than its rounding
    bound = np.maximum(2.0 ** -4 * np.abs(v), 2.0 ** (e - 10)) * (1 + 1e-12)
    sat = np.abs(v) * 2.0 ** -e > 448
    assert np.all((np.abs(d - v) <= bound) | sat)
    assert np.all(np.abs(d[sat]) == 448 * 2.0 ** e)


def test_moe_fp8_mode_exact_on_grid_inputs():
    """Every expert operand whose values lie on its per-tensor grid (max 448 * 2^-j
    in each tensor) is quantised without error, so the gate-up output of the fp8
    mode equals the exact one; the rest of the path differs from the exact MLP
    by no more than FP8 rounding."""
    rng = np.random.default_rng(11)
    T, H, I, E, k = 48, 32, 32, 3, 2
    grid = np.array([v for _, v in CODES if v >= 0])
    x = rng.choice(grid, (T, H)) * rng.choice([-1, 1], (T, H)) / 64
    x[:, 0] = 448.0 / 64                                     # every row holds its group's maximum
    wgu = rng.choice(grid, (E, 2 * I, H)) * rng.choice([-1, 1], (E, 2 * I, H)) / 4096
    wgu[:, 0, 0] = 448.0 / 4096
    wd = rng.standard_normal((E, H, I)) * 0.05
    logits = rng.standard_normal((T, E))
    ids, probs = moe.route_topk(logits, k)
    exact = moe.mlp_fwd(x, ids, probs, wgu, wd, quant=False)
    f8 = moe.mlp_fwd(x, ids, probs, wgu, wd, quant="fp8")
    assert np.array_equal(f8["gu"], exact["gu"])
    rel = np.linalg.norm(f8["y"] - exact["y"]) / np.linalg.norm(exact["y"])
    assert 0 < rel < 0.08


def test_moe_fp8_scales_each_expert_group_separately():
    """Expert 0's tokens carry values ~1e-5, expert 1's ~1: with one scale per
    expert group each group's gate-up output stays within FP8 rounding of the
    exact one (a single scale over all rows would push the small group into
    E4M3's subnormal range and fail the bound)."""
    rng = np.random.default_rng(13)
    T, H, I, E, k = 64, 64, 32, 2, 1
    x = rng.standard_normal((T, H))
    x[:32] *= 1e-5
    logits = np.zeros((T, E))
    logits[:32, 0] = 1.0
    logits[32:, 1] = 1.0
    ids, probs = moe.route_topk(logits, k)
    wgu = rng.standard_normal((E, 2 * I, H)) * 0.1
    wd = rng.standard_normal((E, H, I)) * 0.1
    exact = moe.mlp_fwd(x, ids, probs, wgu, wd, quant=False)
    f8 = moe.mlp_fwd(x, ids, probs, wgu, wd, quant="fp8")
    off = exact["perm"]["offsets"]
    for e in range(E):
        a, b = off[e], off[e + 1]
        r = np.linalg.norm(f8["gu"][a:b] - exact["gu"][a:b]) / np.linalg.norm(exact["gu"][a:b])
        assert r < 0.05, (e, r)
