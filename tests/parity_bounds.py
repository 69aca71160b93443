"""Per-element error bounds for the GPU-vs-oracle parity tests, derived from
the arithmetic of the two sides rather than measured.

The stated tolerance is "at most 2e-2 of the output RMS" for y and the
gradients.  Read strictly per element it is below the storage error of a bf16
output (half a bf16 unit at |y| ~ 1 exceeds 2e-2 of y's RMS on the mid-size
workload), and below the effect of the re-quantisation of intermediates the
GPU computes from other (but equally valid) roundings than the fp64 oracle.
So each tensor is checked two ways:

  1. relative RMS error ||a - r||_2 <= 2e-2 ||r||_2 (the stated tolerance);
  2. per element, |a - r| <= 2e-2 RMS(r) + S + Z * sigma, where
     S     = the bf16 storage of the output and of the rows it is summed
             from: half a bf16 unit is at most 2^-8 |v|, so
             S = 2^-8 (|r| + sum_j |R_j|) (R_j: the k rows of a combine);
     sigma = the spread of the re-quantisation flips of the GEMM operand the
             GPU re-quantises (h in the forward, dGU in the backward).

The flip model.  An operand value v that the GPU holds with a relative
perturbation |dv| <= delta |v| against the oracle's fp64 value is quantised
to a different E4M3 code only if v lies within delta |v| of a rounding
midpoint.  Midpoints are one grid step u(v) apart and u(v) >= 2^-4 |v| for
normal E4M3 codes, so (v spread evenly within its grid cell) the chance of a
flip is p <= 2 delta |v| / u(v) <= 32 delta.  A flip moves the dequantised
value by one step u.  For an output C = sum_n A_n B_n (n over a contraction
of length K) whose A is re-quantised, the flips add independent terms
+-u_n B_n.  The expected number of flips per output is lambda = p K, and:
  * lambda >= 50: their sum is close to normal, with
        sigma^2 <= p * sum_n u_n^2 B_n^2,
    computed from the oracle's own operands and grid steps; the term is
    Z * sigma with Z = 6 (a normal tail of 2e-9 per element);
  * lambda < 50 (rare flips, e.g. of h, whose delta is tiny): at most
    n(lambda) flips happen, n the count a Poisson(lambda) variable (whose
    tail bounds the binomial's) exceeds with chance below 1e-10, and
    each moves C by at most max_n u_n * max_n |B_n|; the term is their
    product.  (One flip of h moves a dW_down element by ~3 % of its RMS: a
    normal 6 sigma with p ~ 3e-5 would understate that.)

delta per re-quantised tensor:
  h   : the GPU computes h = p SiLU(g) u in fp32 from fp32 accumulators; a
        few fp32 roundings and the fast exponential, delta_h = 2^-20.
  dGU : computed from g, u kept in bf16 for the backward and dH parked in
        bf16, each rounded by at most 2^-9 relative, plus the sensitivity of
        the SiLU derivative to g: delta_dGU = 4 * 2^-9.
dprobs (fp32 outputs) are sums of dH * SiLU(g) * u terms whose factors carry
the same bf16 roundings: sigma = delta_dGU * sqrt(sum_i term_i^2).

Only the oracle's values enter a bound; nothing is taken from the GPU run.
"""
from __future__ import annotations

import json
import os

import numpy as np

from oracle import moe, mx

Z = 6.0
FRAC = 2e-2
BF16_HALF_UNIT = 2.0 ** -8
DELTA_H = 2.0 ** -20
DELTA_DGU = 4 * 2.0 ** -9


def flip_prob(delta: float) -> float:
    return min(1.0, 32.0 * delta)


def mx_steps(v: np.ndarray) -> np.ndarray:
    """Grid step of the oracle's MX quantisation at every element of v
    (blocks of 32 along the last axis): 2^e times the E4M3 spacing at the
    scaled value, 2^(e - 9) in the subnormal range and at zero."""
    v = np.asarray(v, dtype=np.float64)
    K = v.shape[-1]
    b = np.abs(v.reshape(v.shape[:-1] + (K // 32, 32)))
    e = mx.block_scale_exponent(b.max(axis=-1))[..., None]
    s = b * np.ldexp(1.0, -e)
    fl = np.where(s > 0, mx.floor_log2(np.where(s > 0, s, 1.0)), mx.E4M3_EMIN)
    fl = np.maximum(fl, mx.E4M3_EMIN)
    return np.ldexp(1.0, fl - mx.E4M3_MBITS + e).reshape(v.shape)


def mx_steps_group_columns(a: np.ndarray) -> np.ndarray:
    """Grid steps of the token-column-wise quantisation of one expert group
    a [m, C] (blocks of 32 tokens from the group's first row), as [m, C]."""
    m, C = a.shape
    mpad = -(-m // 32) * 32
    t = np.zeros((C, mpad))
    t[:, :m] = a.T
    return mx_steps(t)[:, :m].T


def flip_sigma2(u: np.ndarray, b: np.ndarray, delta: float) -> np.ndarray:
    """sigma^2 of C = A B^T (A [m, K] re-quantised with steps u, B [N, K])."""
    return flip_prob(delta) * ((u * u) @ (b * b).T)


LAMBDA_NORMAL = 50.0
TAIL = 1e-10


def rare_flips(lam: float) -> int:
    """Smallest n with P(Poisson(lam) > n) <= 1e-10: more than n flips in one
    output has a negligible chance."""
    if lam <= 0:
        return 0
    term = np.exp(-lam)            # P(N = 0)
    cdf = term
    n = 0
    while 1.0 - cdf > TAIL:
        n += 1
        term *= lam / n
        cdf += term
    return n


def flip_term(var: np.ndarray, m_outer: np.ndarray, lam: float) -> np.ndarray:
    """Per-element flip allowance: Z * sqrt(var) when lam >= 50 flips are
    expected, else n(lam) single-flip maxima (see the module docstring)."""
    if lam >= LAMBDA_NORMAL:
        return Z * np.sqrt(var)
    return rare_flips(lam) * m_outer


def storage(r: np.ndarray, rows_abs_sum: np.ndarray | None = None) -> np.ndarray:
    s = np.abs(r)
    if rows_abs_sum is not None:
        s = s + rows_abs_sum
    return BF16_HALF_UNIT * s


def bound(r: np.ndarray, extra: np.ndarray, frac: float = FRAC) -> np.ndarray:
    rms = float(np.sqrt(np.mean(np.asarray(r, dtype=np.float64) ** 2)))
    return frac * rms + extra


def check(a, r, bnd, name: str, record: dict | None = None, frac: float = FRAC) -> dict:
    """Relative RMS error <= frac (2e-2) and |a - r| <= bnd per element.  Returns
    (and optionally records) max|a - r| / RMS(r), the relative RMS error and
    the largest fraction of the bound used."""
    a = np.asarray(a, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    bnd = np.broadcast_to(np.asarray(bnd, dtype=np.float64), r.shape)
    if r.size == 0:
        return {}
    rms = float(np.sqrt(np.mean(r * r)))
    diff = np.abs(a - r)
    rel_rms = float(np.sqrt(np.mean(diff ** 2)) / rms) if rms > 0 else float(np.sqrt(np.mean(diff ** 2)))
    used = float(np.max(diff / bnd))
    out = {"tensor": name, "max_err_over_rms": float(diff.max() / rms) if rms else 0.0, "rel_rms": rel_rms,
           "bound_used": used, "elements": int(r.size)}
    if record is not None:
        write_record(dict(record, **out))
    assert rel_rms <= frac, f"{name}: relative RMS error {rel_rms:.4g} > {frac}"
    bad = diff > bnd
    assert not bad.any(), (f"{name}: {int(bad.sum())} of {r.size} elements beyond the derived per-element bound "
                           f"(worst {used:.3g}x the bound, max|a-r|/RMS {out['max_err_over_rms']:.3g})")
    return out


def write_record(rec: dict):
    """Append one parity record (JSON line) to $MXG_PARITY_RECORD, if set."""
    path = os.environ.get("MXG_PARITY_RECORD")
    if not path:
        return
    os.makedirs(os.path.dirname(os.path.abspath(path)), exist_ok=True)
    with open(path, "a") as f:
        f.write(json.dumps(rec) + "\n")


# ----------------------------------------------------------- whole-layer bounds
#
# The two variant paths fit the same scheme:
#   bf16 (oracle with quantisation off): no flips; h and dGU are stored in
#     bf16, an error uniform within half a unit (<= 2^-8 |v|), variance
#     (2^-8 v)^2 / 3 per element, so sigma^2 = sum_n (delta v_n)^2 / 3 * B_n^2
#     with delta = 2^-8 for h and 2^-8 + 3 * 2^-9 for dGU (also computed from
#     bf16 g, u and dH); the bar is the test's 5e-3 relative RMS;
#   fp8 (oracle's per-tensor mode, which also rounds h and dGU to bf16 before
#     their quantisation): the flip model on the per-tensor E4M3 grid.  h: the
#     GPU's and the oracle's bf16 h differ (by one bf16 unit) with chance at
#     most 2 delta_h / 2^-8 = 2^-11 and such a difference flips the E4M3 code
#     with chance at most 32 * 2^-7, so p <= 2^-13.  dGU: a relative
#     perturbation of delta_dGU before and one bf16 unit (2^-8) after the
#     bf16 rounding, delta = delta_dGU + 2^-8.  The tensor's one scale moves
#     by a factor two when its largest magnitude, perturbed by delta, can
#     cross a power of two; for such a tensor every code may change, by at
#     most one step of the coarser grid: p = 1 and steps doubled.

DELTA_BF16_H = 2.0 ** -8
DELTA_BF16_DGU = 2.0 ** -8 + 3 * 2.0 ** -9
P_FP8_H = 2.0 ** -13
DELTA_FP8_DGU = DELTA_DGU + 2.0 ** -8


def fp8_steps(v: np.ndarray) -> np.ndarray:
    """Grid step of the per-tensor E4M3 quantisation (one exponent for the
    whole tensor v) at every element."""
    v = np.asarray(v, dtype=np.float64)
    if v.size == 0:
        return v.copy()
    e = int(mx.block_scale_exponent(np.max(np.abs(v))))
    s = np.abs(v) * np.ldexp(1.0, -e)
    fl = np.where(s > 0, mx.floor_log2(np.where(s > 0, s, 1.0)), mx.E4M3_EMIN)
    return np.ldexp(1.0, np.maximum(fl, mx.E4M3_EMIN) - mx.E4M3_MBITS + e)


def flip_allowance(mode: str, which: str, a: np.ndarray, b: np.ndarray, col: bool) -> np.ndarray:
    """Per-element flip (or rounding) allowance of a GEMM over the re-quantised
    (or re-rounded) operand a [m, K] against b [N, K] (col: a and b are
    [tokens, .] and the GEMM contracts the tokens, giving [a-cols, b-cols])."""
    K = a.shape[0] if col else a.shape[1]
    if mode == "bf16":
        # every element rounded: an error uniform within +-delta |v|, no flips
        delta = DELTA_BF16_H if which == "h" else DELTA_BF16_DGU
        var = (delta * a) ** 2 / 3.0
        return Z * np.sqrt(var.T @ (b * b) if col else var @ (b * b).T)
    if mode == "mxfp8":
        u = mx_steps_group_columns(a) if col else mx_steps(a)
        p = flip_prob(DELTA_H if which == "h" else DELTA_DGU)
    else:
        v = moe.bf16_round(a)
        u = fp8_steps(v)
        p = P_FP8_H if which == "h" else flip_prob(DELTA_FP8_DGU)
        delta = DELTA_H if which == "h" else DELTA_FP8_DGU
        amax = float(np.max(np.abs(v))) if v.size else 0.0
        if amax > 0 and np.floor(np.log2(amax * (1 - delta))) != np.floor(np.log2(amax * (1 + delta))):
            p, u = 1.0, 2.0 * u                       # the scale itself may differ by a factor two
    lam = p * K
    if lam >= LAMBDA_NORMAL:
        var = p * u * u
        return flip_term(var.T @ (b * b) if col else var @ (b * b).T, None, lam)
    ab = np.abs(b)
    if col:
        m_outer = np.outer(u.max(axis=0), ab.max(axis=0))
    else:
        m_outer = np.outer(u.max(axis=1), ab.max(axis=1))
    return flip_term(None, m_outer, lam)


def full_bounds(ctx: dict, g: dict | None, weights: dict, dy: np.ndarray | None = None, mode: str = "mxfp8",
                frac: float = FRAC) -> dict:
    """Per-element bounds for y (and, given the backward result g and the
    upstream gradient dy [T, H], dx, dprobs, dW_gate_up, dW_down) of a whole
    layer from the oracle's forward context and each non-empty expert's
    weights as the oracle's GEMMs use them (moe.expert_weights with the same
    quantisation mode).  mode: "mxfp8", "fp8" or "bf16" (see above); frac: the
    relative-RMS bar (also the uniform per-element term)."""
    perm, k, E = ctx["perm"], ctx["k"], ctx["E"]
    off = perm["offsets"]
    R = perm["src_of_row"].size
    T = R // k
    H = ctx["x_perm"].shape[1]
    I = ctx["I"]
    bwd = g is not None
    quantised = mode != "bf16"
    col_in = (lambda v: mx.fake_quant_group_columns(v)) if mode == "mxfp8" else \
        ((lambda v: moe._fq(v, "fp8")) if mode == "fp8" else (lambda v: np.asarray(v, dtype=np.float64)))
    f_y = np.zeros((R, H))
    if bwd:
        f_dx = np.zeros((R, H))
        dp_sig = np.zeros(R)
        f_dwgu = np.zeros((E, 2 * I, H))
        f_dwd = np.zeros((E, H, I))
    tok = perm["src_of_row"] // k
    dp_delta = DELTA_DGU if quantised else 3 * 2.0 ** -9
    for e in range(E):
        a, b = off[e], off[e + 1]
        if b == a:
            continue
        w = weights[e]
        h = ctx["h"][a:b]
        f_y[a:b] = flip_allowance(mode, "h", h, w["wd"], False)
        if not bwd:
            continue
        dgu, x_perm = g["dgu"][a:b], ctx["x_perm"][a:b]
        f_dx[a:b] = flip_allowance(mode, "dgu", dgu, w["wguT"], False)
        gu = ctx["gu"][a:b]
        _, _, terms = moe.dscaled_swiglu(g["dh"][a:b], gu[:, :I], gu[:, I:], ctx["p_perm"][a:b, None])
        dp_sig[a:b] = dp_delta * np.sqrt(np.sum(terms * terms, axis=1))
        f_dwgu[e] = flip_allowance(mode, "dgu", dgu, col_in(x_perm), True)
        dyc = col_in(np.asarray(dy, dtype=np.float64)[tok[a:b]])
        f_dwd[e] = flip_allowance(mode, "h", h, dyc, True).T
    row = perm["row_of_src"].reshape(T, k)
    y_rows_abs = sum(np.abs(ctx["y_perm"][row[:, j]]) for j in range(k))
    out = {"y": bound(ctx["y"], storage(ctx["y"], y_rows_abs) + sum(f_y[row[:, j]] for j in range(k)), frac)}
    if bwd:
        dx_rows_abs = sum(np.abs(g["dx_perm"][row[:, j]]) for j in range(k))
        out["dx"] = bound(g["dx"], storage(g["dx"], dx_rows_abs) + sum(f_dx[row[:, j]] for j in range(k)), frac)
        out["dprobs"] = bound(g["dprobs"], Z * dp_sig[row], frac)
        out["dw_gate_up"] = bound(g["dw_gate_up"], storage(g["dw_gate_up"]) + f_dwgu, frac)
        out["dw_down"] = bound(g["dw_down"], storage(g["dw_down"]) + f_dwd, frac)
    return out
