"""Grouped MoE expert MLP, forward and backward — CPU oracle (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may use
this module.  It shares no code with the CUDA path and never takes an input
from it.  All floating point is fp64; every GEMM operand is MXFP8 (E4M3 codes,
E8M0 scale per 32 values along that GEMM's contraction axis) and dequantised
exactly before an fp64 matmul.

What it follows (page titles abbreviated: [Grouped] = "BioNeMo Uses Grouped
Kernels and MXFP8" (toolai.io); [Overhead] = "How BioNeMo cuts overhead in
biological AI training" (roboticlifestyle.com)):
  route     top-2-of-8 router, outputs combined as a weighted sum:
            [Grouped] Fig. 1.  Probabilities are renormalised over the chosen
            experts (softmax over the chosen logits).
  permute   tokens gathered per expert, one count per expert (split_sizes):
            [Grouped] "Grouping fragmented expert workloads"; [Overhead]
            "Grouping the expert work".  Order inside a group is not given;
            reading: stable in the flat index t*k + j.
  gate-up   GroupedLinear in_features=hidden, out_features=2*intermediate,
            bias=False, one weight per expert: [Grouped] "Grouping fragmented
            expert workloads".  Reading: the first I output columns are the
            gate, the last I the up projection.
  ScaledSwiGLU  h = p * SiLU(g) * u, the routing probability applied once,
            inside the activation: [Grouped] "Fusing precision conversion and
            expert computation"; [Overhead] "Why fused operations matter".
            The combine is then a plain sum of the already-weighted rows.
  down      second GroupedLinear intermediate -> hidden on re-quantised h:
            [Grouped] Fig. 4 ("Quantize", fused block, "Gate Down").
  backward  MXFP8 in forward and backward ([Grouped] "Fusing precision
            conversion and expert computation"); straight-through estimator
            (quantisation is identity for the gradient); every backward GEMM
            operand is MX-quantised along that GEMM's contraction axis; weight
            gradients contract over tokens, so their operands are quantised
            column-wise in blocks of 32 tokens that start at each expert's first
            row (short last block zero-padded).  E4M3 is used for gradients too.

``quant=False`` replaces every quantiser with the identity; the backward is then
the exact gradient of the forward (used by the finite-difference pin).
``quant="fp8"`` replaces every MX quantiser with per-tensor FP8 (oracle/fp8.py):
one scale per expert operand — the expert's weight matrix, and the expert's
rows of x, h, dy and dGU — the same scale in either orientation.  Reading for
that mode: a per-tensor scale needs the whole tensor before any element is
quantised, so h and dGU exist as bf16 tensors between the GEMM that produces
them and their quantisation (as in an unfused FP8 MLP, whose GEMM and
activation outputs are bf16); the oracle rounds them to bf16 there.
"""
from __future__ import annotations

import numpy as np

from . import fp8, mx

PAD = 128   # expert groups start on a multiple of 128 rows in the padded layout


def _fq(v, quant):
    if quant == "fp8":
        return fp8.fake_quant(v)
    return mx.fake_quant(v) if quant else np.asarray(v, dtype=np.float64)


def _fqc(a, quant):
    if quant == "fp8":                  # per-tensor: orientation does not matter
        return fp8.fake_quant(a)
    return mx.fake_quant_group_columns(a) if quant else np.asarray(a, dtype=np.float64)


def _materialised(v, quant):
    """An activation or activation gradient as it is stored before a per-tensor
    FP8 quantisation (bf16); unchanged otherwise."""
    return bf16_round(v) if quant == "fp8" else v


def _fq_groups(v, off, quant):
    """Row-wise quantisation of the permuted activations: MX blocks lie inside a
    row, so the whole matrix is quantised at once; per-tensor FP8 takes one
    tensor per expert group of rows."""
    if quant != "fp8":
        return _fq(v, quant)
    out = np.zeros(v.shape, dtype=np.float64)
    for e in range(len(off) - 1):
        if off[e + 1] > off[e]:
            out[off[e]:off[e + 1]] = fp8.fake_quant(v[off[e]:off[e + 1]])
    return out


def silu(g):
    return g / (1.0 + np.exp(-g))


def sigmoid(g):
    return 1.0 / (1.0 + np.exp(-g))


# ---------------------------------------------------------------- routing ----

def route_topk(logits: np.ndarray, k: int):
    """ids[t, :] = the k largest logits in descending order, ties to the lower
    expert id; probs = softmax over the chosen logits (fp64)."""
    l = np.asarray(logits, dtype=np.float64)
    T, E = l.shape
    work = l.copy()
    ids = np.empty((T, k), dtype=np.int32)
    rows = np.arange(T)
    for j in range(k):
        a = np.argmax(work, axis=1)        # first maximum = lowest id among ties
        ids[:, j] = a
        work[rows, a] = -np.inf
    sel = np.take_along_axis(l, ids.astype(np.int64), axis=1)
    w = np.exp(sel - sel[:, :1])
    probs = w / w.sum(axis=1, keepdims=True)
    return ids, probs


def permute(ids: np.ndarray, E: int, pad: int = PAD) -> dict:
    """Counting sort of flat index f = t*k + j by expert id, stable in f.

    Returns split_sizes[E], offsets[E+1] (exclusive scan), padded_offsets[E+1]
    (each group rounded up to a multiple of ``pad`` rows: a layout of the
    grouped kernels, not part of the method), src_of_row[R] (flat index feeding
    permuted row r) and row_of_src[R] (its inverse).
    """
    flat = np.asarray(ids, dtype=np.int64).reshape(-1)
    R = flat.size
    split = np.zeros(E, dtype=np.int64)
    for f in range(R):                     # histogram
        split[flat[f]] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    padded = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):                     # exclusive scans
        offsets[e + 1] = offsets[e] + split[e]
        padded[e + 1] = padded[e] + (split[e] + pad - 1) // pad * pad
    cursor = offsets[:E].copy()
    src_of_row = np.empty(R, dtype=np.int64)
    row_of_src = np.empty(R, dtype=np.int64)
    for f in range(R):                     # stable scatter
        r = cursor[flat[f]]
        cursor[flat[f]] += 1
        src_of_row[r] = f
        row_of_src[f] = r
    return {"split_sizes": split, "offsets": offsets, "padded_offsets": padded,
            "src_of_row": src_of_row, "row_of_src": row_of_src}


# ------------------------------------------------------ per-expert steps ----

def scaled_swiglu(g, u, p):
    """ScaledSwiGLU: h = p * SiLU(g) * u (p broadcast over columns)."""
    return p * silu(g) * u


def dscaled_swiglu(dh, g, u, p):
    """Gradients of h = p SiLU(g) u: with s = sigmoid(g),
    dg = dh p u s (1 + g (1 - s)), du = dh p g s, and the per-element terms of
    d(prob) = sum_i dh g s u."""
    s = sigmoid(g)
    sl = g * s
    dg = dh * p * u * s * (1.0 + g * (1.0 - s))
    du = dh * p * sl
    return dg, du, dh * sl * u


def expert_weights(w_gate_up_e, w_down_e, quant: bool = True, backward: bool = True) -> dict:
    """One expert's weights, fake-quantised along each GEMM's contraction axis:
    wg [2I,H] along H (gate-up), wd [H,I] along I (down), and for the backward
    wdT [I,H] along H (dgrad-down) and wguT [H,2I] along 2I (dgrad-gate-up)."""
    wgu = np.asarray(w_gate_up_e, dtype=np.float64)
    wd = np.asarray(w_down_e, dtype=np.float64)
    out = {"wg": _fq(wgu, quant), "wd": _fq(wd, quant)}
    if backward:
        out["wdT"] = _fq(wd.T, quant)
        out["wguT"] = _fq(wgu.T, quant)
    return out


def expert_forward_rows(xq_rows, p_rows, w: dict, quant: bool = True):
    """Rows of one expert: GU = Xq Wg^T; h = ScaledSwiGLU(g, u, p); Y = MX(h) Wd^T."""
    gu = xq_rows @ w["wg"].T
    I = gu.shape[1] // 2
    h = scaled_swiglu(gu[:, :I], gu[:, I:], p_rows[:, None])
    y = _fq(_materialised(h, quant), quant) @ w["wd"].T
    return gu, h, y


def expert_backward_rows(dyq_rows, gu, p_rows, w: dict, quant: bool = True):
    """Activation gradients for rows of one expert: dH = dYq WdT^T; dGU from
    dScaledSwiGLU; dX = MX(dGU) WguT^T; per-row d(prob)."""
    I = gu.shape[1] // 2
    dh = dyq_rows @ w["wdT"].T
    dg, du, dpt = dscaled_swiglu(dh, gu[:, :I], gu[:, I:], p_rows[:, None])
    dgu = np.concatenate([dg, du], axis=1)
    dx = _fq(_materialised(dgu, quant), quant) @ w["wguT"].T
    return dh, dgu, dpt.sum(axis=1), dx


def expert_weight_grads(dy_perm_e, h_e, dgu_e, x_perm_e, quant: bool = True):
    """dW_down = colMX(dY)^T colMX(h) and dW_gate_up = colMX(dGU)^T colMX(X) over
    the expert's tokens (column-wise blocks of 32 tokens from its first row)."""
    dw_d = _fqc(dy_perm_e, quant).T @ _fqc(_materialised(h_e, quant), quant)
    dw_gu = _fqc(_materialised(dgu_e, quant), quant).T @ _fqc(x_perm_e, quant)
    return dw_d, dw_gu


# ---------------------------------------------------------------- forward ----

def mlp_fwd(x, ids, probs, w_gate_up, w_down, quant: bool | str = True) -> dict:
    """Forward of the grouped expert MLP.  Shapes: x [T,H], ids/probs [T,k],
    w_gate_up [E,2I,H], w_down [E,H,I] (any float dtype; computed in fp64).
    Returns y [T,H] and the intermediates the backward and the tests need."""
    x = np.asarray(x, dtype=np.float64)
    T, H = x.shape
    k = ids.shape[1]
    E, N2, H2 = w_gate_up.shape
    assert H2 == H and N2 % 2 == 0
    I = N2 // 2
    perm = permute(ids, E)
    src = perm["src_of_row"]
    tok = src // k
    x_perm = x[tok]
    p_perm = np.asarray(probs, dtype=np.float64).reshape(-1)[src]
    off = perm["offsets"]
    xq = _fq_groups(x_perm, off, quant)              # row-wise along H
    R = src.size
    gu = np.empty((R, 2 * I))
    h = np.empty((R, I))
    y_perm = np.empty((R, H))
    for e in range(E):
        a, b = off[e], off[e + 1]
        if b == a:
            continue
        w = expert_weights(w_gate_up[e], w_down[e], quant, backward=False)
        gu[a:b], h[a:b], y_perm[a:b] = expert_forward_rows(xq[a:b], p_perm[a:b], w, quant)
    y = np.zeros((T, H))
    row = perm["row_of_src"].reshape(T, k)
    for j in range(k):
        y += y_perm[row[:, j]]
    return {"y": y, "gu": gu, "h": h, "y_perm": y_perm, "x_perm": x_perm,
            "p_perm": p_perm, "perm": perm, "I": I, "k": k, "E": E, "quant": quant,
            "w_gate_up": w_gate_up, "w_down": w_down}


# --------------------------------------------------------------- backward ----

def mlp_bwd(ctx: dict, dy) -> dict:
    """Backward (straight-through estimator) of mlp_fwd for upstream gradient
    dy [T,H].  Returns dx [T,H], dw_gate_up [E,2I,H], dw_down [E,H,I],
    dprobs [T,k] and per-row intermediates (dgu, dh)."""
    quant = ctx["quant"]
    perm, I, k, E = ctx["perm"], ctx["I"], ctx["k"], ctx["E"]
    dy = np.asarray(dy, dtype=np.float64)
    T, H = dy.shape
    src = perm["src_of_row"]
    tok = src // k
    dy_perm = dy[tok]
    dyq = _fq_groups(dy_perm, perm["offsets"], quant)   # row-wise along H
    gu, h, x_perm, p_perm = ctx["gu"], ctx["h"], ctx["x_perm"], ctx["p_perm"]
    R = src.size
    dgu = np.empty((R, 2 * I))
    dh = np.empty((R, I))
    dp = np.empty(R)
    dx_perm = np.empty((R, H))
    dw_gu = np.zeros((E, 2 * I, H))
    dw_d = np.zeros((E, H, I))
    off = perm["offsets"]
    for e in range(E):
        a, b = off[e], off[e + 1]
        if b == a:
            continue                                  # empty expert: dW stays 0
        w = expert_weights(ctx["w_gate_up"][e], ctx["w_down"][e], quant)
        dh[a:b], dgu[a:b], dp[a:b], dx_perm[a:b] = expert_backward_rows(dyq[a:b], gu[a:b], p_perm[a:b], w, quant)
        dw_d[e], dw_gu[e] = expert_weight_grads(dy_perm[a:b], h[a:b], dgu[a:b], x_perm[a:b], quant)
    row = perm["row_of_src"].reshape(T, k)
    dx = np.zeros((T, H))
    for j in range(k):
        dx += dx_perm[row[:, j]]
    dprobs = dp[row]
    return {"dx": dx, "dw_gate_up": dw_gu, "dw_down": dw_d, "dprobs": dprobs,
            "dgu": dgu, "dh": dh, "dp": dp, "dx_perm": dx_perm}


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round fp64 values to bf16 (via fp32, ties to even), returned as fp64.
    Only used to present oracle outputs in the precision the outputs are stored
    in, never for a bit-exact check (the two-step rounding can differ from a
    direct fp64 -> bf16 rounding in rare ties)."""
    f = np.asarray(a, dtype=np.float32)      # fp64 -> fp32 (RNE)
    bits = f.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    r = ((bits + 0x7FFF + lsb) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)
