"""The oracle evaluated on samples of a full-size workload (test infrastructure only).

At the Mixtral-layer sizes the oracle cannot produce every output inside a
test.  These functions evaluate the same per-expert steps of oracle.moe on
chosen tokens and chosen weight-gradient rows/columns.  That is exact, not an
approximation, because each sampled output depends only on:
  * the routing and the permutation (computed in full — they are cheap);
  * the fake-quantised weights of the experts involved (row-wise MX is per row);
  * the fake-quantised activations of the rows involved; column-wise MX (wgrad
    operands) is per column over one expert's tokens, so a column subset of it
    equals the same columns of the full quantisation.
Only tests/ may use this module.
"""
from __future__ import annotations

import numpy as np

from . import moe


def rows_forward_backward(tokens, x, dy, probs, row_of_src, expert_of_row, k, weights: dict, quant=True):
    """For each token t in ``tokens``: y[t], dx[t], dprobs[t, :] and the gate-up
    output GU of each of its k rows.  ``weights[e]`` is moe.expert_weights(...)
    for the experts to evaluate: slots routed to an expert missing from
    ``weights`` are skipped (their contributions stay zero and ``done`` is
    False there), so a caller can evaluate the experts one at a time and add
    the results.  Also returned per slot, for error bounds: h, the Y row, dH,
    dGU and the dX row."""
    H = x.shape[1]
    n = len(tokens)
    I = next(iter(weights.values()))["wg"].shape[0] // 2
    y = np.zeros((n, H))
    dx = np.zeros((n, H))
    dprobs = np.zeros((n, k))
    gu_rows = np.zeros((n, k, 2 * I))
    rows = np.zeros((n, k), dtype=np.int64)
    done = np.zeros((n, k), dtype=bool)
    parts = {"h": np.zeros((n, k, I)), "y_rows": np.zeros((n, k, H)), "dh": np.zeros((n, k, I)),
             "dgu": np.zeros((n, k, 2 * I)), "dx_rows": np.zeros((n, k, H))}
    for a, t in enumerate(tokens):
        xq = moe._fq(np.asarray(x[t:t + 1], dtype=np.float64), quant)
        dyq = moe._fq(np.asarray(dy[t:t + 1], dtype=np.float64), quant)
        for j in range(k):
            r = int(row_of_src[t * k + j])
            e = int(expert_of_row[r])
            rows[a, j] = r
            if e not in weights:
                continue
            p = np.array([float(probs[t, j])])
            gu, h, yr = moe.expert_forward_rows(xq, p, weights[e], quant)
            dh, dgu, dp, dxr = moe.expert_backward_rows(dyq, gu, p, weights[e], quant)
            y[a] += yr[0]
            dx[a] += dxr[0]
            dprobs[a, j] = dp[0]
            gu_rows[a, j] = gu[0]
            done[a, j] = True
            parts["h"][a, j], parts["y_rows"][a, j], parts["dh"][a, j] = h[0], yr[0], dh[0]
            parts["dgu"][a, j], parts["dx_rows"][a, j] = dgu[0], dxr[0]
    return {"y": y, "dx": dx, "dprobs": dprobs, "gu": gu_rows, "rows": rows, "done": done, **parts}


def dw_down_columns(x_perm_e, dy_perm_e, p_e, w_gate_up_e, cols, quant=True, parts=False):
    """dW_down[e][:, cols] = colMX(dY_e)^T colMX(h_e[:, cols]); h's columns need
    only the gate rows ``cols`` and the up rows ``I + cols`` of the weight.
    With ``parts``, also returns h[:, cols] and colMX(dY_e) (for error bounds)."""
    cols = np.asarray(cols, dtype=np.int64)
    I = w_gate_up_e.shape[0] // 2
    n = cols.size
    wg = moe._fq(np.asarray(w_gate_up_e[np.concatenate([cols, I + cols])], dtype=np.float64), quant)
    gu = moe._fq(np.asarray(x_perm_e, dtype=np.float64), quant) @ wg.T
    h = moe.scaled_swiglu(gu[:, :n], gu[:, n:], np.asarray(p_e, dtype=np.float64)[:, None])
    dyc = moe._fqc(np.asarray(dy_perm_e, dtype=np.float64), quant)
    dw = dyc.T @ moe._fqc(h, quant)
    return (dw, {"h": h, "dyc": dyc}) if parts else dw


def dw_gate_up_rows(x_perm_e, dy_perm_e, p_e, w_gate_up_e, w_down_e, rows_n, quant=True, parts=False):
    """dW_gate_up[e][rows_n, :] = colMX(dGU_e[:, rows_n])^T colMX(X_e).  Column n
    of dGU (gate part n < I, up part n >= I, j = n mod I) needs g, u of column j
    and dH[:, j] = MX(dY_e) . MX-along-H(W_down[:, j]).  With ``parts``, also
    returns dGU[:, rows_n] and colMX(X_e) (for error bounds)."""
    rows_n = np.asarray(rows_n, dtype=np.int64)
    I = w_gate_up_e.shape[0] // 2
    j = rows_n % I
    n = j.size
    p = np.asarray(p_e, dtype=np.float64)[:, None]
    wg = moe._fq(np.asarray(w_gate_up_e[np.concatenate([j, I + j])], dtype=np.float64), quant)
    gu = moe._fq(np.asarray(x_perm_e, dtype=np.float64), quant) @ wg.T
    wdT_rows = moe._fq(np.asarray(w_down_e, dtype=np.float64)[:, j].T, quant)
    dh = moe._fq(np.asarray(dy_perm_e, dtype=np.float64), quant) @ wdT_rows.T
    dg, du, _ = moe.dscaled_swiglu(dh, gu[:, :n], gu[:, n:], p)
    dgu_cols = np.where((rows_n < I)[None, :], dg, du)
    xc = moe._fqc(np.asarray(x_perm_e, dtype=np.float64), quant)
    dw = moe._fqc(dgu_cols, quant).T @ xc
    return (dw, {"dgu": dgu_cols, "xc": xc}) if parts else dw
