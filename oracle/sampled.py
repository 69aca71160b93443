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
    for every expert the tokens use."""
    H = x.shape[1]
    n = len(tokens)
    I = next(iter(weights.values()))["wg"].shape[0] // 2
    y = np.zeros((n, H))
    dx = np.zeros((n, H))
    dprobs = np.zeros((n, k))
    gu_rows = np.zeros((n, k, 2 * I))
    rows = np.zeros((n, k), dtype=np.int64)
    for a, t in enumerate(tokens):
        xq = moe._fq(np.asarray(x[t:t + 1], dtype=np.float64), quant)
        dyq = moe._fq(np.asarray(dy[t:t + 1], dtype=np.float64), quant)
        for j in range(k):
            r = int(row_of_src[t * k + j])
            e = int(expert_of_row[r])
            p = np.array([float(probs[t, j])])
            gu, h, yr = moe.expert_forward_rows(xq, p, weights[e], quant)
            _, _, dp, dxr = moe.expert_backward_rows(dyq, gu, p, weights[e], quant)
            y[a] += yr[0]
            dx[a] += dxr[0]
            dprobs[a, j] = dp[0]
            gu_rows[a, j] = gu[0]
            rows[a, j] = r
    return {"y": y, "dx": dx, "dprobs": dprobs, "gu": gu_rows, "rows": rows}


def dw_down_columns(x_perm_e, dy_perm_e, p_e, w_gate_up_e, cols, quant=True):
    """dW_down[e][:, cols] = colMX(dY_e)^T colMX(h_e[:, cols]); h's columns need
    only the gate rows ``cols`` and the up rows ``I + cols`` of the weight."""
    cols = np.asarray(cols, dtype=np.int64)
    I = w_gate_up_e.shape[0] // 2
    n = cols.size
    wg = moe._fq(np.asarray(w_gate_up_e[np.concatenate([cols, I + cols])], dtype=np.float64), quant)
    gu = moe._fq(np.asarray(x_perm_e, dtype=np.float64), quant) @ wg.T
    h = moe.scaled_swiglu(gu[:, :n], gu[:, n:], np.asarray(p_e, dtype=np.float64)[:, None])
    return moe._fqc(np.asarray(dy_perm_e, dtype=np.float64), quant).T @ moe._fqc(h, quant)


def dw_gate_up_rows(x_perm_e, dy_perm_e, p_e, w_gate_up_e, w_down_e, rows_n, quant=True):
    """dW_gate_up[e][rows_n, :] = colMX(dGU_e[:, rows_n])^T colMX(X_e).  Column n
    of dGU (gate part n < I, up part n >= I, j = n mod I) needs g, u of column j
    and dH[:, j] = MX(dY_e) . MX-along-H(W_down[:, j])."""
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
    return moe._fqc(dgu_cols, quant).T @ moe._fqc(np.asarray(x_perm_e, dtype=np.float64), quant)
