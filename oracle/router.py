"""MoE router front end, forward and backward — CPU oracle (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may use
this module.  It shares no code with the CUDA path.  fp64 throughout.

What it follows ([Grouped] = "BioNeMo Uses Grouped Kernels and MXFP8"):
  router    each token's hidden state goes through a router that picks two of
            eight experts, and the experts' outputs are summed with the
            router's weights: [Grouped] Fig. 1.  Reading (the page does not
            spell the router out): one linear layer H -> E without bias,
            logits = x W_r^T, followed by the top-k route of moe.route_topk
            (k largest logits, ties to the lower id, softmax over the chosen).
  backward  the choice of experts is piecewise constant, so no gradient flows
            through it; the probabilities are a softmax over the k chosen
            logits, so for token t with chosen experts e_1..e_k
                dlogit[t, e_j] = p_j * (dp_j - sum_i p_i dp_i)
            and 0 for experts not chosen; then
                dx_router = dlogits W_r,    dW_r = dlogits^T x.
"""
from __future__ import annotations

import numpy as np

from . import moe


def router_logits(x, w_router):
    """logits[t, e] = <x[t], W_r[e]> in fp64."""
    return np.asarray(x, dtype=np.float64) @ np.asarray(w_router, dtype=np.float64).T


def router_fwd(x, w_router, k: int):
    """Logits, then the top-k route on them."""
    logits = router_logits(x, w_router)
    ids, probs = moe.route_topk(logits, k)
    return logits, ids, probs


def router_dlogits(ids, probs, dprobs, E: int):
    """Gradient of the loss with respect to the full logits [T, E]."""
    ids = np.asarray(ids, dtype=np.int64)
    p = np.asarray(probs, dtype=np.float64)
    dp = np.asarray(dprobs, dtype=np.float64)
    T, k = ids.shape
    inner = (p * dp).sum(axis=1, keepdims=True)
    dsel = p * (dp - inner)                       # gradient of the chosen logits
    dl = np.zeros((T, E), dtype=np.float64)
    np.put_along_axis(dl, ids, dsel, axis=1)
    return dl


def router_bwd(x, w_router, ids, probs, dprobs) -> dict:
    """dlogits [T, E], dx_router [T, H] (to be added to the MLP's dx) and dW_r [E, H]."""
    w = np.asarray(w_router, dtype=np.float64)
    dl = router_dlogits(ids, probs, dprobs, w.shape[0])
    return {"dlogits": dl, "dx": dl @ w, "dw_router": dl.T @ np.asarray(x, dtype=np.float64)}
