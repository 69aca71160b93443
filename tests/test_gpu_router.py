"""Router front end on the GPU against the router oracle: logits (fp32 sums of
bf16 products) within their rounding bound, the route exact wherever the
oracle's logit gaps exceed that bound (and valid where they do not), and the
backward — the router's term added to dx, dW_r — from the oracle's own route."""
import numpy as np
import pytest
import torch

import synthetic
from gpu_helpers import np_, require_gpu
from oracle import moe, router

pytestmark = pytest.mark.gpu

CASES = [                       # T, H, E, k
    (256, 128, 4, 2),           # tiny layer's router
    (4096, 4096, 8, 2),         # Mixtral: top-2 of 8, H = 4096
    (8192, 2048, 64, 8),        # fine-grained: top-8 of 64
    (96, 256, 256, 32),         # widest route the ABI accepts
    (77, 384, 5, 1),            # ragged token count, odd expert count
]


def _gamma(n):
    """Rounding bound of an n-term fp32 sum of exact products: n u / (1 - n u)."""
    u = 2.0 ** -24
    return n * u / (1 - n * u)


def _inputs(T, H, E, seed):
    x = synthetic.random_bf16((T, H), seed)
    w = synthetic.random_bf16((E, H), seed + 1, std=0.02)
    return x, w


@pytest.mark.parametrize("T,H,E,k", CASES)
def test_router_fwd(T, H, E, k):
    m = require_gpu()
    x, w = _inputs(T, H, E, 100 + E)
    logits, ids, probs = m.mxg_router_fwd(x.cuda(), w.cuda(), k)
    torch.cuda.synchronize()
    X, W = x.double().numpy(), w.double().numpy()
    ref = router.router_logits(X, W)
    bound = _gamma(H) * (np.abs(X) @ np.abs(W).T) + 1e-30   # fp32 accumulation of exact bf16 products
    got = np_(logits)
    assert (np.abs(got - ref) <= bound).all(), float(np.max(np.abs(got - ref) / bound))
    rids, rprobs = moe.route_topk(ref, k)
    gids, gprobs = np_(ids).astype(np.int64), np_(probs)
    srt = -np.sort(-ref, axis=1)
    gaps = srt[:, :min(k + 1, E) - 1] - srt[:, 1:min(k + 1, E)]
    margin = 2 * bound.max(axis=1, keepdims=True)
    clear = (gaps > margin).all(axis=1)
    assert clear.mean() > 0.5
    assert np.array_equal(gids[clear], rids[clear])
    # where the oracle's logits are closer than the rounding bound, the GPU's
    # choice must still be a valid top-k: distinct experts whose logits are
    # within the margin of the oracle's order
    for t in np.nonzero(~clear)[0]:
        assert len(set(gids[t].tolist())) == k
        chosen = ref[t, gids[t]]
        assert (chosen >= srt[t, k - 1] - margin[t, 0]).all()
        assert (np.diff(chosen) <= margin[t, 0]).all()
    # probabilities: softmax over the chosen logits (the GPU's choice)
    sel = np.take_along_axis(ref, gids, axis=1)
    p = np.exp(sel - sel[:, :1])
    p /= p.sum(axis=1, keepdims=True)
    # a logit error d moves each probability by at most 2 p max|d|
    assert (np.abs(gprobs - p) <= 2 * p * bound.max(axis=1, keepdims=True) + 1e-6).all()


@pytest.mark.parametrize("T,H,E,k", CASES)
def test_router_bwd(T, H, E, k):
    m = require_gpu()
    x, w = _inputs(T, H, E, 200 + E)
    X, W = x.double().numpy(), w.double().numpy()
    _, rids, rprobs = router.router_fwd(X, W, k)            # the oracle's own route feeds both sides
    rng = np.random.default_rng(7)
    dprobs = rng.standard_normal((T, k)).astype(np.float32)
    dx0 = synthetic.random_bf16((T, H), 300 + E)
    ids_t = torch.from_numpy(rids.astype(np.int32)).cuda()
    probs_t = torch.from_numpy(rprobs.astype(np.float32)).cuda()
    dx = dx0.cuda().clone()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dw = m.mxg_router_bwd(x.cuda(), w.cuda(), ids_t, probs_t, torch.from_numpy(dprobs).cuda(), dx, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    g = router.router_bwd(X, W, rids, rprobs.astype(np.float32).astype(np.float64), dprobs.astype(np.float64))
    ref_dx = dx0.double().numpy() + g["dx"]
    got_dx = np_(dx)
    assert (np.abs(got_dx - ref_dx) <= 2.0 ** -8 * 1.01 * np.abs(ref_dx) + 1e-6).all()   # one bf16 rounding
    dl = g["dlogits"]
    bound = _gamma(T + 64) * (np.abs(dl).T @ np.abs(X)) + 1e-7 * np.abs(g["dw_router"]) + 1e-30
    got_dw = np_(dw)
    assert (np.abs(got_dw - g["dw_router"]) <= bound).all(), float(np.max(np.abs(got_dw - g["dw_router"]) / bound))
    unused = sorted(set(range(E)) - set(rids.reshape(-1).tolist()))
    for e in unused:
        assert np.all(got_dw[e] == 0.0)


def test_router_bwd_reports_bad_expert_id():
    m = require_gpu()
    T, H, E, k = 64, 256, 8, 2
    x, w = _inputs(T, H, E, 5)
    ids = torch.zeros((T, k), dtype=torch.int32)
    ids[:, 1] = 1
    ids[3, 0] = 999
    probs = torch.full((T, k), 0.5, dtype=torch.float32)
    dprobs = torch.ones((T, k), dtype=torch.float32)
    dx = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.mxg_router_bwd(x.cuda(), w.cuda(), ids.cuda(), probs.cuda(), dprobs.cuda(), dx, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 16                               # MXG_ERR_EXPERT_ID


@pytest.mark.parametrize("T,H,E,k", CASES + [(20000, 256, 16, 3)])
def test_router_fwd_permute_equals_router_then_permute(T, H, E, k):
    """The fused call (the router kernel feeds the permute's histogram) gives
    the same logits, route, split sizes, maps and padded offsets, bit for bit,
    as mxg_router_fwd followed by mxg_route_permute (k = 3: a CTA's entries
    straddle a histogram chunk)."""
    m = require_gpu()
    x, w = _inputs(T, H, E, 200 + E)
    xc, wc = x.cuda(), w.cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lo, ids, probs, pm = m.mxg_router_fwd_permute(xc, wc, k, st)
    lo2, ids2, probs2 = m.mxg_router_fwd(xc, wc, k)
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    pm2 = m.mxg_route_permute(ids2, E, st2)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(st2.item()) == 0
    assert torch.equal(lo, lo2) and torch.equal(ids, ids2) and torch.equal(probs, probs2)
    for name in pm2:
        assert torch.equal(pm[name], pm2[name]), name


@pytest.mark.parametrize("T,H,E,k", CASES + [(1000, 512, 64, 8), (300, 256, 33, 3), (500, 256, 16, 4)])
def test_router_route_equals_route_topk_on_its_logits(T, H, E, k):
    """The router's fused route (one thread per token while E k <= 64, one
    warp per token beyond) is bit-identical to mxg_route_topk (one
    warp per token) on the logits the router wrote: same ids, same
    probabilities (the softmax sums in the same order)."""
    m = require_gpu()
    x, w = _inputs(T, H, E, 400 + E)
    logits, ids, probs = m.mxg_router_fwd(x.cuda(), w.cuda(), k)
    ids2, probs2 = m.mxg_route_topk(logits, k)
    torch.cuda.synchronize()
    assert torch.equal(ids, ids2)
    assert torch.equal(probs, probs2)
