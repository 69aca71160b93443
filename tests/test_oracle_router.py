"""Pins for the router oracle against facts fixed outside it: a brute-force dot
product loop, central finite differences of the routed probabilities, the
zero-sum property of a softmax gradient, and (k = E) the autograd gradient of
torch's softmax."""
import numpy as np
import torch

from oracle import moe, router


def test_logits_brute_force_integers():
    rng = np.random.default_rng(3)
    x = rng.integers(-8, 9, size=(7, 19)).astype(np.float64)
    w = rng.integers(-8, 9, size=(5, 19)).astype(np.float64)
    got = router.router_logits(x, w)
    for t in range(7):
        for e in range(5):
            assert got[t, e] == sum(x[t, h] * w[e, h] for h in range(19))


def _separated_case(T, H, E, k, seed, margin=5e-2):
    """Inputs whose k-th and (k+1)-th logits are at least `margin` apart, so
    small perturbations never change the chosen experts."""
    rng = np.random.default_rng(seed)
    w = rng.standard_normal((E, H)) * 0.3
    xs = []
    while len(xs) < T:
        x = rng.standard_normal(H)
        l = np.sort(x @ w.T)[::-1]
        gaps = -np.diff(l)
        if k < E and gaps[k - 1] < margin:
            continue
        if (gaps[:k] < 1e-6).any():
            continue
        xs.append(x)
    return np.stack(xs), w


def _loss(x, w, k, c, ids_ref):
    _, ids, probs = router.router_fwd(x, w, k)
    assert np.array_equal(ids, ids_ref)
    return float((c * probs).sum())


def test_backward_finite_differences():
    T, H, E, k = 6, 10, 8, 2
    x, w = _separated_case(T, H, E, k, 11)
    _, ids, probs = router.router_fwd(x, w, k)
    c = np.random.default_rng(12).standard_normal((T, k))      # dL/dprobs
    g = router.router_bwd(x, w, ids, probs, c)
    eps = 1e-6
    for (t, h) in [(0, 0), (2, 5), (5, 9), (3, 3)]:
        xp, xm = x.copy(), x.copy()
        xp[t, h] += eps
        xm[t, h] -= eps
        fd = (_loss(xp, w, k, c, ids) - _loss(xm, w, k, c, ids)) / (2 * eps)
        assert abs(fd - g["dx"][t, h]) <= 1e-6 * max(1.0, abs(fd))
    for (e, h) in [(int(ids[0, 0]), 1), (int(ids[4, 1]), 7), (int(ids[2, 0]), 4)]:
        wp, wm = w.copy(), w.copy()
        wp[e, h] += eps
        wm[e, h] -= eps
        fd = (_loss(x, wp, k, c, ids) - _loss(x, wm, k, c, ids)) / (2 * eps)
        assert abs(fd - g["dw_router"][e, h]) <= 1e-6 * max(1.0, abs(fd))
    # an expert nobody chose gets no weight gradient
    unused = sorted(set(range(E)) - set(ids.reshape(-1).tolist()))
    for e in unused:
        assert np.all(g["dw_router"][e] == 0.0)


def test_dlogits_rows_sum_to_zero():
    rng = np.random.default_rng(5)
    logits = rng.standard_normal((50, 64))
    ids, probs = moe.route_topk(logits, 8)
    dl = router.router_dlogits(ids, probs, rng.standard_normal((50, 8)), 64)
    assert np.allclose(dl.sum(axis=1), 0.0, atol=1e-13)
    assert (np.count_nonzero(dl, axis=1) <= 8).all()


def test_all_experts_chosen_is_softmax_autograd():
    rng = np.random.default_rng(9)
    E = 6
    logits = rng.standard_normal((20, E))
    ids, probs = moe.route_topk(logits, E)
    dprobs = rng.standard_normal((20, E))
    got = router.router_dlogits(ids, probs, dprobs, E)
    lt = torch.tensor(logits, dtype=torch.float64, requires_grad=True)
    p = torch.softmax(lt, dim=1)
    # dprobs are given in the route's order (ids); scatter them to expert order
    up = np.zeros((20, E))
    np.put_along_axis(up, ids.astype(np.int64), dprobs, axis=1)
    (p * torch.tensor(up)).sum().backward()
    assert np.allclose(got, lt.grad.numpy(), rtol=1e-12, atol=1e-14)
