"""The weight cache (the MXFP8 weights quantised once, reused by later forward
and backward calls) and fp32 gradient accumulation (main_grad) through the C
ABI.

- A forward/backward that reads the cache runs the same kernels on the same
  bytes as one that quantises the weights itself: every output is compared bit
  for bit with the uncached run, whose parity with the oracle the MLP tests
  establish; y is also checked against the oracle here.
- main_grad: two micro-batches add their weight gradients into fp32 buffers.
  Each addition takes the fp32 GEMM accumulator, whose bf16 rounding is the dW
  of the uncached run, so (main_grad - start) differs from 2 dW by at most two
  bf16 roundings (2^-8 relative each) plus two fp32 additions; slices of
  experts without tokens stay bit-identical; against the oracle, (main_grad -
  start) / 2 meets the MLP's parity bounds for dW (tests/parity_bounds.py)."""
import numpy as np
import pytest
import torch

import synthetic
import parity_bounds as pb
from gpu_helpers import np_, require_gpu
from oracle import moe


def _weights(inp, split):
    return {e: moe.expert_weights(inp["w_gate_up"][e].double().numpy(), inp["w_down"][e].double().numpy())
            for e in range(len(split)) if split[e] > 0}

pytestmark = pytest.mark.gpu

CASES = {
    # T, H, I, E, k: weight-gradient tiles on CTA pairs and on single CTAs of both widths
    "ragged": ((300, 256, 384, 6, 2), dict(seed=5, empty_experts=(1, 4))),
    "ragged_k1": ((200, 128, 128, 3, 1), dict(seed=6)),
    "narrow": ((256, 128, 256, 4, 2), dict(seed=8, empty_experts=(2,))),
}


def _setup(m, name):
    shape, kw = CASES[name]
    inp = synthetic.make_case(*shape, **kw)
    dev = "cuda"
    t = {n: inp[n].to(dev) for n in ("logits", "x", "w_gate_up", "w_down", "dy")}
    return shape, inp, t


def _plain(m, shape, t):
    layer = m.GroupedMLP(*shape)
    ids, probs = layer.route(t["logits"])
    y, split = layer.forward(t["x"], ids, probs, t["w_gate_up"], t["w_down"])
    dx, dwgu, dwd, dprobs = layer.backward(t["dy"])
    torch.cuda.synchronize()
    assert layer.status() == 0
    return {n: v.clone() for n, v in dict(y=y, split=split, dx=dx, dwgu=dwgu, dwd=dwd, dprobs=dprobs).items()}


@pytest.mark.parametrize("name", list(CASES))
def test_cached_weights_bit_identical(name):
    m = require_gpu()
    shape, inp, t = _setup(m, name)
    ref = _plain(m, shape, t)
    layer = m.GroupedMLP(*shape)
    layer.quantize_weights(t["w_gate_up"], t["w_down"])
    ids, probs = layer.route(t["logits"])
    for _ in range(2):                                   # two micro-batches on one cache
        y, split = layer.forward(t["x"], ids, probs)
        dx, dwgu, dwd, dprobs = layer.backward(t["dy"])
    torch.cuda.synchronize()
    assert layer.status() == 0
    got = dict(y=y, split=split, dx=dx, dwgu=dwgu, dwd=dwd, dprobs=dprobs)
    for n in ref:
        assert torch.equal(got[n], ref[n]), n
    T, H, I, E, k = shape
    rids, rprobs = moe.route_topk(inp["logits"].numpy(), k)
    ctx = moe.mlp_fwd(inp["x"].double().numpy(), rids, rprobs, inp["w_gate_up"].double().numpy(),
                      inp["w_down"].double().numpy())
    bnd = pb.full_bounds(ctx, None, _weights(inp, ctx["perm"]["split_sizes"]))
    pb.check(np_(y), ctx["y"], bnd["y"], "y", {"test": "weight_cache", "workload": name, "precision": "mxfp8"})


@pytest.mark.parametrize("name", list(CASES))
def test_main_grad_accumulates_fp32(name):
    m = require_gpu()
    shape, inp, t = _setup(m, name)
    T, H, I, E, k = shape
    ref = _plain(m, shape, t)
    g = torch.Generator().manual_seed(11)
    mg0_gu = torch.randn((E, 2 * I, H), generator=g) * 1e-3
    mg0_d = torch.randn((E, H, I), generator=g) * 1e-3
    mg_gu, mg_d = mg0_gu.cuda(), mg0_d.cuda()
    layer = m.GroupedMLP(*shape)
    layer.quantize_weights(t["w_gate_up"], t["w_down"])
    ids, probs = layer.route(t["logits"])
    for _ in range(2):
        layer.forward(t["x"], ids, probs)
        dx, o_gu, o_d, dprobs = layer.backward(t["dy"], main_grad=(mg_gu, mg_d))
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert o_gu is mg_gu and o_d is mg_d
    assert torch.equal(dx, ref["dx"]) and torch.equal(dprobs, ref["dprobs"])
    split = np_(ref["split"])
    rids, rprobs = moe.route_topk(inp["logits"].numpy(), k)
    ctx = moe.mlp_fwd(inp["x"].double().numpy(), rids, rprobs, inp["w_gate_up"].double().numpy(),
                      inp["w_down"].double().numpy())
    gr = moe.mlp_bwd(ctx, inp["dy"].double().numpy())
    bnd = pb.full_bounds(ctx, gr, _weights(inp, ctx["perm"]["split_sizes"]), inp["dy"].double().numpy())
    for got, start, dw, oracle_dw, nm, key in ((mg_gu, mg0_gu, ref["dwgu"], gr["dw_gate_up"], "dW_gate_up", "dw_gate_up"),
                                               (mg_d, mg0_d, ref["dwd"], gr["dw_down"], "dW_down", "dw_down")):
        a, s0, w = np_(got).astype(np.float64), start.numpy().astype(np.float64), np_(dw)
        inc = a - s0
        bound = 2.0 ** -7 * 1.01 * np.abs(w) + 2.0 ** -22 * (np.abs(s0) + 2 * np.abs(w)) + 1e-30
        worst = float(np.max(np.abs(inc - 2 * w) / bound))
        assert worst <= 1.0, f"{nm}: main_grad increment off 2 dW by {worst:.3g}x the rounding bound"
        for e in np.nonzero(split == 0)[0]:
            assert np.array_equal(a[e], s0[e]), f"{nm}: expert {e} without tokens changed"
        pb.check(inc / 2, oracle_dw, bnd[key], nm, {"test": "main_grad", "workload": name, "precision": "mxfp8"})


def test_weight_cache_holds_the_oracles_codes():
    """The cache's four MXFP8 weight tensors, bit for bit against the MX
    quantiser oracle (the inputs are the same bf16 values): W_gate_up along H
    and along 2I (transposed), W_down along I and along H (transposed)."""
    from gpu_helpers import mma_to_canonical
    from oracle import mx
    m = require_gpu()
    H, I, E = 256, 384, 3
    inp = synthetic.make_case(64, H, I, E, 2, seed=9)
    wgu, wd = inp["w_gate_up"], inp["w_down"]
    cache = m.mxg_mlp_quantize_weights(wgu.cuda(), wd.cuda())
    torch.cuda.synchronize()
    base = cache.buffer.data_ptr()

    def view(which, rows, cols, codes):
        off = m.lib().mxg_mlp_weight_cache_view(base, H, I, E, which) - base
        n = rows * cols if codes else rows * cols // 32
        t = cache.buffer[off:off + n]
        return t.cpu().numpy().reshape(rows, cols) if codes else mma_to_canonical(t, rows, cols // 32)

    W_gu, W_d = wgu.double().numpy(), wd.double().numpy()
    for which, rows, cols, ref in ((0, E * 2 * I, H, [W_gu[e] for e in range(E)]),
                                   (2, E * H, I, [W_d[e] for e in range(E)]),
                                   (4, E * H, 2 * I, [W_gu[e].T for e in range(E)]),
                                   (6, E * I, H, [W_d[e].T for e in range(E)])):
        codes, scales = mx.quantize_blocks(np.concatenate(ref, axis=0))
        assert np.array_equal(view(which, rows, cols, True), codes), which
        assert np.array_equal(view(which + 1, rows, cols, False), scales), which + 1
