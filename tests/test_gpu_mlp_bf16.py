"""The BF16 grouped expert MLP (the like-for-like reference of the MXFP8 path)
through the C ABI against the oracle with quantisation off (the exact fp64
MLP): seeded inputs spanning several tiles, ragged group tails and an empty
expert.  The only rounding on the GPU side is bf16 storage (h, dGU, the
gate-up output kept for the backward, the outputs) and fp32 accumulation, so
the errors are far inside the 2e-2 relative-RMS bar; the test states the
tighter bound it expects (5e-3 relative RMS) and checks every element against
the bound tests/parity_bounds.py derives for bf16 storage."""
import numpy as np
import pytest
import torch

import synthetic
import parity_bounds as pb
from gpu_helpers import np_, require_gpu
from oracle import moe

pytestmark = pytest.mark.gpu

CASES = {
    "ragged": ((500, 256, 512, 5, 2), dict(seed=15, empty_experts=(3,))),
    "mid": ((4096, 1024, 2816, 8, 2), None),
}


def _inputs(name):
    shape, kw = CASES[name]
    if kw is None:
        wl = synthetic.WORKLOADS[name]
        return shape, synthetic.make_inputs(wl)
    return shape, synthetic.make_case(*shape, **kw)


@pytest.mark.parametrize("name", list(CASES))
def test_bf16_mlp_fwd_bwd_matches_exact_oracle(name):
    m = require_gpu()
    shape, inp = _inputs(name)
    T, H, I, E, k = shape
    layer = m.GroupedMLP(T, H, I, E, k, precision="bf16")
    dev = "cuda"
    ids, probs = layer.route(inp["logits"].to(dev))
    y, split = layer.forward(inp["x"].to(dev), ids, probs, inp["w_gate_up"].to(dev), inp["w_down"].to(dev))
    dx, dwgu, dwd, dprobs = layer.backward(inp["dy"].to(dev))
    torch.cuda.synchronize()
    assert layer.status() == 0

    rids, rprobs = moe.route_topk(inp["logits"].numpy(), k)
    ctx = moe.mlp_fwd(inp["x"].double().numpy(), rids, rprobs, inp["w_gate_up"].double().numpy(),
                      inp["w_down"].double().numpy(), quant=False)
    g = moe.mlp_bwd(ctx, inp["dy"].double().numpy())
    assert np.array_equal(np_(ids), rids)
    assert np.array_equal(np_(split), ctx["perm"]["split_sizes"])
    W = {e: moe.expert_weights(inp["w_gate_up"][e].double().numpy(), inp["w_down"][e].double().numpy(), quant=False)
         for e in range(E) if ctx["perm"]["split_sizes"][e] > 0}
    bnd = pb.full_bounds(ctx, g, W, inp["dy"].double().numpy(), mode="bf16", frac=5e-3)
    rec = {"test": "mlp_bf16", "workload": name, "precision": "bf16"}
    report = {}
    for key, got, ref in (("y", y, ctx["y"]), ("dx", dx, g["dx"]), ("dprobs", dprobs, g["dprobs"]),
                          ("dw_gate_up", dwgu, g["dw_gate_up"]), ("dw_down", dwd, g["dw_down"])):
        o = pb.check(np_(got), ref, bnd[key], key, rec, frac=5e-3)
        report[key] = (o["max_err_over_rms"], o["rel_rms"])
    for e in np.nonzero(ctx["perm"]["split_sizes"] == 0)[0]:
        assert not np_(dwgu)[e].any() and not np_(dwd)[e].any()
    print(name, {n: (round(a, 5), round(b, 6)) for n, (a, b) in report.items()})


def test_bf16_rejects_shapes_off_the_pair_tile():
    m = require_gpu()
    with pytest.raises(ValueError):
        m.GroupedMLP(256, 128, 256, 4, 2, precision="bf16")     # H not a multiple of 256
