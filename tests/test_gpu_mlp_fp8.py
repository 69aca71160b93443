"""The per-tensor FP8 grouped expert MLP through the C ABI against the
oracle's fp8 mode (oracle/fp8.py: one power-of-two scale per expert tensor,
2^-(floor(log2 amax) - 8), codes nearest-even of the exactly scaled values).

- amax of x (per expert group), W_gate_up and W_down (per expert): bit-exact
  (a maximum of bf16 values);
- x's codes (transposed, padded layout, one scale per expert group): bit-exact
  (scaling by a power of two is exact on both sides);
- amax of h: within 1e-2 relative (h comes out of an fp32 GEMM on one side and
  fp64 on the other);
- y, dx, dW_gate_up, dW_down, dprobs: relative RMS error within 2e-2 and
  every element within the bound tests/parity_bounds.py derives for the
  per-tensor FP8 path;
- experts without tokens: dW exactly 0."""
import ctypes

import numpy as np
import pytest
import torch

import synthetic
import parity_bounds as pb
from gpu_helpers import np_, require_gpu
from oracle import fp8, moe

pytestmark = pytest.mark.gpu

CASES = {
    "ragged": ((500, 256, 512, 5, 2), dict(seed=15, empty_experts=(3,))),
    "mid": ((4096, 1024, 2816, 8, 2), None),
}


def _inputs(name):
    shape, kw = CASES[name]
    if kw is None:
        return shape, synthetic.make_inputs(synthetic.WORKLOADS[name])
    return shape, synthetic.make_case(*shape, **kw)


def _view(m, layer, which, nbytes, dtype):
    ptr = m.lib().mxg_mlp_fp8_saved_view(ctypes.c_void_p(layer.saved.data_ptr()), layer.T, layer.H, layer.I,
                                         layer.E, layer.k, which)
    off = ptr - layer.saved.data_ptr()
    return layer.saved[off:off + nbytes].view(dtype)


@pytest.mark.parametrize("name", list(CASES))
def test_fp8_mlp_matches_oracle(name):
    m = require_gpu()
    shape, inp = _inputs(name)
    T, H, I, E, k = shape
    layer = m.GroupedMLP(T, H, I, E, k, precision="fp8")
    dev = "cuda"
    ids, probs = layer.route(inp["logits"].to(dev))
    y, split = layer.forward(inp["x"].to(dev), ids, probs, inp["w_gate_up"].to(dev), inp["w_down"].to(dev))
    torch.cuda.synchronize()
    mcap = m.mxg_mlp_row_capacity(T, k, E)
    xqT = np_(_view(m, layer, 0, H * mcap, torch.uint8)).reshape(H, mcap)
    amax = {n: np_(_view(m, layer, w, 4 * E, torch.float32)) for n, w in (("x", 1), ("wgu", 2), ("wd", 3), ("h", 4))}
    poff = np_(_view(m, layer, 5, 4 * (E + 1), torch.int32))
    dx, dwgu, dwd, dprobs = layer.backward(inp["dy"].to(dev))
    torch.cuda.synchronize()
    assert layer.status() == 0

    rids, rprobs = moe.route_topk(inp["logits"].numpy(), k)
    X = inp["x"].float().numpy()
    perm = moe.permute(rids, E, pad=m.mxg_mlp_group_align())
    assert np.array_equal(poff, perm["padded_offsets"])
    off = perm["offsets"]
    x_perm = X[perm["src_of_row"] // k]
    for e in range(E):
        a, b = off[e], off[e + 1]
        ref_amax = np.max(np.abs(x_perm[a:b])) if b > a else 0.0
        assert amax["x"][e] == np.float32(ref_amax), (e, amax["x"][e], ref_amax)
        assert amax["wgu"][e] == np.max(np.abs(inp["w_gate_up"][e].float().numpy()))
        assert amax["wd"][e] == np.max(np.abs(inp["w_down"][e].float().numpy()))
        if b > a:
            codes, _ = fp8.quantize(x_perm[a:b])
            p0 = poff[e]
            assert np.array_equal(xqT[:, p0:p0 + (b - a)], codes.T), f"x codes, expert {e}"
            assert not xqT[:, p0 + (b - a):poff[e + 1]].any()       # padding rows are zero codes

    ctx = moe.mlp_fwd(inp["x"].double().numpy(), rids, rprobs, inp["w_gate_up"].double().numpy(),
                      inp["w_down"].double().numpy(), quant="fp8")
    g = moe.mlp_bwd(ctx, inp["dy"].double().numpy())
    for e in range(E):
        a, b = off[e], off[e + 1]
        if b > a:
            ref = np.max(np.abs(ctx["h"][a:b]))
            assert abs(amax["h"][e] - ref) <= 1e-2 * ref, (e, amax["h"][e], ref)
    assert np.array_equal(np_(split), perm["split_sizes"])
    W = {e: moe.expert_weights(inp["w_gate_up"][e].double().numpy(), inp["w_down"][e].double().numpy(), quant="fp8")
         for e in range(E) if perm["split_sizes"][e] > 0}
    bnd = pb.full_bounds(ctx, g, W, inp["dy"].double().numpy(), mode="fp8")
    rec = {"test": "mlp_fp8", "workload": name, "precision": "fp8"}
    report = {}
    for key, got, ref in (("y", y, ctx["y"]), ("dx", dx, g["dx"]), ("dprobs", dprobs, g["dprobs"]),
                          ("dw_gate_up", dwgu, g["dw_gate_up"]), ("dw_down", dwd, g["dw_down"])):
        o = pb.check(np_(got), ref, bnd[key], key, rec)
        report[key] = (o["max_err_over_rms"], o["rel_rms"])
    for e in np.nonzero(perm["split_sizes"] == 0)[0]:
        assert not np_(dwgu)[e].any() and not np_(dwd)[e].any()
    print(name, {n: (round(a, 5), round(b, 6)) for n, (a, b) in report.items()})


def test_fp8_rejects_shapes_off_the_pair_tile():
    m = require_gpu()
    with pytest.raises(ValueError):
        m.GroupedMLP(256, 128, 256, 4, 2, precision="fp8")
