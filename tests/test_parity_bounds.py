"""The derived per-element parity bounds (tests/parity_bounds.py), checked on
the CPU before they are applied to a GPU run:

  * they accept a layer computed with the GPU path's storage choices (fp32
    accumulators and activations, GU and dH held in bf16 for the backward,
    bf16 GEMM outputs, the combine summing bf16 rows in fp32): the
    legitimate differences the bounds are derived for;
  * they reject plausible faults planted in that layer: a row taken from the
    wrong token, an expert's gate and up halves swapped in the weight
    gradient, one 32-value block scaled by two (a wrong shared exponent), the
    routing probability left out of one expert's rows.

The simulated layer is test code: oracle arithmetic with the GPU's roundings
inserted.  It never touches the oracle's own outputs."""
import numpy as np
import pytest

import parity_bounds as pb
import synthetic
from oracle import moe, mx


def _f32(a):
    return np.asarray(a, dtype=np.float32).astype(np.float64)


def _gpu_like(x, ids, probs, wgu, wd, dy, ctx):
    """The layer with the GPU path's roundings (see the module docstring)."""
    perm, k, E, I = ctx["perm"], ctx["k"], ctx["E"], ctx["I"]
    T, H = x.shape
    off = perm["offsets"]
    src = perm["src_of_row"]
    tok = src // k
    R = src.size
    p_perm = _f32(probs.reshape(-1)[src])
    y_rows, dx_rows = np.zeros((R, H)), np.zeros((R, H))
    dprow = np.zeros(R)
    dwgu, dwd = np.zeros((E, 2 * I, H)), np.zeros((E, H, I))
    for e in range(E):
        a, b = off[e], off[e + 1]
        if b == a:
            continue
        w = moe.expert_weights(wgu[e], wd[e])
        xq = mx.fake_quant(x[tok[a:b]])
        gu = _f32(xq @ w["wg"].T)                                  # fp32 accumulators
        g32, u32 = gu[:, :I].astype(np.float32), gu[:, I:].astype(np.float32)
        p32 = p_perm[a:b, None].astype(np.float32)
        h = (p32 * (g32 / (np.float32(1) + np.exp(-g32))) * u32).astype(np.float64)
        y_rows[a:b] = moe.bf16_round(mx.fake_quant(h) @ w["wd"].T)
        gu_saved = moe.bf16_round(gu)                               # GU kept in bf16
        dyq = mx.fake_quant(dy[tok[a:b]])
        dh = moe.bf16_round(_f32(dyq @ w["wdT"].T))                  # dH parked in bf16
        dg, du, terms = moe.dscaled_swiglu(dh, gu_saved[:, :I], gu_saved[:, I:], p_perm[a:b, None])
        dgu = _f32(np.concatenate([dg, du], axis=1))
        dprow[a:b] = _f32(terms.sum(axis=1))
        dx_rows[a:b] = moe.bf16_round(mx.fake_quant(dgu) @ w["wguT"].T)
        dwgu[e] = moe.bf16_round(mx.fake_quant_group_columns(dgu).T @ mx.fake_quant_group_columns(x[tok[a:b]]))
        dwd[e] = moe.bf16_round(mx.fake_quant_group_columns(dy[tok[a:b]]).T @ mx.fake_quant_group_columns(h))
    row = perm["row_of_src"].reshape(T, k)
    y = moe.bf16_round(sum(y_rows[row[:, j]].astype(np.float32) for j in range(k)))
    dx = moe.bf16_round(sum(dx_rows[row[:, j]].astype(np.float32) for j in range(k)))
    return {"y": y, "dx": dx, "dprobs": dprow[row], "dw_gate_up": dwgu, "dw_down": dwd, "dx_rows": dx_rows}


@pytest.fixture(scope="module")
def layer():
    T, H, I, E, k = 384, 256, 384, 4, 2
    c = synthetic.make_case(T, H, I, E, k, seed=21, empty_experts=(2,))
    x, wgu, wd, dy = (c[n].double().numpy() for n in ("x", "w_gate_up", "w_down", "dy"))
    ids, probs = moe.route_topk(c["logits"].numpy(), k)
    ctx = moe.mlp_fwd(x, ids, probs, wgu, wd)
    g = moe.mlp_bwd(ctx, dy)
    W = {e: moe.expert_weights(wgu[e], wd[e]) for e in range(E) if ctx["perm"]["split_sizes"][e] > 0}
    bounds = pb.full_bounds(ctx, g, W, dy)
    sim = _gpu_like(x, ids, probs, wgu, wd, dy, ctx)
    ref = {"y": ctx["y"], "dx": g["dx"], "dprobs": g["dprobs"], "dw_gate_up": g["dw_gate_up"],
           "dw_down": g["dw_down"]}
    return {"ctx": ctx, "g": g, "bounds": bounds, "sim": sim, "ref": ref, "shape": (T, H, I, E, k), "dy": dy}


@pytest.mark.parametrize("name", ["y", "dx", "dprobs", "dw_gate_up", "dw_down"])
def test_bounds_accept_the_gpu_storage_choices(layer, name):
    out = pb.check(layer["sim"][name], layer["ref"][name], layer["bounds"][name], name)
    assert out["bound_used"] < 1.0


def test_bounds_accept_a_single_flip_of_h(layer):
    """One token-column code of h one E4M3 step off (the rare flip an fp32
    versus fp64 h can cause) moves a whole dW_down column by dY * step: the
    bound, derived for rare flips, accepts it."""
    ctx = layer["ctx"]
    perm = ctx["perm"]
    e = 0
    a, b = perm["offsets"][e], perm["offsets"][e + 1]
    h = ctx["h"][a:b]
    u = pb.mx_steps_group_columns(h)
    tok = perm["src_of_row"][a:b] // ctx["k"]
    dyc = mx.fake_quant_group_columns(layer["dy"][tok])
    t, i = np.unravel_index(np.argmax(np.abs(h) * np.abs(dyc).max(axis=1, keepdims=True)), h.shape)
    d = layer["sim"]["dw_down"].copy()
    d[e][:, i] += u[t, i] * dyc[t]
    pb.check(d, layer["ref"]["dw_down"], layer["bounds"]["dw_down"], "dw_down")


def _rejected(a, r, bnd, name):
    with pytest.raises(AssertionError):
        pb.check(a, r, bnd, name)


def test_bounds_reject_a_row_from_the_wrong_token(layer):
    y = layer["sim"]["y"].copy()
    y[[5, 6]] = y[[6, 5]]
    _rejected(y, layer["ref"]["y"], layer["bounds"]["y"], "y")
    dx = layer["sim"]["dx"].copy()
    dx[17] = dx[18]
    _rejected(dx, layer["ref"]["dx"], layer["bounds"]["dx"], "dx")


def test_bounds_reject_swapped_gate_and_up_in_the_weight_gradient(layer):
    I = layer["shape"][2]
    d = layer["sim"]["dw_gate_up"].copy()
    d[0] = np.concatenate([d[0][I:], d[0][:I]])
    _rejected(d, layer["ref"]["dw_gate_up"], layer["bounds"]["dw_gate_up"], "dw_gate_up")


def test_bounds_reject_one_block_with_a_wrong_shared_exponent(layer):
    for name, sl in (("dx", (np.s_[40], np.s_[64:96])), ("dw_down", (1, np.s_[7], np.s_[32:64])),
                     ("y", (np.s_[3], np.s_[0:32]))):
        a = layer["sim"][name].copy()
        a[sl] *= 2.0
        _rejected(a, layer["ref"][name], layer["bounds"][name], name)


def test_bounds_reject_a_missing_routing_probability(layer):
    ctx = layer["ctx"]
    perm, k = ctx["perm"], ctx["k"]
    e = 1
    rows = np.arange(perm["offsets"][e], perm["offsets"][e + 1])
    p = ctx["p_perm"][rows]
    # dprobs of the expert's rows without the probability in dh's chain: divide by p
    dp = layer["sim"]["dprobs"].copy()
    flat = perm["src_of_row"][rows]
    dp.reshape(-1)[flat] = dp.reshape(-1)[flat] / p
    _rejected(dp, layer["ref"]["dprobs"], layer["bounds"]["dprobs"], "dprobs")
    # y with the expert's rows unweighted
    T = perm["row_of_src"].size // k
    y = layer["sim"]["y"].copy()
    tokens = flat // k
    y[tokens] = y[tokens] + (1.0 / p[:, None] - 1.0) * ctx["y_perm"][rows]
    _rejected(y, layer["ref"]["y"], layer["bounds"]["y"], "y")
