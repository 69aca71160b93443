"""Whole-path parity: route -> grouped MLP forward -> backward through the C ABI
against the oracle, element by element, on seeded inputs that span several
tiles, ragged group tails and empty experts.

Tolerances: ids, split_sizes and padded offsets bit-exact; gate-up outputs
within 1e-2 relative (floor |ref| >= 1); y, dx, dW_gate_up, dW_down and dprobs
with a relative RMS error of at most 2e-2 and, per element, within the bound
tests/parity_bounds.py derives (2e-2 of the RMS, the bf16 storage of the
output and of the rows it sums, and the spread of the re-quantisation flips of
h and dGU); dW of an empty expert exactly zero."""
import numpy as np
import pytest
import torch

import synthetic
import parity_bounds as pb
from gpu_helpers import assert_rel_close, codes_equal_up_to_zero_sign, mma_to_canonical, np_, require_gpu
from oracle import moe, mx

pytestmark = pytest.mark.gpu


def _inputs(name):
    if name == "ragged":
        return (300, 256, 384, 6, 2), synthetic.make_case(300, 256, 384, 6, 2, seed=5, empty_experts=(1, 4))
    if name == "ragged_k1":
        return (200, 128, 128, 3, 1), synthetic.make_case(200, 128, 128, 3, 1, seed=6)
    if name == "wide_e256":      # the largest expert count, top-8: ~16 rows per expert, each in its own tile
        return (512, 256, 256, 256, 8), synthetic.make_case(512, 256, 256, 256, 8, seed=7)
    if name == "all_experts":    # k = E: every token goes to every expert
        return (256, 128, 256, 4, 4), synthetic.make_case(256, 128, 256, 4, 4, seed=8)
    if name == "top32":          # the largest k: 32 of 64 experts per token, combines over 32 rows
        return (128, 128, 128, 64, 32), synthetic.make_case(128, 128, 128, 64, 32, seed=9)
    if name == "one_token":      # a single token: two one-row groups, every tile mostly padding
        return (1, 128, 128, 4, 2), synthetic.make_case(1, 128, 128, 4, 2, seed=10)
    wl = synthetic.WORKLOADS[name]
    inp = synthetic.make_inputs(wl)
    if "dy" not in inp:          # the forward-only workload still gets a backward check here
        inp["dy"] = synthetic.random_bf16((wl.T, wl.H), 77)
    return (wl.T, wl.H, wl.I, wl.E, wl.k), inp


def run_gpu(m, shape, inp):
    T, H, I, E, k = shape
    layer = m.GroupedMLP(T, H, I, E, k)
    dev = "cuda"
    logits, x = inp["logits"].to(dev), inp["x"].to(dev)
    wgu, wd, dy = inp["w_gate_up"].to(dev), inp["w_down"].to(dev), inp["dy"].to(dev)
    ids, probs = layer.route(logits)
    y, split = layer.forward(x, ids, probs, wgu, wd, save_for_backward=True)
    mcap0 = layer.padded_rows_capacity()
    off = m.mxg_mlp_workspace_view(layer.workspace, T, H, I, E, k, 4) - layer.workspace.data_ptr()
    yperm = layer.workspace[off:off + 2 * mcap0 * H].clone()
    gu = layer.gu_view().clone()
    poff = layer.padded_offsets().clone()
    mcap = layer.padded_rows_capacity()
    views = {}
    for name, which, rows in (("xc", 3, H), ("sxc", 4, H), ("hc", 5, I), ("shc", 6, I)):
        ptr = m.mxg_mlp_saved_view(layer.saved, T, H, I, E, k, which)
        off = ptr - layer.saved.data_ptr()
        n = rows * mcap if name in ("xc", "hc") else rows * mcap // 32
        views[name] = layer.saved[off:off + n].clone()
    dx, dwgu, dwd, dprobs = layer.backward(dy)
    torch.cuda.synchronize()
    off = m.mxg_mlp_workspace_view(layer.workspace, T, H, I, E, k, 5) - layer.workspace.data_ptr()
    dxperm = layer.workspace[off:off + 2 * mcap0 * H].clone()
    for name, which, n in (("dguq", 0, mcap * 2 * I), ("sdguq", 1, mcap * 2 * I // 32), ("dguc", 2, 2 * I * mcap),
                           ("sdguc", 3, 2 * I * mcap // 32)):
        off = m.mxg_mlp_workspace_view(layer.workspace, T, H, I, E, k, which) - layer.workspace.data_ptr()
        views[name] = layer.workspace[off:off + n].clone()
    out = {"ids": ids, "probs": probs, "y": y, "split": split, "gu": gu, "poff": poff, "dx": dx,
           "dwgu": dwgu, "dwd": dwd, "dprobs": dprobs}
    out = {n: np_(v) for n, v in out.items()}
    out["status"] = layer.status()
    out["mcap"] = mcap
    # the combine is fused into the down / dgrad-gate-up epilogues: recompute it
    # from their rows with the combine's arithmetic (fp32 sum in slot order, one
    # bf16 rounding) for a bit-exact comparison
    rows = layer.padded_rows_capacity()
    poff_np = out["poff"]
    perm = moe.permute(out["ids"].astype(np.int64), E, pad=m.mxg_mlp_group_align())
    e_of_row = np.repeat(np.arange(E), perm["split_sizes"])
    prow_of_flat = np.empty(T * k, dtype=np.int64)
    prow_of_flat[perm["src_of_row"]] = poff_np[e_of_row] + (np.arange(T * k) - perm["offsets"][e_of_row])
    for name, rows_t in (("y_fused_ref", yperm), ("dx_fused_ref", dxperm)):
        Y = rows_t.view(torch.bfloat16).float().cpu().numpy().reshape(rows, H)
        acc = np.zeros((T, H), dtype=np.float32)
        for j in range(k):
            acc += Y[prow_of_flat.reshape(T, k)[:, j]]
        out[name] = torch.from_numpy(acc).to(torch.bfloat16).double().numpy()
    out.update({n: v.cpu().numpy() for n, v in views.items()})
    return out


@pytest.mark.parametrize("name", ["tiny", "ragged", "ragged_k1", "mid", "wide_e256", "all_experts", "top32",
                                  "one_token"])
def test_mlp_fwd_bwd_matches_oracle(name):
    m = require_gpu()
    shape, inp = _inputs(name)
    T, H, I, E, k = shape
    got = run_gpu(m, shape, inp)
    assert got["status"] == 0

    logits = inp["logits"].numpy()
    ids, probs = moe.route_topk(logits, k)
    ctx = moe.mlp_fwd(inp["x"].double().numpy(), ids, probs, inp["w_gate_up"].double().numpy(),
                      inp["w_down"].double().numpy())
    g = moe.mlp_bwd(ctx, inp["dy"].double().numpy())
    perm = ctx["perm"]

    assert np.array_equal(got["ids"], ids)
    assert np.array_equal(got["split"], perm["split_sizes"])
    poff = moe.permute(ids, E, pad=m.mxg_mlp_group_align())["padded_offsets"]
    assert np.array_equal(got["poff"], poff)

    # gate-up output (before the activation), in the padded row layout
    e_of_row = np.repeat(np.arange(E), perm["split_sizes"])
    prow = poff[e_of_row] + (np.arange(T * k) - perm["offsets"][e_of_row])
    assert_rel_close(got["gu"][prow], ctx["gu"], tol=1e-2, floor=1.0, name="gate-up")

    assert np.array_equal(got["y"], got["y_fused_ref"]), "fused combine (forward) differs from the combine arithmetic"
    assert np.array_equal(got["dx"], got["dx_fused_ref"]), "fused combine (backward) differs from the combine arithmetic"
    report = {}
    W = {e: moe.expert_weights(inp["w_gate_up"][e].double().numpy(), inp["w_down"][e].double().numpy())
         for e in range(E) if perm["split_sizes"][e] > 0}
    bnd = pb.full_bounds(ctx, g, W, inp["dy"].double().numpy())
    rec = {"test": "mlp", "workload": name, "precision": "mxfp8"}
    for key, gkey, ref in (("y", "y", ctx["y"]), ("dx", "dx", g["dx"]), ("dprobs", "dprobs", g["dprobs"]),
                           ("dw_gate_up", "dwgu", g["dw_gate_up"]), ("dw_down", "dwd", g["dw_down"])):
        o = pb.check(got[gkey], ref, bnd[key], key, rec)
        report[key] = (o["max_err_over_rms"], o["rel_rms"])
    for e in np.nonzero(perm["split_sizes"] == 0)[0]:
        assert not got["dwgu"][e].any() and not got["dwd"][e].any()

    # token-column-wise MXFP8 kept for the weight gradients: x's (an input) bit
    # for bit; h's (re-quantised from the GEMM's fp32 h) as the fraction of
    # codes and scales that differ from the oracle's quantisation of its fp64 h
    mcap = got["mcap"]
    xc, hc = got["xc"].reshape(H, mcap), got["hc"].reshape(I, mcap)
    sxc = mma_to_canonical(torch.from_numpy(got["sxc"]), H, mcap // 32)
    shc = mma_to_canonical(torch.from_numpy(got["shc"]), I, mcap // 32)
    diff_codes = diff_scales = n_codes = n_scales = 0
    for e in range(E):
        a, b = perm["offsets"][e], perm["offsets"][e + 1]
        if b == a:
            continue
        p0 = poff[e]
        codes, scales = mx.quantize_group_columns(ctx["x_perm"][a:b])
        w = codes.shape[1]
        d, z = codes_equal_up_to_zero_sign(xc[:, p0:p0 + w], codes)
        assert d == 0, f"x column codes, expert {e}: {d} differ"
        assert np.array_equal(sxc[:, p0 // 32:(p0 + w) // 32], scales), f"x column scales, expert {e}"
        codes, scales = mx.quantize_group_columns(ctx["h"][a:b])
        d, z = codes_equal_up_to_zero_sign(hc[:, p0:p0 + w], codes)
        diff_codes += d
        n_codes += codes.size
        diff_scales += int((shc[:, p0 // 32:(p0 + w) // 32] != scales).sum())
        n_scales += scales.size
    frac = diff_codes / n_codes
    report["h column codes differing"] = (frac, diff_scales / n_scales)
    pb.write_record(dict(rec, tensor="h column codes", codes_differing=frac, scales_differing=diff_scales / n_scales))
    assert frac < 1e-3 and diff_scales / n_scales < 1e-3, (frac, diff_scales / n_scales)

    # dGU's fused re-quantisation (both orientations) against the oracle's MX
    # of its fp64 dGU, as fractions of differing codes and scales.  The kernel
    # computes dGU from bf16 g|u (GU is kept in bf16 for the backward) and a
    # bf16-staged dH, a relative perturbation of up to ~3 bf16 half-ulps
    # (3 * 2^-9, 0.6 %) against E4M3 steps of 2^-3 relative, so at most ~5 % of
    # codes can land on the neighbouring value; measured 1.6-3.2 % (scales
    # 0.1-0.3 %), each such code one E4M3 step off.
    dguq, dguc = got["dguq"].reshape(mcap, 2 * I), got["dguc"].reshape(2 * I, mcap)
    sdguq = mma_to_canonical(torch.from_numpy(got["sdguq"]), mcap, 2 * I // 32)
    sdguc = mma_to_canonical(torch.from_numpy(got["sdguc"]), 2 * I, mcap // 32)
    codes_r, scales_r = mx.quantize_blocks(g["dgu"])
    dr, _ = codes_equal_up_to_zero_sign(dguq[prow], codes_r)
    dsr = int((sdguq[prow] != scales_r).sum())
    dc = dsc = nc = nsc = 0
    for e in range(E):
        a, b = perm["offsets"][e], perm["offsets"][e + 1]
        if b == a:
            continue
        p0 = poff[e]
        codes, scales = mx.quantize_group_columns(g["dgu"][a:b])
        w = codes.shape[1]
        d, _ = codes_equal_up_to_zero_sign(dguc[:, p0:p0 + w], codes)
        dc += d
        nc += codes.size
        dsc += int((sdguc[:, p0 // 32:(p0 + w) // 32] != scales).sum())
        nsc += scales.size
    report["dGU row codes differing"] = (dr / codes_r.size, dsr / scales_r.size)
    report["dGU column codes differing"] = (dc / nc, dsc / nsc)
    pb.write_record(dict(rec, tensor="dGU row codes", codes_differing=dr / codes_r.size,
                         scales_differing=dsr / scales_r.size))
    pb.write_record(dict(rec, tensor="dGU column codes", codes_differing=dc / nc, scales_differing=dsc / nsc))
    assert dr / codes_r.size < 5e-2 and dc / nc < 5e-2, (dr / codes_r.size, dc / nc)
    print(name, {n: (round(a, 6), round(b, 6)) for n, (a, b) in report.items()})
