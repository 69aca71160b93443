"""The C-ABI entries around grouped tokens, through the C ABI:

  * mxg_mxfp8_quantize_grouped: row-wise and token-column-wise MXFP8 of rows in
    groups (blocks restarting at every group's first row), canonical and
    tensor-core layouts, bit-exact against the quantiser oracle per group;
    padded offsets exact; padding codes zero; bad offsets reported;
  * mxg_gather_rows and mxg_combine: bit-exact against numpy on the same
    values (a gather is a copy; the combine is an fp32 sum in slot order with
    one bf16 rounding); indices outside the buffer reported;
  * mxg_grouped_mlp_fwd_grouped (+ the backward with k = 1) on pre-grouped
    rows: against the oracle (derived bounds), and bit for bit against the
    regular MLP call's own permuted rows, weight gradients and dprobs, which
    is the equivalence an expert-parallel split relies on."""
import numpy as np
import pytest
import torch

import parity_bounds as pb
import synthetic
from gpu_helpers import mma_to_canonical, np_, require_gpu
from oracle import moe, mx

pytestmark = pytest.mark.gpu


def _bf16(rng, shape, scale=1.0):
    return torch.from_numpy((rng.standard_normal(shape) * scale).astype(np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("layout", [0, 1])
def test_grouped_quantiser_blocks_restart_per_group(layout):
    m = require_gpu()
    rng = np.random.default_rng(31 + layout)
    sizes = np.array([37, 0, 128, 5, 300, 0, 64, 1])        # ragged, empty, aligned, tiny
    rows, cols = int(sizes.sum()), 256
    x = _bf16(rng, (rows, cols))
    x[40:48, :] = 0                                          # an all-zero stretch inside a group
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = m.mxg_mxfp8_quantize_grouped(x.cuda(), torch.from_numpy(off).cuda(), st, layout=layout)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    al = 128 if layout == 1 else 32
    poff = np_(out["padded_offsets"])
    assert np.array_equal(poff, np.concatenate([[0], np.cumsum(-(-sizes // al) * al)]))
    cap = out["capacity"]
    qr, qc = np_(out["q_row"]), np_(out["q_col"])
    if layout == 1:
        sr = mma_to_canonical(out["s_row"], cap, cols // 32)
        sc = mma_to_canonical(out["s_col"], cols, cap // 32)
    else:
        sr = np_(out["s_row"]).reshape(cap, cols // 32)
        sc = np_(out["s_col"]).reshape(cols, cap // 32)
    X = x.double().numpy()
    for g in range(sizes.size):
        a, b, p0, p1 = off[g], off[g + 1], poff[g], poff[g + 1]
        if b == a:
            assert p1 == p0
            continue
        codes, scales = mx.quantize_blocks(X[a:b])
        assert np.array_equal(qr[p0:p0 + (b - a)], codes), g
        assert np.array_equal(sr[p0:p0 + (b - a)], scales), g
        assert not qr[p0 + (b - a):p1].any()                 # padding rows: zero codes
        codes, scales = mx.quantize_group_columns(X[a:b])    # blocks from the group's first row
        w = codes.shape[1]
        assert np.array_equal(qc[:, p0:p0 + w], codes), g
        assert np.array_equal(sc[:, p0 // 32:(p0 + w) // 32], scales), g
        assert not qc[:, p0 + w:p1].any()


def test_grouped_quantiser_reports_bad_offsets():
    m = require_gpu()
    x = torch.zeros((64, 128), dtype=torch.bfloat16, device="cuda")
    for off in ([0, 40, 30, 64], [0, 32, 60], [5, 32, 64]):       # decreasing; not ending at rows; not from 0
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = m.mxg_mxfp8_quantize_grouped(x, torch.tensor(off, dtype=torch.int32, device="cuda"), st)
        torch.cuda.synchronize()
        assert int(st.item()) == 17, off                          # MXG_ERR_OFFSETS
        assert not out["padded_offsets"].any()


def test_gather_rows_and_combine_bit_exact():
    m = require_gpu()
    rng = np.random.default_rng(32)
    T, H, k = 300, 384, 3
    x = _bf16(rng, (T, H))
    src_of_row = rng.permutation(T * k).astype(np.int32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = m.mxg_gather_rows(x.cuda(), torch.from_numpy(src_of_row).cuda(), st, div=k)
    probs = torch.from_numpy(rng.random(T * k).astype(np.float32))
    gp = m.mxg_gather_rows(probs.cuda(), torch.from_numpy(src_of_row).cuda(), st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(g.cpu(), x[torch.from_numpy(src_of_row // k).long()])
    assert torch.equal(gp.cpu(), probs[torch.from_numpy(src_of_row).long()])
    # combine: rows in permuted order back to tokens
    row_of_src = np.empty(T * k, dtype=np.int32)
    row_of_src[src_of_row] = np.arange(T * k)
    rows = _bf16(rng, (T * k, H))
    y = m.mxg_combine(rows.cuda(), torch.from_numpy(row_of_src).cuda(), k, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    R32 = rows.float().numpy()
    acc = np.zeros((T, H), dtype=np.float32)
    for j in range(k):
        acc += R32[row_of_src.reshape(T, k)[:, j]]
    assert torch.equal(y.cpu(), torch.from_numpy(acc).to(torch.bfloat16))
    # indices outside the source: zero rows / skipped, reported
    bad = torch.from_numpy(np.array([0, T * k + 5, -3], dtype=np.int32)).cuda()
    st.zero_()
    gb = m.mxg_gather_rows(x.cuda(), bad, st, div=k)
    torch.cuda.synchronize()
    assert int(st.item()) == 19 and not gb[1].any() and not gb[2].any()
    assert torch.equal(gb[0].cpu(), x[0])
    st.zero_()
    m.mxg_combine(rows.cuda(), torch.tensor([0, 1, T * k], dtype=torch.int32, device="cuda"), 3, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 19


@pytest.mark.parametrize("name", ["ragged", "mid"])
def test_pregrouped_mlp_matches_oracle_and_the_regular_call(name):
    m = require_gpu()
    if name == "ragged":
        T, H, I, E, k = 300, 256, 384, 6, 2
        inp = synthetic.make_case(T, H, I, E, k, seed=5, empty_experts=(1, 4))
    else:
        wl = synthetic.WORKLOADS[name]
        T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.k
        inp = synthetic.make_inputs(wl)
    dev = "cuda"
    d = {n: inp[n].to(dev) for n in ("logits", "x", "w_gate_up", "w_down", "dy")}
    # the regular call (tokens + ids): its permuted rows are the reference layout
    layer = m.GroupedMLP(T, H, I, E, k)
    ids, probs = layer.route(d["logits"])
    y_reg, split = layer.forward(d["x"], ids, probs, d["w_gate_up"], d["w_down"])
    mcap = layer.padded_rows_capacity()
    off = m.mxg_mlp_workspace_view(layer.workspace, T, H, I, E, k, 4) - layer.workspace.data_ptr()
    yperm = layer.workspace[off:off + 2 * mcap * H].view(torch.bfloat16).view(mcap, H).clone()
    poff = layer.padded_offsets().clone()
    dx_reg, dwgu_reg, dwd_reg, dprobs_reg = (t.clone() for t in layer.backward(d["dy"]))
    off = m.mxg_mlp_workspace_view(layer.workspace, T, H, I, E, k, 5) - layer.workspace.data_ptr()
    dxperm = layer.workspace[off:off + 2 * mcap * H].view(torch.bfloat16).view(mcap, H).clone()
    torch.cuda.synchronize()
    assert layer.status() == 0

    # the same tokens, permuted by the caller and handed over grouped
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    pm = m.mxg_route_permute(ids, E, st)
    x_g = m.mxg_gather_rows(d["x"], pm["src_of_row"], st, div=k)
    p_g = m.mxg_gather_rows(probs.reshape(-1), pm["src_of_row"], st)
    dy_g = m.mxg_gather_rows(d["dy"], pm["src_of_row"], st, div=k)
    R = T * k
    ex = m.GroupedExperts(R, H, I, E)
    y_g = ex.forward(x_g, pm["split_sizes"], p_g, d["w_gate_up"], d["w_down"])
    dx_g, dwgu_g, dwd_g, dp_g = ex.backward(dy_g)
    y_c = m.mxg_combine(y_g, pm["row_of_src"], k, st)
    dx_c = m.mxg_combine(dx_g, pm["row_of_src"], k, st)
    dprobs_c = m.mxg_gather_rows(dp_g.reshape(-1), pm["row_of_src"], st).reshape(T, k)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and ex.status() == 0

    # bit for bit against the regular call
    split_np = np_(pm["split_sizes"]).astype(np.int64)
    e_of_row = np.repeat(np.arange(E), split_np)
    offs = np.concatenate([[0], np.cumsum(split_np)])
    prow = torch.from_numpy(np_(poff).astype(np.int64)[e_of_row] + (np.arange(R) - offs[e_of_row])).cuda()
    assert torch.equal(y_g, yperm[prow]), "per-row outputs differ from the regular call's permuted rows"
    assert torch.equal(dx_g, dxperm[prow])
    assert torch.equal(y_c, y_reg) and torch.equal(dx_c, dx_reg)
    assert torch.equal(dwgu_g, dwgu_reg) and torch.equal(dwd_g, dwd_reg)
    assert torch.equal(dprobs_c, dprobs_reg)

    # against the oracle on the grouped rows (k = 1, ids from the split sizes)
    xg, dyg = np_(x_g), np_(dy_g)
    ids1 = e_of_row.reshape(R, 1).astype(np.int32)
    pg = np_(p_g).reshape(R, 1)
    ctx = moe.mlp_fwd(xg, ids1, pg, inp["w_gate_up"].double().numpy(), inp["w_down"].double().numpy())
    gr = moe.mlp_bwd(ctx, dyg)
    W = {e: moe.expert_weights(inp["w_gate_up"][e].double().numpy(), inp["w_down"][e].double().numpy())
         for e in range(E) if split_np[e] > 0}
    bnd = pb.full_bounds(ctx, gr, W, dyg)
    rec = {"test": "pregrouped", "workload": name, "precision": "mxfp8"}
    for key, got, ref in (("y", y_g, ctx["y"]), ("dx", dx_g, gr["dx"]), ("dprobs", dp_g, gr["dprobs"]),
                          ("dw_gate_up", dwgu_g, gr["dw_gate_up"]), ("dw_down", dwd_g, gr["dw_down"])):
        pb.check(np_(got), ref, bnd[key], key, rec)


def test_pregrouped_reports_bad_split_sizes():
    m = require_gpu()
    T, H, I, E = 256, 128, 256, 4
    rng = np.random.default_rng(33)
    x = _bf16(rng, (T, H)).cuda()
    w = synthetic.make_case(16, H, I, E, 1, seed=3)
    ex = m.GroupedExperts(T, H, I, E)
    p = torch.ones(T, device="cuda")
    ex.forward(x, torch.tensor([100, 100, 50, 5], dtype=torch.int32, device="cuda"), p,
               w["w_gate_up"].cuda(), w["w_down"].cuda())                 # sums to 255, not 256
    torch.cuda.synchronize()
    assert ex.status() == 17                                              # MXG_ERR_OFFSETS


def test_pregrouped_mx_forward_equals_the_bf16_rows_forward():
    """The inference forward on grouped rows given as row-wise MXFP8 codes and
    scales (mxg_grouped_mlp_fwd_grouped_mx) gives the same y, bit for bit, as
    the forward on the bf16 rows those codes come from."""
    m = require_gpu()
    T, H, I, E, k = 300, 256, 384, 6, 2
    inp = synthetic.make_case(T, H, I, E, k, seed=35, empty_experts=(2,))
    d = {n: inp[n].cuda() for n in ("logits", "x", "w_gate_up", "w_down")}
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ids, probs = m.mxg_route_topk(d["logits"], k)
    pm = m.mxg_route_permute(ids, E, st)
    R = T * k
    x_g = m.mxg_gather_rows(d["x"], pm["src_of_row"], st, div=k)
    p_g = m.mxg_gather_rows(probs.reshape(-1), pm["src_of_row"], st)
    off = torch.tensor([0, R], dtype=torch.int32, device="cuda")
    q = m.mxg_mxfp8_quantize_grouped(x_g, off, st, row=True, col=False)
    xq, xs = q["q_row"][:R], q["s_row"].view(-1, H // 32)[:R]
    ex = m.GroupedExperts(R, H, I, E)
    y_ref = ex.forward(x_g, pm["split_sizes"], p_g, d["w_gate_up"], d["w_down"], save_for_backward=False).clone()
    y_mx = ex.forward_mx(xq, xs, pm["split_sizes"], p_g, d["w_gate_up"], d["w_down"]).clone()
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and ex.status() == 0
    assert torch.equal(y_mx, y_ref)


def test_pregrouped_all_rows_in_one_expert():
    """Every pre-grouped row belongs to one expert (the others get none): the
    forward and backward match the oracle on those rows, and the idle experts'
    weight gradients are exact zeros."""
    m = require_gpu()
    R, H, I, E, hot = 200, 128, 256, 4, 2
    case = synthetic.make_case(R, H, I, E, 1, seed=12)
    split = torch.zeros(E, dtype=torch.int32)
    split[hot] = R
    p = torch.from_numpy(np.random.default_rng(12).uniform(0.1, 1.0, R).astype(np.float32))
    dev = "cuda"
    ex = m.GroupedExperts(R, H, I, E)
    y = ex.forward(case["x"].to(dev), split.to(dev), p.to(dev), case["w_gate_up"].to(dev), case["w_down"].to(dev))
    dx, dwgu, dwd, dp = ex.backward(case["dy"].to(dev))
    torch.cuda.synchronize()
    assert ex.status() == 0
    for e in range(E):
        if e != hot:
            assert not np_(dwgu[e]).any() and not np_(dwd[e]).any()
    ids1 = np.full((R, 1), hot, dtype=np.int32)
    xg, dyg = case["x"].double().numpy(), case["dy"].double().numpy()
    ctx = moe.mlp_fwd(xg, ids1, p.double().numpy().reshape(R, 1), case["w_gate_up"].double().numpy(),
                      case["w_down"].double().numpy())
    gr = moe.mlp_bwd(ctx, dyg)
    W = {hot: moe.expert_weights(case["w_gate_up"][hot].double().numpy(), case["w_down"][hot].double().numpy())}
    bnd = pb.full_bounds(ctx, gr, W, dyg)
    rec = {"test": "pregrouped", "workload": "one_expert", "precision": "mxfp8"}
    for key, got, ref in (("y", y, ctx["y"]), ("dx", dx, gr["dx"]), ("dprobs", dp, gr["dprobs"]),
                          ("dw_gate_up", dwgu, gr["dw_gate_up"]), ("dw_down", dwd, gr["dw_down"])):
        pb.check(np_(got), ref, bnd[key], key, rec)
