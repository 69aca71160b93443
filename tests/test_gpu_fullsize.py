"""Full-size parity on the three large workloads (Mixtral layer, its Zipf-skewed
variant, fine-grained 64 experts top-8), in the launch configuration bench.py
times: the whole route -> forward -> backward runs on the GPU; the oracle
checks the integer outputs in full and the floating-point outputs on seeded
samples it can evaluate exactly (oracle.sampled):
  * ids, split_sizes, padded offsets and the padded row map: bit-exact, all;
  * sampled rows: for every expert with tokens, 8 of its rows, half of them in
    the expert's last 256-row tile (the ragged tile when the split is not a
    multiple of 256); the tokens owning them bring all their k rows;
  * gate-up outputs of those rows: 1e-2 relative (floor 1);
  * y, dx, dprobs of those tokens and, for every expert with tokens, sampled
    columns of dW_down and rows of dW_gate_up: relative RMS error at most 2e-2
    over the sample and every element within the bound tests/parity_bounds.py
    derives (the RMS being the sample's);
  * dW of every empty expert: exactly zero.
The oracle holds one expert's weights at a time."""
import numpy as np
import pytest
import torch

import parity_bounds as pb
import synthetic
from gpu_helpers import assert_rel_close, np_, require_gpu
from oracle import moe, sampled

pytestmark = pytest.mark.gpu

ROWS_PER_EXPERT = 8
DW_SLICES_PER_EXPERT = 8


@pytest.fixture(scope="module")
def pool():
    from oracle_pool import WeightQuantPool
    p = WeightQuantPool()
    yield p
    p.close()


def _pick_rows(perm, split, align, rng):
    """Permuted rows to sample: per non-empty expert, half from its last tile."""
    rows = []
    for e in np.nonzero(split > 0)[0]:
        a, b = int(perm["offsets"][e]), int(perm["offsets"][e + 1])
        last0 = a + ((b - a - 1) // align) * align
        n_last = min(ROWS_PER_EXPERT // 2, b - last0)
        last = rng.choice(np.arange(last0, b), size=n_last, replace=False)
        rest = np.setdiff1d(np.arange(a, b), last)
        rows.append(last)
        rows.append(rng.choice(rest, size=min(ROWS_PER_EXPERT - n_last, rest.size), replace=False))
    return np.sort(np.concatenate(rows))


@pytest.mark.parametrize("name", ["mixtral", "skew", "fine"])
def test_fullsize_sampled(name, pool):
    m = require_gpu()
    wl = synthetic.WORKLOADS[name]
    inp = synthetic.make_inputs(wl)
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.k

    layer = m.GroupedMLP(T, H, I, E, k)
    d = {n: v.cuda() for n, v in inp.items() if isinstance(v, torch.Tensor)}
    ids_g, probs_g = layer.route(d["logits"])
    layer.forward(d["x"], ids_g, probs_g, d["w_gate_up"], d["w_down"])
    poff_g = layer.padded_offsets().clone()
    base = layer.saved.data_ptr()
    off = m.mxg_mlp_saved_view(layer.saved, T, H, I, E, k, 2) - base
    prow_g = layer.saved[off:off + 4 * T * k].view(torch.int32).clone()
    gu_g = layer.gu_view()
    layer.backward(d["dy"])
    torch.cuda.synchronize()
    assert layer.status() == 0

    # --- integer outputs, in full
    ids, probs = moe.route_topk(inp["logits"].numpy(), k)
    assert np.array_equal(np_(ids_g), ids)
    align = m.mxg_mlp_group_align()
    perm = moe.permute(ids, E, pad=align)
    split = perm["split_sizes"]
    assert np.array_equal(np_(layer.split_sizes), split)
    assert np.array_equal(np_(poff_g), perm["padded_offsets"])
    expert_of_row = np.repeat(np.arange(E), split)
    rows = perm["row_of_src"]
    prow = perm["padded_offsets"][expert_of_row[rows]] + (rows - perm["offsets"][expert_of_row[rows]])
    assert np.array_equal(np_(prow_g), prow)

    # --- sampled tokens: every non-empty expert, its last tile included
    rng = np.random.default_rng(4242 + wl.index)
    tokens = np.unique(perm["src_of_row"][_pick_rows(perm, split, align, rng)] // k)
    x, dy = inp["x"].double().numpy(), inp["dy"].double().numpy()
    tok = perm["src_of_row"] // k
    p_perm = probs.reshape(-1)[perm["src_of_row"]]
    n = tokens.size
    acc = {"y": np.zeros((n, H)), "dx": np.zeros((n, H)), "dprobs": np.zeros((n, k)), "gu": np.zeros((n, k, 2 * I))}
    extra = {"y_rows": np.zeros((n, H)), "dx_rows": np.zeros((n, H)), "f_y": np.zeros((n, H)),
             "f_dx": np.zeros((n, H)), "dp_sig": np.zeros((n, k))}
    done = np.zeros((n, k), dtype=bool)
    dwd_got, dwd_ref, dwd_extra = [], [], []
    dwgu_got, dwgu_ref, dwgu_extra = [], [], []
    for e in [int(v) for v in np.nonzero(split > 0)[0]]:
        W = pool.expert_weights(inp["w_gate_up"][e], inp["w_down"][e])
        s = sampled.rows_forward_backward(tokens, x, dy, probs, rows, expert_of_row, k, {e: W})
        for key in acc:
            acc[key] = acc[key] + s[key]
        done |= s["done"]
        for a, j in zip(*np.nonzero(s["done"])):
            extra["y_rows"][a] += np.abs(s["y_rows"][a, j])
            extra["dx_rows"][a] += np.abs(s["dx_rows"][a, j])
            extra["f_y"][a] += pb.flip_allowance("mxfp8", "h", s["h"][a, j][None], W["wd"], False)[0]
            extra["f_dx"][a] += pb.flip_allowance("mxfp8", "dgu", s["dgu"][a, j][None], W["wguT"], False)[0]
            g_, u_ = s["gu"][a, j, :I], s["gu"][a, j, I:]
            _, _, terms = moe.dscaled_swiglu(s["dh"][a, j], g_, u_, probs[tokens[a], j])
            extra["dp_sig"][a, j] = pb.DELTA_DGU * np.sqrt(np.sum(terms * terms))
        del W
        # weight-gradient slices of this expert
        a0, b0 = perm["offsets"][e], perm["offsets"][e + 1]
        xe, dye, pe = x[tok[a0:b0]], dy[tok[a0:b0]], p_perm[a0:b0]
        cols = np.sort(rng.choice(I, size=DW_SLICES_PER_EXPERT, replace=False))
        ref, parts = sampled.dw_down_columns(xe, dye, pe, inp["w_gate_up"][e].double().numpy(), cols, parts=True)
        dwd_ref.append(ref)
        dwd_got.append(np_(layer.dw_down[e][:, torch.from_numpy(cols).cuda()]))
        dwd_extra.append(pb.storage(ref) + pb.flip_allowance("mxfp8", "h", parts["h"], parts["dyc"], True).T)
        half = DW_SLICES_PER_EXPERT // 2
        rows_n = np.sort(np.concatenate([rng.choice(I, half, replace=False), I + rng.choice(I, half, replace=False)]))
        ref, parts = sampled.dw_gate_up_rows(xe, dye, pe, inp["w_gate_up"][e].double().numpy(),
                                             inp["w_down"][e].double().numpy(), rows_n, parts=True)
        dwgu_ref.append(ref)
        dwgu_got.append(np_(layer.dw_gate_up[e][torch.from_numpy(rows_n).cuda()]))
        dwgu_extra.append(pb.storage(ref) + pb.flip_allowance("mxfp8", "dgu", parts["dgu"], parts["xc"], True))
    assert done.all()

    rec = {"test": "fullsize_sampled", "workload": name, "precision": "mxfp8", "sampled_tokens": int(n)}
    tt = torch.from_numpy(tokens).cuda()
    y_ref, dx_ref = acc["y"], acc["dx"]
    pb.check(np_(layer.y[tt]), y_ref,
             pb.bound(y_ref, pb.storage(y_ref, extra["y_rows"]) + extra["f_y"]), "y", rec)
    pb.check(np_(layer.dx[tt]), dx_ref,
             pb.bound(dx_ref, pb.storage(dx_ref, extra["dx_rows"]) + extra["f_dx"]), "dx", rec)
    pb.check(np_(layer.dprobs[tt]), acc["dprobs"], pb.bound(acc["dprobs"], pb.Z * extra["dp_sig"]), "dprobs", rec)
    dwd_ref_all = np.concatenate([r.ravel() for r in dwd_ref])
    pb.check(np.concatenate([g_.ravel() for g_ in dwd_got]), dwd_ref_all,
             pb.bound(dwd_ref_all, np.concatenate([b_.ravel() for b_ in dwd_extra])), "dw_down", rec)
    dwgu_ref_all = np.concatenate([r.ravel() for r in dwgu_ref])
    pb.check(np.concatenate([g_.ravel() for g_ in dwgu_got]), dwgu_ref_all,
             pb.bound(dwgu_ref_all, np.concatenate([b_.ravel() for b_ in dwgu_extra])), "dw_gate_up", rec)

    # gate-up rows of the sampled tokens (padded row layout)
    srows = perm["row_of_src"].reshape(T, k)[tokens]                  # permuted rows [n, k]
    pr = perm["padded_offsets"][expert_of_row[srows]] + (srows - perm["offsets"][expert_of_row[srows]])
    gu = np_(gu_g[torch.from_numpy(pr.reshape(-1)).cuda()])
    assert_rel_close(gu, acc["gu"].reshape(-1, 2 * I), tol=1e-2, floor=1.0, name=f"{name} gate-up")
    # the sample reached every non-empty expert's last tile
    last_tile_rows = 0
    for e in np.nonzero(split > 0)[0]:
        a0, b0 = perm["offsets"][e], perm["offsets"][e + 1]
        last_tile_rows += int(np.sum((srows >= a0 + ((b0 - a0 - 1) // align) * align) & (srows < b0)) > 0)
    assert last_tile_rows == int(np.sum(split > 0))
    pb.write_record(dict(rec, tensor="coverage", experts=int(np.sum(split > 0)), last_tiles=last_tile_rows))
    for e in np.nonzero(split == 0)[0]:
        assert not bool(layer.dw_gate_up[int(e)].any()) and not bool(layer.dw_down[int(e)].any())
