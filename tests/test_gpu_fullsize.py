"""Full-size parity on the three large workloads (Mixtral layer, its Zipf-skewed
variant, fine-grained 64 experts top-8), in the launch configuration bench.py
times: the whole route -> forward -> backward runs on the GPU; the oracle
checks the integer outputs in full and the floating-point outputs on seeded
samples it can evaluate exactly (oracle.sampled):
  * ids, split_sizes, padded offsets and the padded row map: bit-exact, all;
  * gate-up outputs of the sampled tokens' rows: 1e-2 relative (floor 1);
  * y, dx, dprobs of the sampled tokens and sampled columns of dW_down / rows of
    dW_gate_up: error at most 2e-2 of the reference RMS (relative RMS error over
    the sample, plus the per-element guard);
  * dW of every empty expert: exactly zero."""
import numpy as np
import pytest
import torch

import synthetic
from gpu_helpers import assert_rel_close, assert_rms_close, np_, require_gpu
from oracle import moe, sampled

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pool():
    from oracle_pool import WeightQuantPool
    p = WeightQuantPool()
    yield p
    p.close()


def _pick(wl, ids, split, rng):
    """Sampled tokens and the experts their rows use."""
    if wl.k == 2:
        # tokens routed to the two most loaded experts (both of their rows)
        S = np.argsort(-split, kind="stable")[:2]
        cand = np.nonzero(np.isin(ids[:, 0], S) & np.isin(ids[:, 1], S))[0]
        tokens = np.sort(rng.choice(cand, size=min(24, cand.size), replace=False))
    else:
        tokens = np.sort(rng.choice(wl.T, size=6, replace=False))
    experts = np.unique(ids[tokens])
    return tokens, experts


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
    perm = moe.permute(ids, E, pad=m.mxg_mlp_group_align())
    split = perm["split_sizes"]
    assert np.array_equal(np_(layer.split_sizes), split)
    assert np.array_equal(np_(poff_g), perm["padded_offsets"])
    expert_of_row = np.repeat(np.arange(E), split)
    rows = perm["row_of_src"]
    prow = perm["padded_offsets"][expert_of_row[rows]] + (rows - perm["offsets"][expert_of_row[rows]])
    assert np.array_equal(np_(prow_g), prow)

    # --- sampled floating-point outputs
    rng = np.random.default_rng(4242 + wl.index)
    tokens, experts = _pick(wl, ids, split, rng)
    W = {int(e): pool.expert_weights(inp["w_gate_up"][e], inp["w_down"][e]) for e in experts}
    x, dy = inp["x"].double().numpy(), inp["dy"].double().numpy()
    s = sampled.rows_forward_backward(tokens, x, dy, probs, rows, expert_of_row, k, W)
    tt = torch.from_numpy(tokens).cuda()
    assert_rms_close(np_(layer.y[tt]), s["y"], 2e-2, f"{name} y")
    assert_rms_close(np_(layer.dx[tt]), s["dx"], 2e-2, f"{name} dx")
    assert_rms_close(np_(layer.dprobs[tt]), s["dprobs"], 2e-2, f"{name} dprobs")
    # padded row of each permuted row r (the map above is indexed by flat index)
    prow_of_row = perm["padded_offsets"][expert_of_row] + (np.arange(T * k) - perm["offsets"][expert_of_row])
    pr = prow_of_row[s["rows"].reshape(-1)]
    gu = np_(gu_g[torch.from_numpy(pr).cuda()])
    assert_rel_close(gu, s["gu"].reshape(-1, 2 * I), tol=1e-2, floor=1.0, name=f"{name} gate-up")

    tok = perm["src_of_row"] // k
    p_perm = probs.reshape(-1)[perm["src_of_row"]]
    for e in [int(v) for v in experts[:2] if split[v] > 0]:
        a, b = perm["offsets"][e], perm["offsets"][e + 1]
        xe, dye, pe = x[tok[a:b]], dy[tok[a:b]], p_perm[a:b]
        cols = np.sort(rng.choice(I, size=12, replace=False))
        ref = sampled.dw_down_columns(xe, dye, pe, inp["w_gate_up"][e].double().numpy(), cols)
        got = np_(layer.dw_down[e][:, torch.from_numpy(cols).cuda()])
        assert_rms_close(got, ref, 2e-2, f"{name} dW_down[{e}]")
        rows_n = np.sort(np.concatenate([rng.choice(I, 6, replace=False), I + rng.choice(I, 6, replace=False)]))
        ref = sampled.dw_gate_up_rows(xe, dye, pe, inp["w_gate_up"][e].double().numpy(),
                                      inp["w_down"][e].double().numpy(), rows_n)
        got = np_(layer.dw_gate_up[e][torch.from_numpy(rows_n).cuda()])
        assert_rms_close(got, ref, 2e-2, f"{name} dW_gate_up[{e}]")
    for e in np.nonzero(split == 0)[0]:
        assert not bool(layer.dw_gate_up[int(e)].any()) and not bool(layer.dw_down[int(e)].any())
