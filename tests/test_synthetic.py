"""The seeded input recipe (synthetic.py): deterministic per seed, the stated
value distributions, and the skewed workload's structure (two empty experts,
Zipf weights over the other six, splits that are not multiples of 128, top-2 of
the drawn logits returning the drawn pair)."""
import numpy as np
import torch

import synthetic
from oracle import moe


def test_same_seed_same_inputs():
    a = synthetic.make_case(64, 128, 128, 4, 2, seed=9)
    b = synthetic.make_case(64, 128, 128, 4, 2, seed=9)
    c = synthetic.make_case(64, 128, 128, 4, 2, seed=10)
    for key in ("logits", "x", "w_gate_up", "w_down", "dy"):
        assert torch.equal(a[key], b[key]), key
        assert not torch.equal(a[key], c[key]), key


def test_value_distributions():
    inp = synthetic.make_case(2048, 256, 256, 4, 2, seed=3)
    x = inp["x"].float()
    w = inp["w_gate_up"].float()
    assert abs(x.mean().item()) < 0.02 and abs(x.std().item() - 1.0) < 0.02
    assert abs(w.std().item() - synthetic.WEIGHT_STD) < 0.001
    assert inp["x"].dtype == torch.bfloat16 and inp["logits"].dtype == torch.float32


def test_skew_workload_structure():
    wl = synthetic.WORKLOADS["skew"]
    inp = synthetic.make_inputs(wl, with_weights=False)
    counts = inp["drawn_counts"]
    assert len(inp["empty_experts"]) == 2 and all(counts[e] == 0 for e in inp["empty_experts"])
    live = counts[counts > 0]
    assert live.size == wl.E - 2 and counts.sum() == wl.T * wl.k
    assert all(c % 128 != 0 for c in live)
    assert 0.3 < live.max() / counts.sum() < 0.5          # the top-ranked expert takes ~40 % of the rows
    ids, _ = moe.route_topk(inp["logits"].numpy(), wl.k)
    assert np.array_equal(np.bincount(ids.ravel(), minlength=wl.E), counts)
