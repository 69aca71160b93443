"""bench.py times the step stage by stage (one `_stage` call per kernel group,
events in between).  Running every forward and backward stage in order must
do exactly the work of the full calls: the outputs are bit-identical, for the
MXFP8 path and both precision variants."""
import pytest
import torch

import synthetic
from gpu_helpers import require_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("precision", ["mxfp8", "bf16", "fp8"])
def test_stagewise_step_equals_full_calls(precision):
    m = require_gpu()
    T, H, I, E, k = 500, 256, 512, 5, 2
    inp = synthetic.make_case(T, H, I, E, k, seed=31, empty_experts=(3,))
    d = {n: inp[n].cuda() for n in ("logits", "x", "w_gate_up", "w_down", "dy")}
    results = []
    for staged in (False, True):
        layer = m.GroupedMLP(T, H, I, E, k, precision=precision)
        ids, probs = layer.route(d["logits"])
        if staged:
            for st in range(len(m.FWD_STAGES)):
                layer.forward(d["x"], ids, probs, d["w_gate_up"], d["w_down"], stage=st)
            for st in range(len(m.BWD_STAGES)):
                layer.backward(d["dy"], stage=st)
        else:
            layer.forward(d["x"], ids, probs, d["w_gate_up"], d["w_down"])
            layer.backward(d["dy"])
        torch.cuda.synchronize()
        assert layer.status() == 0
        results.append([t.clone() for t in (layer.y, layer.split_sizes, layer.dx, layer.dw_gate_up, layer.dw_down,
                                            layer.dprobs)])
    for a, b in zip(*results):
        assert torch.equal(a, b)


@pytest.mark.parametrize("precision", ["mxfp8", "bf16", "fp8"])
def test_inference_forward_equals_training_forward(precision):
    """save_for_backward = 0 skips what only the backward needs (transposed
    weights, token-column-wise activations, the saved g|u); y and split_sizes
    are bit-identical to a forward that saves."""
    m = require_gpu()
    T, H, I, E, k = 500, 256, 512, 5, 2
    inp = synthetic.make_case(T, H, I, E, k, seed=33, empty_experts=(1,))
    d = {n: inp[n].cuda() for n in ("logits", "x", "w_gate_up", "w_down")}
    outs = []
    for save in (True, False):
        layer = m.GroupedMLP(T, H, I, E, k, precision=precision)
        ids, probs = layer.route(d["logits"])
        y, split = layer.forward(d["x"], ids, probs, d["w_gate_up"], d["w_down"], save_for_backward=save)
        torch.cuda.synchronize()
        assert layer.status() == 0
        outs.append((y.clone(), split.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
