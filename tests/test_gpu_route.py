"""Routing and permute parity: ids and every permutation index bit-exact
against the oracle, probabilities to fp32 rounding; invalid ids reported."""
import numpy as np
import pytest
import torch

from gpu_helpers import np_, require_gpu
from oracle import moe

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,E,k", [(256, 4, 2), (4096, 8, 2), (8192, 64, 8), (1000, 256, 32), (77, 5, 1)])
def test_topk_and_permute_bit_exact(T, E, k):
    m = require_gpu()
    rng = np.random.default_rng(T + E + k)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[: T // 10, 1] = logits[: T // 10, 0]          # planted exact ties
    logits[T // 10: T // 5] = 0.5                         # whole rows tied
    lg = torch.from_numpy(logits).cuda()
    ids, probs = m.mxg_route_topk(lg, k)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    perm = m.mxg_route_permute(ids, E, st)
    torch.cuda.synchronize()
    ref_ids, ref_probs = moe.route_topk(logits, k)
    assert np.array_equal(np_(ids), ref_ids)
    np.testing.assert_allclose(np_(probs), ref_probs, rtol=2e-6, atol=1e-7)
    ref = moe.permute(ref_ids, E)
    assert int(st.item()) == 0
    assert np.array_equal(np_(perm["split_sizes"]), ref["split_sizes"])
    assert np.array_equal(np_(perm["padded_offsets"]), ref["padded_offsets"])
    assert np.array_equal(np_(perm["src_of_row"]), ref["src_of_row"])
    assert np.array_equal(np_(perm["row_of_src"]), ref["row_of_src"])


def test_permute_reports_bad_expert_id():
    m = require_gpu()
    ids = torch.tensor([[0, 1], [2, 7], [1, 3], [9, 0]], dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    perm = m.mxg_route_permute(ids, 4, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 16                           # MXG_ERR_EXPERT_ID
    row_of_src = np_(perm["row_of_src"])
    assert row_of_src[3] == -1 and row_of_src[6] == -1    # dropped entries
    assert int(np_(perm["split_sizes"]).sum()) == 6


@pytest.mark.parametrize("T,E,k", [(4096, 8, 2), (1000, 16, 4), (300, 64, 1), (77, 5, 3)])
def test_thread_route_equals_warp_route(T, E, k):
    """While E k <= 64 the route runs one thread per token; padding the logits
    with experts that are never chosen (E + 60 columns of -1e30) sends the same
    rows through the one-warp-per-token route.  Ids and probabilities must be
    bit-identical (same picks, same softmax summation order)."""
    m = require_gpu()
    rng = np.random.default_rng(7 * T + E)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[: T // 8, -1] = logits[: T // 8, 0]            # ties go to the lower id on both routes
    padded = np.concatenate([logits, np.full((T, 60), -1e30, np.float32)], axis=1)
    assert E * k <= 64 < (E + 60) * k
    ids_t, probs_t = m.mxg_route_topk(torch.from_numpy(logits).cuda(), k)
    ids_w, probs_w = m.mxg_route_topk(torch.from_numpy(padded).cuda(), k)
    torch.cuda.synchronize()
    assert torch.equal(ids_t, ids_w)
    assert torch.equal(probs_t, probs_w)
