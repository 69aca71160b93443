"""The expert-parallel layer (mxfp8_grouped_gemm_gb300.ep) on the GPU with G
virtual ranks in one process: each rank is a host thread running its own
route, permute, gathers, grouped expert MLP and combine kernels; the
all-to-all steps are done on the host between kernel launches (every rank
synchronises the device before it hands rows over), so no kernel ever waits
on another.  Compared bit for bit with the single-GPU MLP over all ranks'
tokens (the same kernels on the same rows in the same order): y, dx and
dprobs of every rank's tokens, and every rank's experts' dW_gate_up and
dW_down ("BioNeMo Uses Grouped Kernels and MXFP8", "Launching the recipe":
expert parallelism).  The inference payload (each token's row-wise MXFP8
codes and scales instead of its bf16 row) gives the same y."""
import threading

import numpy as np
import pytest
import torch

import synthetic
from gpu_helpers import require_gpu

pytestmark = pytest.mark.gpu


class ThreadComm:
    """All-to-all between G threads of one process (device tensors)."""

    def __init__(self, world: int):
        self.world = world
        self.barrier = threading.Barrier(world)
        self.slots = [[None] * world for _ in range(world)]

    def rank_view(self, rank):
        comm = self

        class View:
            def __init__(self):
                self.rank, self.world = rank, comm.world

            def all_to_all_counts(self, send):
                return comm._exchange(rank, [np.asarray(send[g]).copy() for g in range(comm.world)], np.stack)

            def all_to_all_rows(self, send, send_splits, recv_splits):
                torch.cuda.synchronize()
                off = np.concatenate([[0], np.cumsum(send_splits)])
                chunks = [send[off[g]:off[g + 1]] for g in range(comm.world)]
                out = comm._exchange(rank, chunks, lambda parts: torch.cat(parts, 0))
                assert out.shape[0] == sum(recv_splits)
                return out
        return View()

    def _exchange(self, rank, chunks, join):
        for g in range(self.world):
            self.slots[rank][g] = chunks[g]
        self.barrier.wait()
        got = join([self.slots[s][rank] for s in range(self.world)])
        if isinstance(got, torch.Tensor):
            got = got.clone()
            torch.cuda.synchronize()
        self.barrier.wait()
        return got


@pytest.mark.parametrize("G,payload", [(2, "bf16"), (4, "bf16"), (2, "mxfp8")])
def test_expert_parallel_on_virtual_ranks_equals_single_gpu(G, payload):
    m = require_gpu()
    from mxfp8_grouped_gemm_gb300 import ep
    T_loc, H, I, E, k = 256, 256, 384, 8, 2
    T = G * T_loc
    inp = synthetic.make_case(T, H, I, E, k, seed=50 + G, empty_experts=(3,))
    d = {n: inp[n].cuda() for n in ("logits", "x", "w_gate_up", "w_down", "dy")}

    ref = m.GroupedMLP(T, H, I, E, k)
    ids, probs = ref.route(d["logits"])
    y_ref, _ = ref.forward(d["x"], ids, probs, d["w_gate_up"], d["w_down"])
    dx_ref, dwgu_ref, dwd_ref, dprobs_ref = ref.backward(d["dy"])
    torch.cuda.synchronize()
    assert ref.status() == 0

    comm = ThreadComm(G)
    n = E // G
    out, errors = {}, []

    def run(rank):
        try:
            torch.cuda.set_device(0)
            sl = slice(rank * T_loc, (rank + 1) * T_loc)
            mine = slice(rank * n, (rank + 1) * n)
            layer = ep.ExpertParallelMLP(comm.rank_view(rank), T_loc, H, I, E, k)
            y = layer.forward(d["x"][sl], ids[sl].contiguous(), probs[sl].contiguous(),
                              d["w_gate_up"][mine].contiguous(), d["w_down"][mine].contiguous(), payload=payload)
            if payload == "mxfp8":                  # inference: the forward only
                torch.cuda.synchronize()
                layer.ops.check()
                out[rank] = (y,)
                return
            dx, dwgu, dwd, dprobs = layer.backward(d["dy"][sl].contiguous())
            torch.cuda.synchronize()
            layer.ops.check()
            out[rank] = (y, dx, dwgu, dwd, dprobs)
        except BaseException as exc:          # reported by the main thread
            errors.append(exc)
            comm.barrier.abort()

    threads = [threading.Thread(target=run, args=(r,)) for r in range(G)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not errors, errors[0]
    for r in range(G):
        sl = slice(r * T_loc, (r + 1) * T_loc)
        assert torch.equal(out[r][0], y_ref[sl]), r
        if payload == "mxfp8":
            continue
        y, dx, dwgu, dwd, dprobs = out[r]
        assert torch.equal(dx, dx_ref[sl]), r
        assert torch.equal(dprobs, dprobs_ref[sl]), r
        assert torch.equal(dwgu, dwgu_ref[r * n:(r + 1) * n]), r
        assert torch.equal(dwd, dwd_ref[r * n:(r + 1) * n]), r
