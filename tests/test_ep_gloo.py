"""Expert parallelism as CPU ranks (gloo): world sizes 2 and 4, E/G experts per
rank, every rank routing its own tokens; the dispatch (counts all-to-all, then
all-to-all-v of the token rows and probabilities), the receive-side reorder,
the return of the output rows and the combine run through
mxfp8_grouped_gemm_gb300.ep with the oracle standing in for the kernels
(tests/ep_oracle_ops.py).  Compared with the single-rank oracle over all
ranks' tokens ("BioNeMo Uses Grouped Kernels and MXFP8", "Launching the
recipe": expert parallelism, data x expert parallel sizes = GPU count):
  * bit-exact: split sizes, the rows each rank receives (in the single-rank
    grouped order), their MXFP8 codes and scales (row-wise and per-expert
    token-column-wise);
  * y, dx, dprobs per rank and each rank's experts' dW_gate_up, dW_down:
    the same fp64 arithmetic on the same rows, equal to 1e-12 relative
    (BLAS may block the products differently for differently placed rows).
Not measured across GPUs: the exchange runs here between CPU ranks, and the
single-GPU test (test_gpu_ep.py) runs the ranks as virtual ranks on one device."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import synthetic
from oracle import moe, mx


def _port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _case(G, T_loc, H, I, E, k, seed):
    inp = synthetic.make_case(G * T_loc, H, I, E, k, seed=seed, empty_experts=(E - 1,))
    return {n: (v.double().numpy() if n != "logits" else v.numpy()) for n, v in inp.items()
            if isinstance(v, torch.Tensor)}


def _rank(rank, G, port, shape, seed, out_q, payload="bf16"):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    from ep_oracle_ops import OracleOps
    from mxfp8_grouped_gemm_gb300 import ep
    os.environ["MASTER_ADDR"], os.environ["MASTER_PORT"] = "127.0.0.1", str(port)
    dist.init_process_group("gloo", rank=rank, world_size=G)
    try:
        T_loc, H, I, E, k = shape
        c = _case(G, T_loc, H, I, E, k, seed)
        sl = slice(rank * T_loc, (rank + 1) * T_loc)
        ids, probs = moe.route_topk(c["logits"][sl], k)
        comm = ep.TorchComm(device="cpu")
        n = E // G
        layer = ep.ExpertParallelMLP(comm, T_loc, H, I, E, k, ops=OracleOps(H, I, n))
        mine = slice(rank * n, (rank + 1) * n)
        y = layer.forward(torch.from_numpy(c["x"][sl]), torch.from_numpy(ids), torch.from_numpy(probs),
                          c["w_gate_up"][mine], c["w_down"][mine], payload=payload)
        if payload == "mxfp8":
            out_q.put((rank, {"y": y.numpy(), "split": layer._ctx["split"], **layer.ops.seen_mx}))
            return
        dx, dwgu, dwd, dprobs = layer.backward(torch.from_numpy(c["dy"][sl]))
        seen = layer.ops.seen
        out_q.put((rank, {"y": y.numpy(), "dx": dx.numpy(), "dwgu": dwgu.numpy(), "dwd": dwd.numpy(),
                          "dprobs": dprobs.numpy(), "split": layer._ctx["split"],
                          "counts_recv": layer._ctx["counts_recv"], **seen}))
    finally:
        dist.destroy_process_group()


def _run_ranks(G, shape, seed, payload="bf16"):
    ctx_mp = mp.get_context("spawn")
    q = ctx_mp.Queue()
    port = _port()
    procs = [ctx_mp.Process(target=_rank, args=(r, G, port, shape, seed, q, payload)) for r in range(G)]
    for p in procs:
        p.start()
    res = {}
    import queue
    while len(res) < G:
        try:
            r, o = q.get(timeout=5)
            res[r] = o
        except queue.Empty:
            dead = [p.exitcode for p in procs if p.exitcode not in (None, 0)]
            if dead:
                for p in procs:
                    p.kill()
                pytest.fail(f"a rank exited with {dead[0]}")
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return res


@pytest.mark.parametrize("G", [2, 4])
def test_expert_parallel_equals_single_rank(G):
    T_loc, H, I, E, k = 96, 64, 96, 8, 2
    seed = 40 + G
    res = _run_ranks(G, (T_loc, H, I, E, k), seed)

    c = _case(G, T_loc, H, I, E, k, seed)
    ids, probs = moe.route_topk(c["logits"], k)
    ctx = moe.mlp_fwd(c["x"], ids, probs, c["w_gate_up"], c["w_down"])
    g = moe.mlp_bwd(ctx, c["dy"])
    perm = ctx["perm"]
    n = E // G
    for r in range(G):
        o = res[r]
        sl = slice(r * T_loc, (r + 1) * T_loc)
        # this rank's tokens' split sizes, and what it received for its experts
        ids_r, _ = moe.route_topk(c["logits"][sl], k)
        assert np.array_equal(o["split"], np.bincount(ids_r.reshape(-1), minlength=E))
        assert np.array_equal(o["split_local"], perm["split_sizes"][r * n:(r + 1) * n])
        a, b = perm["offsets"][r * n], perm["offsets"][(r + 1) * n]
        assert np.array_equal(o["x_grouped"], ctx["x_perm"][a:b])            # the single-rank grouped rows
        codes, scales = mx.quantize_blocks(ctx["x_perm"][a:b])
        assert np.array_equal(o["row_codes"][0], codes) and np.array_equal(o["row_codes"][1], scales)
        for e in range(n):
            ea, eb = perm["offsets"][r * n + e], perm["offsets"][r * n + e + 1]
            if eb == ea:
                assert o["col_codes"][e] is None
                continue
            cc, cs = mx.quantize_group_columns(ctx["x_perm"][ea:eb])
            assert np.array_equal(o["col_codes"][e][0], cc) and np.array_equal(o["col_codes"][e][1], cs)
        np.testing.assert_allclose(o["y"], ctx["y"][sl], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(o["dx"], g["dx"][sl], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(o["dprobs"], g["dprobs"][sl], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(o["dwgu"], g["dw_gate_up"][r * n:(r + 1) * n], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(o["dwd"], g["dw_down"][r * n:(r + 1) * n], rtol=1e-12, atol=1e-14)
    # the empty expert (E - 1) lives on the last rank: its dW is exactly zero
    assert not res[G - 1]["dwgu"][-1].any() and not res[G - 1]["dwd"][-1].any()


def test_receive_order_and_partition():
    from mxfp8_grouped_gemm_gb300 import ep
    assert [list(r) for r in ep.partition(8, 4)] == [[0, 1], [2, 3], [4, 5], [6, 7]]
    with pytest.raises(ValueError):
        ep.partition(6, 4)
    counts = np.array([[2, 0, 1], [1, 3, 0]])                 # from source 0, 1 for local experts 0..2
    order = ep.receive_order(counts)
    # received: s0: e0 e0 e2 | s1: e0 e1 e1 e1 -> grouped: e0 (s0 s0 s1), e1 (s1 s1 s1), e2 (s0)
    assert order.tolist() == [0, 1, 3, 4, 5, 6, 2]
    assert np.array_equal(ep.inverse(order)[order], np.arange(7))


def test_expert_parallel_mxfp8_payload_inference():
    """The inference forward that ships each token's row-wise MXFP8 codes and
    scales: every rank receives, bit for bit, the codes and scales the single
    rank computes for its experts' grouped rows, and y equals the single-rank
    oracle's."""
    G, T_loc, H, I, E, k = 2, 96, 64, 96, 8, 2
    seed = 47
    res = _run_ranks(G, (T_loc, H, I, E, k), seed, payload="mxfp8")
    c = _case(G, T_loc, H, I, E, k, seed)
    ids, probs = moe.route_topk(c["logits"], k)
    ctx = moe.mlp_fwd(c["x"], ids, probs, c["w_gate_up"], c["w_down"])
    perm = ctx["perm"]
    n = E // G
    for r in range(G):
        o = res[r]
        a, b = perm["offsets"][r * n], perm["offsets"][(r + 1) * n]
        codes, scales = mx.quantize_blocks(ctx["x_perm"][a:b])
        assert np.array_equal(o["codes"], codes) and np.array_equal(o["scales"], scales)
        sl = slice(r * T_loc, (r + 1) * T_loc)
        np.testing.assert_allclose(o["y"], ctx["y"][sl], rtol=1e-12, atol=1e-14)
