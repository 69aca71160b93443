"""Expert parallelism for the grouped expert MLP: the E experts of one MoE
layer spread over G ranks, E/G consecutive experts each, and every rank's
tokens exchanged with the ranks that hold their experts.  The recipe scales
Mixtral training this way ("BioNeMo Uses Grouped Kernels and MXFP8",
"Launching the recipe": expert parallelism of 8, data x expert parallel
sizes equal to the GPU count; "How BioNeMo cuts overhead in biological AI
training", "What NVIDIA measured").

One rank's forward (tokens of this rank, experts of every rank):
  1. permute its tokens by expert (mxg_route_permute): rows come out grouped
     by expert and therefore by the rank that holds the expert;
  2. exchange the row counts: rank s sends rank g the E/G counts of g's
     experts (an all-to-all of G x E/G integers, on the host side);
  3. gather the token rows and their routing probabilities in permuted order
     (mxg_gather_rows) and all-to-all-v them; rows arrive grouped by source
     rank, inside each source by local expert;
  4. reorder them expert-major (for each local expert: source 0, 1, ...), which
     is the order a single GPU holding every expert would give them (its
     counting sort is stable in the global flat index t*k + j, tokens of rank
     s being s*T + t); one gather with an index built from the count matrix;
  5. the grouped MLP on the local experts (mxg_grouped_mlp_fwd_grouped, one
     count per local expert);
  6. the inverse reorder of the output rows and the all-to-all-v back;
  7. the combine on the source rank (mxg_combine).
The backward mirrors it: dy rows go out like x rows (step 3-4), dx rows and the
per-row d(probability) come back (6-7); each rank keeps its own experts'
weight gradients.

The dispatched payload for training is the bf16 rows: the wgrad operand of
W_gate_up is x quantised in blocks of 32 tokens of an expert's group, and
that group is only complete on the receiving rank, so the quantisation has
to happen there from the bf16 values.  An inference forward (payload
"mxfp8") ships the F3 output instead: each token's row-wise MXFP8 codes and
E8M0 scales (H + H/32 bytes instead of 2H), quantised once per token on the
source rank; row-wise blocks lie inside a row, so these are the codes the
receiving rank would have computed, and the forward is the same bit for bit.

The exchange runs through a communicator object (TorchComm wraps a
torch.distributed process group: NCCL for CUDA tensors, gloo for CPU ones);
the compute through an ops object (CudaOps: the library's kernels).  Both
are parameters so the same control flow can run with host-side stand-ins;
the package itself has no CPU path.
"""
from __future__ import annotations

import numpy as np
import torch

from . import _lib
from .layer import GroupedExperts


class TorchComm:
    """All-to-all exchanges over a torch.distributed process group."""

    def __init__(self, group=None, device: torch.device | str = "cpu"):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)
        self.device = torch.device(device)

    def all_to_all_counts(self, send: np.ndarray) -> np.ndarray:
        """send [G, n] int64: row g goes to rank g; returns [G, n], row s from rank s."""
        t = torch.from_numpy(np.ascontiguousarray(send, dtype=np.int64)).to(self.device)
        out = torch.empty_like(t)
        self.dist.all_to_all_single(out, t, group=self.group)
        return out.cpu().numpy()

    def all_to_all_rows(self, send: torch.Tensor, send_splits: list[int], recv_splits: list[int]) -> torch.Tensor:
        """Rows send[sum(send_splits[:g]) : ...+send_splits[g]] go to rank g;
        returns the rows received, source rank by source rank."""
        out = torch.empty((int(sum(recv_splits)),) + tuple(send.shape[1:]), dtype=send.dtype, device=send.device)
        self.dist.all_to_all_single(out, send.contiguous(), [int(v) for v in recv_splits],
                                    [int(v) for v in send_splits], group=self.group)
        return out


class CudaOps:
    """The library's kernels for the steps of the expert-parallel layer."""

    def __init__(self, max_rows: int, H: int, I: int, E_local: int, device="cuda"):
        self.device = torch.device(device)
        self.H, self.I, self.E_local = H, I, E_local
        self.experts = GroupedExperts(max(max_rows, 1), H, I, E_local, device=self.device)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)

    def permute(self, ids: torch.Tensor, E: int) -> dict:
        return _lib.mxg_route_permute(ids, E, self.status)

    def quantize_rows(self, x: torch.Tensor):
        """Row-wise MXFP8 of x [T, H] (blocks of 32 along H): codes uint8
        [T, H] and canonical scales uint8 [T, H/32]."""
        T, H = x.shape
        off = torch.tensor([0, T], dtype=torch.int32, device=self.device)
        q = _lib.mxg_mxfp8_quantize_grouped(x, off, self.status, row=True, col=False)
        return q["q_row"][:T], q["s_row"].view(-1, H // 32)[:T]

    def counts_to_host(self, split_sizes: torch.Tensor) -> np.ndarray:
        return split_sizes.cpu().numpy().astype(np.int64)

    def index(self, idx: np.ndarray) -> torch.Tensor:
        return torch.from_numpy(np.ascontiguousarray(idx, dtype=np.int32)).to(self.device)

    def gather(self, src: torch.Tensor, index: torch.Tensor, div: int = 1) -> torch.Tensor:
        if index.numel() == 0:
            return src.new_empty((0,) + tuple(src.shape[1:]))
        return _lib.mxg_gather_rows(src, index, self.status, div=div)

    def combine(self, rows: torch.Tensor, row_of_src: torch.Tensor, k: int) -> torch.Tensor:
        T = row_of_src.numel() // k
        if rows.shape[0] == 0:
            return torch.zeros((T, self.H), dtype=torch.bfloat16, device=self.device)
        return _lib.mxg_combine(rows, row_of_src, k, self.status)

    def experts_forward(self, x_rows, split_local: np.ndarray, probs_rows, w_gate_up, w_down):
        self._R = x_rows.shape[0]
        if self._R == 0:
            return x_rows.new_empty((0, self.H))
        split = torch.from_numpy(split_local.astype(np.int32)).to(self.device)
        return self.experts.forward(x_rows, split, probs_rows, w_gate_up, w_down).clone()

    def experts_forward_mx(self, xq_rows, xs_rows, split_local: np.ndarray, probs_rows, w_gate_up, w_down):
        self._R = -1                                  # inference: nothing saved for a backward
        if xq_rows.shape[0] == 0:
            return torch.empty((0, self.H), dtype=torch.bfloat16, device=self.device)
        split = torch.from_numpy(split_local.astype(np.int32)).to(self.device)
        return self.experts.forward_mx(xq_rows, xs_rows, split, probs_rows, w_gate_up, w_down).clone()

    def experts_backward(self, dy_rows):
        if self._R == 0:
            z = torch.zeros
            return (dy_rows.new_empty((0, self.H)),
                    z((self.E_local, 2 * self.I, self.H), dtype=torch.bfloat16, device=self.device),
                    z((self.E_local, self.H, self.I), dtype=torch.bfloat16, device=self.device),
                    torch.empty((0,), dtype=torch.float32, device=self.device))
        dx, dwgu, dwd, dp = self.experts.backward(dy_rows)
        return dx.clone(), dwgu.clone(), dwd.clone(), dp.reshape(-1).clone()

    def check(self):
        for st in (int(self.status.item()), self.experts.status()):
            if st != 0:
                raise _lib.MxgError("expert-parallel step", st)


def partition(E: int, world: int) -> list[range]:
    """Experts of each rank: E/G consecutive ids (E divisible by G)."""
    if E % world:
        raise ValueError(f"{E} experts do not split evenly over {world} ranks")
    n = E // world
    return [range(g * n, (g + 1) * n) for g in range(world)]


def receive_order(counts_recv: np.ndarray) -> np.ndarray:
    """Index that reorders rows received source-major (source s: its rows of
    local expert 0, 1, ... in turn) into expert-major order (local expert e:
    source 0's rows, then source 1's, ...): grouped[new] = received[order[new]]."""
    G, n = counts_recv.shape
    base = np.zeros((G, n), dtype=np.int64)           # start of (s, e) in the received buffer
    flat = counts_recv.reshape(-1)
    starts = np.concatenate([[0], np.cumsum(flat)[:-1]])
    base[:] = starts.reshape(G, n)
    parts = [np.arange(base[s, e], base[s, e] + counts_recv[s, e]) for e in range(n) for s in range(G)]
    return np.concatenate(parts).astype(np.int64) if parts else np.zeros(0, dtype=np.int64)


def inverse(order: np.ndarray) -> np.ndarray:
    inv = np.empty_like(order)
    inv[order] = np.arange(order.size)
    return inv


class ExpertParallelMLP:
    """One rank's share of an expert-parallel grouped MLP layer.

    comm : TorchComm (or an object with the same two methods)
    ops  : CudaOps (or an object with the same methods); built for this rank's
           experts when None
    Every rank holds T tokens (its data-parallel batch) and the weights of its
    E/G experts: w_gate_up [E/G, 2I, H], w_down [E/G, H, I]."""

    def __init__(self, comm, T: int, H: int, I: int, E: int, k: int, ops=None, device="cuda"):
        self.comm = comm
        self.G, self.rank = comm.world, comm.rank
        self.T, self.H, self.I, self.E, self.k = T, H, I, E, k
        self.experts_of = partition(E, self.G)
        self.E_local = E // self.G
        # a rank receives at most min(k, E/G) rows of each token of every rank
        self.max_rows = self.G * T * min(k, self.E_local)
        self.ops = ops if ops is not None else CudaOps(self.max_rows, H, I, self.E_local, device=device)

    # ---------------------------------------------------------------- forward
    def forward(self, x, ids, probs, w_gate_up, w_down, payload: str = "bf16"):
        """payload "bf16": the rows as bf16 (training); "mxfp8": each token's
        row-wise codes and scales (inference: no backward after it)."""
        if payload not in ("bf16", "mxfp8"):
            raise ValueError(f"payload must be 'bf16' or 'mxfp8', got {payload!r}")
        ops, G, n, k = self.ops, self.G, self.E_local, self.k
        perm = ops.permute(ids, self.E)
        split = ops.counts_to_host(perm["split_sizes"])                 # [E] rows per expert, this rank's tokens
        counts_send = split.reshape(G, n)
        counts_recv = self.comm.all_to_all_counts(counts_send)          # [G, n]: from source s, per local expert
        send_splits = counts_send.sum(axis=1).tolist()
        recv_splits = counts_recv.sum(axis=1).tolist()
        p_rows = ops.gather(probs.reshape(-1), perm["src_of_row"])    # permuted order = destination order
        p_recv = self.comm.all_to_all_rows(p_rows, send_splits, recv_splits)
        order = receive_order(counts_recv)
        order_t = ops.index(order)
        p_g = ops.gather(p_recv, order_t)
        split_local = counts_recv.sum(axis=0)                           # rows per local expert
        x_g = None
        if payload == "bf16":
            x_rows = ops.gather(x, perm["src_of_row"], div=k)
            x_g = ops.gather(self.comm.all_to_all_rows(x_rows, send_splits, recv_splits), order_t)
            y_g = ops.experts_forward(x_g, split_local, p_g, w_gate_up, w_down)
        else:
            xq_tok, xs_tok = ops.quantize_rows(x)                      # once per token, on the source rank
            q_rows = ops.gather(xq_tok, perm["src_of_row"], div=k)
            s_rows = ops.gather(xs_tok, perm["src_of_row"], div=k)
            q_g = ops.gather(self.comm.all_to_all_rows(q_rows, send_splits, recv_splits), order_t)
            s_g = ops.gather(self.comm.all_to_all_rows(s_rows, send_splits, recv_splits), order_t)
            y_g = ops.experts_forward_mx(q_g, s_g, split_local, p_g, w_gate_up, w_down)
        back_t = ops.index(inverse(order))
        y_back = self.comm.all_to_all_rows(ops.gather(y_g, back_t), recv_splits, send_splits)
        y = ops.combine(y_back, perm["row_of_src"], k)
        self._ctx = {"perm": perm, "send_splits": send_splits, "recv_splits": recv_splits, "order_t": order_t,
                     "back_t": back_t, "split": split, "counts_recv": counts_recv, "x_grouped": x_g,
                     "split_local": split_local, "payload": payload}
        return y

    # --------------------------------------------------------------- backward
    def backward(self, dy):
        ops, c, k = self.ops, self._ctx, self.k
        if c["payload"] != "bf16":
            raise RuntimeError("a forward with the mxfp8 payload is inference only: it has no backward")
        perm = c["perm"]
        dy_rows = ops.gather(dy, perm["src_of_row"], div=k)
        dy_recv = self.comm.all_to_all_rows(dy_rows, c["send_splits"], c["recv_splits"])
        dy_g = ops.gather(dy_recv, c["order_t"])
        dx_g, dw_gate_up, dw_down, dp_g = ops.experts_backward(dy_g)
        dx_back = self.comm.all_to_all_rows(ops.gather(dx_g, c["back_t"]), c["recv_splits"], c["send_splits"])
        dp_back = self.comm.all_to_all_rows(ops.gather(dp_g, c["back_t"]), c["recv_splits"], c["send_splits"])
        dx = ops.combine(dx_back, perm["row_of_src"], k)
        dprobs = ops.gather(dp_back, perm["row_of_src"]).reshape(-1, k)
        return dx, dw_gate_up, dw_down, dprobs
