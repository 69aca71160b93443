"""Host-side stand-in for the expert-parallel layer's compute steps, built on
the CPU oracle (test infrastructure only: the package has no CPU path).

Same methods as mxfp8_grouped_gemm_gb300.ep.CudaOps, in fp64 numpy on CPU
tensors: the permute is oracle.moe.permute, the gathers are plain indexing,
the combine a plain sum, and the experts' forward and backward are
oracle.moe.mlp_fwd / mlp_bwd on the grouped rows with k = 1 (each row its own
token, its expert given by position).  The exchanged tensors are the ones the
GPU path exchanges (rows of x, dy, y, dx and the per-row probabilities), so
the expert-parallel control flow and its all-to-all steps run unchanged."""
from __future__ import annotations

import numpy as np
import torch

from oracle import moe, mx


class OracleOps:
    def __init__(self, H: int, I: int, E_local: int):
        self.H, self.I, self.E_local = H, I, E_local
        self.seen = {}

    def permute(self, ids, E):
        p = moe.permute(ids.numpy(), E)
        return {n: torch.from_numpy(np.asarray(v)) for n, v in p.items()}

    def counts_to_host(self, split_sizes):
        return split_sizes.numpy().astype(np.int64)

    def index(self, idx):
        return torch.from_numpy(np.asarray(idx, dtype=np.int64))

    def gather(self, src, index, div=1):
        return src[index.long() // div]

    def combine(self, rows, row_of_src, k):
        r = row_of_src.numpy().reshape(-1, k)
        R = rows.numpy()
        y = np.zeros((r.shape[0], R.shape[1]))
        for j in range(k):
            y += R[r[:, j]]
        return torch.from_numpy(y)

    def experts_forward(self, x_rows, split_local, probs_rows, w_gate_up, w_down):
        R = x_rows.shape[0]
        ids = np.repeat(np.arange(self.E_local), split_local).reshape(R, 1).astype(np.int32)
        x = x_rows.numpy()
        self.seen = {"x_grouped": x.copy(), "split_local": np.asarray(split_local).copy()}
        self.ctx = moe.mlp_fwd(x, ids, probs_rows.numpy().reshape(R, 1), np.asarray(w_gate_up),
                               np.asarray(w_down))
        # the MXFP8 codes the experts' GEMMs read: row-wise of every row, and
        # token-column-wise per local expert group
        self.seen["row_codes"] = mx.quantize_blocks(x)
        off = np.concatenate([[0], np.cumsum(split_local)])
        self.seen["col_codes"] = [mx.quantize_group_columns(x[off[e]:off[e + 1]]) if off[e + 1] > off[e] else None
                                  for e in range(self.E_local)]
        return torch.from_numpy(self.ctx["y"])

    def quantize_rows(self, x):
        c, s = mx.quantize_blocks(x.numpy())
        return torch.from_numpy(c), torch.from_numpy(s)

    def experts_forward_mx(self, xq_rows, xs_rows, split_local, probs_rows, w_gate_up, w_down):
        # the dequantised rows lie on the MX grid with the same block maxima,
        # so the oracle's quantisation reproduces exactly these codes
        x = mx.dequantize_blocks(xq_rows.numpy(), xs_rows.numpy())
        self.seen_mx = {"codes": xq_rows.numpy().copy(), "scales": xs_rows.numpy().copy()}
        return self.experts_forward(torch.from_numpy(x), split_local, probs_rows, w_gate_up, w_down)

    def experts_backward(self, dy_rows):
        g = moe.mlp_bwd(self.ctx, dy_rows.numpy())
        return (torch.from_numpy(g["dx"]), torch.from_numpy(g["dw_gate_up"]), torch.from_numpy(g["dw_down"]),
                torch.from_numpy(g["dprobs"].reshape(-1)))

    def check(self):
        pass
