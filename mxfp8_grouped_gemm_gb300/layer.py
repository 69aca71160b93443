"""GroupedMLP: owns the caller-side buffers (saved activations, scratch,
device status word) of one grouped expert MLP shape and runs the library's
route -> forward -> backward calls on the current stream."""
from __future__ import annotations

import torch

from . import _lib


def precision_is_not_mx(layer) -> bool:
    return layer.precision != "mxfp8"


def gu_rows_from_tiles(t: torch.Tensor, m_cap: int, I: int) -> torch.Tensor:
    """[m_cap, 2I] rows from the MXFP8 path's saved g|u tiles (flat, m_cap*2I
    values): the tile of rows 32rb.. and gate columns 32cb.. (cb < I/32) starts
    at element (rb*I/32 + cb)*2048 and holds the gate block, then the up block,
    each as two 16-column halves of 32 rows x 16 values."""
    t = t.view(m_cap // 32, I // 32, 2, 2, 32, 16)          # [rb][cb][gate/up][half][row][16]
    return t.permute(0, 4, 2, 1, 3, 5).reshape(m_cap, 2 * I)  # [rb][row][gate/up][cb][half][16]


class GroupedMLP:
    """precision "mxfp8" (the path), "bf16" (the like-for-like BF16 reference) or
    "fp8" (per-tensor FP8, one scale per expert tensor); bf16 and fp8 need H and
    I multiples of 256."""

    def __init__(self, T: int, H: int, I: int, E: int, k: int, device="cuda", precision: str = "mxfp8"):
        if precision not in ("mxfp8", "bf16", "fp8"):
            raise ValueError(f"precision must be 'mxfp8', 'bf16' or 'fp8', got {precision!r}")
        self.T, self.H, self.I, self.E, self.k = T, H, I, E, k
        self.precision = precision
        self.bf16 = precision == "bf16"
        self.fp8 = precision == "fp8"
        self.device = torch.device(device)
        if self.bf16:
            saved = _lib.mxg_mlp_bf16_saved_bytes(T, H, I, E, k)
            ws = _lib.mxg_mlp_bf16_workspace_bytes(T, H, I, E, k)
        elif self.fp8:
            saved = _lib.mxg_mlp_fp8_saved_bytes(T, H, I, E, k)
            ws = _lib.mxg_mlp_fp8_workspace_bytes(T, H, I, E, k)
        else:
            saved = _lib.mxg_mlp_saved_bytes(T, H, I, E, k)
            ws = _lib.mxg_mlp_workspace_bytes(T, H, I, E, k)
        if saved == 0 or ws == 0:
            raise ValueError(f"unsupported {precision} shape T={T} H={H} I={I} E={E} k={k} "
                             f"(H, I multiples of {128 if precision == 'mxfp8' else 256}; k <= E <= 256)")
        self.saved = torch.empty(saved, dtype=torch.uint8, device=self.device)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=self.device)
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.ids = torch.empty((T, k), dtype=torch.int32, device=self.device)
        self.probs = torch.empty((T, k), dtype=torch.float32, device=self.device)
        self.y = torch.empty((T, H), dtype=torch.bfloat16, device=self.device)
        self.split_sizes = torch.empty(E, dtype=torch.int32, device=self.device)
        self.dx = torch.empty((T, H), dtype=torch.bfloat16, device=self.device)
        self.dw_gate_up = torch.empty((E, 2 * I, H), dtype=torch.bfloat16, device=self.device)
        self.dw_down = torch.empty((E, H, I), dtype=torch.bfloat16, device=self.device)
        self.dprobs = torch.empty((T, k), dtype=torch.float32, device=self.device)
        self.weight_cache = None          # MXFP8 weights kept across micro-batches (quantize_weights)
        self._fwd_cached = False

    def route(self, logits, stream=None):
        """Top-k routing into this object's ids/probs buffers."""
        return _lib.mxg_route_topk(logits, self.k, self.ids, self.probs, stream=stream)

    def quantize_weights(self, w_gate_up, w_down, stream=None):
        """Quantise the weights once into this layer's weight cache (MXFP8 path):
        forward calls given no weights then read it, e.g. for every micro-batch
        of one optimizer step."""
        if precision_is_not_mx(self):
            raise NotImplementedError("the weight cache holds MXFP8 weights")
        self.weight_cache = _lib.mxg_mlp_quantize_weights(w_gate_up, w_down, self.weight_cache, stream=stream)
        return self.weight_cache

    def forward(self, x, ids, probs, w_gate_up=None, w_down=None, save_for_backward=True, stream=None, stage=None,
                y=None):
        """w_gate_up / w_down None: use the weight cache (quantize_weights)."""
        cached = w_gate_up is None and w_down is None
        if cached and self.weight_cache is None:
            raise ValueError("no weights given and no weight cache: call quantize_weights first")
        self._fwd_cached = cached
        return _lib.mxg_grouped_mlp_fwd(x, ids, probs, w_gate_up, w_down, self.saved, self.workspace,
                                        self.dev_status, y=self.y if y is None else y,
                                        split_sizes=self.split_sizes, save_for_backward=save_for_backward,
                                        stream=stream, stage=stage, bf16=self.bf16, fp8=self.fp8,
                                        weight_cache=self.weight_cache if cached else None)

    def backward(self, dy, stream=None, stage=None, dx=None, main_grad=None):
        """main_grad = (fp32 [E, 2I, H], fp32 [E, H, I]): add the weight gradients
        into these (returned in place of dW_gate_up, dW_down)."""
        return _lib.mxg_grouped_mlp_bwd(dy, self.saved, self.workspace, self.dev_status, self.E, self.I, self.k,
                                        dx=self.dx if dx is None else dx,
                                        dw_gate_up=None if main_grad is not None else self.dw_gate_up,
                                        dw_down=None if main_grad is not None else self.dw_down,
                                        dprobs=self.dprobs, stream=stream, stage=stage, bf16=self.bf16,
                                        fp8=self.fp8, weight_cache=self.weight_cache if self._fwd_cached else None,
                                        main_grad=main_grad)

    def step(self, logits, x, w_gate_up, w_down, dy, stream=None):
        """One pass of the whole path: route, forward (saving for backward), backward."""
        ids, probs = self.route(logits, stream=stream)
        self.forward(x, ids, probs, w_gate_up, w_down, True, stream=stream)
        return self.backward(dy, stream=stream)

    def status(self) -> int:
        return int(self.dev_status.item())

    def gu_view(self) -> torch.Tensor:
        """The gate-up GEMM output kept in the saved buffer (MXFP8 path), as a
        bf16 [m_cap, 2I] tensor in row order (gate columns, then up columns):
        a copy of the buffer's 32 x 32 tiles (gu_rows_from_tiles)."""
        if precision_is_not_mx(self):
            raise NotImplementedError("gu_view reads the MXFP8 path's saved layout")
        base = self.saved.data_ptr()
        off = _lib.mxg_mlp_saved_view(self.saved, self.T, self.H, self.I, self.E, self.k, 0) - base
        m_cap = self.padded_rows_capacity()
        return gu_rows_from_tiles(self.saved[off:off + m_cap * 2 * self.I * 2].view(torch.bfloat16), m_cap, self.I)

    def padded_offsets(self) -> torch.Tensor:
        if precision_is_not_mx(self):
            raise NotImplementedError("padded_offsets reads the MXFP8 path's saved layout")
        base = self.saved.data_ptr()
        off = _lib.mxg_mlp_saved_view(self.saved, self.T, self.H, self.I, self.E, self.k, 1) - base
        return self.saved[off:off + 4 * (self.E + 1)].view(torch.int32)

    def padded_rows_capacity(self) -> int:
        return _lib.mxg_mlp_row_capacity(self.T, self.k, self.E)


class GroupedExperts:
    """The expert MLP on rows that arrive already grouped by expert (the
    GroupedLinear call with split_sizes: an expert-parallel dispatcher's
    output, or rows the caller permuted).  Buffers are sized for up to
    ``max_rows`` rows; each call passes its own row count."""

    def __init__(self, max_rows: int, H: int, I: int, E: int, device="cuda"):
        self.R_max, self.H, self.I, self.E = max_rows, H, I, E
        self.device = torch.device(device)
        saved = _lib.mxg_mlp_grouped_saved_bytes(max_rows, H, I, E)
        ws = _lib.mxg_mlp_grouped_workspace_bytes(max_rows, H, I, E)
        if saved == 0 or ws == 0:
            raise ValueError(f"unsupported grouped shape R={max_rows} H={H} I={I} E={E}")
        self.saved = torch.empty(saved, dtype=torch.uint8, device=self.device)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=self.device)
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.weight_cache = None
        self._R = 0
        self._cached = False

    def quantize_weights(self, w_gate_up, w_down, stream=None):
        self.weight_cache = _lib.mxg_mlp_quantize_weights(w_gate_up, w_down, self.weight_cache, stream=stream)
        return self.weight_cache

    def forward(self, x, split_sizes, probs, w_gate_up=None, w_down=None, save_for_backward=True, y=None,
                stream=None):
        """x bf16 [R, H] grouped by expert, split_sizes int32 [E] (device),
        probs fp32 [R] -> per-row outputs y [R, H]."""
        R = x.shape[0]
        if R > self.R_max:
            raise ValueError(f"{R} rows exceed the buffers' {self.R_max}")
        cached = w_gate_up is None and w_down is None
        if cached and self.weight_cache is None:
            raise ValueError("no weights given and no weight cache: call quantize_weights first")
        self._R, self._cached = R, cached
        return _lib.mxg_grouped_mlp_fwd_grouped(x, split_sizes, probs.reshape(R), w_gate_up, w_down, self.saved,
                                                self.workspace, self.dev_status, y=y,
                                                save_for_backward=save_for_backward,
                                                weight_cache=self.weight_cache if cached else None, stream=stream)

    def forward_mx(self, xq, xs, split_sizes, probs, w_gate_up=None, w_down=None, y=None, stream=None):
        """Inference forward on grouped rows given as row-wise MXFP8 (codes xq
        uint8 [R, H], canonical scales xs uint8 [R, H/32]); no backward."""
        R = xq.shape[0]
        if R > self.R_max:
            raise ValueError(f"{R} rows exceed the buffers' {self.R_max}")
        cached = w_gate_up is None and w_down is None
        if cached and self.weight_cache is None:
            raise ValueError("no weights given and no weight cache: call quantize_weights first")
        self._R = -1                                   # nothing saved for a backward
        return _lib.mxg_grouped_mlp_fwd_grouped_mx(xq, xs, split_sizes, probs.reshape(R), w_gate_up, w_down,
                                                   self.saved, self.workspace, self.dev_status, self.H, y=y,
                                                   weight_cache=self.weight_cache if cached else None,
                                                   stream=stream)

    def backward(self, dy, dx=None, dw_gate_up=None, dw_down=None, dprobs=None, main_grad=None, stream=None):
        """dy bf16 [R, H] (per row) -> dx [R, H], dW_gate_up, dW_down, dprobs [R, 1]."""
        R = dy.shape[0]
        if R != self._R:
            raise ValueError("backward rows differ from the forward's")
        return _lib.mxg_grouped_mlp_bwd(dy, self.saved, self.workspace, self.dev_status, self.E, self.I, 1, dx=dx,
                                        dw_gate_up=dw_gate_up, dw_down=dw_down, dprobs=dprobs, stream=stream,
                                        weight_cache=self.weight_cache if self._cached else None,
                                        main_grad=main_grad)

    def status(self) -> int:
        return int(self.dev_status.item())
