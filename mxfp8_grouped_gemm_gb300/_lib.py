"""ctypes binding of libmxg.so (include/mxg.h).  Argument marshalling only:
every step of the path runs in the library's CUDA kernels.  The functions
carry the C names; torch tensors provide device memory and the stream.

There is no fallback: if the library is missing or the tensors are not CUDA
tensors, the call raises."""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmxg.so")

MXG_LAYOUT_CANONICAL = 0
MXG_LAYOUT_MMA = 1

STATUS = {
    0: "MXG_OK", 1: "MXG_ERR_ARG", 2: "MXG_ERR_SHAPE", 3: "MXG_ERR_ALIGN", 4: "MXG_ERR_ARCH",
    5: "MXG_ERR_WORKSPACE", 6: "MXG_ERR_CUDA", 16: "MXG_ERR_EXPERT_ID", 17: "MXG_ERR_OFFSETS",
    18: "MXG_ERR_TIMEOUT", 19: "MXG_ERR_INDEX",
}

EXPORTS = [
    "mxg_status_string", "mxg_device_supported", "mxg_launch_count", "mxg_route_topk",
    "mxg_route_permute_workspace_bytes", "mxg_route_permute", "mxg_mxfp8_quantize", "mxg_grouped_gemm",
    "mxg_grouped_gemm_wgrad", "mxg_mlp_saved_bytes", "mxg_mlp_workspace_bytes", "mxg_grouped_mlp_fwd",
    "mxg_grouped_mlp_bwd", "mxg_mlp_saved_view", "mxg_grouped_mlp_fwd_stage", "mxg_grouped_mlp_bwd_stage",
    "mxg_route_permute_noalloc_max_entries", "mxg_route_permute_noalloc", "mxg_mlp_group_align",
    "mxg_mlp_row_capacity", "mxg_debug_grouped_gemm_stall", "mxg_router_fwd", "mxg_router_bwd_workspace_bytes",
    "mxg_router_bwd", "mxg_mlp_bf16_saved_bytes", "mxg_mlp_bf16_workspace_bytes", "mxg_grouped_mlp_bf16_fwd",
    "mxg_grouped_mlp_bf16_bwd", "mxg_grouped_mlp_bf16_fwd_stage", "mxg_grouped_mlp_bf16_bwd_stage",
    "mxg_mlp_weight_cache_bytes", "mxg_mlp_quantize_weights", "mxg_mlp_saved_bytes_cached",
    "mxg_mlp_fp8_saved_bytes", "mxg_mlp_fp8_workspace_bytes", "mxg_grouped_mlp_fp8_fwd", "mxg_grouped_mlp_fp8_bwd",
    "mxg_grouped_mlp_fp8_fwd_stage", "mxg_grouped_mlp_fp8_bwd_stage", "mxg_mlp_fp8_saved_view",
    "mxg_mlp_workspace_view", "mxg_mlp_weight_cache_view", "mxg_bench_mxfp8_mma_peak",
    "mxg_mxfp8_grouped_rows_capacity", "mxg_mxfp8_quantize_grouped", "mxg_gather_rows", "mxg_combine",
    "mxg_mlp_grouped_saved_bytes", "mxg_mlp_grouped_workspace_bytes", "mxg_grouped_mlp_fwd_grouped",
    "mxg_router_fwd_permute", "mxg_grouped_mlp_fwd_grouped_mx",
]

FWD_STAGES = ["permute", "quant_weights", "quant_x", "gate_up", "down", "combine"]
BWD_STAGES = ["quant_dy", "dgrad_down", "wgrad_down", "dgrad_gate_up", "wgrad_gate_up", "combine_dx", "dprobs"]


class MxgError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} -> {STATUS.get(code, code)}: {status_string(code)}")


class MlpFwdArgs(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("x", ctypes.c_void_p), ("ids", ctypes.c_void_p),
                ("probs", ctypes.c_void_p), ("w_gate_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p),
                ("y", ctypes.c_void_p), ("split_sizes", ctypes.c_void_p), ("saved", ctypes.c_void_p),
                ("saved_bytes", ctypes.c_uint64), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_uint64), ("save_for_backward", ctypes.c_int32),
                ("dev_status", ctypes.c_void_p), ("weight_cache", ctypes.c_void_p),
                ("weight_cache_bytes", ctypes.c_uint64)]


class MlpGroupedFwdArgs(ctypes.Structure):
    _fields_ = [("R", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32), ("E", ctypes.c_int32),
                ("x", ctypes.c_void_p), ("split_sizes", ctypes.c_void_p), ("probs", ctypes.c_void_p),
                ("w_gate_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("saved", ctypes.c_void_p), ("saved_bytes", ctypes.c_uint64), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_uint64), ("save_for_backward", ctypes.c_int32),
                ("dev_status", ctypes.c_void_p), ("weight_cache", ctypes.c_void_p),
                ("weight_cache_bytes", ctypes.c_uint64)]


class MlpGroupedFwdMxArgs(ctypes.Structure):
    _fields_ = [("R", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32), ("E", ctypes.c_int32),
                ("xq", ctypes.c_void_p), ("xs", ctypes.c_void_p), ("split_sizes", ctypes.c_void_p),
                ("probs", ctypes.c_void_p), ("w_gate_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p),
                ("y", ctypes.c_void_p), ("saved", ctypes.c_void_p), ("saved_bytes", ctypes.c_uint64),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_uint64), ("dev_status", ctypes.c_void_p),
                ("weight_cache", ctypes.c_void_p), ("weight_cache_bytes", ctypes.c_uint64)]


class MlpBwdArgs(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("dy", ctypes.c_void_p), ("saved", ctypes.c_void_p),
                ("saved_bytes", ctypes.c_uint64), ("dx", ctypes.c_void_p), ("dw_gate_up", ctypes.c_void_p),
                ("dw_down", ctypes.c_void_p), ("dprobs", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_uint64), ("dev_status", ctypes.c_void_p),
                ("weight_cache", ctypes.c_void_p), ("weight_cache_bytes", ctypes.c_uint64),
                ("main_grad_gate_up", ctypes.c_void_p), ("main_grad_down", ctypes.c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libmxg.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python -m mxfp8_grouped_gemm_gb300.build`")
    L = ctypes.CDLL(LIB_PATH)
    I32, I64, U64, SZ, P = ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_size_t, ctypes.c_void_p
    sig = {
        "mxg_status_string": (ctypes.c_char_p, [I32]),
        "mxg_device_supported": (I32, []),
        "mxg_launch_count": (U64, []),
        "mxg_route_topk": (I32, [P, I32, I32, I32, P, P, P]),
        "mxg_route_permute_workspace_bytes": (SZ, [I32, I32, I32]),
        "mxg_route_permute": (I32, [P, I32, I32, I32, P, P, P, P, P, SZ, P, P]),
        "mxg_mxfp8_quantize": (I32, [P, I32, I32, P, P, P, P, I32, P]),
        "mxg_grouped_gemm": (I32, [P, P, P, P, P, I32, I32, I32, I32, P, P, P]),
        "mxg_grouped_gemm_wgrad": (I32, [P, P, P, P, P, I32, I32, I32, I32, P, P, P]),
        "mxg_debug_grouped_gemm_stall": (I32, [P, P, P, P, P, I32, I32, I32, I32, P, U64, P, P]),
        "mxg_mlp_saved_bytes": (SZ, [I32, I32, I32, I32, I32]),
        "mxg_mlp_group_align": (I32, []),
        "mxg_mlp_row_capacity": (SZ, [I32, I32, I32]),
        "mxg_mlp_workspace_bytes": (SZ, [I32, I32, I32, I32, I32]),
        "mxg_grouped_mlp_fwd": (I32, [ctypes.POINTER(MlpFwdArgs), P]),
        "mxg_grouped_mlp_bwd": (I32, [ctypes.POINTER(MlpBwdArgs), P]),
        "mxg_mlp_saved_view": (P, [P, I32, I32, I32, I32, I32, I32]),
        "mxg_grouped_mlp_fwd_stage": (I32, [ctypes.POINTER(MlpFwdArgs), I32, P]),
        "mxg_route_permute_noalloc_max_entries": (SZ, [I32]),
        "mxg_route_permute_noalloc": (I32, [P, I32, I32, I32, P, P, P, P, P, P]),
        "mxg_grouped_mlp_bwd_stage": (I32, [ctypes.POINTER(MlpBwdArgs), I32, P]),
        "mxg_router_fwd": (I32, [P, P, I32, I32, I32, I32, P, P, P, P]),
        "mxg_mlp_bf16_saved_bytes": (SZ, [I32, I32, I32, I32, I32]),
        "mxg_mlp_bf16_workspace_bytes": (SZ, [I32, I32, I32, I32, I32]),
        "mxg_grouped_mlp_bf16_fwd": (I32, [ctypes.POINTER(MlpFwdArgs), P]),
        "mxg_grouped_mlp_bf16_bwd": (I32, [ctypes.POINTER(MlpBwdArgs), P]),
        "mxg_grouped_mlp_bf16_fwd_stage": (I32, [ctypes.POINTER(MlpFwdArgs), I32, P]),
        "mxg_grouped_mlp_bf16_bwd_stage": (I32, [ctypes.POINTER(MlpBwdArgs), I32, P]),
        "mxg_router_bwd_workspace_bytes": (SZ, [I32, I32, I32, I32]),
        "mxg_router_bwd": (I32, [P, P, P, P, P, I32, I32, I32, I32, P, P, P, SZ, P, P]),
        "mxg_mlp_weight_cache_bytes": (SZ, [I32, I32, I32]),
        "mxg_mlp_quantize_weights": (I32, [P, P, I32, I32, I32, P, SZ, P]),
        "mxg_mlp_saved_bytes_cached": (SZ, [I32, I32, I32, I32, I32]),
        "mxg_mlp_fp8_saved_bytes": (SZ, [I32, I32, I32, I32, I32]),
        "mxg_mlp_fp8_workspace_bytes": (SZ, [I32, I32, I32, I32, I32]),
        "mxg_grouped_mlp_fp8_fwd": (I32, [ctypes.POINTER(MlpFwdArgs), P]),
        "mxg_grouped_mlp_fp8_bwd": (I32, [ctypes.POINTER(MlpBwdArgs), P]),
        "mxg_grouped_mlp_fp8_fwd_stage": (I32, [ctypes.POINTER(MlpFwdArgs), I32, P]),
        "mxg_grouped_mlp_fp8_bwd_stage": (I32, [ctypes.POINTER(MlpBwdArgs), I32, P]),
        "mxg_mlp_fp8_saved_view": (P, [P, I32, I32, I32, I32, I32, I32]),
        "mxg_mlp_workspace_view": (P, [P, I32, I32, I32, I32, I32, I32]),
        "mxg_mlp_weight_cache_view": (P, [P, I32, I32, I32, I32]),
        "mxg_bench_mxfp8_mma_peak": (I32, [I32, ctypes.POINTER(ctypes.c_double), P, P]),
        "mxg_mxfp8_grouped_rows_capacity": (SZ, [I32, I32, I32]),
        "mxg_mxfp8_quantize_grouped": (I32, [P, I32, I32, P, I32, P, P, P, P, P, I32, P, P]),
        "mxg_gather_rows": (I32, [P, I64, I64, P, I32, I64, P, P, P]),
        "mxg_combine": (I32, [P, I64, P, I32, I32, I32, P, P, P]),
        "mxg_mlp_grouped_saved_bytes": (SZ, [I32, I32, I32, I32]),
        "mxg_mlp_grouped_workspace_bytes": (SZ, [I32, I32, I32, I32]),
        "mxg_grouped_mlp_fwd_grouped": (I32, [ctypes.POINTER(MlpGroupedFwdArgs), P]),
        "mxg_router_fwd_permute": (I32, [P, P, I32, I32, I32, I32, P, P, P, P, P, P, P, P, SZ, P, P]),
        "mxg_grouped_mlp_fwd_grouped_mx": (I32, [ctypes.POINTER(MlpGroupedFwdMxArgs), P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def status_string(code: int) -> str:
    return lib().mxg_status_string(int(code)).decode()


def _check(fn: str, code: int):
    if code != 0:
        raise MxgError(fn, code)


def _ptr(t: torch.Tensor | None, dtype=None, name: str = "tensor") -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _bits(t: torch.Tensor | None) -> torch.Tensor | None:
    return t.view(torch.int16) if t is not None and t.dtype == torch.bfloat16 else t


# ------------------------------------------------------------------ entries --

def mxg_device_supported() -> bool:
    return bool(lib().mxg_device_supported())


def mxg_launch_count() -> int:
    return int(lib().mxg_launch_count())


def mxg_route_topk(logits: torch.Tensor, k: int, ids=None, probs=None, stream=None):
    T, E = logits.shape
    ids = torch.empty((T, k), dtype=torch.int32, device=logits.device) if ids is None else ids
    probs = torch.empty((T, k), dtype=torch.float32, device=logits.device) if probs is None else probs
    _check("mxg_route_topk", lib().mxg_route_topk(_ptr(logits, torch.float32, "logits"), T, E, k,
                                                  _ptr(ids, torch.int32, "ids"), _ptr(probs, torch.float32, "probs"),
                                                  _stream(stream)))
    return ids, probs


def mxg_router_fwd(x: torch.Tensor, w_router: torch.Tensor, k: int, logits=None, ids=None, probs=None, stream=None):
    """logits = x W_r^T (fp32 out) and the top-k route on them."""
    T, H = x.shape
    E = w_router.shape[0]
    dev = x.device
    logits = torch.empty((T, E), dtype=torch.float32, device=dev) if logits is None else logits
    ids = torch.empty((T, k), dtype=torch.int32, device=dev) if ids is None else ids
    probs = torch.empty((T, k), dtype=torch.float32, device=dev) if probs is None else probs
    _check("mxg_router_fwd", lib().mxg_router_fwd(_ptr(x, torch.bfloat16, "x"), _ptr(w_router, torch.bfloat16, "w_router"),
                                                  T, H, E, k, _ptr(logits, torch.float32, "logits"),
                                                  _ptr(ids, torch.int32, "ids"), _ptr(probs, torch.float32, "probs"),
                                                  _stream(stream)))
    return logits, ids, probs


def mxg_router_bwd_workspace_bytes(T, H, E, k) -> int:
    return int(lib().mxg_router_bwd_workspace_bytes(T, H, E, k))


def mxg_router_bwd(x, w_router, ids, probs, dprobs, dx, dev_status, dw_router=None, workspace=None, stream=None):
    """Adds the router's term to dx (in place) and returns dW_r (fp32)."""
    T, H = x.shape
    E = w_router.shape[0]
    k = ids.shape[1]
    dev = x.device
    dw_router = torch.empty((E, H), dtype=torch.float32, device=dev) if dw_router is None else dw_router
    nbytes = mxg_router_bwd_workspace_bytes(T, H, E, k)
    workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev) if workspace is None else workspace
    _check("mxg_router_bwd", lib().mxg_router_bwd(
        _ptr(x, torch.bfloat16, "x"), _ptr(w_router, torch.bfloat16, "w_router"), _ptr(ids, torch.int32, "ids"),
        _ptr(probs, torch.float32, "probs"), _ptr(dprobs, torch.float32, "dprobs"), T, H, E, k,
        _ptr(dx, torch.bfloat16, "dx"), _ptr(dw_router, torch.float32, "dw_router"), _ptr(workspace), workspace.numel(),
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)))
    return dw_router


def mxg_route_permute(ids: torch.Tensor, E: int, dev_status: torch.Tensor, stream=None) -> dict:
    T, k = ids.shape
    dev = ids.device
    ws_bytes = int(lib().mxg_route_permute_workspace_bytes(T, k, E))
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    out = {"split_sizes": torch.empty(E, dtype=torch.int32, device=dev),
           "src_of_row": torch.empty(T * k, dtype=torch.int32, device=dev),
           "row_of_src": torch.empty(T * k, dtype=torch.int32, device=dev),
           "padded_offsets": torch.empty(E + 1, dtype=torch.int32, device=dev)}
    _check("mxg_route_permute", lib().mxg_route_permute(
        _ptr(ids, torch.int32, "ids"), T, k, E, _ptr(out["split_sizes"]), _ptr(out["src_of_row"]),
        _ptr(out["row_of_src"]), _ptr(out["padded_offsets"]), _ptr(ws), ws_bytes,
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)))
    return out


def mxfp8_scale_bytes(rows: int, cols: int) -> int:
    return rows * cols // 32


def mxg_mxfp8_quantize(x: torch.Tensor, row: bool = True, col: bool = False, layout: int = MXG_LAYOUT_CANONICAL,
                       stream=None) -> dict:
    """x bf16 [rows, cols] -> {'q_row','s_row'} and/or {'q_col','s_col'} (uint8)."""
    rows, cols = x.shape
    dev = x.device
    out = {}
    if row:
        out["q_row"] = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
        out["s_row"] = torch.empty(rows * cols // 32, dtype=torch.uint8, device=dev)
    if col:
        out["q_col"] = torch.empty((cols, rows), dtype=torch.uint8, device=dev)
        out["s_col"] = torch.empty(rows * cols // 32, dtype=torch.uint8, device=dev)
    _check("mxg_mxfp8_quantize", lib().mxg_mxfp8_quantize(
        _ptr(_bits(x), None, "x"), rows, cols, _ptr(out.get("q_row")), _ptr(out.get("s_row")),
        _ptr(out.get("q_col")), _ptr(out.get("s_col")), layout, _stream(stream)))
    return out


def mxg_grouped_gemm(a, sa, b, sb, padded_offsets, E: int, N: int, K: int, dev_status, d=None, stream=None):
    m_cap = a.shape[0]
    d = torch.empty((m_cap, N), dtype=torch.bfloat16, device=a.device) if d is None else d
    _check("mxg_grouped_gemm", lib().mxg_grouped_gemm(
        _ptr(a, torch.uint8, "a"), _ptr(sa, torch.uint8, "sa"), _ptr(b, torch.uint8, "b"), _ptr(sb, torch.uint8, "sb"),
        _ptr(padded_offsets, torch.int32, "padded_offsets"), E, m_cap, N, K, _ptr(_bits(d)),
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)))
    return d


def mxg_grouped_gemm_wgrad(a, sa, b, sb, padded_offsets, E: int, dev_status, d=None, stream=None):
    M, t_cap = a.shape
    N = b.shape[0]
    d = torch.empty((E, M, N), dtype=torch.bfloat16, device=a.device) if d is None else d
    _check("mxg_grouped_gemm_wgrad", lib().mxg_grouped_gemm_wgrad(
        _ptr(a, torch.uint8, "a"), _ptr(sa, torch.uint8, "sa"), _ptr(b, torch.uint8, "b"), _ptr(sb, torch.uint8, "sb"),
        _ptr(padded_offsets, torch.int32, "padded_offsets"), E, M, N, t_cap, _ptr(_bits(d)),
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)))
    return d


def mxg_mlp_group_align() -> int:
    return int(lib().mxg_mlp_group_align())


def mxg_mlp_row_capacity(T, k, E) -> int:
    return int(lib().mxg_mlp_row_capacity(T, k, E))


def mxg_mlp_saved_bytes(T, H, I, E, k) -> int:
    return int(lib().mxg_mlp_saved_bytes(T, H, I, E, k))


def mxg_mlp_workspace_bytes(T, H, I, E, k) -> int:
    return int(lib().mxg_mlp_workspace_bytes(T, H, I, E, k))


def mxg_mlp_bf16_saved_bytes(T, H, I, E, k) -> int:
    return int(lib().mxg_mlp_bf16_saved_bytes(T, H, I, E, k))


def mxg_mlp_bf16_workspace_bytes(T, H, I, E, k) -> int:
    return int(lib().mxg_mlp_bf16_workspace_bytes(T, H, I, E, k))


def mxg_mlp_fp8_saved_bytes(T, H, I, E, k) -> int:
    return int(lib().mxg_mlp_fp8_saved_bytes(T, H, I, E, k))


def mxg_mlp_fp8_workspace_bytes(T, H, I, E, k) -> int:
    return int(lib().mxg_mlp_fp8_workspace_bytes(T, H, I, E, k))


def mxg_mlp_saved_view(saved: torch.Tensor, T, H, I, E, k, which: int) -> int:
    return int(lib().mxg_mlp_saved_view(_ptr(saved), T, H, I, E, k, which) or 0)


def mxg_mlp_workspace_view(workspace: torch.Tensor, T, H, I, E, k, which: int) -> int:
    return int(lib().mxg_mlp_workspace_view(_ptr(workspace), T, H, I, E, k, which) or 0)


class WeightCache:
    """The MXFP8 weights of one expert MLP (all four orientations), written by
    mxg_mlp_quantize_weights and read by forward / backward calls until the
    weights change."""

    def __init__(self, H: int, I: int, E: int, device="cuda"):
        n = int(lib().mxg_mlp_weight_cache_bytes(H, I, E))
        if n == 0:
            raise ValueError(f"unsupported weight shape H={H} I={I} E={E}")
        self.H, self.I, self.E = H, I, E
        self.buffer = torch.empty(n, dtype=torch.uint8, device=device)


def mxg_mlp_saved_bytes_cached(T, H, I, E, k) -> int:
    return int(lib().mxg_mlp_saved_bytes_cached(T, H, I, E, k))


def mxg_mlp_quantize_weights(w_gate_up, w_down, cache: WeightCache | None = None, stream=None) -> WeightCache:
    """Quantise the bf16 expert weights into a weight cache (allocated if not given)."""
    E, N2, H = w_gate_up.shape
    I = N2 // 2
    if tuple(w_down.shape) != (E, H, I):
        raise ValueError(f"w_down must be [E, H, I] = {(E, H, I)}, got {tuple(w_down.shape)}")
    cache = WeightCache(H, I, E, w_gate_up.device) if cache is None else cache
    if (cache.H, cache.I, cache.E) != (H, I, E):
        raise ValueError("weight cache was made for another shape")
    _check("mxg_mlp_quantize_weights",
           lib().mxg_mlp_quantize_weights(_ptr(_bits(w_gate_up), torch.int16, "w_gate_up"),
                                          _ptr(_bits(w_down), torch.int16, "w_down"), H, I, E,
                                          _ptr(cache.buffer, torch.uint8, "cache"), cache.buffer.numel(),
                                          _stream(stream)))
    return cache


def mxg_grouped_mlp_fwd(x, ids, probs, w_gate_up, w_down, saved, workspace, dev_status, y=None, split_sizes=None,
                        save_for_backward: bool = True, stream=None, stage: int | None = None, bf16: bool = False,
                        weight_cache: WeightCache | None = None, fp8: bool = False):
    """Full forward, or one stage of it (FWD_STAGES index) when ``stage`` is given
    (``bf16``: the BF16 path, mxg_grouped_mlp_bf16_fwd).  With ``weight_cache``
    the weights are read from it and w_gate_up / w_down may be None."""
    T, H = x.shape
    k = ids.shape[1]
    if weight_cache is not None:
        E, I = weight_cache.E, weight_cache.I
    else:
        E, N2, _ = w_gate_up.shape
        I = N2 // 2
    y = torch.empty((T, H), dtype=torch.bfloat16, device=x.device) if y is None else y
    split_sizes = torch.empty(E, dtype=torch.int32, device=x.device) if split_sizes is None else split_sizes
    a = MlpFwdArgs(T, H, I, E, k, _ptr(_bits(x), torch.int16, "x"), _ptr(ids, torch.int32, "ids"),
                   _ptr(probs, torch.float32, "probs"), _ptr(_bits(w_gate_up), torch.int16, "w_gate_up"),
                   _ptr(_bits(w_down), torch.int16, "w_down"), _ptr(_bits(y)), _ptr(split_sizes, torch.int32),
                   _ptr(saved, torch.uint8, "saved"), saved.numel(), _ptr(workspace, torch.uint8, "workspace"),
                   workspace.numel(), 1 if save_for_backward else 0, _ptr(dev_status, torch.int32, "dev_status"),
                   None if weight_cache is None else _ptr(weight_cache.buffer, torch.uint8, "weight_cache"),
                   0 if weight_cache is None else weight_cache.buffer.numel())
    name = "mxg_grouped_mlp_bf16_fwd" if bf16 else ("mxg_grouped_mlp_fp8_fwd" if fp8 else "mxg_grouped_mlp_fwd")
    if stage is None:
        _check(name, getattr(lib(), name)(ctypes.byref(a), _stream(stream)))
    else:
        _check(name + "_stage", getattr(lib(), name + "_stage")(ctypes.byref(a), stage, _stream(stream)))
    return y, split_sizes


def mxg_grouped_mlp_bwd(dy, saved, workspace, dev_status, E: int, I: int, k: int, dx=None, dw_gate_up=None,
                        dw_down=None, dprobs=None, stream=None, stage: int | None = None, bf16: bool = False,
                        weight_cache: WeightCache | None = None, main_grad=None, fp8: bool = False):
    """Full backward, or one stage of it (BWD_STAGES index) when ``stage`` is given
    (``bf16``: the BF16 path, mxg_grouped_mlp_bf16_bwd).  ``weight_cache``: the
    cache the forward used.  ``main_grad`` = (fp32 [E, 2I, H], fp32 [E, H, I]):
    the weight gradients are added into these and returned in place of dW."""
    T, H = dy.shape
    dev = dy.device
    dx = torch.empty((T, H), dtype=torch.bfloat16, device=dev) if dx is None else dx
    if main_grad is not None:
        mg_gu, mg_d = main_grad
        if tuple(mg_gu.shape) != (E, 2 * I, H) or tuple(mg_d.shape) != (E, H, I):
            raise ValueError("main_grad must be fp32 [E, 2I, H] and [E, H, I]")
        dw_gate_up = dw_down = None
    else:
        mg_gu = mg_d = None
        dw_gate_up = torch.empty((E, 2 * I, H), dtype=torch.bfloat16, device=dev) if dw_gate_up is None else dw_gate_up
        dw_down = torch.empty((E, H, I), dtype=torch.bfloat16, device=dev) if dw_down is None else dw_down
    dprobs = torch.empty((T, k), dtype=torch.float32, device=dev) if dprobs is None else dprobs
    a = MlpBwdArgs(T, H, I, E, k, _ptr(_bits(dy), torch.int16, "dy"), _ptr(saved, torch.uint8, "saved"),
                   saved.numel(), _ptr(_bits(dx)), _ptr(_bits(dw_gate_up)), _ptr(_bits(dw_down)),
                   _ptr(dprobs, torch.float32), _ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
                   _ptr(dev_status, torch.int32, "dev_status"),
                   None if weight_cache is None else _ptr(weight_cache.buffer, torch.uint8, "weight_cache"),
                   0 if weight_cache is None else weight_cache.buffer.numel(),
                   _ptr(mg_gu, torch.float32, "main_grad_gate_up"), _ptr(mg_d, torch.float32, "main_grad_down"))
    name = "mxg_grouped_mlp_bf16_bwd" if bf16 else ("mxg_grouped_mlp_fp8_bwd" if fp8 else "mxg_grouped_mlp_bwd")
    if stage is None:
        _check(name, getattr(lib(), name)(ctypes.byref(a), _stream(stream)))
    else:
        _check(name + "_stage", getattr(lib(), name + "_stage")(ctypes.byref(a), stage, _stream(stream)))
    if main_grad is not None:
        return dx, mg_gu, mg_d, dprobs
    return dx, dw_gate_up, dw_down, dprobs


def mxg_bench_mxfp8_mma_peak(steps: int, dev_status: torch.Tensor, stream=None) -> float:
    """Enqueue the MXFP8 MMA-only peak loop; returns the launch's flop count
    (time it with events on the same stream)."""
    flops = ctypes.c_double(0.0)
    _check("mxg_bench_mxfp8_mma_peak", lib().mxg_bench_mxfp8_mma_peak(
        int(steps), ctypes.byref(flops), _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)))
    return float(flops.value)


def mxg_mxfp8_grouped_rows_capacity(rows: int, groups: int, layout: int = MXG_LAYOUT_CANONICAL) -> int:
    return int(lib().mxg_mxfp8_grouped_rows_capacity(rows, groups, layout))


def mxg_mxfp8_quantize_grouped(x: torch.Tensor, group_offsets: torch.Tensor, dev_status: torch.Tensor,
                               row: bool = True, col: bool = True, layout: int = MXG_LAYOUT_CANONICAL,
                               stream=None) -> dict:
    """x bf16 [rows, cols] in groups (group_offsets int32 [groups+1]) -> the
    padded group layout: 'padded_offsets', and 'q_row','s_row' / 'q_col','s_col'."""
    rows, cols = x.shape
    groups = group_offsets.numel() - 1
    cap = mxg_mxfp8_grouped_rows_capacity(rows, groups, layout)
    if cap == 0:
        raise ValueError(f"unsupported grouped quantisation rows={rows} groups={groups}")
    dev = x.device
    out = {"padded_offsets": torch.empty(groups + 1, dtype=torch.int32, device=dev), "capacity": cap}
    if row:
        out["q_row"] = torch.empty((cap, cols), dtype=torch.uint8, device=dev)
        out["s_row"] = torch.empty(cap * cols // 32, dtype=torch.uint8, device=dev)
    if col:
        out["q_col"] = torch.empty((cols, cap), dtype=torch.uint8, device=dev)
        out["s_col"] = torch.empty(cap * cols // 32, dtype=torch.uint8, device=dev)
    _check("mxg_mxfp8_quantize_grouped", lib().mxg_mxfp8_quantize_grouped(
        _ptr(_bits(x), None, "x"), rows, cols, _ptr(group_offsets, torch.int32, "group_offsets"), groups,
        _ptr(out["padded_offsets"]), _ptr(out.get("q_row")), _ptr(out.get("s_row")), _ptr(out.get("q_col")),
        _ptr(out.get("s_col")), layout, _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)))
    return out


def mxg_gather_rows(src: torch.Tensor, index: torch.Tensor, dev_status: torch.Tensor, div: int = 1,
                    out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """out[r] = src[index[r] // div] (rows of src's trailing dimensions)."""
    src_rows = src.shape[0]
    row_bytes = src[0].numel() * src.element_size() if src.dim() > 1 else src.element_size()
    rows = index.numel()
    out = torch.empty((rows,) + tuple(src.shape[1:]), dtype=src.dtype, device=src.device) if out is None else out
    _check("mxg_gather_rows", lib().mxg_gather_rows(
        _ptr(src, None, "src"), src_rows, row_bytes, _ptr(index, torch.int32, "index"), div, rows,
        _ptr(out, src.dtype, "out"), _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)))
    return out


def mxg_combine(rows: torch.Tensor, row_of_src: torch.Tensor, k: int, dev_status: torch.Tensor,
                y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y[t] = sum_j rows[row_of_src[t*k + j]] (fp32 sum in slot order, bf16 out)."""
    src_rows, H = rows.shape
    T = row_of_src.numel() // k
    y = torch.empty((T, H), dtype=torch.bfloat16, device=rows.device) if y is None else y
    _check("mxg_combine", lib().mxg_combine(
        _ptr(_bits(rows), torch.int16, "rows"), src_rows, _ptr(row_of_src, torch.int32, "row_of_src"), T, k, H,
        _ptr(_bits(y), torch.int16, "y"), _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)))
    return y


def mxg_mlp_grouped_saved_bytes(R, H, I, E) -> int:
    return int(lib().mxg_mlp_grouped_saved_bytes(R, H, I, E))


def mxg_mlp_grouped_workspace_bytes(R, H, I, E) -> int:
    return int(lib().mxg_mlp_grouped_workspace_bytes(R, H, I, E))


def mxg_grouped_mlp_fwd_grouped(x, split_sizes, probs, w_gate_up, w_down, saved, workspace, dev_status, y=None,
                                save_for_backward: bool = True, weight_cache: WeightCache | None = None,
                                stream=None):
    """Forward on rows already grouped by expert (split_sizes int32 [E] on the
    device, probs fp32 [R]); returns the per-row outputs y [R, H]."""
    R, H = x.shape
    if weight_cache is not None:
        E, I = weight_cache.E, weight_cache.I
    else:
        E, N2, _ = w_gate_up.shape
        I = N2 // 2
    y = torch.empty((R, H), dtype=torch.bfloat16, device=x.device) if y is None else y
    a = MlpGroupedFwdArgs(R, H, I, E, _ptr(_bits(x), torch.int16, "x"), _ptr(split_sizes, torch.int32, "split_sizes"),
                          _ptr(probs, torch.float32, "probs"), _ptr(_bits(w_gate_up), torch.int16, "w_gate_up"),
                          _ptr(_bits(w_down), torch.int16, "w_down"), _ptr(_bits(y), torch.int16, "y"),
                          _ptr(saved, torch.uint8, "saved"), saved.numel(), _ptr(workspace, torch.uint8, "workspace"),
                          workspace.numel(), 1 if save_for_backward else 0,
                          _ptr(dev_status, torch.int32, "dev_status"),
                          None if weight_cache is None else _ptr(weight_cache.buffer, torch.uint8, "weight_cache"),
                          0 if weight_cache is None else weight_cache.buffer.numel())
    _check("mxg_grouped_mlp_fwd_grouped", lib().mxg_grouped_mlp_fwd_grouped(ctypes.byref(a), _stream(stream)))
    return y


def mxg_router_fwd_permute(x: torch.Tensor, w_router: torch.Tensor, k: int, dev_status: torch.Tensor, stream=None):
    """Router logits + route + permute in one call; returns (logits, ids,
    probs, permute dict as mxg_route_permute)."""
    T, H = x.shape
    E = w_router.shape[0]
    dev = x.device
    logits = torch.empty((T, E), dtype=torch.float32, device=dev)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    probs = torch.empty((T, k), dtype=torch.float32, device=dev)
    ws_bytes = int(lib().mxg_route_permute_workspace_bytes(T, k, E))
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    out = {"split_sizes": torch.empty(E, dtype=torch.int32, device=dev),
           "src_of_row": torch.empty(T * k, dtype=torch.int32, device=dev),
           "row_of_src": torch.empty(T * k, dtype=torch.int32, device=dev),
           "padded_offsets": torch.empty(E + 1, dtype=torch.int32, device=dev)}
    _check("mxg_router_fwd_permute", lib().mxg_router_fwd_permute(
        _ptr(x, torch.bfloat16, "x"), _ptr(w_router, torch.bfloat16, "w_router"), T, H, E, k,
        _ptr(logits), _ptr(ids), _ptr(probs), _ptr(out["split_sizes"]), _ptr(out["src_of_row"]),
        _ptr(out["row_of_src"]), _ptr(out["padded_offsets"]), _ptr(ws), ws_bytes,
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)))
    return logits, ids, probs, out


def mxg_grouped_mlp_fwd_grouped_mx(xq, xs, split_sizes, probs, w_gate_up, w_down, saved, workspace, dev_status,
                                   H: int, y=None, weight_cache: WeightCache | None = None, stream=None):
    """Inference forward on grouped rows given as row-wise MXFP8: codes xq uint8
    [R, H] and canonical scales xs uint8 [R, H/32]; returns y [R, H]."""
    R = xq.shape[0]
    if weight_cache is not None:
        E, I = weight_cache.E, weight_cache.I
    else:
        E, N2, _ = w_gate_up.shape
        I = N2 // 2
    y = torch.empty((R, H), dtype=torch.bfloat16, device=xq.device) if y is None else y
    a = MlpGroupedFwdMxArgs(R, H, I, E, _ptr(xq, torch.uint8, "xq"), _ptr(xs, torch.uint8, "xs"),
                            _ptr(split_sizes, torch.int32, "split_sizes"), _ptr(probs, torch.float32, "probs"),
                            _ptr(_bits(w_gate_up), torch.int16, "w_gate_up"), _ptr(_bits(w_down), torch.int16, "w_down"),
                            _ptr(_bits(y), torch.int16, "y"), _ptr(saved, torch.uint8, "saved"), saved.numel(),
                            _ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
                            _ptr(dev_status, torch.int32, "dev_status"),
                            None if weight_cache is None else _ptr(weight_cache.buffer, torch.uint8, "weight_cache"),
                            0 if weight_cache is None else weight_cache.buffer.numel())
    _check("mxg_grouped_mlp_fwd_grouped_mx", lib().mxg_grouped_mlp_fwd_grouped_mx(ctypes.byref(a), _stream(stream)))
    return y
