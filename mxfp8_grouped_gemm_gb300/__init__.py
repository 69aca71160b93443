"""mxfp8_grouped_gemm_gb300 — grouped MXFP8 MoE expert MLP for GB300 (sm_103a).

The compute lives in libmxg.so (C ABI, include/mxg.h); this package is its
ctypes binding plus a small helper that owns the caller-side buffers.
"""
from ._lib import (  # noqa: F401
    BWD_STAGES, EXPORTS, FWD_STAGES, LIB_PATH, MXG_LAYOUT_CANONICAL, MXG_LAYOUT_MMA, MlpBwdArgs, MlpFwdArgs, MxgError, lib,
    mxg_device_supported, mxg_grouped_gemm, mxg_grouped_gemm_wgrad, mxg_grouped_mlp_bwd, mxg_grouped_mlp_fwd,
    mxg_launch_count, mxg_mlp_group_align, mxg_mlp_row_capacity, mxg_mlp_saved_bytes, mxg_mlp_saved_view, mxg_mlp_workspace_bytes, mxg_mlp_workspace_view, mxg_mxfp8_quantize,
    mxg_route_permute, mxg_route_topk, mxg_router_bwd, mxg_router_bwd_workspace_bytes, mxg_router_fwd, status_string,
    WeightCache, mxg_mlp_quantize_weights, mxg_mlp_saved_bytes_cached, mxg_bench_mxfp8_mma_peak,
    mxg_mxfp8_grouped_rows_capacity, mxg_mxfp8_quantize_grouped, mxg_gather_rows, mxg_combine,
    mxg_mlp_grouped_saved_bytes, mxg_mlp_grouped_workspace_bytes, mxg_grouped_mlp_fwd_grouped,
    mxg_router_fwd_permute, mxg_grouped_mlp_fwd_grouped_mx,
)
from .layer import GroupedExperts, GroupedMLP  # noqa: F401
