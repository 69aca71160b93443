"""Helpers shared by the GPU parity tests: device fixture, tolerance checks,
and the documented MMA scale layout written out from include/mxg.h."""
import numpy as np
import pytest
import torch


def require_gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    import mxfp8_grouped_gemm_gb300 as m
    from mxfp8_grouped_gemm_gb300 import build
    build.build()
    if not m.mxg_device_supported():
        pytest.fail("current device is not sm_103 (GB300)")
    return m


def np_(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        t = t.double()
    return t.numpy()


def mma_index(rows: int, nblocks: int) -> np.ndarray:
    """Byte offset of (row r, block b) in the tensor-core scale layout, from the
    formula documented for MXG_LAYOUT_MMA in include/mxg.h."""
    r = np.arange(rows)[:, None]
    b = np.arange(nblocks)[None, :]
    return ((b // 4) * (rows // 128) + r // 128) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (b % 4)


def mma_to_canonical(s: torch.Tensor, rows: int, nblocks: int) -> np.ndarray:
    flat = s.detach().cpu().numpy().reshape(-1)
    return flat[mma_index(rows, nblocks)]


def assert_rel_close(a, r, tol=1e-2, floor=1.0, name=""):
    a = np.asarray(a, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    bound = tol * np.maximum(np.abs(r), floor)
    bad = np.abs(a - r) > bound
    assert not bad.any(), f"{name}: {int(bad.sum())} elements outside {tol}*max(|r|,{floor}); " \
                          f"worst {float(np.max(np.abs(a - r) / bound)):.3g}x"


def codes_equal_up_to_zero_sign(a: np.ndarray, b: np.ndarray):
    """Bit-exact E4M3 comparison; +0 (0x00) and -0 (0x80) count as equal but the
    number of such cases is returned so the test can report it."""
    a = a.astype(np.uint8)
    b = b.astype(np.uint8)
    zero_sign = ((a == 0x80) & (b == 0x00)) | ((a == 0x00) & (b == 0x80))
    diff = (a != b) & ~zero_sign
    return int(diff.sum()), int(zero_sign.sum())
