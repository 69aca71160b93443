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


def assert_rms_close(a, r, frac=2e-2, name="", guard=0.5):
    """The stated tolerance read as a relative RMS error: ||a - r||_2 <= frac *
    ||r||_2 (the error is at most `frac` of the output RMS).  A per-element
    guard |a - r| <= guard * RMS(r) + 2^-7 |r| catches localised faults (a
    wrong row or tile) that an RMS can hide; it sits above the largest single
    re-quantisation flip of a heavy-tailed product (one E4M3 step of the largest
    dGU value of an expert times a large x, measured up to ~0.35 RMS on few-token
    experts).  Returns (max|a-r| / RMS, rel RMS)."""
    a = np.asarray(a, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    if r.size == 0:
        return 0.0, 0.0
    rms = float(np.sqrt(np.mean(r * r)))
    diff = np.abs(a - r)
    err = float(np.max(diff))
    rel_rms = float(np.sqrt(np.mean(diff ** 2)) / rms) if rms > 0 else float(np.sqrt(np.mean(diff ** 2)))
    assert rel_rms <= frac, f"{name}: relative RMS error {rel_rms:.4g} > {frac} (max|a-r|/RMS {err / rms:.3g})"
    bad = diff > guard * rms + 2.0 ** -7 * np.abs(r)
    assert not bad.any(), f"{name}: {int(bad.sum())} elements beyond the per-element guard (max|a-r|/RMS {err / rms:.3g})"
    return (err / rms if rms else 0.0), rel_rms


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
