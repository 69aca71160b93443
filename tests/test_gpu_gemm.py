"""Grouped MXFP8 GEMM parity (tcgen05 block-scaled path) against the oracle's
fp64 product of the dequantised operands: one tile, several tiles, ragged and
empty groups, both tile widths, and the token-grouped weight-gradient shape."""
import numpy as np
import pytest
import torch

import synthetic
from gpu_helpers import assert_rel_close, np_, require_gpu
from oracle import mx

pytestmark = pytest.mark.gpu


def _quant_mma(m, x):
    out = m.mxg_mxfp8_quantize(x.cuda(), row=True, col=False, layout=m.MXG_LAYOUT_MMA)
    return out["q_row"], out["s_row"]


@pytest.mark.parametrize("sizes,N,K", [
    ([128], 128, 128),                   # one tile, one K step
    ([128], 256, 128),                   # one tile, BN = 256
    ([256], 128, 1024),                  # two row tiles, eight K steps (pipeline wrap)
    ([256, 0, 128, 384], 256, 512),      # ragged and empty groups
    ([128, 128, 128], 384, 256),         # N not a multiple of 256 -> BN = 128
])
def test_grouped_gemm(sizes, N, K):
    m = require_gpu()
    E = len(sizes)
    poff = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    m_cap = int(poff[-1]) + 128
    a = synthetic.random_bf16((m_cap, K), 1000 + K)
    b = synthetic.random_bf16((E * N, K), 2000 + N, std=0.5)
    qa, sa = _quant_mma(m, a)
    qb, sb = _quant_mma(m, b)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = torch.full((m_cap, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    m.mxg_grouped_gemm(qa, sa, qb, sb, torch.from_numpy(poff).cuda(), E, N, K, st, d=d)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = np_(d)
    A = mx.fake_quant(a.double().numpy())
    B = mx.fake_quant(b.double().numpy())
    for e in range(E):
        r0, r1 = poff[e], poff[e + 1]
        if r1 == r0:
            continue
        ref = A[r0:r1] @ B[e * N:(e + 1) * N].T
        assert_rel_close(got[r0:r1], ref, tol=1e-2, floor=1.0, name=f"group {e}")
    assert np.isnan(got[poff[-1]:]).all()            # rows outside the groups untouched


def test_grouped_gemm_bad_offsets_reported():
    m = require_gpu()
    qa = torch.zeros((256, 128), dtype=torch.uint8, device="cuda")
    sa = torch.zeros(256 * 4, dtype=torch.uint8, device="cuda")
    qb = torch.zeros((128, 128), dtype=torch.uint8, device="cuda")
    sb = torch.zeros(128 * 4, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    poff = torch.tensor([0, 100], dtype=torch.int32, device="cuda")      # not 128-aligned
    m.mxg_grouped_gemm(qa, sa, qb, sb, poff, 1, 128, 128, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 17                                          # MXG_ERR_OFFSETS


@pytest.mark.parametrize("sizes,M,N", [([128, 0, 256], 256, 256), ([384, 128], 128, 384)])
def test_grouped_gemm_wgrad(sizes, M, N):
    m = require_gpu()
    E = len(sizes)
    poff = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    t_cap = int(poff[-1]) + 128
    # operands stored token-contiguous: A [M][t_cap], B [N][t_cap]
    a = synthetic.random_bf16((M, t_cap), 3000 + M)
    b = synthetic.random_bf16((N, t_cap), 4000 + N)
    qa, sa = _quant_mma(m, a)
    qb, sb = _quant_mma(m, b)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = torch.full((E, M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    m.mxg_grouped_gemm_wgrad(qa, sa, qb, sb, torch.from_numpy(poff).cuda(), E, st, d=d)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = np_(d)
    A = mx.fake_quant(a.double().numpy())
    B = mx.fake_quant(b.double().numpy())
    for e in range(E):
        t0, t1 = poff[e], poff[e + 1]
        if t1 == t0:
            assert np.array_equal(got[e], np.zeros((M, N)))              # exact zeros
            continue
        ref = A[:, t0:t1] @ B[:, t0:t1].T
        assert_rel_close(got[e], ref, tol=1e-2, floor=1.0, name=f"expert {e}")


def test_kernel_wait_timeout_is_reported_and_context_survives():
    """Failure detection without a fault: a producer that never issues its copies
    makes the MMA warp's bounded wait run out; the kernel reports
    MXG_ERR_TIMEOUT, frees its tensor memory and returns, and a normal GEMM
    afterwards still gives correct results."""
    m = require_gpu()
    L = m.lib()
    E, N, K = 1, 128, 256
    poff = torch.tensor([0, 256], dtype=torch.int32, device="cuda")
    a = synthetic.random_bf16((256, K), 11)
    b = synthetic.random_bf16((N, K), 12)
    qa, sa = _quant_mma(m, a)
    qb, sb = _quant_mma(m, b)
    d = torch.zeros((256, N), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = L.mxg_debug_grouped_gemm_stall(qa.data_ptr(), sa.data_ptr(), qb.data_ptr(), sb.data_ptr(), poff.data_ptr(),
                                        E, 256, N, K, d.data_ptr(), 20_000_000, st.data_ptr(),
                                        torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(st.item()) == 18                                          # MXG_ERR_TIMEOUT
    st.zero_()
    m.mxg_grouped_gemm(qa, sa, qb, sb, poff, E, N, K, st, d=d)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = mx.fake_quant(a.double().numpy()) @ mx.fake_quant(b.double().numpy()).T
    assert_rel_close(np_(d), ref, tol=1e-2, floor=1.0, name="after timeout")
