"""MXFP8 quantiser parity: E4M3 codes and E8M0 scales bit-exact against the
oracle on the same bf16 input, both orientations, both scale layouts."""
import numpy as np
import pytest
import torch

import synthetic
from gpu_helpers import codes_equal_up_to_zero_sign, mma_to_canonical, np_, require_gpu
from oracle import mx

pytestmark = pytest.mark.gpu


def _special_matrix(rows, cols, seed):
    """Normal values spread over many binades, plus planted edge blocks."""
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((rows, cols)) * np.exp2(rng.integers(-40, 40, size=(rows, 1)))
    a[0, :32] = 0.0                                   # all-zero block
    a[1, :32] = 0.0
    a[1, 7] = -3.0e-5                                 # single non-zero
    for i, m in enumerate([256.0, 448.0, 464.0, 480.0, 511.0]):
        a[2 + i, :32] = rng.standard_normal(32)
        a[2 + i, 3] = m * 2.0 ** (i * 7 - 10)         # block max at the saturation edges
    a[8, :32] = 1e-40                                 # bf16 subnormals
    a[9, :32] = 3e38                                  # near the bf16 maximum
    a[10, 32:64] = rng.standard_normal(32) * 1e-38
    a[11, :] = 0.0
    a[:, 5] = np.where(np.arange(rows) % 7 == 0, 0.0, a[:, 5])
    return synthetic.to_bf16(a.astype(np.float32))


@pytest.mark.parametrize("rows,cols", [(32, 128), (128, 256), (384, 640), (1024, 1024)])
def test_quantize_canonical_bit_exact(rows, cols):
    m = require_gpu()
    x = _special_matrix(rows, cols, rows + cols)
    out = m.mxg_mxfp8_quantize(x.cuda(), row=True, col=True, layout=m.MXG_LAYOUT_CANONICAL)
    torch.cuda.synchronize()
    xd = x.double().numpy()
    qr, sr = mx.quantize_blocks(xd)
    qc, sc = mx.quantize_blocks(xd.T)           # column-wise = row-wise of the transpose
    nd, nz = codes_equal_up_to_zero_sign(np_(out["q_row"]), qr)
    assert nd == 0, f"{nd} row-wise codes differ"
    assert np.array_equal(np_(out["s_row"]).reshape(rows, cols // 32), sr)
    nd2, nz2 = codes_equal_up_to_zero_sign(np_(out["q_col"]), qc)
    assert nd2 == 0, f"{nd2} column-wise codes differ"
    assert np.array_equal(np_(out["s_col"]).reshape(cols, rows // 32), sc)
    print(f"zero-sign-only differences: row {nz}, col {nz2}")


def test_quantize_mma_layout_is_a_permutation():
    m = require_gpu()
    rows, cols = 256, 512
    x = synthetic.random_bf16((rows, cols), 99)
    a = m.mxg_mxfp8_quantize(x.cuda(), row=True, col=True, layout=m.MXG_LAYOUT_CANONICAL)
    b = m.mxg_mxfp8_quantize(x.cuda(), row=True, col=True, layout=m.MXG_LAYOUT_MMA)
    torch.cuda.synchronize()
    assert torch.equal(a["q_row"], b["q_row"]) and torch.equal(a["q_col"], b["q_col"])
    assert np.array_equal(mma_to_canonical(b["s_row"], rows, cols // 32), np_(a["s_row"]).reshape(rows, -1))
    assert np.array_equal(mma_to_canonical(b["s_col"], cols, rows // 32), np_(a["s_col"]).reshape(cols, -1))
