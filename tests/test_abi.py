"""Host-side checks of the C ABI (no GPU needed): the library builds and loads,
exports every function include/mxg.h declares, and rejects bad arguments on
the host before anything is launched."""
import ctypes
import os
import re
import subprocess

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "mxg.h")


@pytest.fixture(scope="module")
def L():
    from mxfp8_grouped_gemm_gb300 import build
    build.build()
    import mxfp8_grouped_gemm_gb300 as m
    return m.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mxg_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_path():
    names = declared_functions()
    for n in ["mxg_route_topk", "mxg_route_permute", "mxg_mxfp8_quantize", "mxg_grouped_gemm",
              "mxg_grouped_gemm_wgrad", "mxg_grouped_mlp_fwd", "mxg_grouped_mlp_bwd"]:
        assert n in names


def test_exports_every_declared_symbol(L):
    from mxfp8_grouped_gemm_gb300 import EXPORTS, LIB_PATH
    out = subprocess.run(["nm", "-D", "--defined-only", LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (mxg_\w+)", out))
    for n in declared_functions():
        assert n in exported, n
        assert hasattr(L, n)
    assert set(EXPORTS) == set(declared_functions())


def test_status_strings(L):
    import mxfp8_grouped_gemm_gb300 as m
    for code in [0, 1, 2, 3, 4, 5, 6, 16, 17, 18]:
        s = m.status_string(code)
        assert s and s != "unknown status"
    assert m.status_string(12345) == "unknown status"


FAKE = 0x10000          # 16-byte aligned, never dereferenced: the calls fail validation first
MISALIGNED = 0x10008


def test_route_topk_validation(L):
    assert L.mxg_route_topk(None, 4, 8, 2, FAKE, FAKE, None) == 1
    assert L.mxg_route_topk(FAKE, 0, 8, 2, FAKE, FAKE, None) == 1
    assert L.mxg_route_topk(FAKE, 4, 8, 9, FAKE, FAKE, None) == 2       # k > E
    assert L.mxg_route_topk(FAKE, 4, 300, 2, FAKE, FAKE, None) == 2     # E > 256
    assert L.mxg_route_topk(MISALIGNED, 4, 8, 2, FAKE, FAKE, None) == 3


def test_permute_validation(L):
    args = [FAKE, 16, 2, 8, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, FAKE, None]
    a = list(args); a[0] = None
    assert L.mxg_route_permute(*a) == 1
    a = list(args); a[2] = 9
    assert L.mxg_route_permute(*a) == 2
    a = list(args); a[4] = MISALIGNED
    assert L.mxg_route_permute(*a) == 3
    a = list(args); a[9] = 4
    assert L.mxg_route_permute(*a) == 5
    assert L.mxg_route_permute_workspace_bytes(16, 2, 8) > 0
    assert L.mxg_route_permute_workspace_bytes(0, 2, 8) == 0


def test_quantize_validation(L):
    assert L.mxg_mxfp8_quantize(None, 32, 128, FAKE, FAKE, None, None, 0, None) == 1
    assert L.mxg_mxfp8_quantize(FAKE, 32, 128, None, None, None, None, 0, None) == 1   # nothing requested
    assert L.mxg_mxfp8_quantize(FAKE, 32, 128, FAKE, None, None, None, 0, None) == 1   # codes without scales
    assert L.mxg_mxfp8_quantize(FAKE, 32, 128, FAKE, FAKE, None, None, 7, None) == 1   # bad layout
    assert L.mxg_mxfp8_quantize(FAKE, 33, 128, FAKE, FAKE, None, None, 0, None) == 2
    assert L.mxg_mxfp8_quantize(FAKE, 32, 96, FAKE, FAKE, None, None, 0, None) == 2
    assert L.mxg_mxfp8_quantize(FAKE, 32, 128, FAKE, FAKE, None, None, 1, None) == 2   # MMA layout needs 128 rows
    assert L.mxg_mxfp8_quantize(MISALIGNED, 32, 128, FAKE, FAKE, None, None, 0, None) == 3


def test_gemm_validation(L):
    base = [FAKE, FAKE, FAKE, FAKE, FAKE, 4, 512, 256, 256, FAKE, FAKE, None]
    a = list(base); a[0] = None
    assert L.mxg_grouped_gemm(*a) == 1
    a = list(base); a[8] = 200
    assert L.mxg_grouped_gemm(*a) == 2
    a = list(base); a[7] = 192
    assert L.mxg_grouped_gemm(*a) == 2
    a = list(base); a[6] = 500
    assert L.mxg_grouped_gemm(*a) == 2
    a = list(base); a[9] = MISALIGNED
    assert L.mxg_grouped_gemm(*a) == 3
    w = [FAKE, FAKE, FAKE, FAKE, FAKE, 4, 256, 256, 512, FAKE, FAKE, None]
    a = list(w); a[8] = 100
    assert L.mxg_grouped_gemm_wgrad(*a) == 2


def test_bf16_mlp_sizes_and_validation(L):
    assert L.mxg_mlp_bf16_saved_bytes(256, 256, 512, 4, 2) > 0
    assert L.mxg_mlp_bf16_workspace_bytes(256, 256, 512, 4, 2) > 0
    assert L.mxg_mlp_bf16_saved_bytes(256, 128, 512, 4, 2) == 0      # H not a multiple of 256
    assert L.mxg_mlp_bf16_saved_bytes(256, 256, 384, 4, 2) == 0      # I not a multiple of 256
    import mxfp8_grouped_gemm_gb300 as m
    a = m.MlpFwdArgs(256, 128, 512, 4, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, FAKE, 1 << 30, 1, FAKE)
    assert L.mxg_grouped_mlp_bf16_fwd(ctypes.byref(a), None) == 2
    a = m.MlpFwdArgs(256, 256, 512, 4, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, FAKE, 1 << 30, 1, FAKE)
    assert L.mxg_grouped_mlp_bf16_fwd(ctypes.byref(a), None) == 5      # saved buffer too small
    b = m.MlpBwdArgs(256, 256, 512, 4, 2, MISALIGNED, FAKE, 1 << 30, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, FAKE)
    assert L.mxg_grouped_mlp_bf16_bwd(ctypes.byref(b), None) == 3
    assert L.mxg_grouped_mlp_bf16_fwd_stage(ctypes.byref(a), 99, None) == 1


def test_router_validation(L):
    f = [FAKE, FAKE, 64, 256, 8, 2, FAKE, FAKE, FAKE, None]
    a = list(f); a[0] = None
    assert L.mxg_router_fwd(*a) == 1
    a = list(f); a[3] = 200                    # H not a multiple of 128
    assert L.mxg_router_fwd(*a) == 2
    a = list(f); a[5] = 9                      # k > E
    assert L.mxg_router_fwd(*a) == 2
    a = list(f); a[1] = MISALIGNED
    assert L.mxg_router_fwd(*a) == 3
    ws = L.mxg_router_bwd_workspace_bytes(64, 256, 8, 2)
    assert ws >= 64 * 2 * 4
    b = [FAKE, FAKE, FAKE, FAKE, FAKE, 64, 256, 8, 2, FAKE, FAKE, FAKE, ws, FAKE, None]
    a = list(b); a[9] = None
    assert L.mxg_router_bwd(*a) == 1
    a = list(b); a[6] = 192
    assert L.mxg_router_bwd(*a) == 2
    a = list(b); a[9] = MISALIGNED
    assert L.mxg_router_bwd(*a) == 3
    a = list(b); a[12] = ws - 1
    assert L.mxg_router_bwd(*a) == 5


def test_mlp_sizes_and_validation(L):
    import mxfp8_grouped_gemm_gb300 as m
    assert m.mxg_mlp_saved_bytes(256, 128, 256, 4, 2) > 0
    assert m.mxg_mlp_workspace_bytes(256, 128, 256, 4, 2) > 0
    assert m.mxg_mlp_saved_bytes(256, 100, 256, 4, 2) == 0          # H % 128
    assert m.mxg_mlp_saved_bytes(256, 128, 256, 4, 5) == 0          # k > E
    assert m.mxg_mlp_saved_bytes(512, 128, 256, 4, 2) > m.mxg_mlp_saved_bytes(256, 128, 256, 4, 2)
    align = m.mxg_mlp_group_align()
    assert align in (128, 256)
    assert m.mxg_mlp_row_capacity(300, 2, 6) == (600 + align - 1) // align * align + align * 6
    args = m.MlpFwdArgs(256, 128, 256, 4, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40, FAKE,
                        1 << 40, 1, FAKE)
    bad = m.MlpFwdArgs.from_buffer_copy(args)
    bad.x = None
    assert L.mxg_grouped_mlp_fwd(ctypes.byref(bad), None) == 1
    bad = m.MlpFwdArgs.from_buffer_copy(args)
    bad.H = 96
    assert L.mxg_grouped_mlp_fwd(ctypes.byref(bad), None) == 2
    bad = m.MlpFwdArgs.from_buffer_copy(args)
    bad.y = MISALIGNED
    assert L.mxg_grouped_mlp_fwd(ctypes.byref(bad), None) == 3
    bad = m.MlpFwdArgs.from_buffer_copy(args)
    bad.saved_bytes = 100
    assert L.mxg_grouped_mlp_fwd(ctypes.byref(bad), None) == 5
    assert L.mxg_grouped_mlp_fwd(None, None) == 1
    b = m.MlpBwdArgs(256, 128, 256, 4, 2, FAKE, FAKE, 1 << 40, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40, FAKE)
    bad = m.MlpBwdArgs.from_buffer_copy(b)
    bad.dprobs = None
    assert L.mxg_grouped_mlp_bwd(ctypes.byref(bad), None) == 1
    bad = m.MlpBwdArgs.from_buffer_copy(b)
    bad.workspace_bytes = 1
    assert L.mxg_grouped_mlp_bwd(ctypes.byref(bad), None) == 5


def test_struct_layout_matches_header(tmp_path):
    """ctypes mirrors of the argument structs agree with the C compiler's layout."""
    import mxfp8_grouped_gemm_gb300 as m
    src = tmp_path / "layout.c"
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "mxg.h"', "int main(void) {"]
    for cname, cls in [("mxg_mlp_fwd_args", m.MlpFwdArgs), ("mxg_mlp_bwd_args", m.MlpBwdArgs)]:
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for f, _ in cls._fields_:
            lines.append(f'printf("{cname} {f} %zu\\n", offsetof({cname}, {f}));')
    lines.append("return 0; }")
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    table = {}
    for line in got:
        if line:
            s, f, v = line.split()
            table[(s, f)] = int(v)
    for cname, cls in [("mxg_mlp_fwd_args", m.MlpFwdArgs), ("mxg_mlp_bwd_args", m.MlpBwdArgs)]:
        assert table[(cname, "size")] == ctypes.sizeof(cls)
        for f, _ in cls._fields_:
            assert table[(cname, f)] == getattr(cls, f).offset, (cname, f)


def test_weight_cache_and_main_grad_validation(L):
    import mxfp8_grouped_gemm_gb300 as m
    H, I, E = 128, 256, 4

    def carve(*sizes):
        off = 0
        for n in sizes:
            off = (off + n + 255) // 256 * 256
        return off
    gu, d = E * 2 * I * H, E * H * I
    assert L.mxg_mlp_weight_cache_bytes(H, I, E) == carve(gu, gu // 32, d, d // 32, gu, gu // 32, d, d // 32)
    assert L.mxg_mlp_weight_cache_bytes(100, I, E) == 0
    full, cached = L.mxg_mlp_saved_bytes(256, H, I, E, 2), L.mxg_mlp_saved_bytes_cached(256, H, I, E, 2)
    assert 0 < cached < full
    assert full - cached == carve(gu, gu // 32, d, d // 32)          # the transposed weights move to the cache
    cb = L.mxg_mlp_weight_cache_bytes(H, I, E)
    q = [FAKE, FAKE, H, I, E, FAKE, cb, None]
    a = list(q); a[0] = None
    assert L.mxg_mlp_quantize_weights(*a) == 1
    a = list(q); a[2] = 96
    assert L.mxg_mlp_quantize_weights(*a) == 2
    a = list(q); a[5] = MISALIGNED
    assert L.mxg_mlp_quantize_weights(*a) == 3
    a = list(q); a[6] = cb - 1
    assert L.mxg_mlp_quantize_weights(*a) == 5
    # forward with a cache: weights may be NULL; the cached saved size suffices, a short cache does not
    f = m.MlpFwdArgs(256, H, I, E, 2, FAKE, FAKE, FAKE, None, None, FAKE, FAKE, FAKE, cached, FAKE, 1 << 40, 1,
                     FAKE, FAKE, cb)
    bad = m.MlpFwdArgs.from_buffer_copy(f); bad.saved_bytes = cached - 1
    assert L.mxg_grouped_mlp_fwd(ctypes.byref(bad), None) == 5
    bad = m.MlpFwdArgs.from_buffer_copy(f); bad.weight_cache_bytes = cb - 1
    assert L.mxg_grouped_mlp_fwd(ctypes.byref(bad), None) == 5
    bad = m.MlpFwdArgs.from_buffer_copy(f); bad.weight_cache = None          # no weights at all
    assert L.mxg_grouped_mlp_fwd(ctypes.byref(bad), None) == 1
    bad = m.MlpFwdArgs.from_buffer_copy(f); bad.weight_cache = MISALIGNED
    assert L.mxg_grouped_mlp_fwd(ctypes.byref(bad), None) == 3
    # backward: main_grad both or neither; with it dW may be NULL
    b = m.MlpBwdArgs(256, H, I, E, 2, FAKE, FAKE, 1 << 40, FAKE, None, None, FAKE, FAKE, 1 << 40, FAKE, None, 0,
                     FAKE, None)
    assert L.mxg_grouped_mlp_bwd(ctypes.byref(b), None) == 1
    bad = m.MlpBwdArgs.from_buffer_copy(b); bad.main_grad_down = MISALIGNED
    assert L.mxg_grouped_mlp_bwd(ctypes.byref(bad), None) == 3
    bad = m.MlpBwdArgs.from_buffer_copy(b); bad.main_grad_down = FAKE; bad.weight_cache = FAKE
    bad.weight_cache_bytes = cb - 1; bad.saved_bytes = cached
    assert L.mxg_grouped_mlp_bwd(ctypes.byref(bad), None) == 5
    # the BF16 path takes neither
    H2, I2 = 256, 512
    f2 = m.MlpFwdArgs(256, H2, I2, E, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40, FAKE, 1 << 40, 1,
                      FAKE, FAKE, 1 << 40)
    assert L.mxg_grouped_mlp_bf16_fwd(ctypes.byref(f2), None) == 1
    b2 = m.MlpBwdArgs(256, H2, I2, E, 2, FAKE, FAKE, 1 << 40, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40, FAKE, None, 0,
                      FAKE, FAKE)
    assert L.mxg_grouped_mlp_bf16_bwd(ctypes.byref(b2), None) == 1


def test_fp8_mlp_sizes_and_validation(L):
    import mxfp8_grouped_gemm_gb300 as m
    assert L.mxg_mlp_fp8_saved_bytes(256, 256, 512, 4, 2) > 0
    assert L.mxg_mlp_fp8_workspace_bytes(256, 256, 512, 4, 2) > 0
    assert L.mxg_mlp_fp8_saved_bytes(256, 128, 512, 4, 2) == 0       # H not a multiple of 256
    assert L.mxg_mlp_fp8_saved_bytes(256, 256, 384, 4, 2) == 0       # I not a multiple of 256
    a = m.MlpFwdArgs(256, 128, 512, 4, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, FAKE, 1 << 30, 1,
                     FAKE, None, 0)
    assert L.mxg_grouped_mlp_fp8_fwd(ctypes.byref(a), None) == 2
    a = m.MlpFwdArgs(256, 256, 512, 4, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, FAKE, 1 << 30, 1, FAKE,
                     None, 0)
    assert L.mxg_grouped_mlp_fp8_fwd(ctypes.byref(a), None) == 5      # saved buffer too small
    bad = m.MlpFwdArgs.from_buffer_copy(a); bad.x = MISALIGNED; bad.saved_bytes = 1 << 30
    assert L.mxg_grouped_mlp_fp8_fwd(ctypes.byref(bad), None) == 3
    bad = m.MlpFwdArgs.from_buffer_copy(a); bad.weight_cache = FAKE
    assert L.mxg_grouped_mlp_fp8_fwd(ctypes.byref(bad), None) == 1    # the weight cache is MXFP8-only
    b = m.MlpBwdArgs(256, 256, 512, 4, 2, FAKE, FAKE, 1 << 30, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, FAKE, None, 0,
                     FAKE, FAKE)
    assert L.mxg_grouped_mlp_fp8_bwd(ctypes.byref(b), None) == 1      # main_grad is MXFP8-only
    assert L.mxg_grouped_mlp_fp8_fwd_stage(ctypes.byref(a), 99, None) == 1
    assert L.mxg_mlp_fp8_saved_view(None, 256, 256, 512, 4, 2, 0) is None
    assert L.mxg_mlp_fp8_saved_view(FAKE, 256, 256, 512, 4, 2, 9) is None


def test_saved_gu_tile_layout_reads_back_in_row_order():
    """The saved g|u tiles (documented in include/mxg.h, saved view 0) read
    back as [m_cap, 2I] rows: every element placed by the header's formula
    lands at its (row, column)."""
    import torch
    from mxfp8_grouped_gemm_gb300.layer import gu_rows_from_tiles
    m_cap, I = 96, 64
    want = torch.arange(m_cap * 2 * I, dtype=torch.float64).view(m_cap, 2 * I)
    flat = torch.full((m_cap * 2 * I,), -1.0, dtype=torch.float64)
    for row in range(m_cap):
        for col in range(2 * I):
            gate_up, j = divmod(col, I)
            rb, r = divmod(row, 32)
            cb, c = divmod(j, 32)
            h, c16 = divmod(c, 16)
            off = (rb * (I // 32) + cb) * 2048 + gate_up * 1024 + h * 512 + r * 16 + c16
            flat[off] = want[row, col]
    assert bool((flat >= 0).all())
    assert torch.equal(gu_rows_from_tiles(flat, m_cap, I), want)
