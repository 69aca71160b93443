"""Guard bytes around every buffer a call writes: each output, the saved and
workspace buffers and the status word sit inside a larger allocation whose
4 KB before and after hold a known pattern, checked after the calls.  A
kernel that writes past its buffer's end (or before its start) changes the
pattern.  The results must also equal, bit for bit, the same calls on plain
allocations.  Covers the MXFP8 path (ragged groups, an empty expert, with
and without the weight cache and fp32 main_grad), the BF16 and FP8 paths,
the pre-grouped call, the standalone permute, grouped quantiser, gather and
combine."""
import numpy as np
import pytest
import torch

import synthetic
from gpu_helpers import require_gpu

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5


class Guarded:
    def __init__(self):
        self.bufs = []

    def new(self, shape, dtype, fill=None):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        n_al = -(-n // 256) * 256
        buf = torch.full((GUARD + n_al + GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        inner = buf[GUARD:GUARD + n].view(dtype).view(shape)
        if fill is not None:
            inner.fill_(fill)
        self.bufs.append((buf, n))
        return inner

    def check(self):
        torch.cuda.synchronize()
        for buf, n in self.bufs:
            assert bool((buf[:GUARD] == PATTERN).all()), "guard bytes before a buffer changed"
            assert bool((buf[GUARD + n:] == PATTERN).all()), "guard bytes after a buffer changed"


@pytest.mark.parametrize("precision", ["mxfp8", "bf16", "fp8"])
def test_mlp_writes_stay_inside_their_buffers(precision):
    m = require_gpu()
    from mxfp8_grouped_gemm_gb300 import _lib
    T, H, I, E, k = 300, 256, 512, 6, 2
    inp = synthetic.make_case(T, H, I, E, k, seed=61, empty_experts=(2,))
    d = {n: inp[n].cuda() for n in ("logits", "x", "w_gate_up", "w_down", "dy")}
    ref = m.GroupedMLP(T, H, I, E, k, precision=precision)
    ids, probs = ref.route(d["logits"])
    ref.forward(d["x"], ids, probs, d["w_gate_up"], d["w_down"])
    want = [t.clone() for t in (ref.y, ref.split_sizes) + tuple(ref.backward(d["dy"]))]

    g = Guarded()
    sizes = {"mxfp8": (_lib.mxg_mlp_saved_bytes, _lib.mxg_mlp_workspace_bytes),
             "bf16": (_lib.mxg_mlp_bf16_saved_bytes, _lib.mxg_mlp_bf16_workspace_bytes),
             "fp8": (_lib.mxg_mlp_fp8_saved_bytes, _lib.mxg_mlp_fp8_workspace_bytes)}[precision]
    saved = g.new((sizes[0](T, H, I, E, k),), torch.uint8)
    ws = g.new((sizes[1](T, H, I, E, k),), torch.uint8)
    st = g.new((1,), torch.int32, 0)
    y, split = g.new((T, H), torch.bfloat16), g.new((E,), torch.int32)
    dx, dprobs = g.new((T, H), torch.bfloat16), g.new((T, k), torch.float32)
    dwgu, dwd = g.new((E, 2 * I, H), torch.bfloat16), g.new((E, H, I), torch.bfloat16)
    kw = {"bf16": precision == "bf16", "fp8": precision == "fp8"}
    _lib.mxg_grouped_mlp_fwd(d["x"], ids, probs, d["w_gate_up"], d["w_down"], saved, ws, st, y=y, split_sizes=split,
                             **kw)
    _lib.mxg_grouped_mlp_bwd(d["dy"], saved, ws, st, E, I, k, dx=dx, dw_gate_up=dwgu, dw_down=dwd, dprobs=dprobs,
                             **kw)
    g.check()
    assert int(st.item()) == 0
    for got, w in zip((y, split, dx, dwgu, dwd, dprobs), want):
        assert torch.equal(got, w)

    if precision == "mxfp8":
        # the weight cache and fp32 main_grad accumulation
        cache = _lib.WeightCache(H, I, E)
        cache.buffer = g.new((cache.buffer.numel(),), torch.uint8)
        _lib.mxg_mlp_quantize_weights(d["w_gate_up"], d["w_down"], cache)
        saved_c = g.new((_lib.mxg_mlp_saved_bytes_cached(T, H, I, E, k),), torch.uint8)
        mg = (g.new((E, 2 * I, H), torch.float32, 0.0), g.new((E, H, I), torch.float32, 0.0))
        _lib.mxg_grouped_mlp_fwd(d["x"], ids, probs, None, None, saved_c, ws, st, y=y, split_sizes=split,
                                 weight_cache=cache)
        _lib.mxg_grouped_mlp_bwd(d["dy"], saved_c, ws, st, E, I, k, dx=dx, dprobs=dprobs, weight_cache=cache,
                                 main_grad=mg)
        g.check()
        assert int(st.item()) == 0
        assert torch.equal(y, want[0]) and torch.equal(dx, want[2])


def test_pregrouped_and_row_entries_stay_inside_their_buffers():
    m = require_gpu()
    from mxfp8_grouped_gemm_gb300 import _lib
    T, H, I, E, k = 200, 256, 256, 5, 2
    inp = synthetic.make_case(T, H, I, E, k, seed=62, empty_experts=(0,))
    d = {n: inp[n].cuda() for n in ("logits", "x", "w_gate_up", "w_down", "dy")}
    st0 = torch.zeros(1, dtype=torch.int32, device="cuda")
    ids, probs = m.mxg_route_topk(d["logits"], k)
    pm = m.mxg_route_permute(ids, E, st0)
    R = T * k
    g = Guarded()
    st = g.new((1,), torch.int32, 0)
    # gather and combine
    xg = g.new((R, H), torch.bfloat16)
    _lib.mxg_gather_rows(d["x"], pm["src_of_row"], st, div=k, out=xg)
    pg = g.new((R,), torch.float32)
    _lib.mxg_gather_rows(probs.reshape(-1), pm["src_of_row"], st, out=pg)
    # the pre-grouped forward / backward
    saved = g.new((_lib.mxg_mlp_grouped_saved_bytes(R, H, I, E),), torch.uint8)
    ws = g.new((_lib.mxg_mlp_grouped_workspace_bytes(R, H, I, E),), torch.uint8)
    yg = g.new((R, H), torch.bfloat16)
    _lib.mxg_grouped_mlp_fwd_grouped(xg, pm["split_sizes"], pg, d["w_gate_up"], d["w_down"], saved, ws, st, y=yg)
    dyg = m.mxg_gather_rows(d["dy"], pm["src_of_row"], st0, div=k)
    dxg, dpg = g.new((R, H), torch.bfloat16), g.new((R, 1), torch.float32)
    dwgu, dwd = g.new((E, 2 * I, H), torch.bfloat16), g.new((E, H, I), torch.bfloat16)
    _lib.mxg_grouped_mlp_bwd(dyg, saved, ws, st, E, I, 1, dx=dxg, dw_gate_up=dwgu, dw_down=dwd, dprobs=dpg)
    y = g.new((T, H), torch.bfloat16)
    _lib.mxg_combine(yg, pm["row_of_src"], k, st, y=y)
    g.check()
    assert int(st.item()) == 0 and int(st0.item()) == 0
    ref = m.GroupedMLP(T, H, I, E, k)
    y_ref, _ = ref.forward(d["x"], ids, probs, d["w_gate_up"], d["w_down"])
    assert torch.equal(y, y_ref)


def test_standalone_quantisers_stay_inside_their_buffers():
    m = require_gpu()
    from mxfp8_grouped_gemm_gb300 import _lib
    rng = np.random.default_rng(63)
    rows, cols = 300, 256
    x = torch.from_numpy(rng.standard_normal((rows, cols)).astype(np.float32)).to(torch.bfloat16).cuda()
    off = torch.tensor([0, 37, 37, 200, 300], dtype=torch.int32, device="cuda")
    for layout in (0, 1):
        g = Guarded()
        st = g.new((1,), torch.int32, 0)
        cap = _lib.mxg_mxfp8_grouped_rows_capacity(rows, 4, layout)
        poff = g.new((5,), torch.int32)
        qr, sr = g.new((cap, cols), torch.uint8), g.new((cap * cols // 32,), torch.uint8)
        qc, sc = g.new((cols, cap), torch.uint8), g.new((cap * cols // 32,), torch.uint8)
        rc = _lib.lib().mxg_mxfp8_quantize_grouped(x.data_ptr(), rows, cols, off.data_ptr(), 4, poff.data_ptr(),
                                                   qr.data_ptr(), sr.data_ptr(), qc.data_ptr(), sc.data_ptr(),
                                                   layout, st.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert rc == 0
        g.check()
        assert int(st.item()) == 0
    # the ungrouped quantiser and the permute
    g = Guarded()
    xs = x[:256].contiguous()
    qr, sr = g.new((256, cols), torch.uint8), g.new((256 * cols // 32,), torch.uint8)
    qc, sc = g.new((cols, 256), torch.uint8), g.new((256 * cols // 32,), torch.uint8)
    rc = _lib.lib().mxg_mxfp8_quantize(xs.data_ptr(), 256, cols, qr.data_ptr(), sr.data_ptr(), qc.data_ptr(),
                                       sc.data_ptr(), 1, torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    T, E, k = 1000, 16, 4
    logits = torch.from_numpy(rng.standard_normal((T, E)).astype(np.float32)).cuda()
    ids, probs = m.mxg_route_topk(logits, k)
    st = g.new((1,), torch.int32, 0)
    wsb = _lib.lib().mxg_route_permute_workspace_bytes(T, k, E)
    ws = g.new((wsb,), torch.uint8)
    outs = [g.new((E,), torch.int32), g.new((T * k,), torch.int32), g.new((T * k,), torch.int32),
            g.new((E + 1,), torch.int32)]
    rc = _lib.lib().mxg_route_permute(ids.data_ptr(), T, k, E, *[o.data_ptr() for o in outs], ws.data_ptr(), wsb,
                                      st.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    g.check()
    assert int(st.item()) == 0
