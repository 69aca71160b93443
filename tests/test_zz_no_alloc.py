"""The permute entry point that takes no scratch buffer (for callers that cannot
allocate device memory where they route tokens).  Called through the C ABI and
checked against the regular entry point (which takes caller scratch) on two
calls in a row; the outputs are integer indices, so they must match exactly.
Collected last so a failure here leaves every other test already run."""
import ctypes

import numpy as np
import pytest
import torch

from gpu_helpers import require_gpu

pytestmark = pytest.mark.gpu


def _noalloc(L, ids, E, st):
    T, k = ids.shape
    dev = ids.device
    out = {"split_sizes": torch.full((E,), -7, dtype=torch.int32, device=dev),
           "src_of_row": torch.full((T * k,), -7, dtype=torch.int32, device=dev),
           "row_of_src": torch.full((T * k,), -7, dtype=torch.int32, device=dev),
           "padded_offsets": torch.full((E + 1,), -7, dtype=torch.int32, device=dev)}
    rc = L.mxg_route_permute_noalloc(ids.data_ptr(), T, k, E, out["split_sizes"].data_ptr(),
                                     out["src_of_row"].data_ptr(), out["row_of_src"].data_ptr(),
                                     out["padded_offsets"].data_ptr(), st.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream)
    assert rc == 0, rc
    return out


def test_noalloc_permute_matches_regular_entry_twice():
    m = require_gpu()
    L = m.lib()
    cases = [(4096, 8, 2, 1), (8192, 64, 8, 2), (300, 5, 1, 3)]
    for T, E, k, seed in cases:
        rng = np.random.default_rng(seed)
        logits = torch.from_numpy(rng.standard_normal((T, E)).astype(np.float32)).cuda()
        ids, _ = m.mxg_route_topk(logits, k)
        st_ref = torch.zeros(1, dtype=torch.int32, device="cuda")
        ref = m.mxg_route_permute(ids, E, st_ref)
        for call in range(2):                        # two calls in a row share the scratch
            st = torch.zeros(1, dtype=torch.int32, device="cuda")
            got = _noalloc(L, ids, E, st)
            torch.cuda.synchronize()
            assert int(st.item()) == 0 and int(st_ref.item()) == 0
            for name in ref:
                assert torch.equal(got[name], ref[name]), (T, E, k, call, name)


def test_noalloc_permute_at_its_size_limit():
    """E = 256 with exactly mxg_route_permute_noalloc_max_entries(256) routed
    entries: the scratch's per-chunk counts and bases fill the static array to
    its end; results must still equal the regular entry point's, and one more
    entry is rejected on the host."""
    m = require_gpu()
    L = m.lib()
    E, k = 256, 8
    limit = int(L.mxg_route_permute_noalloc_max_entries(E))
    assert limit % k == 0
    T = limit // k
    rng = np.random.default_rng(11)
    logits = torch.from_numpy(rng.standard_normal((T, E)).astype(np.float32)).cuda()
    ids, _ = m.mxg_route_topk(logits, k)
    st_ref = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = m.mxg_route_permute(ids, E, st_ref)
    for call in range(2):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        got = _noalloc(L, ids, E, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0 and int(st_ref.item()) == 0
        for name in ref:
            assert torch.equal(got[name], ref[name]), (call, name)
    fake = ctypes.c_void_p(0x10000)
    rc = L.mxg_route_permute_noalloc(fake, limit + 1, 1, E, fake, fake, fake, fake, fake, None)
    assert rc == 5                                   # MXG_ERR_WORKSPACE, nothing launched


def test_noalloc_permute_leaves_device_memory_unchanged():
    """After a first call on the device, a call changes neither the free device
    memory nor torch's allocated bytes: the entry point allocates nothing."""
    m = require_gpu()
    L = m.lib()
    T, E, k = 2048, 8, 2
    rng = np.random.default_rng(12)
    logits = torch.from_numpy(rng.standard_normal((T, E)).astype(np.float32)).cuda()
    ids, _ = m.mxg_route_topk(logits, k)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    _noalloc(L, ids, E, st)                          # first call on this device: address lookup, module load
    out = {"split_sizes": torch.empty(E, dtype=torch.int32, device="cuda"),
           "src_of_row": torch.empty(T * k, dtype=torch.int32, device="cuda"),
           "row_of_src": torch.empty(T * k, dtype=torch.int32, device="cuda"),
           "padded_offsets": torch.empty(E + 1, dtype=torch.int32, device="cuda")}
    torch.cuda.synchronize()
    free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    rc = L.mxg_route_permute_noalloc(ids.data_ptr(), T, k, E, out["split_sizes"].data_ptr(),
                                     out["src_of_row"].data_ptr(), out["row_of_src"].data_ptr(),
                                     out["padded_offsets"].data_ptr(), st.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0 and int(st.item()) == 0
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_allocated() == alloc0


def test_noalloc_permute_rejects_oversize_on_host():
    m = require_gpu()
    L = m.lib()
    E, k = 8, 2
    limit = L.mxg_route_permute_noalloc_max_entries(E)
    T = limit // k + 1
    fake = ctypes.c_void_p(0x10000)
    rc = L.mxg_route_permute_noalloc(fake, T, k, E, fake, fake, fake, fake, fake, None)
    assert rc == 5                                   # MXG_ERR_WORKSPACE, nothing launched
