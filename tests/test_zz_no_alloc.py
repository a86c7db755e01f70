"""The allocation-free entry point (qsa_select_paged_tokens_noalloc).

For callers that cannot allocate device memory on their hot path: the call
borrows a scratch buffer that lives inside the library.  It must give the same
answer as the workspace entry point, on two calls in a row (the buffer keeps
the previous call's contents), and refuse work that does not fit the buffer.
This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from block_sparse_attention_select_gb300 import qsa
from block_sparse_attention_select_gb300 import workloads as W

from gpu_util import ATOL, RTOL, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()
    return qsa.load()


def _noalloc(lib, d, wl, k):
    oi = torch.full((wl.rows, k), -7, dtype=torch.int32, device="cuda")
    ov = torch.full((wl.rows, k), 7.0, dtype=torch.float32, device="cuda")
    st = lib.qsa_select_paged_tokens_noalloc(
        ctypes.c_void_p(d["q"].data_ptr()), ctypes.c_void_p(d["w"].data_ptr()), wl.rows, wl.heads,
        ctypes.byref(d["keys"].c), ctypes.c_void_p(d["row_req"].data_ptr()),
        ctypes.c_void_p(d["row_visible"].data_ptr()), k, ctypes.c_void_p(oi.data_ptr()),
        ctypes.c_void_p(ov.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == qsa.QSA_OK, qsa.status_string(st)
    return oi.cpu().numpy(), ov.cpu().numpy()


@pytest.mark.parametrize("which", ["tiny", "gauss"])
def test_noalloc_matches_workspace_entry_point_on_two_calls(lib, which):
    if which == "tiny":
        wl = W.tiny()
    else:
        wl = W.make_workload("noalloc", seed=31, ctx_tokens=[20000, 9000], rows_per_req=[40, 24],
                             k=256)
    d = to_device(wl)
    ri, rv = qsa.select_paged_tokens(d["q"], d["w"], d["keys"], d["row_req"], d["row_visible"],
                                     wl.k)
    ri, rv = ri.cpu().numpy(), rv.cpu().numpy()
    for _ in range(2):
        gi, gv = _noalloc(lib, d, wl, wl.k)
        np.testing.assert_array_equal(gi, ri)
        fin = np.isfinite(rv)
        np.testing.assert_array_equal(np.isfinite(gv), fin)
        np.testing.assert_allclose(gv[fin], rv[fin], rtol=RTOL, atol=ATOL)
    assert qsa.get_device_status() == qsa.QSA_OK


def test_noalloc_refuses_work_beyond_its_buffer(lib):
    wl = W.tiny()
    d = to_device(wl)
    rows = 1 << 20                     # far more rows than the buffer can plan for
    big = qsa.PagedKeysC(d["keys"].c.k_cache, d["keys"].c.num_pages, 16, 128,
                         d["keys"].c.block_table, 1, 4096)
    st = lib.qsa_select_paged_tokens_noalloc(
        ctypes.c_void_p(d["q"].data_ptr()), ctypes.c_void_p(d["w"].data_ptr()), rows, 4,
        ctypes.byref(big), ctypes.c_void_p(d["row_req"].data_ptr()),
        ctypes.c_void_p(d["row_visible"].data_ptr()), 64, ctypes.c_void_p(0), None, None)
    assert st == qsa.QSA_ERR_STATIC_LIMIT
    assert qsa.last_launch_count() == 0
