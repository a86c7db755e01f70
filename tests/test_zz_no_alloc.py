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

from gpu_util import to_device

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


def _workspace_call(d, wl, path):
    qsa.set_config(qsa.QSA_CFG_PATH, path)
    try:
        ri, rv = qsa.select_paged_tokens(d["q"], d["w"], d["keys"], d["row_req"], d["row_visible"], wl.k)
    finally:
        qsa.set_config(qsa.QSA_CFG_PATH, qsa.PATH_AUTO)
    return ri.cpu().numpy(), rv.cpu().numpy()


def _noalloc_on_path(lib, d, wl, path):
    qsa.set_config(qsa.QSA_CFG_PATH, path)
    try:
        return _noalloc(lib, d, wl, wl.k)
    finally:
        qsa.set_config(qsa.QSA_CFG_PATH, qsa.PATH_AUTO)


def test_noalloc_tiny_matches_oracle(lib):
    import oracle
    wl = W.tiny()
    d = to_device(wl)
    oi, ov, _ = oracle.select_paged_tokens(wl.q, wl.w, wl.k_cache, wl.block_table, wl.row_req,
                                           wl.row_visible, wl.k, ld=wl.ld)
    for path in (qsa.PATH_AUTO, qsa.PATH_FILTER):
        for _ in range(2):
            gi, gv = _noalloc_on_path(lib, d, wl, path)
            np.testing.assert_array_equal(gi, oi)
            np.testing.assert_array_equal(gv, ov)
    assert qsa.get_device_status() == qsa.QSA_OK


# Two different batches in turn, each twice: the shared buffer then holds the
# other batch's (or the same batch's) leftovers when a call starts.  "long"
# takes the sampled-threshold filter path on its own (7,500 positions, k 512);
# "short" (fewer rows and positions) is run on both paths.
_BATCHES = {
    "long": dict(seed=31, ctx_tokens=[30000], rows_per_req=[100], k=512),
    "short": dict(seed=32, ctx_tokens=[20000, 9000], rows_per_req=[40, 24], k=256),
}


@pytest.mark.parametrize("path", [qsa.PATH_AUTO, qsa.PATH_FILTER, qsa.PATH_DENSE])
def test_noalloc_matches_workspace_entry_point_on_two_calls(lib, path):
    wls = {n: W.make_workload(f"noalloc_{n}", **kw) for n, kw in _BATCHES.items()}
    devs = {n: to_device(wl) for n, wl in wls.items()}
    want = {n: _workspace_call(devs[n], wl, path) for n, wl in wls.items()}
    for n in ("long", "short", "long", "short", "short"):
        gi, gv = _noalloc_on_path(lib, devs[n], wls[n], path)
        np.testing.assert_array_equal(gi, want[n][0])        # same kernels, same inputs: bit for bit
        np.testing.assert_array_equal(gv, want[n][1])
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
