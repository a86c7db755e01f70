"""GPU parity of the sparse-attention consumer (qsa_sparse_attention) with the
oracle in oracle/consumer.py, on the same seeded inputs.

Tolerance: the kernel accumulates in FP32 (scores over 256 products, an online
softmax with FP32 exponentials, 4 * k + 3 weighted values) and the oracle in
FP64.  The outputs are convex combinations of FP16 values of magnitude ~1-4,
and the FP32 path is good to ~1e-6 relative per step, so |gpu - oracle| <=
2e-4 + 2e-4 * |oracle| leaves a wide margin while a wrong token, head or
weight moves the output by far more.
"""
import numpy as np
import pytest
import torch

from block_sparse_attention_select_gb300 import qsa, workloads as W
from oracle import consumer as C

pytestmark = pytest.mark.gpu


def _run(inp, scale=None, sel=None, block_table=None):
    dev = "cuda"
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    bt = inp.block_table if block_table is None else block_table
    out = qsa.sparse_attention(t(inp.q), t(inp.k_cache), t(inp.v_cache), t(bt), t(inp.row_req),
                               t(inp.row_token), t(inp.sel if sel is None else sel), scale=scale)
    return out.cpu().numpy().astype(np.float64), qsa.get_device_status()


def _oracle(inp, scale=None, sel=None, block_table=None):
    bt = inp.block_table if block_table is None else block_table
    return C.sparse_attention(inp.q, inp.k_cache, inp.v_cache, bt, inp.row_req, inp.row_token,
                              inp.sel if sel is None else sel, scale)


def _close(got, want):
    np.testing.assert_allclose(got, want, rtol=2e-4, atol=2e-4)


@pytest.mark.parametrize("scale", [None, 1.0])
def test_consumer_matches_oracle(scale):
    inp = W.make_consumer_inputs("c", seed=21, ctx_tokens=[300, 130, 75, 9], rows_per_req=[6, 3, 4, 2], k=16)
    got, st = _run(inp, scale)
    assert st == qsa.QSA_OK, qsa.status_string(st)
    _close(got, _oracle(inp, scale))


def test_consumer_every_position_selected():
    inp = W.make_consumer_inputs("c", seed=22, ctx_tokens=[300, 130], rows_per_req=[6, 3], k=80)
    got, st = _run(inp, 1.0)
    assert st == qsa.QSA_OK, qsa.status_string(st)
    _close(got, _oracle(inp, 1.0))


def test_consumer_k2048_long_context():
    """k = 2,048 positions (8,192 raw tokens per row, 257 chunks) over a 40,000-token context."""
    inp = W.make_consumer_inputs("c", seed=23, ctx_tokens=[40_000], rows_per_req=[6], k=2048)
    got, st = _run(inp)
    assert st == qsa.QSA_OK, qsa.status_string(st)
    _close(got, _oracle(inp))


def test_consumer_bad_page_is_flagged():
    inp = W.make_consumer_inputs("c", seed=24, ctx_tokens=[300], rows_per_req=[2], k=16)
    bt = inp.block_table.copy()
    bt[0, 0] = inp.k_cache.shape[0] + 7                  # tokens 0..63: outside the cache
    sel = inp.sel.copy()
    sel[:, 0] = 3                                         # every row reads a token of page 0
    _, st = _run(inp, sel=sel, block_table=bt)
    assert st == qsa.QSA_ERR_BAD_PAGE
