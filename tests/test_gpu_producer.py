"""GPU parity of the index-key producer (qsa_index_key_produce, qsa_rope_table)
with the oracle in oracle/producer.py, on the same seeded inputs.

Tolerance: the kernel pools, normalises and rotates in FP32 (cos / sin from
the FP64-built table), the oracle in FP64; both round the key to FP16.  The
FP32 path differs from FP64 by a few parts in 1e7, so the two FP16 results
are equal or one FP16 step apart (the exact value near a rounding midpoint):
|gpu - oracle| <= spacing_fp16(|oracle|) + 2e-6.  Slots the call does not
write must come back bit-identical.
"""
import numpy as np
import pytest
import torch

from block_sparse_attention_select_gb300 import qsa, workloads as W
from oracle import producer as P

pytestmark = pytest.mark.gpu


def _fp16_close(got, want):
    g = got.astype(np.float64)
    w = want.astype(np.float64)
    tol = np.spacing(np.abs(want).astype(np.float16)).astype(np.float64) + 2e-6
    bad = np.abs(g - w) > tol
    assert not bad.any(), f"{int(bad.sum())} values off, worst {np.max(np.abs(g - w)):.3g}"


def _run(inp, rope_dim=None, table_blocks=None):
    rope_dim = inp.rope_dim if rope_dim is None else rope_dim
    dev = "cuda"
    kc = torch.from_numpy(inp.k_cache.copy()).to(dev)
    keys = qsa.PagedKeys(kc, torch.from_numpy(inp.block_table).to(dev))
    blocks_needed = int(((inp.pos_start.astype(np.int64) + np.diff(inp.seq_start)) // 4).max()) + 1
    nb = blocks_needed if table_blocks is None else table_blocks
    tab = qsa.rope_table(nb, rope_dim, inp.theta) if rope_dim > 0 else None
    pl = torch.from_numpy(inp.pool_logit).to(dev) if inp.pool_logit is not None else None
    qsa.index_key_produce(torch.from_numpy(inp.x).to(dev), torch.from_numpy(inp.seq_start).to(dev),
                          torch.from_numpy(inp.pos_start).to(dev), inp.max_tokens,
                          torch.from_numpy(inp.norm_weight).to(dev), tab, keys, pool_logit=pl,
                          eps=inp.eps, rope_dim=rope_dim, window=inp.window)
    status = qsa.get_device_status()
    return kc.cpu().numpy(), status


def _oracle(inp, rope_dim=None):
    rope_dim = inp.rope_dim if rope_dim is None else rope_dim
    return P.produce(inp.x, inp.pool_logit, inp.seq_start, inp.pos_start, inp.norm_weight, inp.eps,
                     rope_dim, inp.theta, inp.window, inp.k_cache, inp.block_table)


def _compare(inp, got, want, done):
    written = np.zeros(inp.k_cache.shape[:2], bool)
    for b, i in done:
        written[inp.block_table[b, i // 16], i % 16] = True
    _fp16_close(got[written], want[written])
    np.testing.assert_array_equal(got[~written], inp.k_cache[~written])


@pytest.mark.parametrize("window,logits", [(4, False), (4, True), (8, False), (8, True)])
@pytest.mark.parametrize("rope_dim", [0, 64, 128])
def test_producer_matches_oracle(window, logits, rope_dim):
    inp = W.producer_small(window=window, logits=logits)
    got, st = _run(inp, rope_dim=rope_dim)
    assert st == qsa.QSA_OK, qsa.status_string(st)
    want, done = _oracle(inp, rope_dim=rope_dim)
    assert len(done) > 80
    _compare(inp, got, want, done)


def test_rope_table_matches_fp64():
    n, rd, theta = 5000, 64, 10000.0
    tab = qsa.rope_table(n, rd, theta).cpu().numpy().astype(np.float64)
    i = np.arange(n, dtype=np.float64)[:, None]
    j = np.arange(rd // 2, dtype=np.float64)[None, :]
    ang = 4.0 * i * np.power(theta, -2.0 * j / rd)
    want = np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32).astype(np.float64)
    # the device's and numpy's FP64 pow / sincos may differ by an ulp or two:
    # at angles up to 4 * 5000 that is ~1e-11 absolute, which matters (against
    # an FP32 ulp) only for cos / sin near zero, and the rotation error is
    # absolute: one FP32 step of the value plus 1e-10
    diff = np.abs(tab - want)
    tol = np.spacing(np.abs(want).astype(np.float32)).astype(np.float64) + 1e-10
    assert np.all(diff <= tol), f"worst {diff.max():.3g}"
    assert np.mean(diff == 0) > 0.99                  # almost all equal after rounding to FP32


def test_producer_bad_page_is_flagged_and_skipped():
    inp = W.producer_small()
    bt = inp.block_table.copy()
    first = P.produced_blocks(int(inp.pos_start[1]), int(inp.seq_start[2] - inp.seq_start[1]), inp.window)[0]
    bt[1, first // 16] = inp.k_cache.shape[0] + 5  # the page of request 1's first block: outside the cache
    inp.block_table = bt
    got, st = _run(inp)
    assert st == qsa.QSA_ERR_BAD_PAGE
    want, done = _oracle(inp)                      # the oracle skips that page's blocks too
    _compare(inp, got, want, done)


def test_producer_short_rope_table_is_flagged():
    inp = W.producer_small()
    got, st = _run(inp, table_blocks=10)           # request 6 reaches block 324
    assert st == qsa.QSA_ERR_INVALID_ARG
    want, done = _oracle(inp)
    ok = [(b, i) for b, i in done if i < 10]       # blocks past the table are skipped
    assert 0 < len(ok) < len(done)
    _compare(inp, got, want, ok)


@pytest.mark.parametrize("window", [4, 8])
def test_producer_full_context(window):
    """The whole 184,320-token context of one request: 46,080 keys."""
    inp = W.producer_context(window=window, logits=window == 8)
    got, st = _run(inp)
    assert st == qsa.QSA_OK, qsa.status_string(st)
    want, done = _oracle(inp)
    assert len(done) == 46_080
    _compare(inp, got, want, done)


def test_producer_chunk_at_the_end_of_a_long_context():
    inp = W.producer_chunk()
    got, st = _run(inp)
    assert st == qsa.QSA_OK, qsa.status_string(st)
    want, done = _oracle(inp)
    assert len(done) == 404
    _compare(inp, got, want, done)
