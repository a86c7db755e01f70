"""GPU parity of the M3-style block scorer (qsa_block_select) against its
oracle (oracle/block_scorer.py, numpy float64).

A block's score is the maximum raw-token dot product over its visible tokens,
per query row and KV head; the top-k blocks are ordered by score, then block
index.  Integer-valued inputs make every FP32 dot product exact, so indices
and values must match bit for bit; on Gaussian inputs the values must agree
within |g - o| <= 1e-3 |o| + 1e-6 and the selected sets may differ only at
near-ties of the cut.
"""
import numpy as np
import pytest
import torch

from oracle import block_scorer as BS
from block_sparse_attention_select_gb300 import qsa
from block_sparse_attention_select_gb300 import workloads as W

from gpu_util import ATOL, RTOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    qsa.load()
    assert torch.cuda.is_available()
    yield
    assert qsa.get_device_status() == qsa.QSA_OK


def _run(inp, k=None, block_table=None):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    bt = inp.block_table if block_table is None else block_table
    gi, gv = qsa.block_select(t(inp.q), t(inp.k_cache), t(bt), t(inp.row_req), t(inp.row_token),
                              inp.k if k is None else k)
    return gi.cpu().numpy(), gv.cpu().numpy()


def _oracle_scores(inp, r, h):
    b, tok = int(inp.row_req[r]), int(inp.row_token[r])
    pages = inp.block_table[b, : tok // 128 + 1]
    keys = inp.k_cache[pages].reshape(-1, inp.k_cache.shape[2], 128)
    return BS.block_scores(inp.q[r, h], keys[:, h], tok)


CASES = [
    # (ctx tokens per request, rows per request, k, heads, dist)
    ([3000, 700, 129], [300, 5, 2], 8, 1, "int"),
    ([5000, 1000], [40, 300], 12, 2, "int"),
    ([2000, 4100, 260], [70, 9, 3], 16, 4, "int"),
    ([9000], [600], 20, 2, "int"),
    ([6000, 3000], [100, 40], 16, 2, "gauss"),
]


@pytest.mark.parametrize("case", CASES, ids=[f"c{i}" for i in range(len(CASES))])
def test_block_scorer_against_oracle(case):
    ctx, rows, k, heads, dist = case
    inp = W.make_block_scorer_inputs("blk", seed=sum(ctx) % 997, ctx_tokens=ctx, rows_per_req=rows, k=k,
                                     heads=heads, dist=dist)
    gi, gv = _run(inp)
    oi, ov = BS.select_blocks(inp.q, inp.k_cache, inp.block_table, inp.row_req, inp.row_token, k)
    assert qsa.get_device_status() == qsa.QSA_OK
    if dist == "int":
        np.testing.assert_array_equal(gi, oi)
        np.testing.assert_array_equal(gv, ov.astype(np.float32))
        return
    _check_gauss(inp, gi, gv, oi, range(gi.shape[0]), k)


def _check_gauss(inp, gi, gv, oi, rows, k):
    """Rows `rows` of the GPU result (gi, gv: [R, H, k]) against the oracle's
    selection oi ([len(rows), H, k]): values within tolerance of the oracle's
    block scores, sets equal up to near-ties of the cut."""
    H = gi.shape[1]
    for j, r in enumerate(rows):
        for h in range(H):
            sc = _oracle_scores(inp, r, h)
            n = min(k, len(sc))
            assert np.all(gi[r, h, n:] == -1) and np.all(np.isneginf(gv[r, h, n:]))
            sel = gi[r, h, :n]
            assert len(np.unique(sel)) == n and np.all((sel >= 0) & (sel < len(sc)))
            o = sc[sel]
            assert np.all(np.abs(gv[r, h, :n] - o) <= RTOL * np.abs(o) + ATOL), (r, h)
            assert np.all(np.diff(gv[r, h, :n].astype(np.float64)) <= 0)
            kth = sc[oi[j, h, n - 1]]
            for c in set(sel.tolist()) ^ set(oi[j, h, :n].tolist()):
                assert abs(sc[c] - kth) <= RTOL * abs(kth) + ATOL, (r, h, c)


def test_block_scorer_group_half_boundaries():
    # A group holds up to 256 rows of one request and head as two MMA halves of
    # 128: requests of 128 rows (one half), 129 (a second half of one row) and
    # 257 (a full group, then a group of one row).
    inp = W.make_block_scorer_inputs("halves", seed=11, ctx_tokens=[1500, 1400, 2600], rows_per_req=[129, 128, 257],
                                     k=10, heads=2, dist="int")
    gi, gv = _run(inp)
    oi, ov = BS.select_blocks(inp.q, inp.k_cache, inp.block_table, inp.row_req, inp.row_token, inp.k)
    assert qsa.get_device_status() == qsa.QSA_OK
    np.testing.assert_array_equal(gi, oi)
    np.testing.assert_array_equal(gv, ov.astype(np.float32))


@pytest.mark.parametrize("dist", ["int", "gauss"])
def test_block_scorer_full_size(dist):
    # The benchmarked shape (1,616 rows at the end of a 184,320-token context,
    # 2 KV heads, top 16 of 1,440 blocks): every row checked for k distinct
    # visible blocks in non-increasing score order; sampled rows, among them
    # both sides of a half and of a group boundary and the last, 80-row group,
    # against the oracle.
    inp = W.make_block_scorer_inputs(f"blocks_full_{dist}", seed=41, ctx_tokens=[184_320], rows_per_req=[1616],
                                     k=16, heads=2, dist=dist)
    gi, gv = _run(inp)
    assert qsa.get_device_status() == qsa.QSA_OK
    R, H, k = gi.shape
    nvis = (inp.row_token.astype(np.int64) // 128 + 1)[:, None, None]
    assert np.all(gi >= 0) and np.all(gi < nvis)
    assert np.all(np.diff(np.sort(gi, axis=2), axis=2) > 0)
    assert np.all(np.diff(gv.astype(np.float64), axis=2) <= 0)
    rows = sorted(set(np.linspace(0, R - 1, 10).astype(int).tolist()) | {127, 128, 255, 256, 767, 768, 1535, 1536, 1600})
    oi, ov = BS.select_blocks(inp.q[rows], inp.k_cache, inp.block_table, inp.row_req[rows], inp.row_token[rows], k)
    if dist == "int":
        np.testing.assert_array_equal(gi[rows], oi)
        np.testing.assert_array_equal(gv[rows], ov.astype(np.float32))
    else:
        _check_gauss(inp, gi, gv, oi, rows, k)


def test_block_scorer_k_above_visible_blocks_and_ties():
    # every dot product 0 (q = 0): all visible blocks tie, in index order, and
    # k exceeds the visible count of the short rows
    inp = W.make_block_scorer_inputs("tie", seed=3, ctx_tokens=[1000, 200], rows_per_req=[20, 6], k=9, heads=2,
                                     dist="int")
    inp.q[:] = 0
    gi, gv = _run(inp)
    oi, ov = BS.select_blocks(inp.q, inp.k_cache, inp.block_table, inp.row_req, inp.row_token, inp.k)
    np.testing.assert_array_equal(gi, oi)
    np.testing.assert_array_equal(gv, ov.astype(np.float32))
    assert np.any(gi == -1)


def test_block_scorer_bad_page_is_reported():
    inp = W.make_block_scorer_inputs("bp", seed=4, ctx_tokens=[2000], rows_per_req=[5], k=4, heads=2, dist="int")
    bt = inp.block_table.copy()
    bt[0, 2] = inp.k_cache.shape[0] + 50
    _run(inp, block_table=bt)
    assert qsa.get_device_status() == qsa.QSA_ERR_BAD_PAGE
    assert qsa.get_device_status() == qsa.QSA_OK


@pytest.mark.parametrize("seed", range(6))
def test_block_scorer_random_shapes(seed):
    # seeded random batches: 1-4 requests of 1-700 rows over 3-6,000-token
    # contexts, 1, 3, 8 or 16 heads, k from 1 to 16; integer data, bit-exact
    # on every row of a small batch, else on 60 rows that include both sides
    # of the 128-row half and 256-row group boundaries; every row checked for
    # distinct visible blocks in score order
    rng = np.random.default_rng(900 + seed)
    nreq = int(rng.integers(1, 5))
    ctx = [int(c) for c in rng.integers(3, 6000, size=nreq)]
    rows = [int(rng.integers(1, min(c, 700) + 1)) for c in ctx]
    heads = int(rng.choice([1, 3, 8, 16]))
    k = int(rng.integers(1, 17))
    inp = W.make_block_scorer_inputs(f"rand{seed}", seed=seed, ctx_tokens=ctx, rows_per_req=rows, k=k,
                                     heads=heads, dist="int")
    gi, gv = _run(inp)
    assert qsa.get_device_status() == qsa.QSA_OK
    R = gi.shape[0]
    nvis = np.minimum(inp.row_token.astype(np.int64) // 128 + 1, k)[:, None]
    for h in range(heads):
        sel, val = gi[:, h], gv[:, h].astype(np.float64)
        n_ok = (sel >= 0).sum(axis=1)
        assert np.all(n_ok == nvis[:, 0])
        assert np.all(np.diff(np.where(sel >= 0, val, -3e38), axis=1) <= 0)     # padding: a finite floor
    if R <= 120:
        sample = list(range(R))
    else:
        edges = {0, 127, 128, 255, 256, 383, 384, 511, 512, R - 1}
        sample = sorted({e for e in edges if e < R} | set(rng.choice(R, 60 - len(edges), replace=False).tolist()))
    oi, ov = BS.select_blocks(inp.q[sample], inp.k_cache, inp.block_table, inp.row_req[sample],
                              inp.row_token[sample], k)
    np.testing.assert_array_equal(gi[sample], oi)
    np.testing.assert_array_equal(gv[sample], ov.astype(np.float32))
