"""Pins of the M3-style block scorer oracle (the second workload) against what
the pages and the mathematics fix ("spec(MODEL-MM-QWEN4-EXP) ...": the block
score is the maximum of the raw-token dot products over a 128-token block, no
pooling, no ReLU, no head reduction, one block set per KV head):

* block scores equal np.matmul followed by a blockwise max, future tokens
  masked, and a scalar brute force on a small case;
* the top-k order equals np.lexsort on (block index, -score), -1 padded;
* causality, head independence, positive-scale invariance, all-ties order,
  and paging invariance.
"""
import numpy as np

from oracle import block_scorer as S
from block_sparse_attention_select_gb300 import workloads as W


def _inp(**kw):
    a = dict(seed=5, ctx_tokens=[900, 300], rows_per_req=[5, 3], k=4)
    a.update(kw)
    return W.make_block_scorer_inputs("s", **a)


def _keys(inp, b, n):
    pages = inp.block_table[b, : (n + 127) // 128]
    return inp.k_cache[pages].reshape(-1, inp.k_cache.shape[2], 128)[:n]


def test_scores_equal_matmul_then_blockwise_max():
    inp = _inp()
    for r in range(len(inp.row_token)):
        b, t = int(inp.row_req[r]), int(inp.row_token[r])
        keys = _keys(inp, b, t + 1).astype(np.float64)
        for h in range(2):
            full = np.matmul(keys[:, h], inp.q[r, h].astype(np.float64))
            nb = t // 128 + 1
            pad = np.full(nb * 128, -np.inf)
            pad[: t + 1] = full
            want = pad.reshape(nb, 128).max(axis=1)
            np.testing.assert_array_equal(S.block_scores(inp.q[r, h], _keys(inp, b, 128 * nb)[:, h], t), want)


def test_scores_brute_force_scalar():
    inp = _inp(ctx_tokens=[260], rows_per_req=[1], k=3)
    t = int(inp.row_token[0])
    keys = _keys(inp, 0, 384)
    got = S.block_scores(inp.q[0, 1], keys[:, 1], t)
    want = []
    for c in range(t // 128 + 1):
        best = None
        for p in range(128 * c, min(128 * c + 128, t + 1)):
            s = 0.0
            for d in range(128):
                s += float(inp.q[0, 1, d]) * float(keys[p, 1, d])
            best = s if best is None or s > best else best
        want.append(best)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_top_order_matches_lexsort_and_pads():
    rng = np.random.default_rng(3)
    for n in (1, 5, 40):
        sc = np.round(rng.standard_normal(n), 1)                 # rounded: ties happen
        for k in (1, 3, 8, 64):
            got = S.top_blocks(sc, k)
            order = np.lexsort((np.arange(n), -sc))[:k]
            assert got[: len(order)].tolist() == order.tolist()
            assert np.all(got[len(order):] == -1)


def test_causality_heads_and_scale():
    inp = _inp()
    idx, val = S.select_blocks(inp.q, inp.k_cache, inp.block_table, inp.row_req, inp.row_token, inp.k)
    # tokens after a row's own token do not matter: overwrite request 0's last page past token 896
    kc = inp.k_cache.copy()
    last = inp.block_table[0, 7]                                  # tokens 896 .. 1023
    kc[last, 1:] = 7.0                                            # token 897 onward (row tokens are 895..899)
    i2, _ = S.select_blocks(inp.q, kc, inp.block_table, inp.row_req, inp.row_token, inp.k)
    rows = inp.row_token <= 896
    np.testing.assert_array_equal(i2[rows], idx[rows])
    # head 1's keys do not move head 0's blocks
    kc = inp.k_cache.copy()
    kc[:, :, 1] = 0
    i3, _ = S.select_blocks(inp.q, kc, inp.block_table, inp.row_req, inp.row_token, inp.k)
    np.testing.assert_array_equal(i3[:, 0], idx[:, 0])
    # a positive scale of the queries keeps every selection
    q4 = (inp.q.astype(np.float32) * 2).astype(np.float16)
    i4, v4 = S.select_blocks(q4, inp.k_cache, inp.block_table, inp.row_req, inp.row_token, inp.k)
    np.testing.assert_array_equal(i4, idx)
    np.testing.assert_allclose(v4, 2 * val, rtol=1e-12)


def test_all_ties_take_the_lowest_blocks_and_pad():
    inp = _inp(ctx_tokens=[700], rows_per_req=[2], k=8, dist="int")
    kc = np.ones_like(inp.k_cache)
    q = np.ones_like(inp.q)
    idx, _ = S.select_blocks(q, kc, inp.block_table, inp.row_req, inp.row_token, 8)
    assert idx[0, 0].tolist() == [0, 1, 2, 3, 4, 5, -1, -1]      # token 698: blocks 0..5


def test_paging_invariance():
    inp = _inp()
    idx, val = S.select_blocks(inp.q, inp.k_cache, inp.block_table, inp.row_req, inp.row_token, inp.k)
    rng = np.random.default_rng(9)
    perm = rng.permutation(inp.k_cache.shape[0])
    inv = np.argsort(perm)
    kc2 = inp.k_cache[perm]                                       # page p now at inv[p]
    bt2 = np.where(inp.block_table >= 0, inv[np.maximum(inp.block_table, 0)], -1).astype(np.int32)
    i2, v2 = S.select_blocks(inp.q, kc2, bt2, inp.row_req, inp.row_token, inp.k)
    np.testing.assert_array_equal(i2, idx)
    np.testing.assert_array_equal(v2, val)
