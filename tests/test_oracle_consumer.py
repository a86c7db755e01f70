"""Pins of the sparse-attention consumer oracle (the step after the indexer)
against what the pages and the mathematics fix, independent of its own code:

* every visible position selected = causal attention over the row's whole
  prefix, checked against torch's scaled_dot_product_attention (float64, CPU)
  on contiguous K / V;
* the selection is a set: order, duplicates and -1 entries do not matter;
* GQA: query head h reads KV head h // 12 (24 query heads over 2 KV heads,
  "spec(MODEL-MM-QWEN4-EXP) ...");
* each output is a convex combination of the attended values;
* one selected position, brute force with scalar loops;
* the paged layout: token p of request b at page block_table[b][p // 64],
  slot p % 64;
* the attended tokens: the 4 raw tokens of each selected position ("attends
  raw tokens selected at ratio-4 granularity") plus the unfinished block.
"""
import math

import numpy as np
import pytest

from oracle import consumer as C
from block_sparse_attention_select_gb300 import workloads as W

torch = pytest.importorskip("torch")


def _inputs(**kw):
    a = dict(seed=1, ctx_tokens=[300, 130], rows_per_req=[6, 3], k=16, all_selected_rows=0)
    a.update(kw)
    return W.make_consumer_inputs("c", **a)


def _contiguous(cache, block_table, b, n):
    """Request b's first n tokens of a paged cache, by walking its pages."""
    rows = []
    for pg in range((n + 63) // 64):
        rows.append(cache[block_table[b, pg]])
    return np.concatenate(rows, axis=0)[:n]


def test_attended_tokens_rule():
    assert C.attended_tokens(np.array([0]), 10).tolist() == [0, 1, 2, 3, 8, 9, 10]
    assert C.attended_tokens(np.array([1, -1, 1]), 7).tolist() == [4, 5, 6, 7]   # 7 ends block 1
    assert C.attended_tokens(np.array([-1, -1]), 2).tolist() == [0, 1, 2]       # nothing complete yet
    assert C.attended_tokens(np.arange(3), 11).tolist() == list(range(12))


def test_all_selected_is_causal_attention():
    inp = _inputs(k=80, all_selected_rows=0)      # k >= every row's visible count: all selected
    out = C.sparse_attention(inp.q, inp.k_cache, inp.v_cache, inp.block_table, inp.row_req, inp.row_token,
                             inp.sel)
    checked = 0
    for r in range(len(inp.row_token)):
        b, t = int(inp.row_req[r]), int(inp.row_token[r])
        v = (t + 1) // 4
        if set(inp.sel[r][inp.sel[r] >= 0].tolist()) != set(range(v)):
            continue
        K = _contiguous(inp.k_cache, inp.block_table, b, t + 1)      # [t+1, 2, 256]
        V = _contiguous(inp.v_cache, inp.block_table, b, t + 1)
        q = torch.from_numpy(inp.q[r].astype(np.float64))[None, :, None, :]          # [1, 24, 1, 256]
        k = torch.from_numpy(K.astype(np.float64)).permute(1, 0, 2).repeat_interleave(12, 0)[None]
        vv = torch.from_numpy(V.astype(np.float64)).permute(1, 0, 2).repeat_interleave(12, 0)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, vv)[0, :, 0].numpy()
        np.testing.assert_allclose(out[r], ref, rtol=1e-10, atol=1e-12)
        checked += 1
    assert checked == len(inp.row_token) == 9


def test_selection_is_a_set():
    inp = _inputs(all_selected_rows=0)
    base = C.sparse_attention(inp.q, inp.k_cache, inp.v_cache, inp.block_table, inp.row_req, inp.row_token,
                              inp.sel)
    rng = np.random.default_rng(4)
    sel2 = np.full((inp.sel.shape[0], inp.sel.shape[1] * 2 + 3), -1, dtype=np.int32)
    for r in range(inp.sel.shape[0]):
        s = inp.sel[r][inp.sel[r] >= 0]
        s = np.concatenate([s, s[: len(s) // 2]])                  # duplicates
        rng.shuffle(s)
        sel2[r, : len(s)] = s
    other = C.sparse_attention(inp.q, inp.k_cache, inp.v_cache, inp.block_table, inp.row_req, inp.row_token,
                               sel2)
    np.testing.assert_allclose(other, base, rtol=1e-12, atol=1e-14)


def test_gqa_head_mapping():
    inp = _inputs()
    base = C.sparse_attention(inp.q, inp.k_cache, inp.v_cache, inp.block_table, inp.row_req, inp.row_token,
                              inp.sel)
    v0 = inp.v_cache.copy()
    v0[:, :, 1, :] = 0
    z = C.sparse_attention(inp.q, inp.k_cache, v0, inp.block_table, inp.row_req, inp.row_token, inp.sel)
    assert np.all(z[:, 12:] == 0.0)
    np.testing.assert_array_equal(z[:, :12], base[:, :12])


def test_outputs_are_convex_combinations():
    inp = _inputs(all_selected_rows=0)
    out = C.sparse_attention(inp.q, inp.k_cache, inp.v_cache, inp.block_table, inp.row_req, inp.row_token,
                             inp.sel)
    for r in range(len(inp.row_token)):
        toks = C.attended_tokens(inp.sel[r], int(inp.row_token[r]))
        vv = C.gather(inp.v_cache, inp.block_table, int(inp.row_req[r]), toks).astype(np.float64)
        for h in (0, 13):
            g = h // 12
            assert np.all(out[r, h] <= vv[:, g].max(axis=0) + 1e-12)
            assert np.all(out[r, h] >= vv[:, g].min(axis=0) - 1e-12)


def test_single_position_brute_force():
    inp = _inputs(ctx_tokens=[200], rows_per_req=[1], k=4, all_selected_rows=0)
    t = int(inp.row_token[0])                                        # 199: ends block 49, no tail
    sel = np.array([[37, -1, -1, -1]], dtype=np.int32)
    out = C.sparse_attention(inp.q, inp.k_cache, inp.v_cache, inp.block_table, inp.row_req, inp.row_token, sel)
    K = _contiguous(inp.k_cache, inp.block_table, 0, t + 1)
    V = _contiguous(inp.v_cache, inp.block_table, 0, t + 1)
    for h in (0, 11, 12, 23):
        g = h // 12
        s = [sum(float(inp.q[0, h, d]) * float(K[p, g, d]) for d in range(256)) / 16.0 for p in range(148, 152)]
        m = max(s)
        w = [math.exp(x - m) for x in s]
        want = [sum(w[i] * float(V[148 + i, g, d]) for i in range(4)) / sum(w) for d in range(256)]
        np.testing.assert_allclose(out[0, h], want, rtol=1e-9, atol=1e-12)


def test_paged_gather_layout():
    inp = _inputs()
    toks = np.array([0, 63, 64, 65, 128, 299])
    got = C.gather(inp.k_cache, inp.block_table, 0, toks)
    flat = _contiguous(inp.k_cache, inp.block_table, 0, 300)
    np.testing.assert_array_equal(got, flat[toks])
