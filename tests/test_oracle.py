"""Pins for the CPU oracle, against things other than the oracle itself.

Each test ties one part of the oracle to a fact fixed by the pages or by
mathematics: a hand-worked example, the IEEE binary16 definition (through
numpy's own conversion), dense-matrix special cases (np.matmul, exact on
integer data), algebraic identities of ReLU, paging invariance, a brute-force
selector and numpy's lexicographic sort.  A dropped term, a wrong sign, index
or operand order in the oracle fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from block_sparse_attention_select_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f(x):
    return -np.inf if x == "-inf" else float(x)


# ---------------------------------------------------------------- golden ----

def test_hand_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "hand_example.json")))
    q = np.array(g["q"], dtype=np.float16)
    w = np.array(g["w"], dtype=np.float32)
    kc = np.array(g["k_cache"], dtype=np.float16)
    bt = np.array(g["block_table"], dtype=np.int32)
    rr = np.array(g["row_req"], dtype=np.int32)
    rv = np.array(g["row_visible"], dtype=np.int32)
    lg = oracle.score(q, w, kc, bt, rr, rv, ld=6)
    exp = np.array([[_f(x) for x in row] for row in g["expected_logits"]], dtype=np.float32)
    np.testing.assert_array_equal(lg, exp)
    idx, val = oracle.select(lg, rv, g["k"])
    np.testing.assert_array_equal(idx, np.array(g["expected_idx"], dtype=np.int32))
    np.testing.assert_array_equal(val, np.array([[_f(x) for x in r] for r in g["expected_val"]],
                                                dtype=np.float32))
    bidx, bval = oracle.select_bruteforce(lg, rv, g["k"])
    np.testing.assert_array_equal(bidx, idx)


# ------------------------------------------------------------- binary16 ----

def test_half_to_float_matches_ieee_binary16_everywhere():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle.half_to_float(int(b)) for b in bits], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


# ----------------------------------------------------------- visibility ----

@pytest.mark.parametrize("ratio", [1, 2, 4, 8])
def test_visible_positions_counts_completed_blocks(ratio):
    # brute force: compressed position p (tokens ratio*p .. ratio*p+ratio-1) is
    # visible at token t once its last token exists, i.e. (position+1) % ratio == 0
    # has fired for it.
    for t in range(0, 300):
        n = sum(1 for p in range(0, 400) if ratio * p + ratio - 1 <= t)
        assert oracle.visible_positions(t, ratio) == n


def test_workload_visibility_matches_oracle_rule():
    wl = W.tiny()
    for t, v in zip(wl.row_token, wl.row_visible):
        assert oracle.visible_positions(int(t), 4) == int(v)


# --------------------------------------------------------------- scorer ----

def _dense_case(seed, R=5, H=3, D=24, npos=40, P=4, lo=-4, hi=4):
    rng = np.random.default_rng(seed)
    q = rng.integers(lo, hi + 1, size=(R, H, D)).astype(np.float16)
    keys = rng.integers(lo, hi + 1, size=(npos, D)).astype(np.float16)
    pages = -(-npos // P)
    kc = np.zeros((pages, P, D), dtype=np.float16)
    kc.reshape(-1, D)[:npos] = keys
    bt = np.arange(pages, dtype=np.int32)[None, :]
    rr = np.zeros(R, dtype=np.int32)
    rv = rng.integers(0, npos + 1, size=R).astype(np.int32)
    rv[0] = npos
    return q, keys, kc, bt, rr, rv


def test_score_single_head_is_relu_of_dense_matmul():
    # identity block table + one-hot weights: logit = max(q_h . k_j, 0), and
    # L(q) - L(-q) = q_h . k_j, L(q) + L(-q) = |q_h . k_j| (np.matmul, exact on ints).
    q, keys, kc, bt, rr, rv = _dense_case(1)
    R, H, D = q.shape
    for h in range(H):
        w = np.zeros((R, H), np.float32)
        w[:, h] = 1.0
        lp = oracle.score(q, w, kc, bt, rr, rv, ld=keys.shape[0])
        ln = oracle.score(-q, w, kc, bt, rr, rv, ld=keys.shape[0])
        dot = np.matmul(q[:, h, :].astype(np.float64), keys.astype(np.float64).T)
        for r in range(R):
            V = rv[r]
            np.testing.assert_array_equal(lp[r, :V] - ln[r, :V], dot[r, :V])
            np.testing.assert_array_equal(lp[r, :V] + ln[r, :V], np.abs(dot[r, :V]))
            assert np.all(lp[r, :V] >= 0)
            assert np.all(np.isneginf(lp[r, V:]))


def test_score_is_linear_in_head_weights():
    # ReLU is applied per head before weighting: doubling / summing weights
    # scales / sums logits exactly (dyadic weights, integer data).
    q, keys, kc, bt, rr, rv = _dense_case(2)
    R, H, _ = q.shape
    rng = np.random.default_rng(3)
    wa = rng.choice(np.array([0.25, 0.5, 1, 2], np.float32), size=(R, H))
    wb = rng.choice(np.array([-1, 0.5, 1, 4], np.float32), size=(R, H))
    la = oracle.score(q, wa, kc, bt, rr, rv, ld=keys.shape[0])
    lb = oracle.score(q, wb, kc, bt, rr, rv, ld=keys.shape[0])
    lab = oracle.score(q, wa + wb, kc, bt, rr, rv, ld=keys.shape[0])
    for r in range(R):
        V = rv[r]
        np.testing.assert_array_equal(lab[r, :V], la[r, :V] + lb[r, :V])
    # weights of other rows do not leak into row r
    wc = wa.copy()
    wc[1:] = 7.0
    lc = oracle.score(q, wc, kc, bt, rr, rv, ld=keys.shape[0])
    np.testing.assert_array_equal(lc[0], la[0])


def test_score_relu_precedes_head_sum():
    # One head positive, one negative on the same key: a relu after the sum
    # would give max(a+b,0); relu per head gives max(a,0)+max(b,0).
    q = np.zeros((1, 2, 4), np.float16)
    q[0, 0, 0] = 3
    q[0, 1, 0] = -2
    kc = np.zeros((1, 4, 4), np.float16)
    kc[0, 0, 0] = 1
    lg = oracle.score(q, np.ones((1, 2), np.float32), kc, np.zeros((1, 1), np.int32),
                      np.zeros(1, np.int32), np.array([1], np.int32), ld=1)
    assert lg[0, 0] == 3.0


def test_score_paging_invariance_and_request_routing():
    # Two requests with different keys; permuting the physical pages (and the
    # block tables with them) must not change any logit, and each row must read
    # its own request's pages only.
    rng = np.random.default_rng(5)
    P, D, H = 4, 16, 2
    npos = [29, 18]
    keys = [rng.integers(-4, 5, size=(n, D)).astype(np.float16) for n in npos]
    pages = [-(-n // P) for n in npos]
    kc = np.zeros((sum(pages), P, D), np.float16)
    bt = np.full((2, max(pages)), -1, np.int32)
    off = 0
    for b in range(2):
        flat = np.zeros((pages[b] * P, D), np.float16)
        flat[:npos[b]] = keys[b]
        kc[off:off + pages[b]] = flat.reshape(pages[b], P, D)
        bt[b, :pages[b]] = np.arange(off, off + pages[b])
        off += pages[b]
    R = 6
    q = rng.integers(-4, 5, size=(R, H, D)).astype(np.float16)
    w = np.ones((R, H), np.float32)
    rr = np.array([0, 0, 1, 0, 1, 1], np.int32)
    rv = np.array([29, 13, 18, 0, 5, 17], np.int32)
    ld = 32
    base = oracle.score(q, w, kc, bt, rr, rv, ld=ld)
    perm = rng.permutation(kc.shape[0])
    inv = np.empty_like(perm)
    inv[perm] = np.arange(len(perm))
    kc2 = kc[perm]                        # physical page p now lives at slot inv[p]
    bt2 = np.where(bt >= 0, inv[np.maximum(bt, 0)], -1).astype(np.int32)
    np.testing.assert_array_equal(oracle.score(q, w, kc2, bt2, rr, rv, ld=ld), base)
    for r in range(R):
        b, V = rr[r], rv[r]
        dots = np.matmul(q[r].astype(np.float64), keys[b].astype(np.float64).T)
        ref = np.maximum(dots, 0).sum(axis=0)[:V]
        np.testing.assert_array_equal(base[r, :V], ref)
        assert np.all(np.isneginf(base[r, V:]))


def test_score_fp32_accumulation_within_summation_bound():
    # Gaussian FP16 data: the FP32 result lies within the standard bound for a
    # sequential binary32 sum, |err| <= n*u/(1-n*u) * sum|terms| (u = 2^-24),
    # of the float64 value (products are exact in binary32).
    wl = W.make_workload("g", seed=7, ctx_tokens=[512], rows_per_req=[9], k=16,
                         shuffle_pages=False)
    lg = oracle.score(wl.q, wl.w, wl.k_cache, wl.block_table, wl.row_req, wl.row_visible, wl.ld)
    keys = wl.k_cache.reshape(-1, 128).astype(np.float64)
    D = 128
    u = 2.0 ** -24
    gam = lambda n: n * u / (1 - n * u)
    for r in range(wl.rows):
        V = wl.row_visible[r]
        qr = wl.q[r].astype(np.float64)
        dots = qr @ keys[:V].T                       # [H, V]
        absd = np.abs(qr) @ np.abs(keys[:V]).T
        ref = (wl.w[r].astype(np.float64)[:, None] * np.maximum(dots, 0)).sum(axis=0)
        # dot error propagates through relu and the weight; then H more adds.
        bound = (np.abs(wl.w[r]).astype(np.float64)[:, None] * absd * gam(D)).sum(axis=0) \
            + gam(wl.heads + 1) * (np.abs(wl.w[r]).astype(np.float64)[:, None]
                                   * np.abs(dots)).sum(axis=0) + 1e-30
        assert np.all(np.abs(lg[r, :V].astype(np.float64) - ref) <= bound)


def test_score_zero_query_or_zero_weight_gives_plus_zero():
    for qd, wd in (("zero", "gauss"), ("gauss", "zero")):
        wl = W.make_workload("z", seed=9, ctx_tokens=[256], rows_per_req=[3], k=8, dist=qd,
                             wdist=wd)
        lg = oracle.score(wl.q, wl.w, wl.k_cache, wl.block_table, wl.row_req, wl.row_visible,
                          wl.ld)
        for r in range(wl.rows):
            V = wl.row_visible[r]
            assert np.all(lg[r, :V] == 0) and not np.any(np.signbit(lg[r, :V]))


def test_score_negative_weights_never_give_negative_zero():
    wl = W.make_workload("n", seed=11, ctx_tokens=[256], rows_per_req=[4], k=8, dist="int4")
    w = -np.abs(wl.w)
    lg = oracle.score(wl.q, w, wl.k_cache, wl.block_table, wl.row_req, wl.row_visible, wl.ld)
    fin = np.isfinite(lg)
    assert not np.any(np.signbit(lg[fin]) & (lg[fin] == 0))
    assert np.all(lg[fin] <= 0)


# ------------------------------------------------------------- selector ----

def _check_invariants(lg, rv, k, idx, val):
    R = lg.shape[0]
    for r in range(R):
        V = int(rv[r])
        n = min(k, V)
        sel = idx[r, :n]
        assert np.all(idx[r, n:] == -1) and np.all(np.isneginf(val[r, n:]))
        assert len(set(sel.tolist())) == n
        assert np.all((sel >= 0) & (sel < V))
        np.testing.assert_array_equal(val[r, :n], lg[r, sel])
        keys = list(zip(-val[r, :n].astype(np.float64), sel))
        assert keys == sorted(keys) and len(set(keys)) == n          # strictly ordered
        if n < V:
            mask = np.ones(V, bool)
            mask[sel] = False
            uns = np.nonzero(mask)[0]
            assert lg[r, sel].min() >= lg[r, uns].max()
            cut = lg[r, sel].min()
            tied_sel = sel[lg[r, sel] == cut]
            tied_uns = uns[lg[r, uns] == cut]
            if len(tied_uns):
                assert tied_sel.max() < tied_uns.min()


@pytest.mark.parametrize("seed", range(6))
def test_select_matches_bruteforce_with_heavy_ties(seed):
    rng = np.random.default_rng(100 + seed)
    R, ld = 7, 50
    lg = rng.integers(-3, 4, size=(R, ld)).astype(np.float32) * np.float32(0.5)
    rv = rng.integers(0, ld + 1, size=R).astype(np.int32)
    rv[0], rv[1] = ld, 0
    for k in (1, 5, 16, 50, 64):
        idx, val = oracle.select(lg, rv, k)
        bidx, bval = oracle.select_bruteforce(lg, rv, k)
        np.testing.assert_array_equal(idx, bidx)
        np.testing.assert_array_equal(val, bval)
        _check_invariants(lg, rv, k, idx, val)


def test_select_matches_numpy_lexsort():
    rng = np.random.default_rng(7)
    R, ld, k = 12, 3000, 257
    lg = (rng.standard_normal((R, ld)).astype(np.float32) * 4).round(1).astype(np.float32)
    rv = rng.integers(0, ld + 1, size=R).astype(np.int32)
    idx, val = oracle.select(lg, rv, k)
    for r in range(R):
        V = rv[r]
        order = np.lexsort((np.arange(V), -lg[r, :V].astype(np.float64)))[:k]
        n = min(k, V)
        np.testing.assert_array_equal(idx[r, :n], order)
        assert np.all(idx[r, n:] == -1)
    _check_invariants(lg, rv, k, idx, val)


def test_select_closed_forms():
    # all-equal scores: pure tie rule -> 0..k-1 ascending
    lg = np.zeros((2, 100), np.float32)
    rv = np.array([100, 37], np.int32)
    idx, _ = oracle.select(lg, rv, 40)
    np.testing.assert_array_equal(idx[0], np.arange(40))
    np.testing.assert_array_equal(idx[1], np.r_[np.arange(37), [-1, -1, -1]])
    # strictly increasing scores: the last k indices, descending
    lg = np.tile(np.arange(100, dtype=np.float32), (1, 1))
    idx, _ = oracle.select(lg, np.array([100], np.int32), 10)
    np.testing.assert_array_equal(idx[0], np.arange(99, 89, -1))
    # k = V: a full sort; k = 1: argmax with the lowest index among equals
    rng = np.random.default_rng(1)
    lg = rng.integers(0, 5, size=(1, 64)).astype(np.float32)
    idx, _ = oracle.select(lg, np.array([64], np.int32), 64)
    assert sorted(idx[0].tolist()) == list(range(64))
    idx1, _ = oracle.select(lg, np.array([64], np.int32), 1)
    assert idx1[0, 0] == int(np.argmax(lg[0]))          # np.argmax returns the first max


def test_step_on_tiny_workload_is_consistent():
    wl = W.tiny()
    idx, val, lg = oracle.select_paged_tokens(wl.q, wl.w, wl.k_cache, wl.block_table, wl.row_req,
                                              wl.row_visible, wl.k, ld=wl.ld)
    _check_invariants(lg, wl.row_visible, wl.k, idx, val)
    # integer data: the FP32 logits are exact, so they equal the float64 dense value
    keys = wl.k_cache.reshape(-1, 128).astype(np.float64)
    for r in range(wl.rows):
        V = wl.row_visible[r]
        d = wl.q[r].astype(np.float64) @ keys[:V].T
        ref = (wl.w[r].astype(np.float64)[:, None] * np.maximum(d, 0)).sum(0)
        np.testing.assert_array_equal(lg[r, :V], ref)


def test_threads_do_not_change_results():
    wl = W.make_workload("t", seed=21, ctx_tokens=[2048, 1500], rows_per_req=[7, 5], k=33)
    a = oracle.select_paged_tokens(wl.q, wl.w, wl.k_cache, wl.block_table, wl.row_req,
                                   wl.row_visible, wl.k, ld=wl.ld, nthreads=1)
    b = oracle.select_paged_tokens(wl.q, wl.w, wl.k_cache, wl.block_table, wl.row_req,
                                   wl.row_visible, wl.k, ld=wl.ld, nthreads=4)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
