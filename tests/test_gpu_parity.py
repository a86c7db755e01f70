"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Integer-valued inputs must match bit for bit (indices and values); Gaussian
inputs must give logits within |g - o| <= 1e-3 |o| + 1e-6 and selections that
differ from the oracle's only at near-ties of the cutoff (within the same
tolerance), with the disagreement rate reported.  Selections are also
compared bit-exactly with the oracle's selector run on the GPU's own logits.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_select_gb300 import qsa
from block_sparse_attention_select_gb300 import workloads as W

from gpu_util import (assert_logits_close, assert_values_at_selection, check_sorted_valid, gpu_logits,
                      gpu_select, near_tie_disagreement, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    qsa.load()
    assert torch.cuda.is_available()
    yield
    assert qsa.get_device_status() == qsa.QSA_OK


def _oracle_rows(wl, rows, ld=None):
    rows = np.asarray(rows)
    ld = wl.ld if ld is None else ld
    lg = oracle.score(wl.q[rows], wl.w[rows], wl.k_cache, wl.block_table, wl.row_req[rows],
                      wl.row_visible[rows], ld)
    idx, val = oracle.select(lg, wl.row_visible[rows], wl.k)
    return lg, idx, val


# ------------------------------------------------------------ tiny, exact ----

@pytest.mark.parametrize("path", [qsa.PATH_DENSE, qsa.PATH_FILTER])
def test_tiny_config_bit_exact(path):
    wl = W.tiny()
    oi, ov, ol = oracle.select_paged_tokens(wl.q, wl.w, wl.k_cache, wl.block_table, wl.row_req,
                                            wl.row_visible, wl.k, ld=wl.ld)
    gi, gv = gpu_select(wl, path=path)
    np.testing.assert_array_equal(gi, oi)
    np.testing.assert_array_equal(gv, ov)


def test_tiny_config_logits_bit_exact():
    wl = W.tiny()
    ol = oracle.score(wl.q, wl.w, wl.k_cache, wl.block_table, wl.row_req, wl.row_visible, wl.ld)
    np.testing.assert_array_equal(gpu_logits(wl), ol)
    # a wider logit row than the cache: the tail is -inf
    ol2 = oracle.score(wl.q, wl.w, wl.k_cache, wl.block_table, wl.row_req, wl.row_visible, 300)
    np.testing.assert_array_equal(gpu_logits(wl, ld=300), ol2)


# ------------------------------------------------- ragged, multi-request ----

CASES = [
    # (ctx tokens per request, rows per request, k, dist, H, page positions)
    ([3000, 777, 5], [70, 3, 1], 33, "int4", 4, 16),
    ([1030, 2050], [130, 65], 100, "int4", 2, 16),
    ([4100], [40], 64, "int4", 8, 16),
    ([2600, 900], [300, 20], 17, "int4", 1, 16),
    ([6000, 1000], [5, 9], 128, "int4", 4, 8),
    ([6000], [9], 128, "int4", 4, 32),
    ([9000], [11], 128, "int4", 4, 128),
    ([9000], [11], 96, "int4", 4, 256),
    ([20000, 9000], [90, 45], 256, "gauss", 4, 16),
    # a few rows per request: the narrow scorer (decode-like batches)
    ([5000, 3000, 12000, 800, 20000], [1, 2, 1, 1, 3], 128, "int4", 4, 16),
    ([7000, 900, 15000], [2, 1, 1], 96, "int4", 8, 16),
    ([30000, 2000, 11000, 6000], [1, 1, 2, 1], 512, "gauss", 4, 16),
    # rows longer than 65,536 positions: the candidate selector's 32-bit positions
    ([282000, 5000], [3, 2], 400, "int4", 4, 64),
]


@pytest.mark.parametrize("case", CASES, ids=[f"c{i}" for i in range(len(CASES))])
@pytest.mark.parametrize("path", [qsa.PATH_DENSE, qsa.PATH_FILTER])
def test_ragged_cases_against_oracle(case, path):
    ctx, rows, k, dist, H, P = case
    wl = W.make_workload("ragged", seed=hash((tuple(ctx), k, H, P)) % 1000, ctx_tokens=ctx,
                         rows_per_req=rows, k=k, dist=dist, heads=H, page_positions=P)
    d = to_device(wl)
    ol, oi, ov = _oracle_rows(wl, np.arange(wl.rows))
    gl = gpu_logits(wl, d)
    gi, gv = gpu_select(wl, d, path=path)
    check_sorted_valid(gi, gv, wl.row_visible, k)
    if dist == "int4":
        np.testing.assert_array_equal(gl, ol)
        np.testing.assert_array_equal(gi, oi)
        np.testing.assert_array_equal(gv, ov)
    else:
        assert_logits_close(gl, ol, wl.row_visible)
        # exact against the oracle's selector on the GPU's own logits
        ei, ev = oracle.select(gl, wl.row_visible, k)
        np.testing.assert_array_equal(gi, ei)
        np.testing.assert_array_equal(gv, ev)
        rate, same = near_tie_disagreement(gi, oi, ol, wl.row_visible, k)
        print(f"disagreement rate {rate:.2e}, identical rows {same:.3f}")


@pytest.mark.parametrize("dist,wdist", [("int4", "int4_signed"), ("gauss", "gauss_signed")])
@pytest.mark.parametrize("path", [qsa.PATH_DENSE, qsa.PATH_FILTER])
def test_mixed_sign_weights(dist, wdist, path):
    # Negative head weights: scores of either sign, a negative weight times a
    # clipped head gives -0 (which must tie with +0), and many scores below 0.
    wl = W.make_workload("signed", seed=21, ctx_tokens=[24000, 3000, 9000], rows_per_req=[40, 7, 20],
                         k=300, dist=dist, wdist=wdist)
    assert (wl.w < 0).any() and (wl.w > 0).any()
    d = to_device(wl)
    ol, oi, ov = _oracle_rows(wl, np.arange(wl.rows))
    gl = gpu_logits(wl, d)
    gi, gv = gpu_select(wl, d, path=path)
    check_sorted_valid(gi, gv, wl.row_visible, wl.k)
    if dist == "int4":
        np.testing.assert_array_equal(gl, ol)
        np.testing.assert_array_equal(gi, oi)
        np.testing.assert_array_equal(gv, ov)
    else:
        assert_logits_close(gl, ol, wl.row_visible)
        ei, ev = oracle.select(gl, wl.row_visible, wl.k)
        np.testing.assert_array_equal(gi, ei)
        np.testing.assert_array_equal(gv, ev)
        near_tie_disagreement(gi, oi, ol, wl.row_visible, wl.k)
    assert not np.any(np.signbit(gv[gv == 0]))          # the zeros come back as +0


@pytest.mark.parametrize("csize", [1, 2, 4, 8])
@pytest.mark.parametrize("dist,k", [("int4", 512), ("tern", 300)])
def test_cluster_selector_matches_oracle(csize, dist, k):
    # Few rows: the candidate selector splits each row over a thread-block
    # cluster (sizes forced here, capped by the device's own query) and merges
    # the slices through distributed shared memory.  Integer data: bit-exact.
    wl = W.make_workload("cl", seed=41 + k, ctx_tokens=[30000, 2000, 60000, 9000], rows_per_req=[3, 2, 1, 4],
                         k=k, dist=dist)
    oi, ov, _ = oracle.select_paged_tokens(wl.q, wl.w, wl.k_cache, wl.block_table, wl.row_req,
                                           wl.row_visible, wl.k, ld=wl.ld)
    qsa.set_config(qsa.QSA_CFG_CLUSTER, csize)
    try:
        gi, gv = gpu_select(wl, path=qsa.PATH_FILTER)
        used = qsa.last_cluster_size()
    finally:
        qsa.set_config(qsa.QSA_CFG_CLUSTER, 0)
    assert 1 <= used <= csize and used & (used - 1) == 0
    np.testing.assert_array_equal(gi, oi)
    np.testing.assert_array_equal(gv, ov)


@pytest.mark.parametrize("csize", [1, 4])
def test_decode_batch_full_rows_on_cluster_and_plain_selectors(csize):
    # the 64-row decode batch, every row, through both candidate selectors:
    # exactly the oracle's selection on the GPU's own logits
    wl = W.CONFIGS["decode"]()
    d = to_device(wl)
    gl = gpu_logits(wl, d)
    ei, ev = oracle.select(gl, wl.row_visible, wl.k)
    qsa.set_config(qsa.QSA_CFG_CLUSTER, csize)
    try:
        gi, gv = gpu_select(wl, d, path=qsa.PATH_FILTER)
        used = qsa.last_cluster_size()
    finally:
        qsa.set_config(qsa.QSA_CFG_CLUSTER, 0)
    assert used == csize or (csize > 1 and 1 < used < csize)
    np.testing.assert_array_equal(gi, ei)
    np.testing.assert_array_equal(gv, ev)


def test_filter_path_falls_back_when_sampling_misleads():
    # Scores are high only in sampled key tiles (every 2nd tile for k=256), so
    # the sample threshold keeps fewer than k candidates and rows must take the
    # dense fallback.  Integer data: the result must still be exact.
    k, H, npos = 256, 1, 6000
    wl = W.make_workload("fb", seed=1, ctx_tokens=[4 * npos], rows_per_req=[7], k=k,
                         dist="zero", wdist="ones", heads=H, shuffle_pages=False)
    keys = wl.k_cache.reshape(-1, 128)
    j = np.arange(keys.shape[0])
    keys[:, 0] = ((j % 97) + np.where((j // 128) % 2 == 0, 100, 0)).astype(np.float16)
    wl.q[:, 0, 0] = 1
    oi, ov, _ = oracle.select_paged_tokens(wl.q, wl.w, wl.k_cache, wl.block_table, wl.row_req,
                                           wl.row_visible, k, ld=wl.ld)
    for path in (qsa.PATH_FILTER, qsa.PATH_DENSE):
        gi, gv = gpu_select(wl, path=path)
        np.testing.assert_array_equal(gi, oi)
        np.testing.assert_array_equal(gv, ov)


@pytest.mark.parametrize("ctx", [40000, 280000])
def test_filter_path_falls_back_on_candidate_overflow(ctx):
    # every score equal (w = 0): the threshold admits every position, more than
    # the candidate capacity -> fallback; the answer is the pure tie order
    # (280,000 tokens: rows past 65,536 positions, 32-bit candidate positions)
    k = 300
    wl = W.make_workload("of", seed=2, ctx_tokens=[ctx], rows_per_req=[5], k=k,
                         dist="int4", wdist="zero")
    gi, gv = gpu_select(wl, path=qsa.PATH_FILTER)
    for r in range(wl.rows):
        n = min(k, wl.row_visible[r])
        np.testing.assert_array_equal(gi[r, :n], np.arange(n))
        assert np.all(gv[r, :n] == 0) and not np.any(np.signbit(gv[r, :n]))


def test_zero_visible_rows_and_k_above_visible():
    wl = W.make_workload("z", seed=3, ctx_tokens=[3, 20, 700], rows_per_req=[3, 4, 2], k=200,
                         dist="int4")
    assert (wl.row_visible == 0).any() and (wl.row_visible < 200).all()
    oi, ov, _ = oracle.select_paged_tokens(wl.q, wl.w, wl.k_cache, wl.block_table, wl.row_req,
                                           wl.row_visible, wl.k, ld=wl.ld)
    for path in (qsa.PATH_DENSE, qsa.PATH_FILTER):
        gi, gv = gpu_select(wl, path=path)
        np.testing.assert_array_equal(gi, oi)
        np.testing.assert_array_equal(gv, ov)


def test_k_equals_one_and_max_k():
    wl = W.make_workload("k", seed=4, ctx_tokens=[40000], rows_per_req=[3], k=1, dist="int4")
    d = to_device(wl)
    ol = oracle.score(wl.q, wl.w, wl.k_cache, wl.block_table, wl.row_req, wl.row_visible, wl.ld)
    for k in (1, qsa.QSA_MAX_K):
        oi, ov = oracle.select(ol, wl.row_visible, k)
        gi, gv = gpu_select(wl, d, k=k)
        np.testing.assert_array_equal(gi, oi)
        np.testing.assert_array_equal(gv, ov)


@pytest.mark.parametrize("ctx", [160000, 280000])
def test_filter_path_at_max_k(ctx):
    # The candidate selector at its largest shared-memory footprint (k =
    # QSA_MAX_K): 40,000 positions (16-bit candidate positions) and 70,000
    # (32-bit), both against the oracle.
    k = qsa.QSA_MAX_K
    wl = W.make_workload("kmax", seed=5, ctx_tokens=[ctx], rows_per_req=[3], k=k, dist="int4")
    assert wl.row_visible.min() >= 3 * k
    oi, ov, _ = oracle.select_paged_tokens(wl.q, wl.w, wl.k_cache, wl.block_table, wl.row_req,
                                           wl.row_visible, k, ld=wl.ld)
    gi, gv = gpu_select(wl, path=qsa.PATH_FILTER)
    np.testing.assert_array_equal(gi, oi)
    np.testing.assert_array_equal(gv, ov)


# ---------------------------------------------------- selector on its own ----

@pytest.mark.parametrize("n,k,kind", [(5000, 700, "gauss"), (30000, 2048, "gauss"),
                                      # long rows through the sampled threshold: small k, and
                                      # a gathered set of three values (the order by position)
                                      (50000, 100, "gauss"), (20000, 1000, "few"),
                                      # just past the staging area, and a gathered set too
                                      # large for it (the digit passes take over)
                                      (8200, 4096, "gauss"), (12000, 7000, "gauss"),
                                      (60000, 2048, "ties"), (60000, 4000, "few"),
                                      (9000, 8192, "ties"), (100, 64, "ties"),
                                      # k <= 16: the warp-per-row selector
                                      (1440, 16, "gauss"), (5000, 16, "ties"), (40000, 7, "few"),
                                      (10, 16, "gauss"), (3000, 1, "ties")])
def test_topk_exact_on_oracle_style_logits(n, k, kind):
    rng = np.random.default_rng(n + k)
    R = 9
    if kind == "gauss":
        lg = rng.standard_normal((R, n)).astype(np.float32)
    elif kind == "ties":
        lg = rng.integers(-20, 21, size=(R, n)).astype(np.float32) * np.float32(0.25)
    else:
        lg = rng.integers(0, 3, size=(R, n)).astype(np.float32)
    lg[0, :] = 0.0
    lg[1, ::2] = -0.0                      # -0 ties with +0
    vis = rng.integers(0, n + 1, size=R).astype(np.int32)
    vis[:3] = n
    oi, ov = oracle.select(lg, vis, k)
    gi, gv = qsa.topk_exact(torch.from_numpy(lg).cuda(), torch.from_numpy(vis).cuda(), k)
    gi, gv = gi.cpu().numpy(), gv.cpu().numpy()
    np.testing.assert_array_equal(gi, oi)
    # values: the canonical +0 for either zero
    np.testing.assert_array_equal(gv, ov + np.float32(0.0))


# -------------------------------------------------------- device checks ----

def test_bad_page_id_is_reported_not_faulted():
    wl = W.make_workload("bp", seed=5, ctx_tokens=[2000], rows_per_req=[4], k=16, dist="int4")
    bt = wl.block_table.copy()
    bt[0, 3] = wl.k_cache.shape[0] + 1000
    d = to_device(wl)
    d["keys"] = qsa.PagedKeys(d["keys"].k_cache, torch.from_numpy(bt).cuda())
    qsa.select_paged_tokens(d["q"], d["w"], d["keys"], d["row_req"], d["row_visible"], wl.k)
    assert qsa.get_device_status() == qsa.QSA_ERR_BAD_PAGE
    assert qsa.get_device_status() == qsa.QSA_OK          # read-and-clear
    gi, _ = gpu_select(wl, d=to_device(wl))                # the context is still usable
    assert gi.shape == (wl.rows, wl.k)


def test_row_request_out_of_range_is_reported():
    wl = W.make_workload("rr", seed=6, ctx_tokens=[2000], rows_per_req=[4], k=16, dist="int4")
    d = to_device(wl)
    d["row_req"][1] = 7
    idx, _ = qsa.select_paged_tokens(d["q"], d["w"], d["keys"], d["row_req"], d["row_visible"],
                                     wl.k)
    assert qsa.get_device_status() == qsa.QSA_ERR_INVALID_ARG
    assert torch.all(idx[1] == -1)


def test_deterministic_and_counts_launches():
    wl = W.make_workload("det", seed=7, ctx_tokens=[30000], rows_per_req=[100], k=512)
    d = to_device(wl)
    a = gpu_select(wl, d)
    n = qsa.last_launch_count()
    b = gpu_select(wl, d)
    assert n >= 3
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


# ------------------------------------------------------ full-size configs ----
#
# Every row of each full-size batch is compared with the oracle, except the
# long prefill (16,384 rows x 32,768 positions), where 256 evenly spaced rows
# of each of its four requests are.  Integer-valued batches must match bit for
# bit; on Gaussian ones every returned value must be the oracle's logit at the
# returned position (within the logit tolerance) and the selected sets may
# differ only at near-ties of the cut.  The disagreement rate and the share of
# rows whose selected set is identical (the pages' own comparison) are
# recorded per batch; with QSA_PARITY_OUT set they are written there as JSON.

_PARITY = {}


@pytest.fixture(scope="module", autouse=True)
def _parity_record():
    yield
    path = os.environ.get("QSA_PARITY_OUT")
    if path and _PARITY:
        with open(path, "w") as f:
            json.dump(_PARITY, f, indent=1, sort_keys=True)


def _compared_rows(name, wl):
    if name != "long":
        return np.arange(wl.rows)
    out = []
    for b in range(len(wl.req_positions)):
        rb = np.nonzero(wl.row_req == b)[0]
        out.append(rb[np.linspace(0, len(rb) - 1, 256).astype(np.int64)])
    return np.concatenate(out)


@pytest.mark.parametrize("name", ["bench", "decode", "ties", "long", "bench_k512", "ctx29k", "bench_plus1"])
def test_full_size_config(name):
    wl = W.CONFIGS[name]()
    d = to_device(wl)
    gi, gv = gpu_select(wl, d)
    rows = _compared_rows(name, wl)
    ol, oi, ov = _oracle_rows(wl, rows)
    gi, gv = gi[rows], gv[rows]
    check_sorted_valid(gi, gv, wl.row_visible[rows], wl.k)
    if wl.meta["dist"] in ("int4", "tern"):
        np.testing.assert_array_equal(gi, oi)
        np.testing.assert_array_equal(gv, ov)
        rate, same = 0.0, 1.0
    else:
        assert_values_at_selection(gi, gv, ol)
        rate, same = near_tie_disagreement(gi, oi, ol, wl.row_visible[rows], wl.k)
    _PARITY[wl.name] = {"rows_compared": int(len(rows)), "rows": wl.rows, "k": wl.k,
                        "disagreement_rate": rate, "identical_rows": same,
                        "values": wl.meta["dist"]}
    print(f"{name}: {len(rows)} rows, disagreement rate {rate:.2e}, identical rows {same:.4f}")


@pytest.mark.parametrize("name", ["bench", "ctx29k", "decode"])
def test_full_size_selection_exact_on_gpu_logits(name):
    # The selection itself, apart from scoring rounding: both paths must pick
    # exactly what the oracle's selector picks from the GPU's own logits.
    wl = W.CONFIGS[name]()
    d = to_device(wl)
    gl = gpu_logits(wl, d)
    ei, ev = oracle.select(gl, wl.row_visible, wl.k)
    for path in (qsa.PATH_AUTO, qsa.PATH_DENSE, qsa.PATH_FILTER):
        gi, gv = gpu_select(wl, d, path=path)
        np.testing.assert_array_equal(gi, ei)
        np.testing.assert_array_equal(gv, ev)
