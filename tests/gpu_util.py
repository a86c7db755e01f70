"""Helpers shared by the GPU tests: move a workload to the device, compare
selections with the oracle's under the tolerance of the step."""
from __future__ import annotations

import numpy as np
import torch

from block_sparse_attention_select_gb300 import qsa

RTOL = 1e-3      # logits: |gpu - oracle| <= RTOL * |oracle| + ATOL
ATOL = 1e-6


def to_device(wl, dev="cuda"):
    d = dict(
        q=torch.from_numpy(wl.q).to(dev),
        w=torch.from_numpy(wl.w).to(dev),
        row_req=torch.from_numpy(wl.row_req).to(dev),
        row_visible=torch.from_numpy(wl.row_visible).to(dev),
    )
    d["keys"] = qsa.PagedKeys(torch.from_numpy(wl.k_cache).to(dev),
                              torch.from_numpy(wl.block_table).to(dev))
    return d


def gpu_select(wl, d=None, k=None, path=qsa.PATH_AUTO):
    d = d or to_device(wl)
    qsa.set_config(qsa.QSA_CFG_PATH, path)
    try:
        idx, val = qsa.select_paged_tokens(d["q"], d["w"], d["keys"], d["row_req"],
                                           d["row_visible"], wl.k if k is None else k)
    finally:
        qsa.set_config(qsa.QSA_CFG_PATH, qsa.PATH_AUTO)
    st = qsa.get_device_status()
    assert st == qsa.QSA_OK, qsa.status_string(st)
    return idx.cpu().numpy(), val.cpu().numpy()


def gpu_logits(wl, d=None, ld=None):
    d = d or to_device(wl)
    ld = wl.ld if ld is None else ld
    lg = torch.empty((wl.rows, ld), dtype=torch.float32, device="cuda")
    qsa.index_score(d["q"], d["w"], d["keys"], d["row_req"], d["row_visible"], lg)
    st = qsa.get_device_status()
    assert st == qsa.QSA_OK, qsa.status_string(st)
    return lg.cpu().numpy()


def assert_logits_close(g, o, vis):
    for r in range(g.shape[0]):
        V = int(vis[r])
        gv, ov = g[r, :V].astype(np.float64), o[r, :V].astype(np.float64)
        bad = np.abs(gv - ov) > RTOL * np.abs(ov) + ATOL
        assert not np.any(bad), (r, np.nonzero(bad)[0][:5], gv[bad][:5], ov[bad][:5])
        assert np.all(np.isneginf(g[r, V:]))


def check_sorted_valid(idx, val, vis, k):
    """Structural invariants of one output block (any logits)."""
    for r in range(idx.shape[0]):
        n = min(k, int(vis[r]))
        sel = idx[r, :n]
        assert np.all(idx[r, n:] == -1), r
        assert np.all(np.isneginf(val[r, n:])), r
        assert len(np.unique(sel)) == n, r
        assert np.all((sel >= 0) & (sel < vis[r])), r
        v = val[r, :n].astype(np.float64)
        assert np.all(np.diff(v) <= 0), r
        ties = np.diff(v) == 0
        assert np.all(np.diff(sel.astype(np.int64))[ties] > 0), r


def assert_values_at_selection(g_idx, g_val, o_logits_rows):
    """Each returned value is the oracle's logit at the returned position,
    within the logit tolerance (padding excluded)."""
    sel = g_idx >= 0
    o = np.take_along_axis(o_logits_rows, np.where(sel, g_idx, 0).astype(np.int64), axis=1)
    o, g = o.astype(np.float64), g_val.astype(np.float64)
    bad = sel & (np.abs(g - o) > RTOL * np.abs(o) + ATOL)
    assert not np.any(bad), (np.argwhere(bad)[:5], g[bad][:5], o[bad][:5])


def near_tie_disagreement(g_idx, o_idx, o_logits_rows, vis, k):
    """Rows compared as sets; every position in the symmetric difference must
    score within tolerance of the oracle's k-th score.  Returns the
    disagreement rate |symdiff| / (2 * sum min(k, V)) and the share of rows
    whose selected set is identical."""
    diff, total, same = 0, 0, 0
    for r in range(g_idx.shape[0]):
        n = min(k, int(vis[r]))
        a, b = set(g_idx[r, :n].tolist()), set(o_idx[r, :n].tolist())
        sd = a ^ b
        total += 2 * n
        diff += len(sd)
        same += int(not sd)
        if sd:
            kth = float(o_logits_rows[r][o_idx[r, n - 1]])
            for j in sd:
                oj = float(o_logits_rows[r][j])
                assert abs(oj - kth) <= RTOL * abs(kth) + ATOL, (r, j, oj, kth)
    return diff / max(total, 1), same / max(g_idx.shape[0], 1)
