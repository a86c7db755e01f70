"""CPU oracle for the sparse-attention consumer, the step after the indexer:
each query row attends the raw tokens of the index positions selected for it.

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this module.  The
product path never imports, links or calls it, and it imports nothing from the
product package.  Plain numpy in float64, loops over rows and heads: meant for
small cases.

What the pages fix ("spec(MODEL-MM-QWEN4-EXP) ...", section "The component
deep-dives"): QSA attends raw tokens selected at ratio-4 granularity (not a
pooled key and value, and not whole pages); and, where the same page sets QSA
beside MiniMax-M3 in its op survey, its attention is plain GQA, 24 query heads
over 2 KV heads, head_dim 256.

Readings taken where the pages are silent:
  * row r, a query at token t_r of request b, attends the tokens 4j .. 4j + 3
    of every selected position j (the indexer's output, -1 entries ignored,
    duplicates counted once) and the tokens 4 V_r .. t_r of its current,
    unfinished block (V_r = (t_r + 1) // 4); when every visible position is
    selected that is exactly causal attention over tokens 0 .. t_r;
  * query head h reads KV head h // (H_q / H_kv);
  * weights softmax(scale * q . k), scale = 1 / sqrt(head_dim) by default;
  * the raw K and V caches are paged like the index-key cache, 64 tokens per
    page through the same block table: token p of request b sits at page
    block_table[b][p // 64], slot p % 64.
"""
from __future__ import annotations

import numpy as np

COMPRESS = 4
PAGE_TOKENS = 64


def attended_tokens(sel: np.ndarray, token: int) -> np.ndarray:
    """Sorted token positions a row at token `token` attends, given its
    selected index positions `sel` (int, -1 = none)."""
    toks = set()
    for j in np.asarray(sel).tolist():
        if j >= 0:
            toks.update(range(COMPRESS * j, COMPRESS * j + COMPRESS))
    v = (token + 1) // COMPRESS
    toks.update(range(COMPRESS * v, token + 1))
    return np.array(sorted(toks), dtype=np.int64)


def gather(cache: np.ndarray, block_table: np.ndarray, req: int, tokens: np.ndarray) -> np.ndarray:
    """cache [num_pages, 64, H_kv, D] -> [len(tokens), H_kv, D] of request `req`."""
    pages = block_table[req, tokens // PAGE_TOKENS]
    return cache[pages, tokens % PAGE_TOKENS]


def attend(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """Softmax attention of one query vector over rows of k / v (float64)."""
    s = (k.astype(np.float64) @ q.astype(np.float64)) * scale
    e = np.exp(s - s.max())
    return (e / e.sum()) @ v.astype(np.float64)


def sparse_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, block_table: np.ndarray,
                     row_req: np.ndarray, row_token: np.ndarray, sel: np.ndarray,
                     scale: float | None = None) -> np.ndarray:
    """q: float16 [R, H_q, D]; k_cache / v_cache: float16 [num_pages, 64, H_kv, D];
    block_table: int32 [B, max_pages]; row_req, row_token: [R]; sel: int32 [R, k].
    Returns float64 [R, H_q, D]."""
    R, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    group = Hq // Hkv
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    out = np.zeros((R, Hq, D), dtype=np.float64)
    for r in range(R):
        toks = attended_tokens(sel[r], int(row_token[r]))
        kk = gather(k_cache, block_table, int(row_req[r]), toks)
        vv = gather(v_cache, block_table, int(row_req[r]), toks)
        for h in range(Hq):
            g = h // group
            out[r, h] = attend(q[r, h], kk[:, g], vv[:, g], scale)
    return out
