"""CPU oracle for the second workload: the MiniMax-M3-style block scorer, which
scores KV blocks of raw tokens per KV head and keeps the top-k blocks.

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this module.  The
product path never imports, links or calls it, and it imports nothing from the
product package.  Plain numpy in float64.

What the pages fix ("spec(MODEL-MM-QWEN4-EXP) ...", section "The component
deep-dives", where M3 is set against QSA): the block score is the maximum of
the query-key dot products over the block's raw tokens, with no pooling, no
ReLU and no reduction over heads; index heads equal KV heads, so each query
token gets one block set per KV head; the block is 128 tokens, the KV page
size; a bitonic top-k picks the blocks.

Readings taken where the pages are silent:
  * a query at token t sees the tokens 0 .. t; a block counts when it holds at
    least one of them, and its score is the maximum over those only;
  * the top-k is ordered by score descending, the lower block index first on
    equal scores, padded with -1 (the bitonic network's own tie order is not
    described);
  * index keys are stored per raw token and head, paged 128 tokens to a page:
    token p of request b at page block_table[b][p // 128], slot p % 128.
"""
from __future__ import annotations

import numpy as np

BLOCK = 128


def block_scores(q: np.ndarray, keys: np.ndarray, token: int) -> np.ndarray:
    """q: [D] one head's query; keys: [n, D] that head's keys of tokens 0 .. n-1
    (n > token).  Returns the score of every block holding a visible token."""
    s = keys[: token + 1].astype(np.float64) @ q.astype(np.float64)
    nb = token // BLOCK + 1
    return np.array([s[BLOCK * c: BLOCK * (c + 1)].max() for c in range(nb)])


def top_blocks(scores: np.ndarray, k: int) -> np.ndarray:
    """Block indices by (score desc, index asc), the first k, -1 padded."""
    order = sorted(range(len(scores)), key=lambda c: (-scores[c], c))[:k]
    out = np.full(k, -1, dtype=np.int32)
    out[: len(order)] = order
    return out


def select_blocks(q: np.ndarray, k_cache: np.ndarray, block_table: np.ndarray, row_req: np.ndarray,
                  row_token: np.ndarray, k: int):
    """q: float16 [R, H, D]; k_cache: float16 [num_pages, 128, H, D];
    block_table: int32 [B, max_pages]; row_req, row_token: [R].
    Returns (int32 [R, H, k] block indices, float64 [R, H, k] scores, -inf pad)."""
    R, H, _ = q.shape
    idx = np.full((R, H, k), -1, dtype=np.int32)
    val = np.full((R, H, k), -np.inf)
    for r in range(R):
        b, t = int(row_req[r]), int(row_token[r])
        pages = block_table[b, : t // BLOCK + 1]
        keys = k_cache[pages].reshape(-1, H, k_cache.shape[3])        # tokens 0 .. 128 * pages - 1
        for h in range(H):
            sc = block_scores(q[r, h], keys[:, h], t)
            top = top_blocks(sc, k)
            idx[r, h] = top
            val[r, h, top >= 0] = sc[top[top >= 0]]
    return idx, val
