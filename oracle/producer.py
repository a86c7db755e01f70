"""CPU oracle for the index-key producer, the step before the indexer: each
completed block of four tokens is pooled into one index key, RMS-normalised,
rotated (RoPE) at the block's first token position and stored in its slot of
the paged key cache.

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this module.  The
product path never imports, links or calls it, and it imports nothing from the
product package.  Plain numpy in float64; pure-Python loops over blocks, so it
is meant for the small cases the tests use and bounded samples.

What the pages fix ("spec(MODEL-MM-QWEN4-EXP) ...", section "The component
deep-dives", the list of structural matches with DeepSeek-V4): compress ratio
4, one stored index-key state per four tokens, the state emitted at the token
with (position + 1) % 4 == 0, RMSNorm on the pooled key and RoPE at the
block-start position; the same section notes that the DSv4 compress kernel is
not a mean pool but a learned softmax pool over an overlapping window of eight
tokens, driven by a score channel the QSA checkpoint does not have.

Readings taken where the pages are silent:
  * pool: weights softmax(pool_logit) over the window's tokens, or equal
    weights (the mean) when no logits are given; window W = 4 (the block) or 8
    (the block and the four tokens before it), clipped at position 0;
  * RMSNorm: v / sqrt(mean(v^2) + eps) * g, with a weight vector g;
  * RoPE: the first rope_dim dimensions rotate in pairs (j, j + rope_dim/2)
    by angle P * theta^(-2j / rope_dim), P = 4i the block's first token
    position; the other dimensions pass through;
  * a call with the new tokens [p0, p0 + n) of a request produces block i
    when the block is complete inside them and every existing position of its
    window is among them (the caller passes the window's earlier tokens when
    it wants such a block produced);
  * the stored key is rounded to FP16 (the key cache's type).
"""
from __future__ import annotations

import numpy as np

COMPRESS = 4   # tokens per stored index key


def produced_blocks(pos_start: int, n_tokens: int, window: int) -> list[int]:
    """Blocks a call produces for new tokens [pos_start, pos_start + n_tokens).

    Block i ends at position 4i + 3, the token with (position + 1) % 4 == 0;
    its window starts at max(0, 4i + 4 - window)."""
    out = []
    for p in range(pos_start, pos_start + n_tokens):
        if (p + 1) % COMPRESS != 0:
            continue
        i = (p + 1) // COMPRESS - 1
        if max(0, COMPRESS * i + COMPRESS - window) >= pos_start:
            out.append(i)
    return out


def pool(tokens: np.ndarray, logits: np.ndarray | None) -> np.ndarray:
    """Softmax-weighted sum of the window's token keys (the mean without logits)."""
    x = tokens.astype(np.float64)
    if logits is None:
        a = np.full(x.shape[0], 1.0 / x.shape[0])
    else:
        z = logits.astype(np.float64)
        e = np.exp(z - z.max())
        a = e / e.sum()
    return a @ x


def rms_norm(v: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm on the pooled key."""
    return v / np.sqrt(np.mean(v * v) + eps) * g.astype(np.float64)


def rope(v: np.ndarray, position: int, rope_dim: int, theta: float) -> np.ndarray:
    """Rotary embedding of the first rope_dim dimensions at `position`."""
    h = rope_dim // 2
    out = v.copy()
    if h == 0:
        return out
    j = np.arange(h, dtype=np.float64)
    ang = float(position) * np.power(float(theta), -2.0 * j / rope_dim)
    c, s = np.cos(ang), np.sin(ang)
    a, b = v[:h], v[h:rope_dim]
    out[:h] = a * c - b * s
    out[h:rope_dim] = a * s + b * c
    return out


def block_key(tokens: np.ndarray, logits: np.ndarray | None, block: int, g: np.ndarray, eps: float,
              rope_dim: int, theta: float) -> np.ndarray:
    """The stored key of one block from its window's tokens, in float64."""
    return rope(rms_norm(pool(tokens, logits), g, eps), COMPRESS * block, rope_dim, theta)


def produce(x: np.ndarray, pool_logit: np.ndarray | None, seq_start: np.ndarray, pos_start: np.ndarray,
            norm_weight: np.ndarray, eps: float, rope_dim: int, theta: float, window: int,
            k_cache: np.ndarray, block_table: np.ndarray):
    """Returns (the key cache after the call, the list of (request, block) produced).

    x: float16 [T, D] token keys, request b's tokens at rows seq_start[b] ..
    seq_start[b + 1] - 1 with positions pos_start[b] ..; pool_logit: float32
    [T] or None; k_cache: float16 [num_pages, P, D] (copied, not modified);
    block_table: int32 [num_reqs, max_pages].  A block whose page entry is
    outside the table or the cache is not stored (the library flags it)."""
    cache = k_cache.copy()
    num_pages, P = cache.shape[0], cache.shape[1]
    done = []
    for b in range(len(pos_start)):
        t0, t1 = int(seq_start[b]), int(seq_start[b + 1])
        p0 = int(pos_start[b])
        for i in produced_blocks(p0, t1 - t0, window):
            first = max(0, COMPRESS * i + COMPRESS - window)
            last = COMPRESS * i + COMPRESS - 1
            lo, hi = t0 + first - p0, t0 + last - p0 + 1
            lg = None if pool_logit is None else pool_logit[lo:hi]
            key = block_key(x[lo:hi], lg, i, norm_weight, eps, rope_dim, theta)
            if i // P >= block_table.shape[1]:
                continue
            page = int(block_table[b, i // P])
            if page < 0 or page >= num_pages:
                continue
            cache[page, i % P] = key.astype(np.float16)
            done.append((b, i))
    return cache, done
