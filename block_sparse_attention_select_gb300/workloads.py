"""Seeded synthetic inputs for the QSA indexer step.

This module only draws inputs (numpy PCG64 streams, platform independent); it
holds none of the indexer's arithmetic.  Both the CUDA path and the CPU oracle
are fed the very same bytes from here.

Shapes follow the workloads the pages describe: a key cache of one FP16 index
key (dim 128) per compressed position, compress ratio 4, 64-token pages of 16
positions, an int32 block table per request, and query rows that each see the
compressed positions completed before them.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

COMPRESS_RATIO = 4
PAGE_POSITIONS = 16          # 64-token pages at compress ratio 4
HEAD_DIM = 128


@dataclass
class Workload:
    name: str
    q: np.ndarray             # float16 [R, H, D]
    w: np.ndarray             # float32 [R, H]
    k_cache: np.ndarray       # float16 [num_pages, PAGE_POSITIONS, D]
    block_table: np.ndarray   # int32 [num_reqs, max_pages]
    row_req: np.ndarray       # int32 [R]
    row_visible: np.ndarray   # int32 [R]
    row_token: np.ndarray     # int64 [R] 0-based token position of each query row
    req_positions: np.ndarray  # int32 [num_reqs] compressed positions stored per request
    k: int
    meta: dict = field(default_factory=dict)

    @property
    def rows(self) -> int:
        return int(self.q.shape[0])

    @property
    def heads(self) -> int:
        return int(self.q.shape[1])

    @property
    def ld(self) -> int:
        """Longest row a request's block table can address (logit row stride)."""
        return int(self.block_table.shape[1]) * int(self.k_cache.shape[1])

    @property
    def visible_pairs(self) -> int:
        return int(np.sum(self.row_visible.astype(np.int64)))


def _values(rng: np.random.Generator, shape, dist: str) -> np.ndarray:
    if dist == "int4":
        return rng.integers(-4, 5, size=shape).astype(np.float16)
    if dist == "tern":
        return rng.integers(-1, 2, size=shape).astype(np.float16)
    if dist == "gauss":
        return (rng.standard_normal(size=shape, dtype=np.float32)
                / np.float32(np.sqrt(128.0))).astype(np.float16)
    if dist == "zero":
        return np.zeros(shape, dtype=np.float16)
    raise ValueError(dist)


def _weights(rng: np.random.Generator, shape, dist: str) -> np.ndarray:
    if dist == "int4":
        return rng.choice(np.array([0.25, 0.5, 1.0, 2.0], dtype=np.float32), size=shape)
    if dist in ("tern", "ones"):
        return np.ones(shape, dtype=np.float32)
    if dist == "gauss":
        return rng.random(size=shape, dtype=np.float32)
    if dist == "zero":
        return np.zeros(shape, dtype=np.float32)
    if dist == "int4_signed":
        # dyadic magnitudes with either sign: integer-valued scores stay exact
        mag = rng.choice(np.array([0.25, 0.5, 1.0, 2.0], dtype=np.float32), size=shape)
        return np.where(rng.random(size=shape) < 0.5, -mag, mag).astype(np.float32)
    if dist == "gauss_signed":
        return (2.0 * rng.random(size=shape, dtype=np.float32) - 1.0).astype(np.float32)
    raise ValueError(dist)


def make_workload(name: str, *, seed: int, ctx_tokens, rows_per_req, k: int, heads: int = 4,
                  head_dim: int = HEAD_DIM, page_positions: int = PAGE_POSITIONS,
                  dist: str = "gauss", wdist: str | None = None, shuffle_pages: bool = True,
                  visibility: str = "pages", extra_pages: int = 0) -> Workload:
    """Build one batch.

    ctx_tokens[b]: tokens in request b's context; the request stores
    ctx // 4 compressed positions.  rows_per_req[b]: query rows of request b,
    the last rows of its context (prefill chunk / decode token).
    visibility: "pages" -> V = (t+1) // 4 (a position is stored once its fourth
    token exists); "plus_one" -> V = t // 4 + 1 (the alternative reading).
    """
    rng = np.random.default_rng(seed)
    ctx_tokens = [int(c) for c in ctx_tokens]
    rows_per_req = [int(n) for n in rows_per_req]
    B = len(ctx_tokens)
    assert len(rows_per_req) == B
    P = [c // COMPRESS_RATIO for c in ctx_tokens]
    pages = [-(-p // page_positions) for p in P]
    max_pages = max(1, max(pages) + extra_pages)
    num_pages = max(1, sum(pages))
    phys = rng.permutation(num_pages).astype(np.int32) if shuffle_pages else \
        np.arange(num_pages, dtype=np.int32)
    bt = np.full((B, max_pages), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        bt[b, :pages[b]] = phys[off:off + pages[b]]
        off += pages[b]
    k_cache = _values(rng, (num_pages, page_positions, head_dim), dist)
    row_req, row_tok = [], []
    for b in range(B):
        n = rows_per_req[b]
        row_req += [b] * n
        row_tok += list(range(ctx_tokens[b] - n, ctx_tokens[b]))
    R = len(row_req)
    q = _values(rng, (R, heads, head_dim), dist)
    w = _weights(rng, (R, heads), wdist or dist)
    row_tok = np.asarray(row_tok, dtype=np.int64)
    if visibility == "pages":
        vis = (row_tok + 1) // COMPRESS_RATIO
    elif visibility == "plus_one":
        vis = row_tok // COMPRESS_RATIO + 1
    else:
        raise ValueError(visibility)
    req_arr = np.asarray(row_req, dtype=np.int32)
    vis = np.minimum(vis, np.asarray(P, dtype=np.int64)[req_arr]).astype(np.int32)
    return Workload(name=name, q=q, w=w, k_cache=k_cache, block_table=bt, row_req=req_arr,
                    row_visible=vis, row_token=row_tok, req_positions=np.asarray(P, np.int32),
                    k=int(k), meta=dict(seed=seed, dist=dist, shuffle=shuffle_pages,
                                        visibility=visibility))


# The five synthetic batches (sizes as in the kernel-bench description of the
# pages plus the decode, tie-stress and long-prefill shapes built around it).

def tiny(seed: int = 0) -> Workload:
    """1 request, 64 rows at the end of a 1,024-token context, k 64, integer data."""
    return make_workload("tiny_1x64rows_ctx1024_k64_int", seed=seed, ctx_tokens=[1024],
                         rows_per_req=[64], k=64, dist="int4", shuffle_pages=False)


def bench(seed: int = 1, k: int = 2048, ctx: int = 184_320, visibility: str = "pages") -> Workload:
    """Last 1,616-row chunk of a 184,320-token context (46,080 positions), k 2,048."""
    tag = "" if visibility == "pages" else f"_vis-{visibility}"
    return make_workload(f"prefill_1x1616rows_ctx{ctx}_k{k}{tag}", seed=seed, ctx_tokens=[ctx],
                         rows_per_req=[1616], k=k, dist="gauss", shuffle_pages=False,
                         visibility=visibility)


def decode(seed: int = 2, num_reqs: int = 64) -> Workload:
    """64 requests x 1 row, contexts uniform in [8,192, 131,072] tokens, k 2,048."""
    rng = np.random.default_rng(10_000 + seed)
    ctx = rng.integers(8192, 131072, size=num_reqs, endpoint=True)
    return make_workload(f"decode_{num_reqs}x1row_ctx8k-128k_k2048", seed=seed, ctx_tokens=ctx,
                         rows_per_req=[1] * num_reqs, k=2048, dist="gauss", shuffle_pages=True)


def tie_stress(seed: int = 3) -> Workload:
    """8 requests x 256 rows at the end of 32,768 tokens, ternary data, w = 1, k 512."""
    return make_workload("ties_8x256rows_ctx32768_k512_tern", seed=seed, ctx_tokens=[32768] * 8,
                         rows_per_req=[256] * 8, k=512, dist="tern", shuffle_pages=True)


def long_prefill(seed: int = 4) -> Workload:
    """4 requests x 4,096 rows at the end of 131,072 tokens (32,768 positions), k 2,048."""
    return make_workload("prefill_4x4096rows_ctx131072_k2048", seed=seed,
                         ctx_tokens=[131072] * 4, rows_per_req=[4096] * 4, k=2048,
                         dist="gauss", shuffle_pages=True)


def bench_k512(seed: int = 1) -> Workload:
    """The prefill bench shape with k = 512 positions (the pages' "block top-k 512")."""
    return bench(seed=seed, k=512)


def bench_ctx29k(seed: int = 1) -> Workload:
    """The prefill bench shape at the pages' other context point, 29,000 tokens (7,250 positions)."""
    return bench(seed=seed, ctx=29_000)


def bench_plus_one(seed: int = 1) -> Workload:
    """The prefill bench shape with V_r = t_r // 4 + 1 (the other reading of the visible count)."""
    return bench(seed=seed, visibility="plus_one")


CONFIGS = {
    "tiny": tiny,
    "bench": bench,
    "decode": decode,
    "ties": tie_stress,
    "long": long_prefill,
    "bench_k512": bench_k512,
    "ctx29k": bench_ctx29k,
    "bench_plus1": bench_plus_one,
}


# ------------------------------------------------------------------------
# Inputs of the index-key producer (the step before the indexer): the raw
# per-token index keys of each request's new tokens, optional pooling logits,
# the RMSNorm weight and a paged cache to store into.  Random draws only.

@dataclass
class ProducerInputs:
    name: str
    x: np.ndarray              # float16 [T, D] raw index keys, request after request
    pool_logit: np.ndarray | None   # float32 [T] or None (equal weights)
    seq_start: np.ndarray      # int32 [num_reqs + 1] row offsets into x
    pos_start: np.ndarray      # int32 [num_reqs] position of each request's first new token
    norm_weight: np.ndarray    # float32 [D]
    k_cache: np.ndarray        # float16 [num_pages, PAGE_POSITIONS, D] cache before the call
    block_table: np.ndarray    # int32 [num_reqs, max_pages]
    window: int                # pooling window in tokens (4 or 8)
    rope_dim: int = 64
    theta: float = 10000.0
    eps: float = 1e-6

    @property
    def tokens(self) -> int:
        return int(self.x.shape[0])

    @property
    def max_tokens(self) -> int:
        return int(np.max(np.diff(self.seq_start))) if len(self.pos_start) else 0


def make_producer_inputs(name: str, *, seed: int, new_tokens, pos_start, window: int = 4,
                         logits: bool = False, rope_dim: int = 64, spare_pages: int = 3) -> ProducerInputs:
    """new_tokens[b] tokens for request b starting at position pos_start[b];
    each request's block table covers its last position, pages shuffled over
    a cache with a few spare pages (filled with random keys, never written)."""
    rng = np.random.default_rng(seed)
    new_tokens = np.asarray(new_tokens, dtype=np.int64)
    pos_start = np.asarray(pos_start, dtype=np.int64)
    nreq = len(new_tokens)
    seq_start = np.zeros(nreq + 1, dtype=np.int32)
    seq_start[1:] = np.cumsum(new_tokens)
    T = int(seq_start[-1])
    x = (rng.standard_normal((T, HEAD_DIM)) * 0.5).astype(np.float16)
    pool_logit = (rng.standard_normal(T) * 1.5).astype(np.float32) if logits else None
    norm_weight = (1.0 + 0.1 * rng.standard_normal(HEAD_DIM)).astype(np.float32)
    blocks_end = (pos_start + new_tokens + COMPRESS_RATIO - 1) // COMPRESS_RATIO
    pages_per_req = np.maximum(1, (blocks_end + PAGE_POSITIONS - 1) // PAGE_POSITIONS)
    max_pages = int(pages_per_req.max()) if nreq else 1
    num_pages = int(pages_per_req.sum()) + spare_pages
    perm = rng.permutation(num_pages).astype(np.int32)
    block_table = np.full((max(nreq, 1), max_pages), -1, dtype=np.int32)
    at = 0
    for b in range(nreq):
        n = int(pages_per_req[b])
        block_table[b, :n] = perm[at:at + n]
        at += n
    k_cache = (rng.standard_normal((num_pages, PAGE_POSITIONS, HEAD_DIM)) * 0.25).astype(np.float16)
    return ProducerInputs(name, x, pool_logit, seq_start, pos_start.astype(np.int32), norm_weight,
                          k_cache, block_table, window, rope_dim)


def producer_small(seed: int = 11, window: int = 4, logits: bool = False) -> ProducerInputs:
    """Ragged requests: from position 0, mid-context chunks (aligned and not), a
    decode step that completes a block (passing the block's four tokens), a
    decode token that completes none, an empty request."""
    return make_producer_inputs("producer_small", seed=seed, window=window, logits=logits,
                                new_tokens=[37, 64, 23, 4, 1, 0, 300],
                                pos_start=[0, 128, 70, 12, 17, 40, 1000])


def producer_context(seed: int = 12, window: int = 4, logits: bool = False) -> ProducerInputs:
    """One request's whole 184,320-token context (46,080 index keys)."""
    return make_producer_inputs("producer_ctx184320", seed=seed, window=window, logits=logits,
                                new_tokens=[184_320], pos_start=[0])


def producer_chunk(seed: int = 13, window: int = 4, logits: bool = False) -> ProducerInputs:
    """The new tokens of a 1,616-token prefill chunk at the end of a 184,320-token context."""
    return make_producer_inputs("producer_chunk1616", seed=seed, window=window, logits=logits,
                                new_tokens=[1616], pos_start=[184_320 - 1616])


PRODUCER_CONFIGS = {
    "small": producer_small,
    "context": producer_context,
    "chunk": producer_chunk,
}


# ------------------------------------------------------------------------
# Inputs of the sparse-attention consumer (the step after the indexer): query
# heads, raw K / V caches paged 64 tokens to a page through the index cache's
# block table, and each row's selected index positions.  Random draws only.

CONSUMER_Q_HEADS = 24
CONSUMER_KV_HEADS = 2
CONSUMER_HEAD_DIM = 256
PAGE_TOKENS = PAGE_POSITIONS * COMPRESS_RATIO      # 64


@dataclass
class ConsumerInputs:
    name: str
    q: np.ndarray            # float16 [R, 24, 256]
    k_cache: np.ndarray      # float16 [num_pages, 64, 2, 256]
    v_cache: np.ndarray      # float16 [num_pages, 64, 2, 256]
    block_table: np.ndarray  # int32 [num_reqs, max_pages]
    row_req: np.ndarray      # int32 [R]
    row_token: np.ndarray    # int32 [R] token position of each query row
    sel: np.ndarray          # int32 [R, k] selected index positions (-1 = none)


def make_consumer_inputs(name: str, *, seed: int, ctx_tokens, rows_per_req, k: int,
                         all_selected_rows: int = 0) -> ConsumerInputs:
    """Request b holds ctx_tokens[b] tokens; its last rows_per_req[b] tokens are
    query rows.  Each row's selection is k distinct visible positions drawn at
    random (all of them when fewer are visible); the first all_selected_rows
    rows of request 0 select every visible position."""
    rng = np.random.default_rng(seed)
    ctx = np.asarray(ctx_tokens, dtype=np.int64)
    nreq = len(ctx)
    pages_per_req = (ctx + PAGE_TOKENS - 1) // PAGE_TOKENS
    max_pages = int(pages_per_req.max())
    num_pages = int(pages_per_req.sum()) + 2
    perm = rng.permutation(num_pages).astype(np.int32)
    block_table = np.full((nreq, max_pages), -1, dtype=np.int32)
    at = 0
    for b in range(nreq):
        n = int(pages_per_req[b])
        block_table[b, :n] = perm[at:at + n]
        at += n
    shape = (num_pages, PAGE_TOKENS, CONSUMER_KV_HEADS, CONSUMER_HEAD_DIM)
    k_cache = (rng.standard_normal(shape) * 0.5).astype(np.float16)
    v_cache = rng.standard_normal(shape).astype(np.float16)
    rows_req, rows_tok, sels = [], [], []
    for b in range(nreq):
        for t in range(int(ctx[b]) - int(rows_per_req[b]), int(ctx[b])):
            v = (t + 1) // COMPRESS_RATIO
            if b == 0 and len(rows_tok) < all_selected_rows or v <= k:
                if v > k:
                    raise ValueError("a row selecting every visible position needs k >= its visible count")
                s = np.arange(v)
            else:
                s = np.sort(rng.choice(v, size=k, replace=False))
            row = np.full(k, -1, dtype=np.int32)
            row[:len(s)] = s[:k]
            rows_req.append(b)
            rows_tok.append(t)
            sels.append(row)
    R = len(rows_tok)
    q = (rng.standard_normal((R, CONSUMER_Q_HEADS, CONSUMER_HEAD_DIM)) * 0.5).astype(np.float16)
    return ConsumerInputs(name, q, k_cache, v_cache, block_table, np.array(rows_req, np.int32),
                          np.array(rows_tok, np.int32), np.array(sels, np.int32).reshape(R, k))


# ------------------------------------------------------------------------
# Inputs of the second workload, the M3-style block scorer: per-head index
# queries and per-token, per-head index keys paged 128 tokens to a page.
# Random draws only.

SCORER_BLOCK = 128


@dataclass
class BlockScorerInputs:
    name: str
    q: np.ndarray            # float16 [R, H, 128]
    k_cache: np.ndarray      # float16 [num_pages, 128, H, 128]
    block_table: np.ndarray  # int32 [num_reqs, max_pages]
    row_req: np.ndarray      # int32 [R]
    row_token: np.ndarray    # int32 [R]
    k: int


def make_block_scorer_inputs(name: str, *, seed: int, ctx_tokens, rows_per_req, k: int, heads: int = 2,
                             dist: str = "gauss") -> BlockScorerInputs:
    rng = np.random.default_rng(seed)
    ctx = np.asarray(ctx_tokens, dtype=np.int64)
    nreq = len(ctx)
    pages_per_req = (ctx + SCORER_BLOCK - 1) // SCORER_BLOCK
    num_pages = int(pages_per_req.sum()) + 2
    perm = rng.permutation(num_pages).astype(np.int32)
    block_table = np.full((nreq, int(pages_per_req.max())), -1, dtype=np.int32)
    at = 0
    for b in range(nreq):
        n = int(pages_per_req[b])
        block_table[b, :n] = perm[at:at + n]
        at += n
    shape = (num_pages, SCORER_BLOCK, heads, HEAD_DIM)
    if dist == "int":
        k_cache = rng.integers(-2, 3, size=shape).astype(np.float16)
    else:
        k_cache = (rng.standard_normal(shape) / np.sqrt(HEAD_DIM)).astype(np.float16)
    rows_req, rows_tok = [], []
    for b in range(nreq):
        for t in range(int(ctx[b]) - int(rows_per_req[b]), int(ctx[b])):
            rows_req.append(b)
            rows_tok.append(t)
    R = len(rows_tok)
    if dist == "int":
        q = rng.integers(-2, 3, size=(R, heads, HEAD_DIM)).astype(np.float16)
    else:
        q = rng.standard_normal((R, heads, HEAD_DIM)).astype(np.float16)
    return BlockScorerInputs(name, q, k_cache, block_table, np.array(rows_req, np.int32),
                             np.array(rows_tok, np.int32), k)


def block_scorer_bench(seed: int = 41) -> BlockScorerInputs:
    """The indexer bench's prefill chunk for the block scorer: 1,616 query rows at
    the end of a 184,320-token context, 2 KV heads, the top 16 blocks of 128
    tokens (a 2,048-token budget) per row and head."""
    return make_block_scorer_inputs("blocks_1x1616rows_ctx184320_h2_k16", seed=seed, ctx_tokens=[184_320],
                                    rows_per_req=[1616], k=16, heads=2)
