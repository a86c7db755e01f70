"""Pins of the index-key producer oracle against what the pages and the
mathematics fix, independent of the oracle's own code paths:

* the block boundary: a state per four tokens, emitted at the token with
  (position + 1) % 4 == 0 ("spec(MODEL-MM-QWEN4-EXP) ...", section "The
  component deep-dives"), checked by brute force over windows;
* RoPE: a rotation (pair lengths kept), the angle of a unit vector, and the
  defining property that the dot product of two rotated keys depends only on
  their position difference;
* RMSNorm: unit RMS (g = 1) and invariance to scaling the input;
* softmax pooling: invariance to shifting the logits, the one-token limit,
  constant tokens pool to themselves, the window of eight clipped at
  position 0;
* the paged store: each key lands at block_table[b][i // P], slot i % P, and
  nothing else in the cache changes.
"""
import numpy as np
import pytest

from oracle import producer as P
from block_sparse_attention_select_gb300 import workloads as W

D = 128


def _single(tokens, block, logits=None, g=None, eps=1e-6, rope_dim=64, theta=10000.0):
    g = np.ones(D, np.float32) if g is None else g
    return P.block_key(np.asarray(tokens, np.float16), logits, block, g, eps, rope_dim, theta)


def test_block_boundaries_brute_force():
    for window in (4, 8):
        for p0 in range(0, 13):
            for n in range(0, 14):
                got = P.produced_blocks(p0, n, window)
                new = set(range(p0, p0 + n))
                want = []
                for i in range(0, 10):
                    toks = set(range(4 * i, 4 * i + 4))
                    win = set(range(max(0, 4 * i + 4 - window), 4 * i + 4))
                    if toks & new and win <= new:
                        want.append(i)
                assert got == want, (window, p0, n)
    # worked cases
    assert P.produced_blocks(0, 4, 4) == [0]
    assert P.produced_blocks(0, 3, 4) == []
    assert P.produced_blocks(4, 4, 8) == []          # needs positions 0..3 too
    assert P.produced_blocks(0, 8, 8) == [0, 1]
    assert P.produced_blocks(2, 10, 4) == [1, 2]
    assert P.produced_blocks(15, 1, 4) == []         # the block's other tokens are not given
    assert P.produced_blocks(12, 4, 4) == [3]        # a decode step passes the block's four tokens
    assert P.produced_blocks(17, 1, 4) == []


def test_rope_rotates_a_unit_vector_by_the_stated_angle():
    rope_dim, theta, h = 64, 10000.0, 32
    for j in (0, 1, 7, 31):
        for block in (0, 1, 5, 777):
            u = np.zeros((4, D), np.float16)
            u[:, j] = 1.0
            out = _single(u, block, rope_dim=rope_dim, theta=theta, eps=0.0)
            y = np.sqrt(D)                              # e_j normalised to unit RMS
            assert np.hypot(out[j], out[j + h]) == pytest.approx(y, rel=1e-12)
            ang = 4 * block * theta ** (-2.0 * j / rope_dim)
            got = np.arctan2(out[j + h], out[j])
            assert np.cos(got - ang) == pytest.approx(1.0, abs=1e-12)
            rest = np.delete(out, [j, j + h])
            assert np.all(rest == 0.0)


def test_rope_dot_depends_only_on_position_difference():
    rng = np.random.default_rng(5)
    a = np.repeat(rng.standard_normal((1, D)).astype(np.float16), 4, axis=0)
    b = np.repeat(rng.standard_normal((1, D)).astype(np.float16), 4, axis=0)
    for (i1, i2, shift) in ((3, 10, 17), (0, 1, 1000), (250, 200, 4321)):
        d0 = _single(a, i1) @ _single(b, i2)
        d1 = _single(a, i1 + shift) @ _single(b, i2 + shift)
        assert d1 == pytest.approx(d0, rel=1e-9, abs=1e-9)
    # and it does change with the difference (the rotation is not trivial)
    assert abs(_single(a, 3) @ _single(b, 10) - _single(a, 3) @ _single(b, 11)) > 1e-3


def test_rope_keeps_pair_lengths_and_passes_the_rest():
    rng = np.random.default_rng(6)
    toks = rng.standard_normal((4, D)).astype(np.float16)
    at0 = _single(toks, 0)          # position 0: no rotation
    at9 = _single(toks, 9)
    h = 32
    np.testing.assert_allclose(np.hypot(at9[:h], at9[h:64]), np.hypot(at0[:h], at0[h:64]), rtol=1e-12)
    np.testing.assert_array_equal(at9[64:], at0[64:])


def test_rmsnorm_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(7)
    toks = (rng.standard_normal((4, D)) * 0.5).astype(np.float16)
    out = _single(toks, 0, eps=0.0)
    assert np.sqrt(np.mean(out * out)) == pytest.approx(1.0, rel=1e-12)
    big = (toks.astype(np.float32) * 4).astype(np.float16)     # exact: a power of two
    np.testing.assert_allclose(_single(big, 5, eps=0.0), _single(toks, 5, eps=0.0), rtol=1e-12, atol=1e-12)
    # the weight multiplies dimension by dimension
    g = np.linspace(0.5, 1.5, D).astype(np.float32)
    np.testing.assert_allclose(_single(toks, 0, g=g, eps=0.0), out * g.astype(np.float64), rtol=1e-12)


def test_softmax_pool_shift_and_limits():
    rng = np.random.default_rng(8)
    toks = rng.standard_normal((8, D)).astype(np.float16)
    lg = rng.standard_normal(8)                                   # float64: the shift is exact enough
    base = _single(toks, 3, logits=lg)
    np.testing.assert_allclose(_single(toks, 3, logits=lg + 7.0), base, rtol=1e-12, atol=1e-13)
    # one dominant logit: the key of that token alone
    spike = np.zeros(8, np.float32)
    spike[5] = 80.0
    np.testing.assert_allclose(_single(toks, 3, logits=spike), _single(toks[5:6], 3), rtol=1e-9, atol=1e-12)
    # equal tokens pool to themselves whatever the weights
    same = np.repeat(toks[:1], 8, axis=0)
    np.testing.assert_allclose(_single(same, 3, logits=lg), _single(same[:1], 3), rtol=1e-12, atol=1e-14)
    # no logits = the mean = equal logits
    np.testing.assert_allclose(_single(toks, 3), _single(toks, 3, logits=np.zeros(8)),
                               rtol=1e-12, atol=1e-14)


def test_window_eight_at_block_zero_is_the_block_itself():
    inp = W.make_producer_inputs("w", seed=3, new_tokens=[12], pos_start=[0], window=8, logits=True)
    c8, d8 = P.produce(inp.x, inp.pool_logit, inp.seq_start, inp.pos_start, inp.norm_weight, inp.eps,
                       inp.rope_dim, inp.theta, 8, inp.k_cache, inp.block_table)
    c4, d4 = P.produce(inp.x, inp.pool_logit, inp.seq_start, inp.pos_start, inp.norm_weight, inp.eps,
                       inp.rope_dim, inp.theta, 4, inp.k_cache, inp.block_table)
    assert d8 == d4 == [(0, 0), (0, 1), (0, 2)]
    pg = inp.block_table[0, 0]
    np.testing.assert_array_equal(c8[pg, 0], c4[pg, 0])
    assert not np.array_equal(c8[pg, 1], c4[pg, 1])        # later blocks see the wider window


def test_paged_store_layout_and_untouched_slots():
    inp = W.producer_small()
    cache, done = P.produce(inp.x, inp.pool_logit, inp.seq_start, inp.pos_start, inp.norm_weight, inp.eps,
                            inp.rope_dim, inp.theta, inp.window, inp.k_cache, inp.block_table)
    written = np.zeros(inp.k_cache.shape[:2], bool)
    for b, i in done:
        page, slot = inp.block_table[b, i // 16], i % 16
        assert not written[page, slot]
        written[page, slot] = True
        t0, p0 = inp.seq_start[b], inp.pos_start[b]
        toks = inp.x[t0 + 4 * i - p0: t0 + 4 * i - p0 + 4]
        want = P.block_key(toks, None, i, inp.norm_weight, inp.eps, inp.rope_dim, inp.theta).astype(np.float16)
        np.testing.assert_array_equal(cache[page, slot], want)
    np.testing.assert_array_equal(cache[~written], inp.k_cache[~written])
    # per request, the blocks the boundary rule names
    per_req = {}
    for b, i in done:
        per_req.setdefault(b, []).append(i)
    n = np.diff(inp.seq_start)
    for b in range(len(inp.pos_start)):
        assert per_req.get(b, []) == P.produced_blocks(int(inp.pos_start[b]), int(n[b]), 4)
    assert per_req[3] == [3] and 4 not in per_req and 5 not in per_req   # decode-shaped requests
