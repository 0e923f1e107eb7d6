"""Pins for the oracle's rotary encoding and cache append (the step before the
decode path: "DeepSeek-V3 MLA deep engineering", sec. 3.1 decoupled RoPE -
a position-dependent rotation of the rope parts - and sec. 4.3, only the
latent is stored in the paged cache).

The pages describe RoPE only in words; the oracle takes the standard rotary
encoding (adjacent pairs rotated by position x theta_i, theta_i =
base^(-2i/d)). Pins that a wrong pairing, sign, frequency or position fails:
  * position 0 is the identity;
  * a base chosen so that theta_1 = pi/2 (d = 4): position 1 turns pair 1 by a
    quarter turn, (a, b) -> (-b, a); position 2 by a half turn, (a, b) -> (-a, -b);
  * with d = 2 the single pair turns by exactly `position` radians: position 1
    gives (cos 1, sin 1) for (1, 0) (tabulated values);
  * every pair keeps its length;
  * relative position: <RoPE(q, m), RoPE(k, n)> depends only on m - n (the
    property the pages give as the reason for RoPE: a positional term of t);
  * composition: RoPE(RoPE(x, a), b) = RoPE(x, a + b);
  * cache append: the latent is copied bit-exactly into row t % 64 of block
    table[b][t / 64] with t = seqlen - s_q + s, the rope part is RoPE at t,
    every other slot is untouched, tokens at t < 0 are skipped.
"""
import math

import numpy as np
import pytest

import oracle


def rng(seed):
    return np.random.default_rng(seed)


def test_position_zero_is_identity():
    x = rng(1).standard_normal((5, 64)).astype(np.float32)
    y = oracle.rope(x, np.zeros(5, np.int64))
    assert np.array_equal(y, x.astype(np.float64))


def test_quarter_and_half_turns():
    base = (2.0 / math.pi) ** 2  # theta_1 = base^(-2/4) = pi/2 for d = 4
    x = np.array([[1.0, 2.0, 3.0, 4.0]], np.float32)
    y1 = oracle.rope(x, [1], base)[0]
    assert y1[2:] == pytest.approx([-4.0, 3.0], abs=1e-12)
    y2 = oracle.rope(x, [2], base)[0]
    assert y2[2:] == pytest.approx([-3.0, -4.0], abs=1e-12)
    # pair 0 (theta_0 = 1) turns by 1 and 2 radians
    assert y1[:2] == pytest.approx([math.cos(1) - 2 * math.sin(1), math.sin(1) + 2 * math.cos(1)], abs=1e-12)


def test_single_pair_turns_by_position_radians():
    y = oracle.rope(np.array([[1.0, 0.0]], np.float32), [1])[0]
    assert y == pytest.approx([0.5403023058681398, 0.8414709848078965], abs=1e-15)


def test_pairs_keep_their_length():
    x = rng(2).standard_normal((7, 64)).astype(np.float32)
    pos = rng(3).integers(0, 40000, 7)
    y = oracle.rope(x, pos)
    nx = np.hypot(x[:, 0::2].astype(np.float64), x[:, 1::2])
    ny = np.hypot(y[:, 0::2], y[:, 1::2])
    assert np.allclose(nx, ny, rtol=1e-12)


def test_relative_position():
    q = rng(4).standard_normal((1, 64)).astype(np.float32)
    k = rng(5).standard_normal((1, 64)).astype(np.float32)
    dots = []
    for m, n in ((7, 3), (104, 100), (30004, 30000)):
        dots.append(float(oracle.rope(q, [m])[0] @ oracle.rope(k, [n])[0]))
    assert dots[1] == pytest.approx(dots[0], rel=1e-9)
    assert dots[2] == pytest.approx(dots[0], rel=1e-7)
    # and it does depend on the offset
    other = float(oracle.rope(q, [9])[0] @ oracle.rope(k, [3])[0])
    assert abs(other - dots[0]) > 1e-3


def test_composition():
    x = rng(6).standard_normal((3, 64)).astype(np.float32)
    a, b = np.array([5, 100, 2000]), np.array([11, 7, 300])
    once = oracle.rope(x, a + b)
    # rotate by a, then by b (the second call takes the rounded-to-float result,
    # so compare at float precision)
    twice = oracle.rope(oracle.rope(x, a).astype(np.float32), b)
    assert np.allclose(once, twice, atol=1e-5)


def test_cache_append_slots_and_bits():
    g = rng(7)
    B, s_q = 3, 2
    seqlens = np.array([1, 64, 130], np.int32)
    nblk = [(int(s) + 63) // 64 for s in seqlens]
    pool = sum(nblk) + 2
    perm = g.permutation(pool).astype(np.int32)
    table = np.full((B, max(nblk)), -1, np.int32)
    k = 0
    for b in range(B):
        table[b, :nblk[b]] = perm[k:k + nblk[b]]
        k += nblk[b]
    kv = g.standard_normal((pool, 64, 576)).astype(np.float32)
    new = g.standard_normal((B, s_q, 576)).astype(np.float32)
    out = oracle.cache_append(kv, new, table, seqlens, base=10000.0)
    touched = np.zeros((pool, 64), bool)
    for b in range(B):
        for s in range(s_q):
            t = int(seqlens[b]) - s_q + s
            if t < 0:
                continue
            blk, r = int(table[b, t // 64]), t % 64
            touched[blk, r] = True
            assert np.array_equal(out[blk, r, :512], new[b, s, :512].astype(np.float64))
            assert np.allclose(out[blk, r, 512:], oracle.rope(new[b, s, 512:][None], [t])[0], rtol=0, atol=0)
    # sequence 0 has one token: its s = 0 token (t = -1) is skipped
    assert touched.sum() == 5
    assert np.array_equal(out[~touched], kv[~touched].astype(np.float64))
