"""The float64 reblocking tree (oracle/reblock_f64.py) against the
fixed-order FP32 statement (oracle/reblock.py) under the margin rule.

The two share no arithmetic: the float64 tree uses ordinary dot products,
the FP32 statement its documented summation order.  They must agree on every
decision whose float64 margin exceeds the float32 error bound; where every
margin is that wide they give the same permutation.  The bounds themselves
are checked against the FP32 statement's values, and the check is shown to
catch misplaced tokens.

Source: "Sol-Attn and Spark for MiniMax-H3", section "Spark primitives"
(spark_reblock) and section "Spark inference integration" (power-of-two
fanout, cosine scoring on normalized FP16 vectors).
"""

import numpy as np
import pytest

from oracle import reblock as R
from oracle import reblock_f64 as F

DEPTHS = [F.ANY_ORDER, 8]  # any summation order; the FP32 statement's depth


def _bits(x):
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)


@pytest.mark.parametrize("depth", DEPTHS)
def test_unit_rows_within_their_bound(depth):
    # the FP32 statement's FP16 unit rows equal the float64 ones except at
    # elements the float64 side marks as possibly rounding the other way
    rng = np.random.default_rng(11)
    x = rng.standard_normal((4000, 128)) * np.exp(rng.uniform(-4, 4, (4000, 1)))
    xb = _bits(x)
    u32 = R.unit_fp16(xb).astype(np.float64)
    u64, dev, wild = F.units(xb, depth)
    assert not wild.any()
    diff = np.abs(u32 - u64)
    assert np.all((diff == 0) | (diff <= dev))
    # the window is (depth / 2 + 4) u either side of a midpoint, against an
    # FP16 spacing of at least 2^-11 relative: a small share of elements
    assert np.count_nonzero(dev) < (depth + 8) * 2.0 ** -12 * dev.size


@pytest.mark.parametrize("depth", DEPTHS)
def test_kappa_within_its_bound(depth):
    # kappa of the FP32 statement (its cosines of its FP16 rows) lies within
    # the float64 tree's bound of the float64 kappa
    rng = np.random.default_rng(12)
    T = 3000
    xb = _bits(rng.standard_normal((T, 128)))
    u32 = R.unit_fp16(xb)
    u64, dev, wild = F.units(xb, depth)
    tokens = list(range(T))
    for a, b in [(0, 1), (5, 2999), (17, 400)]:
        k32 = (R.cosines(u32, u32[a]) - R.cosines(u32, u32[b])).astype(np.float32).astype(np.float64)
        k64, B = F.kappa_and_bound(u64, dev, wild, tokens, a, b, depth)
        assert np.all(np.abs(k32 - k64) <= B)
        # tight enough to decide most boundaries (about 2 gamma * 0.64 typically)
        assert np.median(B) < (4e-5 if depth == F.ANY_ORDER else 4e-6)


@pytest.mark.parametrize("depth", DEPTHS)
@pytest.mark.parametrize("T,fanout", [(64 * 7 + 13, 2), (64 * 20 + 1, 8), (64 * 33 + 63, 16),
                                      (64 * 60, 8), (64 * 148 + 33, 8), (64 * 11 + 3, 4)])
def test_fp32_statement_agrees_under_the_margin_rule(T, fanout, depth):
    rng = np.random.default_rng(T + fanout)
    xb = _bits(rng.standard_normal((T, 128)))
    p32, _ = R.reblock_head(xb, fanout)
    p64, nodes = F.reblock_tree(xb, fanout, depth=depth)
    viol, cov = F.check_permutation(p32, p64, nodes, T)
    assert viol == []
    if depth == 8 and T <= 64 * 21:
        assert cov == 1.0


@pytest.mark.parametrize("fanout", [2, 4, 8, 16])
def test_wide_margins_give_the_same_permutation(fanout):
    # tokens on a planar arc, 0.3 degrees apart: every decision is far from
    # its bound, so the two statements must give one permutation
    rng = np.random.default_rng(200 + fanout)
    q, _ = np.linalg.qr(rng.standard_normal((128, 2)))
    n = 64 * 9
    ang = np.deg2rad(5.0 + 170.0 * rng.permutation(n) / n)
    r = np.exp(rng.uniform(np.log(0.1), np.log(10.0), n))
    x = r[:, None] * (np.cos(ang)[:, None] * q[:, 0] + np.sin(ang)[:, None] * q[:, 1])
    xb = _bits(np.concatenate([x, rng.standard_normal((21, 128))]))
    p32, _ = R.reblock_head(xb, fanout)
    for depth in DEPTHS:
        p64, nodes = F.reblock_tree(xb, fanout, depth=depth)
        viol, cov = F.check_permutation(p32, p64, nodes, xb.shape[0])
        assert viol == [] and cov == 1.0
        assert np.array_equal(p32, p64)


def _case():
    rng = np.random.default_rng(31)
    T = 64 * 20 + 5
    xb = _bits(rng.standard_normal((T, 128)))
    p64, nodes = F.reblock_tree(xb, 8, depth=8)
    return xb, T, p64, nodes


def test_the_check_catches_misplaced_tokens():
    xb, T, p64, nodes = _case()
    assert F.check_permutation(p64, p64, nodes, T) == ([], 1.0)
    # two tokens exchanged between leaf blocks (each block re-sorted)
    bad = p64.copy()
    bad[3], bad[64 * 7 + 9] = bad[64 * 7 + 9], bad[3]
    for b in (0, 7):
        bad[64 * b:64 * (b + 1)] = np.sort(bad[64 * b:64 * (b + 1)])
    viol, _ = F.check_permutation(bad, p64, nodes, T)
    assert any("outside child blocks" in v for v in viol)
    # whole blocks in another order
    blocks = p64[:64 * 20].reshape(20, 64)
    viol, _ = F.check_permutation(np.concatenate([blocks[::-1].ravel(), p64[64 * 20:]]), p64, nodes, T)
    assert viol
    # a block out of ascending order, a shuffled remainder, a duplicate
    bad = p64.copy()
    bad[[0, 1]] = bad[[1, 0]]
    assert any("ascending" in v for v in F.check_permutation(bad, p64, nodes, T)[0])
    bad = p64.copy()
    bad[-2:] = bad[-2:][::-1]
    assert any("remainder" in v for v in F.check_permutation(bad, p64, nodes, T)[0])
    bad = p64.copy()
    bad[5] = bad[6]
    assert F.check_permutation(bad, p64, nodes, T)[0] == ["not a permutation of [0, T)"]


def test_the_check_catches_a_different_tree():
    # the same tokens through a tree with another fanout, or with kappa's
    # sign flipped, fail the check against the fanout-8 float64 tree
    xb, T, p64, nodes = _case()
    p4, _ = R.reblock_head(xb, 4)
    assert F.check_permutation(p4, p64, nodes, T)[0]
    orig = R.cosines
    try:
        R.cosines = lambda xh, u: -orig(xh, u)
        flipped = R.reblock_head(xb, 8)[0]
    finally:
        R.cosines = orig
    assert not np.array_equal(flipped, p64)
    assert F.check_permutation(flipped, p64, nodes, T)[0]
