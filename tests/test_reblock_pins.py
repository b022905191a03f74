"""Pins of the reblocking oracles (the fixed-order FP32 statement in
oracle/reblock.py and the float64 tree in oracle/reblock_f64.py) to facts
that do not come from either oracle: hand-worked splits of orthogonal token groups (child
order, the farthest-pair tie rule, stable parent order), the closed form of
tokens on a planar arc (every split is by angle, so the blocks are the runs
of 64 of the angle order), landmark positions (decoy tokens off the landmark
grid never span a split), the power-of-two child counts, and the
permutation's invariants.

Source: "Sol-Attn and Spark for MiniMax-H3", section "Spark primitives"
(spark_reblock) and section "Spark inference integration" (fanout with
power-of-two scheduling, cosine scoring on normalized FP16 vectors).
"""

import math

import numpy as np
import pytest

from oracle import reblock as R
from oracle import reblock_f64 as F

IMPLS = ["fp32", "fp64"]


def _perm(impl, bits, fanout):
    """The permutation of one head by the FP32 statement or the float64 tree."""
    if impl == "fp32":
        return R.reblock_head(bits, fanout)[0]
    return F.reblock_tree(bits, fanout)[0]


def _bits(x):
    """Round FP32 values to BF16 (nearest even) and return the bit patterns."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)


def _decode(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _groups(ng, T):
    """Token group g (rows [64 g, 64 g + 64)) points along axis g; the rest
    along the last axis."""
    x = np.zeros((T, 128), dtype=np.float32)
    for g in range(ng):
        x[64 * g:64 * (g + 1), g] = 1.0
    x[64 * ng:, 127] = 1.0
    return _bits(x)


@pytest.mark.parametrize("child_blocks", [R.child_blocks, F.children_sizes], ids=IMPLS)
def test_child_counts_are_powers_of_two_up_to_the_fanout(child_blocks):
    assert child_blocks(148, 8) == [19, 19, 19, 19, 18, 18, 18, 18]
    assert child_blocks(19, 8) == [3, 3, 3, 2, 2, 2, 2, 2]
    assert child_blocks(3, 8) == [2, 1]
    assert child_blocks(5, 4) == [2, 1, 1, 1]
    assert child_blocks(7, 16) == [2, 2, 2, 1]
    assert child_blocks(20, 16) == [2, 2, 2, 2] + [1] * 12
    assert child_blocks(2, 2) == [1, 1]
    for m in range(2, 300):
        for f in (2, 4, 8, 16):
            s = child_blocks(m, f)
            c = len(s)
            assert c & (c - 1) == 0 and c <= min(f, m) < 2 * c
            assert sum(s) == m and max(s) - min(s) <= 1 and s == sorted(s, reverse=True)


def test_landmarks_sit_on_the_even_grid():
    assert R.landmark_positions(128) == list(range(0, 128, 4))
    assert R.landmark_positions(256) == list(range(0, 256, 8))
    assert R.landmark_positions(64 * 3) == list(range(0, 192, 6))
    assert R.landmark_positions(10, 32) == list(range(10))


@pytest.mark.parametrize("impl", IMPLS)
def test_two_orthogonal_groups_hand_worked(impl):
    # Tokens 0-63 along e0, 64-127 along e1, 5 remainder tokens.  Landmarks
    # are positions 0, 4, ..., 124; every cross pair has cosine 0 (the
    # minimum), the first one is landmarks (0, 16): a = token 0 (e0),
    # b = token 64 (e1).  kappa = cos(t, a) - cos(t, b) is -1 on the e1 group,
    # +1 on the e0 group, so the e1 group is child 0.
    T = 133
    x = _groups(2, T)
    for fanout in (2, 8):
        perm = _perm(impl, x, fanout)
        assert perm.tolist() == list(range(64, 128)) + list(range(64)) + list(range(128, 133))


@pytest.mark.parametrize("impl", IMPLS)
def test_four_orthogonal_groups_hand_worked(impl):
    # Landmarks every 8 tokens: 0-7 in group 0, 8-15 group 1, ...  The first
    # pair with cosine 0 is (0, 8): a = group 0, b = group 1.  kappa: group 1
    # -1, groups 2 and 3 0 (ranked by position), group 0 +1.
    x = _groups(4, 256)
    perm = _perm(impl, x, 4)
    assert perm.tolist() == list(range(64, 128)) + list(range(128, 256)) + list(range(64))
    # with fanout 2 the root splits 2 + 2 blocks: child 0 = groups 1 and 2,
    # child 1 = groups 3 and 0 in parent order (0 then 3).  Child 0 (256
    # -> 128 tokens, landmarks every 4): pair (0, 16) = (group 1, group 2),
    # so group 2 comes first; child 1: pair (group 0, group 3), group 3 first.
    perm = _perm(impl, x, 2)
    assert perm.tolist() == (list(range(128, 192)) + list(range(64, 128))
                             + list(range(192, 256)) + list(range(64)))


def _plane(rng):
    q, _ = np.linalg.qr(rng.standard_normal((128, 2)))
    return q[:, 0], q[:, 1]


def _arc_tokens(rng, n, lo_deg, hi_deg, rem=0):
    """n tokens at evenly spaced angles in [lo, hi) of a random plane, in a
    shuffled order, with random norms; then rem remainder tokens."""
    u1, u2 = _plane(rng)
    ang = np.deg2rad(lo_deg + (hi_deg - lo_deg) * np.arange(n) / n)
    ang = ang[rng.permutation(n)]
    r = np.exp(rng.uniform(np.log(0.05), np.log(20.0), n))
    x = r[:, None] * (np.cos(ang)[:, None] * u1 + np.sin(ang)[:, None] * u2)
    x = np.concatenate([x, rng.standard_normal((rem, 128))])
    bits = _bits(x)
    xd = _decode(bits)
    # the angle each rounded token actually has in the plane
    theta = np.arctan2(xd @ u2, xd @ u1)
    return bits, theta


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("fanout", [2, 4, 8, 16])
def test_planar_arc_blocks_are_runs_of_the_angle_order(fanout, impl):
    # On an arc shorter than 180 degrees the farthest landmarks are the
    # arc's extremes among the landmarks and kappa is monotone in the angle,
    # in every node: each block is 64 tokens consecutive in angle, and inside
    # a block the tokens stay in index order (stable parent order).
    rng = np.random.default_rng(100 + fanout)
    n = 512
    bits, theta = _arc_tokens(rng, n, 5.0, 175.0, rem=7)
    perm = _perm(impl, bits, fanout)
    want = {tuple(sorted(np.argsort(theta[:n])[64 * b:64 * (b + 1)].tolist())) for b in range(n // 64)}
    got = [perm[64 * b:64 * (b + 1)].tolist() for b in range(n // 64)]
    assert {tuple(g) for g in got} == want
    for g in got:
        assert g == sorted(g)
    assert perm[n:].tolist() == list(range(n, n + 7))


@pytest.mark.parametrize("impl", IMPLS)
def test_decoys_off_the_landmark_grid_do_not_span_the_split(impl):
    # 256 tokens, fanout 4: one split of the root into 4 leaves.  254 tokens
    # sit on an evenly spaced grid from 0 to 90 degrees with the two ends at
    # landmark positions 0 and 248 (landmarks are every 8th position), so
    # the farthest landmarks are the ends: a = 0 degrees, b = 90 degrees and
    # kappa = cos(theta - theta_a) - cos(theta - theta_b).  Two decoys at
    # positions 25 and 167 (off the grid) sit at 179 and -89 degrees: were
    # either a landmark, the farthest pair would hold a decoy and the split
    # would turn.
    rng = np.random.default_rng(7)
    u1, u2 = _plane(rng)
    n = 256
    ang = np.empty(n)
    grid_ang = np.deg2rad(90.0 * np.arange(254) / 253)
    rest = np.setdiff1d(np.arange(n), [0, 248, 25, 167])
    ang[0], ang[248] = grid_ang[0], grid_ang[-1]
    ang[rest] = grid_ang[1:-1][rng.permutation(252)]
    ang[25], ang[167] = np.deg2rad(179.0), np.deg2rad(-89.0)
    r = np.exp(rng.uniform(np.log(0.5), np.log(4.0), n))
    bits = _bits(r[:, None] * (np.cos(ang)[:, None] * u1 + np.sin(ang)[:, None] * u2))
    xd = _decode(bits)
    theta = np.arctan2(xd @ u2, xd @ u1)
    kappa = np.cos(theta - theta[0]) - np.cos(theta - theta[248])
    order = np.lexsort((np.arange(n), kappa))
    perm = _perm(impl, bits, 4)
    for b in range(4):
        assert perm[64 * b:64 * (b + 1)].tolist() == sorted(order[64 * b:64 * (b + 1)].tolist())
    assert 25 in perm[:64] and 167 in perm[192:256]


@pytest.mark.parametrize("T,fanout", [(64 * 7 + 13, 2), (64 * 9, 4), (64 * 20 + 1, 8), (64 * 33 + 63, 16), (40, 8), (64, 8)])
def test_permutation_invariants(T, fanout):
    rng = np.random.default_rng(T)
    x = _bits(rng.standard_normal((T, 2, 128)))
    out = R.spark_reblock(x, fanout)
    N = 64 * (T // 64)
    for h in range(2):
        p, iv = out["perm"][h], out["inv"][h]
        assert sorted(p.tolist()) == list(range(T))
        assert np.array_equal(iv[p], np.arange(T)) and np.array_equal(p[iv], np.arange(T))
        assert sorted(p[:N].tolist()) == list(range(N))
        assert p[N:].tolist() == list(range(N, T))
        for blk in out["blocks"][h]:
            assert blk.tolist() == sorted(blk.tolist())  # stable parent order
    assert out["blocks"].shape == (2, N // 64, 64) and out["excluded"].shape == (2, T - N)


@pytest.mark.parametrize("impl", IMPLS)
def test_scale_and_degenerate_rows(impl):
    # a positive scale per token changes nothing (cosine distance); identical
    # rows make every kappa 0, so every split keeps the flat order
    rng = np.random.default_rng(3)
    T = 64 * 6 + 5
    x = rng.standard_normal((T, 128)).astype(np.float32)
    # powers of two keep the BF16 rounding of every row's direction exact
    s = (2.0 ** rng.integers(-6, 7, T)).astype(np.float32)
    p0 = _perm(impl, _bits(x), 8)
    p1 = _perm(impl, _bits(x * s[:, None]), 8)
    assert np.array_equal(p0, p1)
    same = np.tile(_bits(rng.standard_normal(128))[None], (T, 1))
    p2 = _perm(impl, same, 8)
    assert p2.tolist() == list(range(T))
    zero = np.zeros((T, 128), dtype=np.uint16)
    p3 = _perm(impl, zero, 4)
    assert p3.tolist() == list(range(T))


def test_fold_order_and_fp16_units():
    # the fixed summation order, checked against an explicit loop, and the
    # unit rows against a float64 normalisation within FP16 rounding
    rng = np.random.default_rng(5)
    p = rng.standard_normal((3, 128)).astype(np.float32)
    for r in range(3):
        lanes = []
        for l in range(32):
            s = np.float32(0.0)
            s = np.float32(p[r, 4 * l] + p[r, 4 * l + 1])
            s = np.float32(s + p[r, 4 * l + 2])
            s = np.float32(s + p[r, 4 * l + 3])
            lanes.append(s)
        for off in (16, 8, 4, 2, 1):
            lanes = [np.float32(lanes[l] + lanes[l ^ off]) for l in range(32)]
        assert len(set(float(v) for v in lanes)) == 1
        assert R._fold32(p[r]) == lanes[0]
    xb = _bits(rng.standard_normal((50, 128)) * 3)
    xd = _decode(xb)
    u = R.unit_fp16(xb)
    ref = xd / np.linalg.norm(xd, axis=1, keepdims=True)
    assert np.max(np.abs(u - ref)) <= 2.0 ** -11
    assert np.allclose(np.linalg.norm(u, axis=1), 1.0, atol=2e-3)
    assert np.array_equal(u.astype(np.float16).astype(np.float32), u)


def test_tree_depth_used_for_launch_counts_matches_the_recursion():
    # bench.py counts 3 launches per tree level; its depth must be the depth
    # of the recursion the oracle runs (not monotone in m: fanout 8 splits 8
    # blocks in one level, 7 blocks in two)
    import bench

    def depth(m, f):
        return 0 if m == 1 else 1 + max(depth(s, f) for s in R.child_blocks(m, f))

    for f in (2, 4, 8, 16):
        for m in range(1, 400):
            assert bench.reblock_depth(m, f) == depth(m, f), (m, f)
    assert bench.reblock_depth(148, 8) == 4  # the H3 keys: 148 blocks
