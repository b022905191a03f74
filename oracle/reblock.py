"""Plain CPU statement of Spark's token reblocking (the landmark tree).

TEST INFRASTRUCTURE ONLY: imported by the tests and by the benchmark's
CPU-baseline / reference leg, never by the CUDA path; it shares no code with
the CUDA library.  Slow and obviously correct.

Source: "Sol-Attn and Spark for MiniMax-H3" (Spark-H3 README), section "Spark
primitives" (spark_reblock: the permutation, its inverse, the [T // 64, 64]
block indices and the T % 64 excluded remainder; defaults of 64-token leaves,
cosine distance, eight children, 32 midpoint landmarks, flat initial order,
stable parent order), section "Spark inference integration" (fanout 16 with
power-of-two scheduling in the H3 installer; cosine scoring on normalized
FP16 vectors) and section "H3 pipeline integration" (Q and K reordered
independently have no shared locality).

The pages name the tree's ingredients but not its steps.  The reading taken
here, for one head's sample matrix x [T, 128]:

1. N = 64 floor(T / 64) tokens are blocked; the remainder, the last T % 64
   tokens of the flat (raster) order, is excluded and kept at the end of the
   permutation in its own order.
2. Every token becomes an FP16 unit vector (cosine scoring on normalized
   FP16 values); a zero row stays zero.
3. The root node holds tokens [0, N) in flat order.  A node of m > 1 blocks
   of 64 splits into c children, c the largest power of two not above
   min(fanout, m) (power-of-two scheduling); child i takes
   floor(m / c) + [i < m mod c] blocks, so every leaf holds 64 tokens.
4. Landmarks: the L = 32 tokens at positions floor(j n / L), j < L, of the
   node's current order (n tokens).  The two landmarks farthest apart in
   cosine distance (the smallest cosine; ties to the lower landmark pair
   (j, j')) span the split: a = landmark j, b = landmark j'.
5. Each token of the node gets kappa = cos(t, a) - cos(t, b), so tokens near
   b come first.  The node's tokens are ranked by (kappa, position) and the
   first 64 m_0 go to child 0, the next 64 m_1 to child 1, and so on.
6. Inside a child the tokens keep the node's order (stable parent order);
   children follow one another in child order.  Leaves (m = 1) are blocks.

Precision.  The CUDA path takes these decisions in FP32 from FP16 unit
vectors, and so does this file, in the same order of operations, so the
integer result is bit-exact: a dot product of 128 values is summed as 32
partial sums of four consecutive products (left to right), then folded by
a butterfly over offsets 16, 8, 4, 2, 1.  Products of two FP16 values, and
squares of BF16 values, are exact in FP32.
"""

from __future__ import annotations

import numpy as np

BLOCK = 64
HEAD_DIM = 128
LANES = 32


def _fold32(p: np.ndarray) -> np.ndarray:
    """FP32 sum over the last axis (128 products) in the order stated above."""
    p = np.asarray(p, dtype=np.float32).reshape(p.shape[:-1] + (LANES, 4))
    s = ((p[..., 0] + p[..., 1]) + p[..., 2]) + p[..., 3]
    lane = np.arange(LANES)
    for off in (16, 8, 4, 2, 1):
        s = (s + s[..., lane ^ off]).astype(np.float32)
    return s[..., 0]


def unit_fp16(x_bits: np.ndarray) -> np.ndarray:
    """FP16 unit vectors [..., 128] (as float32) of BF16 rows given as bits.

    ss = sum of squares (FP32, the fixed order), r = sqrt(ss) rounded to
    FP32, x / r rounded to FP32 and then to FP16; r = 0 gives a zero row.
    """
    x = (np.asarray(x_bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    ss = _fold32(x * x)
    r = np.sqrt(ss).astype(np.float32)
    safe = np.where(r > 0, r, np.float32(1.0)).astype(np.float32)
    y = (x / safe[..., None]).astype(np.float32)
    y = np.where((r > 0)[..., None], y, np.float32(0.0))
    return y.astype(np.float16).astype(np.float32)


def cosines(xh: np.ndarray, u: np.ndarray) -> np.ndarray:
    """cos(t, u) for every row t of xh [n, 128] against one unit row u."""
    return _fold32(xh * u[None, :].astype(np.float32))


def child_blocks(m: int, fanout: int) -> list:
    """Blocks per child of a node of m blocks (power-of-two scheduling)."""
    c = 1
    while c * 2 <= min(fanout, m):
        c *= 2
    return [m // c + (1 if i < m % c else 0) for i in range(c)]


def landmark_positions(n: int, L: int = 32) -> list:
    """Positions floor(j n / L), j < L, in the node's current order."""
    L = min(L, n)
    return [(j * n) // L for j in range(L)]


def farthest_pair(xh_land: np.ndarray):
    """(j, j') with the smallest cosine among landmark rows, j < j'; ties to
    the lower pair in (j, j') order."""
    best = None
    L = xh_land.shape[0]
    for j in range(L):
        c = cosines(xh_land, xh_land[j])
        for jj in range(j + 1, L):
            if best is None or c[jj] < best[0]:
                best = (c[jj], j, jj)
    return best[1], best[2]


def split_node(xh: np.ndarray, order: list, fanout: int, L: int = 32) -> list:
    """The children (lists of token ids, each in parent order) of one node."""
    n = len(order)
    sizes = child_blocks(n // BLOCK, fanout)
    pos = landmark_positions(n, L)
    rows = xh[np.asarray(order)]
    j, jj = farthest_pair(rows[pos])
    a, b = rows[pos[j]], rows[pos[jj]]
    kappa = (cosines(rows, a) - cosines(rows, b)).astype(np.float32)
    kappa = kappa + np.float32(0.0)  # -0 and +0 are one value
    ranked = sorted(range(n), key=lambda i: (float(kappa[i]), i))
    child_of = np.empty(n, dtype=np.int64)
    start = 0
    for ci, mb in enumerate(sizes):
        for r in ranked[start:start + BLOCK * mb]:
            child_of[r] = ci
        start += BLOCK * mb
    return [[order[i] for i in range(n) if child_of[i] == ci] for ci in range(len(sizes))]


def reblock_head(x_bits: np.ndarray, fanout: int = 8, L: int = 32):
    """Permutation and inverse [T] of one head's rows x_bits [T, 128] (BF16 bits).

    perm[i] is the original token at new position i; inv[perm[i]] = i.
    """
    T = x_bits.shape[0]
    N = BLOCK * (T // BLOCK)
    xh = unit_fp16(x_bits)
    leaves = []

    def rec(order):
        if len(order) == BLOCK:
            leaves.append(order)
            return
        for ch in split_node(xh, order, fanout, L):
            rec(ch)

    if N:
        rec(list(range(N)))
    perm = np.array([t for leaf in leaves for t in leaf] + list(range(N, T)), dtype=np.int64)
    inv = np.empty(T, dtype=np.int64)
    inv[perm] = np.arange(T)
    return perm, inv


def spark_reblock(x_bits: np.ndarray, fanout: int = 8, L: int = 32):
    """All heads of x_bits [T, H, 128]: perm, inv [H, T]; block_indices
    [H, T // 64, 64]; excluded [H, T % 64]."""
    T, H, D = x_bits.shape
    assert D == HEAD_DIM
    perm = np.empty((H, T), dtype=np.int64)
    inv = np.empty((H, T), dtype=np.int64)
    for h in range(H):
        perm[h], inv[h] = reblock_head(x_bits[:, h, :], fanout, L)
    N = BLOCK * (T // BLOCK)
    return {"perm": perm, "inv": inv, "blocks": perm[:, :N].reshape(H, N // BLOCK, BLOCK),
            "excluded": perm[:, N:]}


def reblock_bytes(T: int, H: int) -> int:
    """Algorithmic HBM bytes of one call: the samples read once (BF16) and the
    permutation and its inverse written (int32)."""
    return T * H * HEAD_DIM * 2 + 2 * T * H * 4
