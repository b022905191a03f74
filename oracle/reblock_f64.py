"""Spark's token reblocking (the landmark tree) in plain float64, with the
margin of every decision.

TEST INFRASTRUCTURE ONLY: imported by the tests, never by the CUDA path; it
shares no code with the CUDA library, nor with the FP32 statement in
oracle/reblock.py (each helper below is restated here on purpose).

Source: "Sol-Attn and Spark for MiniMax-H3" (Spark-H3 README), section "Spark
primitives" (spark_reblock: 64-token leaves, cosine distance, midpoint
landmarks, flat initial order, stable parent order, the T % 64 remainder
kept last) and section "Spark inference integration" (power-of-two fanout;
cosine scoring on normalized FP16 vectors).  The tree's steps are the same
reading as oracle/reblock.py states; only the arithmetic differs.

Arithmetic.  Unit vectors: x / ||x|| in float64, rounded once to FP16.
Every cosine is an ordinary float64 dot product (numpy), with no fixed
summation order and no lane structure.  kappa = cos(t, a) - cos(t, b) in
float64.

Margins.  A float32 implementation of the same steps whose sums of 128
terms pass each term through at most `depth` roundings (any order: depth
127; a four-term chain then a five-level tree: depth 8) can differ from this
one in three places, each bounded here (u = 2^-24, gamma_d = d u / (1 - d u)):
  * a unit-vector element whose exact value lies within the float32
    normalisation error ((depth / 2 + 4) u relative: the sum of squares, its
    square root and the division) of an FP16 rounding midpoint may round to
    the other FP16 neighbour;
  * a float32 dot product of 128 exact FP16 products is off by at most
    gamma_depth times the sum of |products|;
  * kappa's float32 subtraction rounds once more (u |kappa|).
A decision is *certain* when its float64 margin exceeds the sum of these
bounds of the values it compares: then every such float32 implementation
takes it the same way.  Node sizes depend only on T, so each node owns a
fixed range of blocks in the permutation, and the check in
`check_permutation` compares another implementation's permutation with this
tree node by node, wherever the decisions that fix a node's token set are
certain (in the spirit of the near-tie rule for block lists).
"""

from __future__ import annotations

import numpy as np

BLOCK = 64
HEAD_DIM = 128
U32 = 2.0 ** -24
ANY_ORDER = 127  # summation depth that covers every order of 128 terms


def gamma(depth: int) -> float:
    return depth * U32 / (1 - depth * U32)


def children_sizes(m: int, fanout: int) -> list:
    """Blocks per child of a node of m blocks: c = the largest power of two
    not above min(fanout, m) children, the first m mod c one block larger."""
    c = 1
    while 2 * c <= min(fanout, m):
        c *= 2
    return [m // c + (1 if i < m % c else 0) for i in range(c)]


def bf16_bits_to_f64(x_bits: np.ndarray) -> np.ndarray:
    return ((np.asarray(x_bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)).astype(np.float64)


def units(x_bits: np.ndarray, depth: int = ANY_ORDER):
    """FP16 unit rows (as float64) of BF16 rows [n, 128], and for each
    element the size of the possible float32 disagreement (the FP16
    neighbour gap where the exact value is that close to a rounding
    midpoint, else 0).  Rows with squares below float32's normal range are
    marked wholly uncertain (`wild`)."""
    x = bf16_bits_to_f64(x_bits)
    ss = np.sum(x * x, axis=-1)
    r = np.sqrt(ss)
    q = np.where(r[..., None] > 0, x / np.where(r > 0, r, 1.0)[..., None], 0.0)
    u16 = q.astype(np.float16)
    u = u16.astype(np.float64)
    # the other FP16 neighbour of q and the midpoint between the two
    other = np.where(u >= q, np.nextafter(u16, np.float16(-np.inf)), np.nextafter(u16, np.float16(np.inf)))
    other = other.astype(np.float64)
    mid = 0.5 * (u + other)
    gap = np.abs(other - u)
    amb = np.abs(q - mid) <= ((depth / 2 + 4) * U32 + 1e-14) * np.abs(q)
    dev = np.where(amb & (q != 0), gap, 0.0)
    tiny = (np.abs(x) > 0) & (np.abs(x) < 2.0 ** -62)
    wild = np.any(tiny, axis=-1)
    return u, dev, wild


def cos_and_bound(u: np.ndarray, dev: np.ndarray, wild: np.ndarray, rows, col, depth: int = ANY_ORDER):
    """cos(t, s) for rows t against one token s (float64) and the bound on a
    float32 implementation's disagreement with it."""
    ut, dt = u[rows], dev[rows]
    us, ds = u[col], dev[col]
    c = ut @ us
    perturb = dt @ np.abs(us) + np.abs(ut) @ ds + dt @ ds
    sabs = np.abs(ut) @ np.abs(us) + perturb
    b = gamma(depth) * sabs + perturb + 1e-12
    b = np.where(wild[rows] | wild[col], 4.0, b)
    return c, b


def kappa_and_bound(u, dev, wild, tokens, a, b, depth: int = ANY_ORDER):
    """kappa = cos(t, a) - cos(t, b) for the tokens (float64) and the bound
    on a float32 implementation's disagreement with it."""
    ca, ba = cos_and_bound(u, dev, wild, tokens, a, depth)
    cb, bb = cos_and_bound(u, dev, wild, tokens, b, depth)
    kappa = ca - cb
    return kappa, ba + bb + U32 * (np.abs(kappa) + ba + bb)


class Node:
    """One node of the tree: its block range, its tokens (ascending), and
    whether its own decisions (the landmark pair, the child boundaries) are
    certain; `child_tokens` / `certain` per child when it was split."""

    def __init__(self, b0, b1, tokens):
        self.b0, self.b1, self.tokens = b0, b1, tokens
        self.pair_certain = True
        self.children = []        # [(b0, b1, tokens, token_certain mask)]


def split(u, dev, wild, node: Node, fanout: int, L: int, depth: int):
    tokens = node.tokens
    n = len(tokens)
    sizes = children_sizes(n // BLOCK, fanout)
    Lc = min(L, n)
    land = [tokens[(j * n) // Lc] for j in range(Lc)]
    # farthest landmark pair: smallest cosine, ties to the lower (j, j')
    cs, bs = [], []
    for j in range(Lc):
        c, b = cos_and_bound(u, dev, wild, land, land[j], depth)
        cs.append(c)
        bs.append(b)
    best = None
    pairs = []
    for j in range(Lc):
        for jj in range(j + 1, Lc):
            pairs.append((cs[j][jj], bs[j][jj], j, jj))
            if best is None or cs[j][jj] < best[0]:
                best = (cs[j][jj], bs[j][jj], j, jj)
    for c, b, j, jj in pairs:
        if (j, jj) != (best[2], best[3]) and not (c - b > best[0] + best[1]):
            node.pair_certain = False
            break
    node.a, node.b = land[best[2]], land[best[3]]
    kappa, B = kappa_and_bound(u, dev, wild, tokens, node.a, node.b, depth)
    rank = np.lexsort((np.arange(n), kappa))   # by kappa, then position
    child_of = np.empty(n, dtype=np.int64)
    bounds = np.cumsum([0] + [BLOCK * m for m in sizes])
    for ci in range(len(sizes)):
        child_of[rank[bounds[ci]:bounds[ci + 1]]] = ci
    # token t is certain in child c = [K_c, K_{c+1}) of the ranking when at
    # most K_{c+1} - 1 others can rank before it and at least K_c must
    lo, hi = np.sort(kappa - B), np.sort(kappa + B)
    possible_before = np.searchsorted(lo, kappa + B, side="right") - 1
    certain_before = np.searchsorted(hi, kappa - B, side="left")
    K0 = bounds[child_of]
    K1 = bounds[child_of + 1]
    tok_certain = (possible_before <= K1 - 1) & (certain_before >= K0)
    if not node.pair_certain:
        tok_certain[:] = False
    b = node.b0
    tok = np.asarray(tokens)
    for ci, m in enumerate(sizes):
        sel = child_of == ci
        node.children.append((b, b + m, [int(t) for t in tok[sel]], tok_certain[sel]))
        b += m


def reblock_tree(x_bits: np.ndarray, fanout: int = 8, L: int = 32, depth: int = ANY_ORDER):
    """The float64 tree of one head's rows x_bits [T, 128] (BF16 bits).

    Returns (perm, nodes): perm[i] is the original token at new position i
    (the remainder last, in flat order); nodes lists every split node whose
    token set is certain, with its children and per-token certainty."""
    T = x_bits.shape[0]
    N = BLOCK * (T // BLOCK)
    u, dev, wild = units(x_bits, depth)
    leaves, nodes = [], []

    def rec(b0, b1, tokens, set_certain):
        if b1 - b0 == 1:
            leaves.append(tokens)
            return
        node = Node(b0, b1, tokens)
        split(u, dev, wild, node, fanout, L, depth)
        if set_certain:
            nodes.append(node)
        for cb0, cb1, ct, cert in node.children:
            rec(cb0, cb1, ct, set_certain and bool(np.all(cert)))

    if N:
        rec(0, N // BLOCK, list(range(N)), True)
    perm = np.array([t for leaf in leaves for t in leaf] + list(range(N, T)), dtype=np.int64)
    return perm, nodes


def check_permutation(perm_other: np.ndarray, perm: np.ndarray, nodes, T: int):
    """Compare another implementation's permutation of one head with the
    float64 tree under the margin rule.

    Always: perm_other is a permutation of [0, T), every block lists its
    tokens in ascending order (stable parent order from a flat root) and
    the remainder comes last in flat order.  For every node whose token set
    is certain: each token whose child is certain sits in that child's
    block range.  Returns (violations, certain_fraction): a list of
    messages (empty when the two agree) and the fraction of blocked tokens
    whose leaf block is certain."""
    viol = []
    N = BLOCK * (T // BLOCK)
    po = np.asarray(perm_other, dtype=np.int64)
    if po.shape != (T,) or not np.array_equal(np.sort(po), np.arange(T)):
        return ["not a permutation of [0, T)"], 0.0
    if not np.array_equal(po[N:], np.arange(N, T)):
        viol.append("remainder not last in flat order")
    blocks = po[:N].reshape(-1, BLOCK) if N else po[:0].reshape(0, BLOCK)
    if N and not np.all(np.diff(blocks, axis=1) > 0):
        viol.append("a block is not in ascending token order")
    inv = np.empty(T, dtype=np.int64)
    inv[po] = np.arange(T)
    blk = inv // BLOCK
    certain_tokens = 0
    for node in nodes:
        for cb0, cb1, ct, cert in node.children:
            ct = np.asarray(ct, dtype=np.int64)
            bad = cert & ((blk[ct] < cb0) | (blk[ct] >= cb1))
            if np.any(bad):
                viol.append(f"node blocks [{node.b0}, {node.b1}): token {int(ct[bad][0])} "
                            f"outside child blocks [{cb0}, {cb1})")
            if cb1 - cb0 == 1 and np.all(cert):
                certain_tokens += len(ct)
    if N == BLOCK:
        certain_tokens = BLOCK  # a single block is fixed by the invariants
    return viol, (certain_tokens / N if N else 1.0)
