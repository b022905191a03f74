"""Plain CPU fp64 statement of Top-K block-sparse routed attention.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the package smoke check
and by the benchmark's CPU-baseline / reference leg, never by the CUDA path.
It is slow and obviously correct, not fast.  It shares no code with the CUDA
library; the seeded inputs come from ``workloads`` and are BF16 bit patterns,
decoded here exactly to float64.

Sources (web pages, cited by title and section):

* [SOL-H3]  "Sol-Attn and Spark for MiniMax-H3" (Spark-H3 README).
* [BIAS]    "Add key bias to chunked Sol-Attn producers" (comfy-kitchen PR).
* [SDNEXT]  SD.Next attention-backends commit (sparse stage, router, flex).

The method, step by step (each function below names the step it states):

1. Q and K are cut into physical 64-token blocks; the target-video prefix is
   sparse and the context suffix is exact ([SOL-H3] "H3 pipeline
   integration").
2. The route centroid of a block is the mean of its Q (or K) rows ([SOL-H3]
   "Spark inference integration": native mean Top-K routing; [SOL-H3] "H3
   pipeline integration": pad mode preserves the block routing centroid).
3. The route score is Qmean . Kmean / sqrt(128), per head.
4. Per video query block, the Top-K key blocks by score, K = ceil(ratio x
   video key blocks); ties go to the lower block index.  The selection runs on
   FP32 score values ([SOL-H3] "Spark inference integration": exact FP32 radix
   boundary selection).
5. Forced exact blocks are added outside the budget: the self block and its
   +-radius neighbours ([SOL-H3] "H3 pipeline integration",
   sol_exact_block_radius) and every context sink block, which never enters
   the candidate set ([BIAS] "Tests and source audit": sinks are inserted
   directly into the exact list and excluded from the routed candidates).
6. Each video query row attends exactly, with softmax, over the union of its
   block list.  An optional per-key additive logit bias (natural-log units)
   is allowed only on sink keys ([BIAS] "Summary", "Contract").
7. Context query rows, and in tail_mode "dense" the rows of a video block cut
   by the video/context boundary, attend densely to every key ([SOL-H3] "H3
   pipeline integration").  In tail_mode "pad" that block runs sparse; its
   centroid is the mean of its real video rows.

Readings of points the pages leave open are stated at the function that takes
them.
"""

from __future__ import annotations

import math
from dataclasses import dataclass
from fractions import Fraction

import numpy as np

BLOCK = 64  # physical block length, [SOL-H3] "H3 pipeline integration"
HEAD_DIM = 128  # [SOL-H3] "Install": contiguous BF16 [batch, tokens, heads, 128]


@dataclass(frozen=True)
class Sizes:
    T: int  # packed tokens
    H: int  # heads
    D: int  # head dimension (128)
    Nv: int  # target-video tokens, the prefix [0, Nv)
    nvk: int  # full video blocks, floor(Nv / 64): the routed key blocks
    tail: int  # video tokens of the block cut by the boundary, Nv - 64 nvk
    nblk: int  # physical key blocks, ceil(T / 64)
    nq: int  # sparse query blocks: nvk, plus the tail block in pad mode
    K: int  # Top-K budget
    R: int  # forced local radius
    tail_mode: str  # "dense" or "pad"
    nsink: int  # sink blocks, nblk - nvk
    maxl: int  # block-list width
    dense_row_start: int  # first query row evaluated densely


def topk_count(topk_ratio: float, nvk: int) -> int:
    """K = ceil(topk_ratio x video key blocks), clamped to nvk.

    Reading: the product is taken on the decimal value of the ratio as
    written (so 0.1 x 30 gives 3, not the 4 that the binary float 0.1 would
    give).  [SOL-H3] "Spark inference integration": ratio 0.1 Top-K.
    """
    r = Fraction(repr(float(topk_ratio)))
    return min(nvk, math.ceil(r * nvk))


def derive_sizes(T, H, video_tokens, topk_ratio, radius, tail_mode, D=HEAD_DIM) -> Sizes:
    """Block bookkeeping of the packed layout ([SOL-H3] "H3 pipeline integration").

    Raises ValueError where the layout is outside the method: D != 128,
    video prefix shorter than one block or longer than T, ratio outside
    (0, 1], negative radius, or pad mode without enough context slots to
    complete the tail block ("The packed context suffix must contain enough
    slots to complete the 64-row block").
    """
    if D != HEAD_DIM:
        raise ValueError("head dimension must be 128")
    if H < 1 or T < 1:
        raise ValueError("empty shape")
    if not (BLOCK <= video_tokens <= T):
        raise ValueError("need 64 <= video_tokens <= T")
    if not (0.0 < topk_ratio <= 1.0):
        raise ValueError("topk_ratio must lie in (0, 1]")
    if radius < 0:
        raise ValueError("radius must be >= 0")
    if tail_mode not in ("dense", "pad"):
        raise ValueError("tail_mode must be 'dense' or 'pad'")
    nvk = video_tokens // BLOCK
    tail = video_tokens - BLOCK * nvk
    nblk = -(-T // BLOCK)
    pad_block = tail_mode == "pad" and tail > 0
    if pad_block and T < BLOCK * (nvk + 1):
        raise ValueError("pad mode needs context slots to complete the tail block")
    nq = nvk + (1 if pad_block else 0)
    K = topk_count(topk_ratio, nvk)
    nsink = nblk - nvk
    maxl = min(nvk, 2 * radius + 1 + K) + nsink
    dense_row_start = BLOCK * nvk if tail_mode == "dense" else video_tokens
    return Sizes(T, H, D, video_tokens, nvk, tail, nblk, nq, K, radius, tail_mode, nsink,
                 maxl, dense_row_start)


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """BF16 bit patterns (uint16) -> exact float64 values."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def query_block_rows(i: int, sz: Sizes) -> range:
    """Real query rows of sparse query block i.

    Full video blocks own 64 rows; the pad-mode tail block owns only its real
    video rows [64 nvk, Nv).  Its non-video slots are filled with the mean Q of
    those rows ([SOL-H3] "H3 pipeline integration"), which leaves the centroid
    unchanged, and their outputs are not kept: context rows are produced by
    the dense path.
    """
    if i < sz.nvk:
        return range(BLOCK * i, BLOCK * i + BLOCK)
    assert i == sz.nvk and sz.nq == sz.nvk + 1
    return range(BLOCK * sz.nvk, sz.Nv)


def centroids(q_bits: np.ndarray, k_bits: np.ndarray, sz: Sizes):
    """Step 2: route centroids, the mean of each block's rows (fp64).

    Qc[h, i] = (1/n_i) sum_{t in rows(i)} Q[t, h, :] for the nq query blocks;
    Kc[h, j] the same over K for the nvk video key blocks.  Only full video
    blocks are routed keys; every later block is a sink (reading: the block
    cut by the boundary holds context tokens, so it is treated as context,
    matching sink_start = video_tokens rounded down to a block).
    """
    H, D = sz.H, sz.D
    Qc = np.zeros((H, sz.nq, D))
    Kc = np.zeros((H, sz.nvk, D))
    for i in range(sz.nq):
        rows = query_block_rows(i, sz)
        Qc[:, i, :] = decode_bf16(q_bits[rows.start:rows.stop]).sum(axis=0) / len(rows)
    for j in range(sz.nvk):
        Kc[:, j, :] = decode_bf16(k_bits[BLOCK * j:BLOCK * j + BLOCK]).sum(axis=0) / BLOCK
    return Qc, Kc


def route_scores(Qc: np.ndarray, Kc: np.ndarray) -> np.ndarray:
    """Step 3: s[h, i, j] = Qc[h, i] . Kc[h, j] / sqrt(D), fp64."""
    D = Qc.shape[-1]
    return np.matmul(Qc, Kc.transpose(0, 2, 1)) / math.sqrt(D)


def local_video_blocks(i: int, R: int, nvk: int) -> list:
    """Step 5: forced local blocks that are video blocks, |j - i| <= R, 0 <= j < nvk.

    Radius 0 forces only the self block, radius 1 the self block and its two
    neighbours ([SOL-H3] "H3 pipeline integration").  Reading: neighbours past
    either end are clipped, never wrapped; a neighbour at or after nvk is a
    sink and already exact.
    """
    return [j for j in range(i - R, i + R + 1) if 0 <= j < nvk]


def select_topk(scores_f32_row: np.ndarray, cand, K: int) -> list:
    """Step 4: the min(K, |cand|) best candidates by (score desc, index asc).

    Reading: forced local blocks are not candidates; the budget K is spent on
    the other video blocks ("These blocks are added outside the Top-K
    budget", [SOL-H3] "H3 pipeline integration").  The comparison is on FP32
    values.
    """
    cand = np.asarray(sorted(cand), dtype=np.int64)
    if cand.size == 0:
        return []
    vals = scores_f32_row[cand].astype(np.float64)
    order = np.lexsort((cand, -vals))  # primary key -score, then index
    return [int(j) for j in cand[order[: min(K, cand.size)]]]


def block_lists(scores: np.ndarray, sz: Sizes):
    """Steps 4-5: per (head, query block) the sorted union of forced local
    video blocks, Top-K routed blocks and all sink blocks.

    Returns idx int32 [H, nq, maxl] padded with -1 and cnt int32 [H, nq].
    """
    s32 = scores.astype(np.float32)
    idx = np.full((sz.H, sz.nq, sz.maxl), -1, dtype=np.int32)
    cnt = np.zeros((sz.H, sz.nq), dtype=np.int32)
    sinks = list(range(sz.nvk, sz.nblk))
    for h in range(sz.H):
        for i in range(sz.nq):
            lv = local_video_blocks(i, sz.R, sz.nvk)
            cand = sorted(set(range(sz.nvk)) - set(lv))
            top = select_topk(s32[h, i], cand, sz.K)
            lst = sorted(set(lv) | set(top) | set(sinks))
            idx[h, i, : len(lst)] = lst
            cnt[h, i] = len(lst)
    return idx, cnt


def plan(q_bits: np.ndarray, k_bits: np.ndarray, sz: Sizes) -> dict:
    """Steps 2-5: centroids, route scores and block lists."""
    Qc, Kc = centroids(q_bits, k_bits, sz)
    s = route_scores(Qc, Kc)
    idx, cnt = block_lists(s, sz)
    return {"Qc": Qc, "Kc": Kc, "scores": s, "idx": idx, "cnt": cnt}


def check_key_bias(bias, sz: Sizes):
    """The key-bias contract ([BIAS] "Contract", "Tests and source audit").

    The carrier is float32 with exactly B*T elements, in natural-log units.
    Biased key blocks must be sink-routed: a nonzero bias on any key of a
    routed video block (u < 64 nvk) is rejected.  Reading: +inf and NaN are
    rejected too; -inf is allowed and removes that key.  Returns the bias as
    float64 [T] (zeros when absent).
    """
    if bias is None:
        return np.zeros(sz.T)
    b = np.asarray(bias)
    if b.dtype != np.float32 or b.size != sz.T:
        raise ValueError("key_bias must be float32 with exactly B*T elements")
    b = b.reshape(-1).astype(np.float64)
    if np.any(np.isnan(b)) or np.any(b == np.inf):
        raise ValueError("key_bias must not hold NaN or +inf")
    if np.any(b[: BLOCK * sz.nvk] != 0.0):
        raise ValueError("key_bias is allowed only on sink keys")
    return b


def row_key_set(t: int, h: int, idx: np.ndarray, cnt: np.ndarray, sz: Sizes) -> np.ndarray:
    """Keys U(t) that query row t attends in head h (sorted token indices)."""
    if t < BLOCK * sz.nvk or (sz.nq > sz.nvk and t < sz.Nv):
        i = min(t // BLOCK, sz.nq - 1)
        blocks = idx[h, i, : cnt[h, i]]
        return np.concatenate([np.arange(BLOCK * b, min(BLOCK * b + BLOCK, sz.T)) for b in blocks])
    return np.arange(sz.T)


def _softmax_attend(q_rows, k_keys, v_keys, b_keys, D):
    """Steps 6-7 for rows sharing one key set: exact softmax attention.

    l[t, u] = q_t . k_u / sqrt(D) + bias_u ;  O[t] = sum_u e^{l - m} v_u / sum_u e^{l - m}
    """
    logits = q_rows @ k_keys.T / math.sqrt(D) + b_keys[None, :]
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    return (p @ v_keys) / p.sum(axis=1, keepdims=True)


def forward(q_bits, k_bits, v_bits, bias, idx, cnt, sz: Sizes, heads=None) -> np.ndarray:
    """Steps 6-7 for every row: O [T, len(heads), D] fp64."""
    b = check_key_bias(bias, sz)
    heads = list(range(sz.H)) if heads is None else list(heads)
    out = np.zeros((sz.T, len(heads), sz.D))
    for hn, h in enumerate(heads):
        q = decode_bf16(q_bits[:, h, :])
        k = decode_bf16(k_bits[:, h, :])
        v = decode_bf16(v_bits[:, h, :])
        for i in range(sz.nq):
            rows = np.arange(query_block_rows(i, sz).start, query_block_rows(i, sz).stop)
            keys = row_key_set(int(rows[0]), h, idx, cnt, sz)
            out[rows, hn] = _softmax_attend(q[rows], k[keys], v[keys], b[keys], sz.D)
        rows = np.arange(sz.dense_row_start, sz.T)
        if rows.size:
            out[rows, hn] = _softmax_attend(q[rows], k, v, b, sz.D)
    return out


def forward_rows(q_bits, k_bits, v_bits, bias, idx, cnt, sz: Sizes, rows, heads) -> np.ndarray:
    """Steps 6-7 for selected (row, head) pairs: O [len(rows), len(heads), D]."""
    b = check_key_bias(bias, sz)
    rows = [int(t) for t in rows]
    out = np.zeros((len(rows), len(heads), sz.D))
    for hn, h in enumerate(heads):
        for rn, t in enumerate(rows):
            keys = row_key_set(t, h, idx, cnt, sz)
            kk = decode_bf16(k_bits[keys, h, :])
            vv = decode_bf16(v_bits[keys, h, :])
            qq = decode_bf16(q_bits[t:t + 1, h, :])
            out[rn, hn] = _softmax_attend(qq, kk, vv, b[keys], sz.D)[0]
    return out


def kept_keys_per_row(idx: np.ndarray, cnt: np.ndarray, sz: Sizes) -> np.ndarray:
    """|U(t)| for every real query row: int64 [H, T]."""
    out = np.zeros((sz.H, sz.T), dtype=np.int64)
    for h in range(sz.H):
        for i in range(sz.nq):
            blocks = idx[h, i, : cnt[h, i]]
            nkeys = sum(min(BLOCK, sz.T - BLOCK * int(b)) for b in blocks)
            r = query_block_rows(i, sz)
            out[h, r.start:r.stop] = nkeys
        out[h, sz.dense_row_start:] = sz.T
    return out


def kept_flops(idx: np.ndarray, cnt: np.ndarray, sz: Sizes) -> int:
    """Kept-block attention work: 4 x D per (real query row, kept key), summed
    over heads (QK^T and PV, one multiply-add each)."""
    return int(kept_keys_per_row(idx, cnt, sz).sum()) * 4 * sz.D


def dense_score_bytes(T: int, H: int) -> int:
    """Bytes of an FP32 score matrix over every (query, key) pair of every
    head: what an eager dense call materialises ([SDNEXT] flex_attention
    paragraph: about 20 GB at 9505 tokens x 56 heads)."""
    return T * T * H * 4
