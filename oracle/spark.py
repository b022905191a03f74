"""Plain CPU fp64 statement of Spark's per-block virtual summaries.

TEST INFRASTRUCTURE ONLY: imported by the tests and by the benchmark's
CPU-baseline leg, never by the CUDA path; it shares no code with the CUDA
library.  Slow and obviously correct.

Source: "Sol-Attn and Spark for MiniMax-H3" (Spark-H3 README), section "Spark
primitives" (spark_reweight, the virtual summaries) and section "Spark
inference integration" (the default numerics of the reweight: BF16 stored
summaries, log-mass taken against the stored BF16 summary key).

For anchor a_p (one query representative of head h) and physical 64-token
block b of K/V, with u running over the real keys of the block only (a
partial final block has fewer than 64):

    s_u  = a_p . k_u / sqrt(128)                       (natural-log units)
    w_u  = exp(s_u) / sum_u' exp(s_u')                 (softmax over the block)
    ak   = sum_u w_u k_u,   av = sum_u w_u v_u         (stored as BF16)
    lm   = logsumexp_u(s_u) - a_p . ak / sqrt(128)     (FP32)

and by default the ak inside lm is the stored, BF16-rounded one.  With the
unrounded ak, lm is the Shannon entropy of w: logsumexp(s) - sum_u w_u s_u.
"""

from __future__ import annotations

import math

import numpy as np

from .oracle import BLOCK, HEAD_DIM, decode_bf16


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Nearest BF16 value (ties to even) of float64 values, as float64.

    Rounds the float64 value straight to 8 significant bits (no detour
    through float32, which could round twice).  Finite inputs only.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                      # x = m * 2^e, 0.5 <= |m| < 1
    scaled = np.ldexp(m, 8)                 # 8 significant bits above the point
    r = np.round(scaled)                    # numpy rounds halves to even
    out = np.ldexp(r, e - 8)
    # below the normal range BF16 has FP32's subnormal spacing 2^-133
    tiny = np.abs(x) < 2.0 ** -126
    out[tiny] = np.round(x[tiny] * 2.0 ** 133) * 2.0 ** -133
    return out


def block_ranges(T: int):
    """Physical 64-token blocks of a length-T sequence, the last one partial
    when T is not a multiple of 64 (its padding is excluded)."""
    return [range(b * BLOCK, min(T, (b + 1) * BLOCK)) for b in range((T + BLOCK - 1) // BLOCK)]


def spark_reweight(a_bits: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray, pre_round=False):
    """Virtual summaries of every (anchor, head, block).

    a_bits: BF16 bits [P, H, 128]; k_bits, v_bits: BF16 bits [T, H, 128].
    Returns dict with
      ak, av     float64 [P, H, nblk, 128]  (unrounded)
      ak16, av16 float64 [P, H, nblk, 128]  (their BF16 values, as stored)
      lm         float64 [P, H, nblk]       (log-mass against ak16, or against
                                             the unrounded ak if pre_round)
    """
    a = decode_bf16(a_bits)
    k = decode_bf16(k_bits)
    v = decode_bf16(v_bits)
    P, H, D = a.shape
    T = k.shape[0]
    assert D == HEAD_DIM and k.shape == (T, H, D) and v.shape == (T, H, D)
    blocks = block_ranges(T)
    nb = len(blocks)
    ak = np.zeros((P, H, nb, D))
    av = np.zeros((P, H, nb, D))
    lm = np.zeros((P, H, nb))
    scale = 1.0 / math.sqrt(D)
    for p in range(P):
        for h in range(H):
            for b, rows in enumerate(blocks):
                kb = k[rows.start:rows.stop, h, :]
                vb = v[rows.start:rows.stop, h, :]
                s = (kb @ a[p, h]) * scale
                m = s.max()
                e = np.exp(s - m)
                w = e / e.sum()
                ak[p, h, b] = w @ kb
                av[p, h, b] = w @ vb
                lse = m + math.log(e.sum())
                lm[p, h, b] = lse  # the key term is subtracted below
    ak16 = round_to_bf16(ak)
    av16 = round_to_bf16(av)
    key = ak if pre_round else ak16
    lm = lm - np.einsum("phbd,phd->phb", key, a) * scale
    return {"ak": ak, "av": av, "ak16": ak16, "av16": av16, "lm": lm}


def reweight_bytes(P: int, T: int, H: int) -> int:
    """Algorithmic HBM bytes of one call: K and V read once, anchors read,
    ak/av (BF16) and lm (FP32) written."""
    nb = (T + BLOCK - 1) // BLOCK
    return 2 * T * H * HEAD_DIM * 2 + P * H * HEAD_DIM * 2 + P * H * nb * (2 * HEAD_DIM * 2 + 4)


# ---------------------------------------------------------------- merged attention
# "Sol-Attn and Spark for MiniMax-H3", section "Spark inference integration":
# one global representative per head, formed by averaging all target-video
# queries and stored as BF16; global-anchor K/V and log-mass summaries merged
# with exact attention.  Read here as: every video key block that a sparse
# query block's list skips enters that block's softmax as one virtual key,
# the summary key ak, with logit q . ak / sqrt(128) + lm and value av.  For a
# query equal to the anchor this reproduces the block's exact contribution,
# since exp(a . ak / sqrt(128) + lm) = sum_u exp(a . k_u / sqrt(128)).

def bf16_bits(x: np.ndarray) -> np.ndarray:
    """BF16 bit patterns of float64 values that are BF16 values."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "not a BF16 value"
    return (u >> 16).astype(np.uint16)


def video_query_anchor(q_bits: np.ndarray, video_tokens: int) -> np.ndarray:
    """BF16 bits [1, H, 128]: per head the mean of the target-video query
    rows t < video_tokens, rounded to BF16."""
    q = decode_bf16(q_bits[:video_tokens])
    return bf16_bits(round_to_bf16(q.mean(axis=0)))[None]


def skipped_blocks(h: int, i: int, idx: np.ndarray, cnt: np.ndarray, nvk: int) -> np.ndarray:
    """Video key blocks j < nvk absent from the list of query block i, head h."""
    listed = set(int(b) for b in idx[h, i, : cnt[h, i]])
    return np.array([j for j in range(nvk) if j not in listed], dtype=np.int64)


def forward_merged(q_bits, k_bits, v_bits, bias, idx, cnt, sz, ak, av, lm, heads=None):
    """Exact attention over each list plus one virtual key per skipped video
    key block: O [T, len(heads), 128] fp64.

    ak, av: [H, nblk, 128] summaries (one anchor per head), lm: [H, nblk].
    Dense rows attend every key exactly and see no virtual key.
    """
    from .oracle import _softmax_attend, check_key_bias, query_block_rows, row_key_set

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
            sk = skipped_blocks(h, i, idx, cnt, sz.nvk)
            # virtual keys after the exact ones; the log-mass is an additive logit
            kk = np.concatenate([k[keys], ak[h, sk]])
            vv = np.concatenate([v[keys], av[h, sk]])
            bb = np.concatenate([b[keys], lm[h, sk]])
            out[rows, hn] = _softmax_attend(q[rows], kk, vv, bb, sz.D)
        rows = np.arange(sz.dense_row_start, sz.T)
        if rows.size:
            out[rows, hn] = _softmax_attend(q[rows], k, v, b, sz.D)
    return out


def spark_forward(q_bits, k_bits, v_bits, bias, sz, plan_out=None):
    """The whole merged path: routing lists, the per-head anchor (mean of the
    video queries), its virtual summaries (stored BF16 values) and the merged
    attention.  Returns dict(o, idx, cnt, a, ak16, av16, lm)."""
    from .oracle import plan

    ref = plan_out if plan_out is not None else plan(q_bits, k_bits, sz)
    a = video_query_anchor(q_bits, sz.Nv)
    s = spark_reweight(a, k_bits, v_bits)
    o = forward_merged(q_bits, k_bits, v_bits, bias, ref["idx"], ref["cnt"], sz,
                       s["ak16"][0], s["av16"][0], s["lm"][0])
    return {"o": o, "idx": ref["idx"], "cnt": ref["cnt"], "a": a, "ak16": s["ak16"][0],
            "av16": s["av16"][0], "lm": s["lm"][0]}
