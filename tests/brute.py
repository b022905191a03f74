"""Independent brute-force formulations used to pin the oracle.

Nothing here calls the oracle's arithmetic.  Each function restates one step
in a different form that is easy to check by hand on tiny inputs:

* ``brute_topk``: exhaustive search over all K-subsets of the candidates for
  the largest exact score sum, ties resolved to the lexicographically
  smallest index tuple (which is "lower block index wins").
* ``token_mask``: the block lists expanded to a token-level boolean mask
  (the "kernel contract against the token-expanded mask" of the SD.Next
  attention-backends commit), with the row classification re-derived here.
* ``masked_dense_attention``: dense fp64 softmax attention with -inf outside
  the mask.
"""

from __future__ import annotations

import itertools
import math
from fractions import Fraction

import numpy as np


def brute_topk(scores_f32_row, cand, K):
    cand = sorted(int(c) for c in cand)
    k = min(K, len(cand))
    if k == 0:
        return []
    exact = {j: Fraction(float(scores_f32_row[j])) for j in cand}
    best_sum, best = None, None
    for sub in itertools.combinations(cand, k):  # tuples come out sorted
        s = sum(exact[j] for j in sub)
        if best is None or s > best_sum or (s == best_sum and sub < best):
            best_sum, best = s, sub
    return list(best)


def row_kind(t, T, Nv, tail_mode):
    """('sparse', block) or ('dense', None) for query row t."""
    nvk = Nv // 64
    if t < 64 * nvk:
        return "sparse", t // 64
    if tail_mode == "pad" and t < Nv:
        return "sparse", nvk
    return "dense", None


def token_mask(idx, cnt, T, Nv, tail_mode):
    """bool [H, T, T]: mask[h, t, u] is True when row t attends key u."""
    H = idx.shape[0]
    mask = np.zeros((H, T, T), dtype=bool)
    kblock = np.arange(T) // 64
    for h in range(H):
        for t in range(T):
            kind, i = row_kind(t, T, Nv, tail_mode)
            if kind == "dense":
                mask[h, t, :] = True
            else:
                blocks = idx[h, i, : cnt[h, i]]
                mask[h, t, :] = np.isin(kblock, blocks)
    return mask


def masked_dense_attention(q, k, v, bias, mask):
    """q, k, v fp64 [T, H, D]; bias fp64 [T]; mask bool [H, T, T] -> O [T, H, D]."""
    T, H, D = q.shape
    out = np.zeros((T, H, D))
    for h in range(H):
        logits = q[:, h, :] @ k[:, h, :].T / math.sqrt(D) + bias[None, :]
        logits = np.where(mask[h], logits, -np.inf)
        m = logits.max(axis=1, keepdims=True)
        p = np.exp(logits - m)
        out[:, h, :] = (p @ v[:, h, :]) / p.sum(axis=1, keepdims=True)
    return out
