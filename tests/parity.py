"""Comparison helpers for GPU-vs-oracle parity (test side only).

Block lists: bit-exact, except where the oracle's route scores put a block
inside the near-tie band of the K-th selected score (FP32 on the GPU vs fp64
in the oracle can order near-equal scores differently).  Band:
  |s - s_K| <= 1e-5 max(|s|, |s_K|) + 1e-7 |Qc| |Kc| / sqrt(128).
Outputs: max |O_gpu - O_oracle| <= 2e-2 and mean <= 2e-3 on BF16 outputs.
"""

from __future__ import annotations

import math

import numpy as np

OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 2e-3


def compare_lists(idx_gpu, cnt_gpu, ref, sz):
    """Returns (n_exact, n_tie, bad) over (head, query block); bad lists the
    (h, i, reason) pairs that violate the rule."""
    idx_o, cnt_o, s = ref["idx"], ref["cnt"], ref["scores"]
    qn = np.linalg.norm(ref["Qc"], axis=-1)  # [H, nq]
    kn = np.linalg.norm(ref["Kc"], axis=-1)  # [H, nvk]
    n_exact = n_tie = 0
    bad = []
    H, nq = cnt_o.shape
    idx_gpu = idx_gpu.reshape(H, nq, -1)
    cnt_gpu = cnt_gpu.reshape(H, nq)
    for h in range(H):
        for i in range(nq):
            a = idx_gpu[h, i]
            b = idx_o[h, i]
            if cnt_gpu[h, i] == cnt_o[h, i] and np.array_equal(a, b):
                n_exact += 1
                continue
            if cnt_gpu[h, i] != cnt_o[h, i]:
                bad.append((h, i, "count"))
                continue
            la = a[: cnt_gpu[h, i]]
            if (a[cnt_gpu[h, i]:] != -1).any() or (np.diff(la) <= 0).any():
                bad.append((h, i, "layout"))
                continue
            diff = set(la.tolist()) ^ set(b[: cnt_o[h, i]].tolist())
            lo, hi = max(0, i - sz.R), min(sz.nvk - 1, i + sz.R)
            chosen = [j for j in b[: cnt_o[h, i]] if j < sz.nvk and not (lo <= j <= hi)]
            if not chosen:
                bad.append((h, i, "no candidates"))
                continue
            sK = min(s[h, i, j] for j in chosen)
            ok = True
            for j in diff:
                if j >= sz.nvk or lo <= j <= hi:
                    ok = False
                    break
                band = 1e-5 * max(abs(s[h, i, j]), abs(sK)) + 1e-7 * qn[h, i] * kn[h, j] / math.sqrt(128)
                if abs(s[h, i, j] - sK) > band:
                    ok = False
                    break
            if ok:
                n_tie += 1
            else:
                bad.append((h, i, f"outside tie band: {sorted(diff)}"))
    return n_exact, n_tie, bad


def same_list_mask(idx_gpu, cnt_gpu, ref):
    """bool [H, nq]: True where the GPU list equals the oracle's exactly."""
    H, nq = ref["cnt"].shape
    a = idx_gpu.reshape(H, nq, -1)
    return (a == ref["idx"]).all(axis=-1) & (cnt_gpu.reshape(H, nq) == ref["cnt"])


def bf16_tensor_to_f64(t):
    """torch bf16 tensor -> float64 numpy (exact)."""
    import torch

    return t.detach().to(torch.float64).cpu().numpy()


def output_errors(o_gpu, o_ref):
    d = np.abs(o_gpu - o_ref)
    return float(d.max()), float(d.mean())


# ---------------------------------------------------------------- oracle outputs, every head
def _oracle_head(args):
    """One head of the oracle's output (runs in a spawned worker)."""
    kind, qh, kh, vh, bias, idx_h, cnt_h, prm = args
    import oracle as O

    sz = O.derive_sizes(prm["T"], 1, prm["video_tokens"], prm["topk_ratio"], prm["radius"], prm["tail_mode"])
    if kind == "exact":
        return O.forward(qh, kh, vh, bias, idx_h, cnt_h, sz)[:, 0]
    a = O.video_query_anchor(qh, sz.Nv)
    s = O.spark_reweight(a, kh, vh)
    return O.forward_merged(qh, kh, vh, bias, idx_h, cnt_h, sz, s["ak16"][0], s["av16"][0], s["lm"][0])[:, 0]


def _reblock_margin_head(args):
    """The margin-rule check of one head's permutation against the float64
    reblocking tree (runs in a spawned worker): (violations, coverage)."""
    bits_h, perm_h, fanout, L, depth = args
    from oracle import reblock_f64 as F

    p64, nodes = F.reblock_tree(bits_h, fanout, L, depth)
    return F.check_permutation(perm_h, p64, nodes, bits_h.shape[0])


def reblock_margin_all(pool, x_bits, perm, fanout, L, depth, heads=None):
    """Margin-rule checks of perm [H, T] against the float64 tree of every
    (or the listed) head of x_bits [T, H, 128]: a list of (head, violations,
    coverage)."""
    heads = list(range(x_bits.shape[1])) if heads is None else list(heads)
    tasks = [(np.ascontiguousarray(x_bits[:, h, :]), np.asarray(perm[h]), fanout, L, depth) for h in heads]
    return [(h, v, c) for h, (v, c) in zip(heads, pool.map(_reblock_margin_head, tasks, chunksize=1))]


def oracle_pool(max_workers=16):
    """A spawned process pool for the oracle (safe after CUDA is initialised),
    one BLAS thread per worker."""
    import multiprocessing as mp
    import os

    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ.setdefault(var, "1")
    n = max(1, min(max_workers, len(os.sched_getaffinity(0))))
    return mp.get_context("spawn").Pool(n)


def oracle_all_heads(pool, kind, arrays, prm, idx, cnt):
    """The oracle's output for every head, O [T, H, 128] fp64, with the
    oracle's own lists; kind is "exact" (oracle.forward) or "merged"
    (oracle.spark: anchor, summaries, forward_merged)."""
    H = idx.shape[0]
    tasks = [(kind, np.ascontiguousarray(arrays["q"][:, [h]]), np.ascontiguousarray(arrays["k"][:, [h]]),
              np.ascontiguousarray(arrays["v"][:, [h]]), arrays["bias"], idx[[h]], cnt[[h]], prm)
             for h in range(H)]
    outs = pool.map(_oracle_head, tasks, chunksize=1)
    return np.stack(outs, axis=1)


def compare_all(o_gpu, o_ref, same, sz):
    """max and mean |O_gpu - O_oracle| over every (row, head, dim) except the
    rows of query blocks whose GPU list differs from the oracle's (near-tie
    rule); also the number of values compared."""
    import oracle as O

    keep = np.ones(o_gpu.shape[:2], dtype=bool)
    for h in range(same.shape[0]):
        for i in range(same.shape[1]):
            if not same[h, i]:
                r = O.oracle.query_block_rows(i, sz)
                keep[r.start:r.stop, h] = False
    d = np.abs(o_gpu - o_ref)[keep]
    return float(d.max()), float(d.mean()), int(d.size)
