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
