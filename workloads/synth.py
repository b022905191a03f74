"""Synthetic packed video-diffusion sequences.

The shapes follow the packed layout of "Sol-Attn and Spark for MiniMax-H3",
section "H3 pipeline integration": a target-video prefix of `video_tokens`
tokens followed by a context suffix, contiguous BF16 [1, T, H, 128].  The H3
sizes (9505 tokens, 56 heads) are the ones quoted in the SD.Next attention
backend commit (eager flex_attention paragraph).  No dataset exists for these
activations, so the value distributions are synthetic:

* ``iid``: Q, K, V i.i.d. N(0, 1).
* ``walk1d``: per head, a 128-dim Gaussian random walk over block index
  (c[0] = 0, c[b] = c[b-1] + 0.3 N(0, I)) through video and context blocks;
  Q[t] = c[block(t)] + 0.5 N(0, I) and K[t] likewise with independent noise;
  V ~ N(0, 1).
* ``walk3d``: video block b maps to (f, y, x) in raster order over a
  frames x height x width block grid; c = Wf[f] + Wy[y] + Wx[x] with three
  independent per-axis walks (first element 0, step 0.3).  Blocks after the
  last full video block continue a 1-D walk of step 0.3 from it.

Key bias kinds: ``none`` (no tensor), ``zero`` (all-zero float32 [T]) and
``sink_normal`` (0.5 N(0, 1) on keys at or after the video boundary, 0 on
video keys).  "N(0, s)" is read as standard deviation s.

All draws come from one numpy PCG64 stream per workload, in a fixed order, and
are rounded once to BF16 (round to nearest even).  Arrays are returned as BF16
bit patterns (uint16) in [T, H, 128] order.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

D_HEAD = 128
BLOCK = 64


@dataclass(frozen=True)
class Workload:
    name: str
    H: int
    T: int
    video_tokens: int
    topk_ratio: float
    radius: int
    tail_mode: str  # "dense" or "pad"
    qk_kind: str  # "iid", "walk1d" or "walk3d"
    bias_kind: str  # "none", "zero" or "sink_normal"
    seed: int
    grid: tuple = field(default=())  # (frames, height, width) for walk3d


WORKLOADS = {
    # 16 video blocks + 2 context blocks, i.i.d. inputs; small enough for the
    # CPU oracle to evaluate every output row in seconds.
    "tiny": Workload("tiny", 2, 1152, 1024, 0.25, 0, "dense", "iid", "none", 0),
    # 128 video blocks + 512 context tokens, all-zero key bias.
    "8k": Workload("8k", 24, 8704, 8192, 0.1, 1, "dense", "walk1d", "zero", 1),
    # MiniMax-H3 shape: 9240 video tokens (144 blocks + 24-token tail, dense
    # tail) + 265 context tokens, 56 heads.
    "h3": Workload("h3", 56, 9505, 9240, 0.1, 1, "dense", "walk1d", "none", 2),
    # 512 video blocks + 1024 context tokens, biased sinks.
    "32k": Workload("32k", 40, 33792, 32768, 0.1, 1, "dense", "walk1d", "sink_normal", 3),
    # 1024 video blocks + 24-token tail (pad tail) + 2048 context tokens,
    # 3-D clustered over a 16 x 8 x 8 block grid, biased sinks.
    "64k": Workload(
        "64k", 24, 67608, 65560, 0.05, 1, "pad", "walk3d", "sink_normal", 4, (16, 8, 8)
    ),
}


def bf16_round_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to BF16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def _walk(rng: np.random.Generator, n: int, H: int, step: float) -> np.ndarray:
    """[H, n, D] Gaussian random walk starting at 0."""
    inc = rng.standard_normal((H, n, D_HEAD), dtype=np.float32) * np.float32(step)
    inc[:, 0, :] = 0.0
    return np.cumsum(inc, axis=1, dtype=np.float32)


def _block_centres(rng, kind, H, T, video_tokens, grid):
    nblk = -(-T // BLOCK)
    if kind == "walk1d":
        return _walk(rng, nblk, H, 0.3)
    if kind == "walk3d":
        f, y, x = grid
        nvid = f * y * x
        nvk = video_tokens // BLOCK
        if nvk != nvid:
            raise ValueError("walk3d grid must cover the full video blocks exactly")
        wf = _walk(rng, f, H, 0.3)
        wy = _walk(rng, y, H, 0.3)
        wx = _walk(rng, x, H, 0.3)
        b = np.arange(nvid)
        cf, cy, cx = b // (y * x), (b // x) % y, b % x
        vid = wf[:, cf] + wy[:, cy] + wx[:, cx]
        rest = nblk - nvid
        if rest > 0:
            inc = rng.standard_normal((H, rest, D_HEAD), dtype=np.float32) * np.float32(0.3)
            tail = vid[:, -1:, :] + np.cumsum(inc, axis=1, dtype=np.float32)
            return np.concatenate([vid, tail], axis=1)
        return vid
    raise ValueError(kind)


def _noisy_tokens(rng, centres, T, H, sigma, chunk=4096):
    """[T, H, D] BF16 bits of centre(block(t)) + sigma N(0, I)."""
    out = np.empty((T, H, D_HEAD), dtype=np.uint16)
    ct = np.ascontiguousarray(centres.transpose(1, 0, 2))  # [nblk, H, D]
    for t0 in range(0, T, chunk):
        t1 = min(T, t0 + chunk)
        x = rng.standard_normal((t1 - t0, H, D_HEAD), dtype=np.float32) * np.float32(sigma)
        if centres is not None:
            x += ct[np.arange(t0, t1) // BLOCK]
        out[t0:t1] = bf16_round_bits(x)
    return out


def _normal_tokens(rng, T, H, chunk=4096):
    out = np.empty((T, H, D_HEAD), dtype=np.uint16)
    for t0 in range(0, T, chunk):
        t1 = min(T, t0 + chunk)
        out[t0:t1] = bf16_round_bits(rng.standard_normal((t1 - t0, H, D_HEAD), dtype=np.float32))
    return out


def make_inputs(
    *,
    T: int,
    H: int,
    video_tokens: int,
    qk_kind: str = "iid",
    bias_kind: str = "none",
    seed: int = 0,
    grid: tuple = (),
):
    """Return dict(q, k, v: uint16 BF16 bits [T, H, 128]; bias: float32 [T] or None)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    if qk_kind == "iid":
        q = _normal_tokens(rng, T, H)
        k = _normal_tokens(rng, T, H)
    else:
        c = _block_centres(rng, qk_kind, H, T, video_tokens, grid)
        q = _noisy_tokens(rng, c, T, H, 0.5)
        k = _noisy_tokens(rng, c, T, H, 0.5)
    v = _normal_tokens(rng, T, H)
    if bias_kind == "none":
        bias = None
    elif bias_kind == "zero":
        bias = np.zeros(T, dtype=np.float32)
    elif bias_kind == "sink_normal":
        bias = np.zeros(T, dtype=np.float32)
        n = T - video_tokens
        bias[video_tokens:] = rng.standard_normal(n, dtype=np.float32) * np.float32(0.5)
    else:
        raise ValueError(bias_kind)
    return {"q": q, "k": k, "v": v, "bias": bias}


def make_workload(name: str):
    """Inputs and parameters of one named workload."""
    w = WORKLOADS[name]
    arrays = make_inputs(
        T=w.T,
        H=w.H,
        video_tokens=w.video_tokens,
        qk_kind=w.qk_kind,
        bias_kind=w.bias_kind,
        seed=w.seed,
        grid=w.grid,
    )
    params = dict(
        T=w.T,
        H=w.H,
        video_tokens=w.video_tokens,
        topk_ratio=w.topk_ratio,
        radius=w.radius,
        tail_mode=w.tail_mode,
        bias_kind=w.bias_kind,
    )
    return arrays, params


# Virtual-summary (spark_reweight) workloads: the K/V of an attention workload
# plus P anchors per head.  The anchors stand in for query representatives
# (the page's default is one per head); they are drawn N(0, scale^2) per
# dimension and rounded to BF16, from their own PCG64 stream.
REWEIGHT_WORKLOADS = {
    # name: (attention workload for K/V, anchors per head, anchor scale, seed)
    "reweight_h3": ("h3", 1, 1.0, 11),
    "reweight_h3_p4": ("h3", 4, 1.0, 12),
    "reweight_32k": ("32k", 1, 1.0, 13),
    "reweight_8k_sharp": ("8k", 2, 4.0, 14),
}


def make_anchors(P: int, H: int, scale: float, seed: int) -> np.ndarray:
    """BF16 bits [P, H, 128] of N(0, scale^2) anchors."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return bf16_round_bits(rng.standard_normal((P, H, D_HEAD), dtype=np.float32) * np.float32(scale))


def make_reweight_workload(name: str):
    """(k, v, a) BF16 bits and the sizes of one named reweight workload."""
    base, P, scale, seed = REWEIGHT_WORKLOADS[name]
    arrays, prm = make_workload(base)
    a = make_anchors(P, prm["H"], scale, seed)
    return {"k": arrays["k"], "v": arrays["v"], "a": a}, dict(T=prm["T"], H=prm["H"], P=P, base=base)
