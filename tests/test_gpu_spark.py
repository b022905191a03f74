"""Parity of the CUDA virtual summaries (sparse_attn_spark_reweight) with the
fp64 oracle (oracle/spark.py).

Source: "Sol-Attn and Spark for MiniMax-H3", section "Spark primitives"
(spark_reweight) and section "Spark inference integration" (BF16 stored
summaries; log-mass against the stored BF16 key).

Tolerances follow from the FP32 arithmetic of the kernel (u = 2^-24):
  * scores: a dot product summed in depth 9 (4 products per lane, then a
    5-level butterfly): |ds| <= g9 * sum_d |a_d k_d| / sqrt(128), g9 = 9u/(1-9u);
  * ak, av: weights carry <= 2 max|ds| + 2^-22 (ex2) relative error and the
    64-term sums g64; the FP32 result is then rounded to BF16, so GPU and
    oracle agree exactly unless the exact value lies within that error of a
    rounding midpoint, where they may differ by one BF16 step;
  * lm: logsumexp carries <= 3 max|ds| + 64u + 2^-22, the key term (a dot
    product with the stored BF16 key) g9 * sum_d |a_d ak_d| / sqrt(128); a
    block whose BF16 key differs by a step in dimension d shifts lm by
    |a_d| * step / sqrt(128).  Bounds are doubled for the library log and
    reciprocal.
"""

import math

import numpy as np
import pytest

import oracle as O
from workloads import make_anchors, make_inputs, make_reweight_workload

pytestmark = pytest.mark.gpu

U = 2.0 ** -24
G9 = 9 * U / (1 - 9 * U)
G64 = 64 * U / (1 - 64 * U)
EX2 = 2.0 ** -22


@pytest.fixture(scope="module")
def bsr():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_sparse_routed_gb300 as m

    m.load_library()
    return m


def _dev(bits):
    import torch

    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _f64(t):
    import torch

    return t.float().cpu().numpy().astype(np.float64) if t.dtype == torch.bfloat16 else t.cpu().numpy().astype(np.float64)


def run(bsr, a, k, v):
    P, H, _ = a.shape
    T = k.shape[0]
    ak, av, lm = bsr.spark_reweight(_dev(a).reshape(1, P, H, 128), _dev(k).reshape(1, T, H, 128),
                                    _dev(v).reshape(1, T, H, 128))
    import torch

    torch.cuda.synchronize()
    return _f64(ak)[0], _f64(av)[0], _f64(lm)[0]


def bf16_step(x):  # noqa: D401
    """Distance from |x| to the next BF16 value above it (one rounding step)."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def check(a_bits, k_bits, v_bits, gpu):
    ak_g, av_g, lm_g = gpu
    ref = O.spark_reweight(a_bits, k_bits, v_bits)
    a = O.decode_bf16(a_bits)
    k = O.decode_bf16(k_bits)
    P, H, _ = a.shape
    blocks = O.block_ranges(k.shape[0])
    # per (p, h, b): max_u sum_d |a_d k_ud| / sqrt(128)
    sabs = np.zeros((P, H, len(blocks)))
    for b, rows in enumerate(blocks):
        sabs[:, :, b] = np.einsum("phd,uhd->phu", np.abs(a), np.abs(k[rows.start:rows.stop])).max(axis=2)
    ds = G9 * sabs / math.sqrt(128.0)
    v = O.decode_bf16(v_bits)
    for name, g16, r16, r, x in (("ak", ak_g, ref["ak16"], ref["ak"], k), ("av", av_g, ref["av16"], ref["av"], v)):
        # the kernel's FP32 value is within `err` of the exact one, and BF16
        # rounding is monotone: its BF16 value lies between the roundings of
        # the two ends of that interval
        xmax = np.zeros((H, len(blocks)))
        for b, rows in enumerate(blocks):
            xmax[:, b] = np.abs(x[rows.start:rows.stop]).max(axis=(0, 2))
        err = 2 * (2 * ds + EX2 + G64) * xmax[None]
        err = np.broadcast_to(err[..., None], r.shape)
        lo, hi = O.round_to_bf16(r - err), O.round_to_bf16(r + err)
        ok = (g16 >= lo) & (g16 <= hi)
        assert np.all(ok), (name, np.argwhere(~ok)[:5])
        assert (g16 != r16).mean() < 0.02, (name, (g16 != r16).mean())
    # lm
    key = np.einsum("phbd,phd->phb", np.abs(ref["ak16"]), np.abs(a)) / math.sqrt(128.0)
    tol = 2 * (3 * ds + 64 * U + EX2 + G9 * key)
    same = np.all(ak_g == ref["ak16"], axis=-1)
    shift = np.einsum("phbd,phd->phb", bf16_step(ref["ak"]), np.abs(a)) / math.sqrt(128.0)
    tol = np.where(same, tol, tol + shift)
    d = np.abs(lm_g - ref["lm"])
    assert np.all(d <= tol), (d.max(), d[same].max() if same.any() else None)
    return ref


@pytest.mark.parametrize("name", ["reweight_h3", "reweight_h3_p4", "reweight_32k", "reweight_8k_sharp"])
def test_reweight_workloads(bsr, name):
    arrays, prm = make_reweight_workload(name)
    gpu = run(bsr, arrays["a"], arrays["k"], arrays["v"])
    check(arrays["a"], arrays["k"], arrays["v"], gpu)


@pytest.mark.parametrize("T,H,P", [(1, 1, 1), (5, 2, 3), (64, 1, 2), (65, 3, 1), (64 * 7 + 33, 5, 2)])
def test_reweight_ragged_sizes(bsr, T, H, P):
    arrays = make_inputs(T=T, H=H, video_tokens=min(T, 64) if T >= 64 else T, qk_kind="iid", seed=T + H)
    a = make_anchors(P, H, 1.5, seed=T * 7 + P)
    gpu = run(bsr, a, arrays["k"], arrays["v"])
    ref = check(a, arrays["k"], arrays["v"], gpu)
    assert gpu[2].shape == (P, H, (T + 63) // 64) and ref["lm"].shape == gpu[2].shape


def test_zero_anchor_gives_block_means_and_log_length(bsr):
    T, H = 64 * 3 + 9, 2
    arrays = make_inputs(T=T, H=H, video_tokens=64, qk_kind="iid", seed=21)
    a = np.zeros((1, H, 128), dtype=np.uint16)
    ak, av, lm = run(bsr, a, arrays["k"], arrays["v"])
    lens = [64, 64, 64, 9]
    for b, n in enumerate(lens):
        assert np.allclose(lm[0, :, b], math.log(n), rtol=0, atol=4 * 64 * U + 4 * EX2)
    check(a, arrays["k"], arrays["v"], (ak, av, lm))


def test_sharp_anchor_selects_one_key(bsr):
    # one key aligned with a large anchor: weights one-hot, lm ~ 0
    T, H = 64, 1
    arrays = make_inputs(T=T, H=H, video_tokens=64, qk_kind="iid", seed=22)
    k = arrays["k"].copy()
    k[40, 0] = np.full(128, 0x4080, dtype=np.uint16)   # 4.0 in every dimension
    a = np.full((1, H, 128), 0x4280, dtype=np.uint16)   # 64.0
    ak, av, lm = run(bsr, a, k, arrays["v"])
    assert np.array_equal(ak[0, 0, 0], O.decode_bf16(k[40, 0]))
    assert np.array_equal(av[0, 0, 0], O.decode_bf16(arrays["v"][40, 0]))
    assert abs(lm[0, 0, 0]) < 1e-3


def test_reweight_rejects_bad_arguments(bsr):
    import torch

    k = torch.zeros((1, 70, 2, 128), dtype=torch.bfloat16, device="cuda")
    a = torch.zeros((1, 1, 2, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        bsr.spark_reweight(a, k, k[:, :69].contiguous())
    with pytest.raises(ValueError):
        bsr.spark_reweight(a.float(), k, k)
