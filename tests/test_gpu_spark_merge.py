"""GPU parity of Spark's merged attention (sparse_attn_spark_fwd) with the
fp64 oracle (oracle/spark.py: spark_forward / forward_merged).

Source: "Sol-Attn and Spark for MiniMax-H3", section "Spark inference
integration" (per-head anchor from all target-video queries, BF16; global
anchor K/V and log-mass summaries merged with exact attention).

The oracle takes its own lists, anchors and summaries.  Every output value
(row, head, dim) of the five workloads is compared, the oracle evaluated
head by head in a spawned process pool; rows whose GPU list differs from the
oracle's (near-tie rule) are left out, as in the exact path's tests.
Outputs must agree within the same max-abs 2e-2 / mean-abs 2e-3.  Anchors: each GPU value must lie between the BF16 roundings of the
exact mean +- its FP32 error bound (recursive sums of 64 rows per thread, 16
thread groups and the 1024-row chunks, then one division).
"""

import math
import os

import numpy as np
import pytest

import oracle as O
from tests import parity
from workloads import WORKLOADS, make_inputs, make_workload

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

U = 2.0 ** -24


@pytest.fixture(scope="module")
def pool():
    p = parity.oracle_pool()
    yield p
    p.close()
    p.join()


@pytest.fixture(scope="module")
def bsr():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from block_sparse_routed_gb300.build import LIB_PATH, build

    if not os.path.exists(LIB_PATH):
        build()
    import block_sparse_routed_gb300 as m

    m.load_library()
    return m


def to_dev(bits, T, H):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).reshape(1, T, H, 128).cuda()


def a256(x):
    return (x + 255) // 256 * 256


def run_spark(bsr, arrays, T, H, Nv, ratio, R, mode, exact_too=False):
    P = bsr.Params(T=T, H=H, video_tokens=Nv, topk_ratio=ratio, radius=R, tail_mode=mode)
    sz = bsr.sparse_attn_query(P)
    q, k, v = (to_dev(arrays[n], T, H) for n in "qkv")
    bias = None if arrays["bias"] is None else torch.from_numpy(arrays["bias"]).cuda()
    idx, cnt = bsr.sparse_attn_plan(P, q, k)
    from block_sparse_routed_gb300 import _native

    ws = torch.empty(_native.sparse_attn_spark_ws_bytes(P.to_c()), dtype=torch.uint8, device="cuda")
    o = bsr.sparse_attn_spark_fwd(P, q, k, v, idx, cnt, key_bias=bias, ws=ws)
    status = bsr.sparse_attn_last_device_status(ws)
    out = {"status": status, "idx": idx.cpu().numpy().reshape(H, sz.nq, sz.maxl),
           "cnt": cnt.cpu().numpy().reshape(H, sz.nq),
           "o": parity.bf16_tensor_to_f64(o.reshape(T, H, 128))}
    # anchors from the documented workspace layout
    off = 256 + a256(T * 4)
    wsb = ws.cpu().numpy()
    out["anchor"] = wsb[off:off + H * 256].view(np.uint16).reshape(H, 128)
    if exact_too:
        o2 = bsr.sparse_attn_fwd(P, q, k, v, idx, cnt, key_bias=bias)
        out["o_exact"] = parity.bf16_tensor_to_f64(o2.reshape(T, H, 128))
    torch.cuda.synchronize()
    return out, sz


def check_anchor(gpu_anchor_bits, q_bits, Nv):
    q = O.decode_bf16(q_bits[:Nv])
    exact = q.mean(axis=0)
    # recursive FP32 sums along 64 rows per thread, 16 thread groups, then
    # the chunks; one rounded division: |err| <= (64 + 16 + nch + 1) u mean|q|
    nch = (Nv + 1023) // 1024
    err = 2 * (64 + 16 + nch + 1) * U * np.abs(q).mean(axis=0)
    lo, hi = O.round_to_bf16(exact - err), O.round_to_bf16(exact + err)
    g = O.decode_bf16(gpu_anchor_bits)
    assert np.all((g >= lo) & (g <= hi))


def oracle_merged(arrays, sz, heads):
    ref = O.plan(arrays["q"], arrays["k"], sz)
    a = O.video_query_anchor(arrays["q"], sz.Nv)
    s = O.spark_reweight(a[:, heads], np.ascontiguousarray(arrays["k"][:, heads]),
                         np.ascontiguousarray(arrays["v"][:, heads]))
    H = sz.H
    ak = np.zeros((H, sz.nblk, 128))
    av = np.zeros((H, sz.nblk, 128))
    lm = np.zeros((H, sz.nblk))
    ak[heads], av[heads], lm[heads] = s["ak16"][0], s["av16"][0], s["lm"][0]
    o = O.forward_merged(arrays["q"], arrays["k"], arrays["v"], arrays["bias"], ref["idx"], ref["cnt"],
                         sz, ak, av, lm, heads=heads)
    return ref, a, o


@pytest.mark.parametrize("name", ["tiny", "8k", "h3", "32k", "64k"])
def test_merged_workloads(bsr, pool, name):
    w = WORKLOADS[name]
    arrays, prm = make_workload(name)
    gpu, _ = run_spark(bsr, arrays, w.T, w.H, w.video_tokens, w.topk_ratio, w.radius, w.tail_mode)
    assert gpu["status"] == 0
    sz = O.derive_sizes(w.T, w.H, w.video_tokens, w.topk_ratio, w.radius, w.tail_mode)
    ref = O.plan(arrays["q"], arrays["k"], sz)
    check_anchor(gpu["anchor"], arrays["q"], sz.Nv)
    same = parity.same_list_mask(gpu["idx"], gpu["cnt"], ref)
    o = parity.oracle_all_heads(pool, "merged", arrays, prm, ref["idx"], ref["cnt"])
    dmax, dmean, n = parity.compare_all(gpu["o"], o, same, sz)
    print(f"[parity] merged {name}: {n} values, max-abs {dmax:.3e}, mean-abs {dmean:.3e}")
    assert n >= 0.99 * sz.T * sz.H * 128
    assert dmax <= parity.OUT_MAX_ABS, dmax
    assert dmean <= parity.OUT_MEAN_ABS, dmean


def test_merged_with_every_block_exact_equals_the_exact_path(bsr):
    # ratio 1: no video block is skipped, the summary keys are all masked
    T, H, Nv = 64 * 12 + 21, 2, 64 * 12
    arrays = make_inputs(T=T, H=H, video_tokens=Nv, qk_kind="walk1d", seed=41)
    gpu, _ = run_spark(bsr, arrays, T, H, Nv, 1.0, 1, "dense", exact_too=True)
    assert np.array_equal(gpu["o"], gpu["o_exact"])


def test_merged_dense_rows_equal_the_exact_path(bsr):
    w = WORKLOADS["8k"]
    arrays, prm = make_workload("8k")
    gpu, sz = run_spark(bsr, arrays, w.T, w.H, w.video_tokens, w.topk_ratio, w.radius, w.tail_mode,
                        exact_too=True)
    r0 = sz.dense_row_start
    assert np.array_equal(gpu["o"][r0:], gpu["o_exact"][r0:])
    assert not np.array_equal(gpu["o"][:r0], gpu["o_exact"][:r0])


@pytest.mark.parametrize("T,Nv,mode", [(64 * 6 + 40, 64 * 5 + 20, "pad"), (64 * 70 + 3, 64 * 70, "dense")])
def test_merged_ragged(bsr, T, Nv, mode):
    H = 3
    arrays = make_inputs(T=T, H=H, video_tokens=Nv, qk_kind="walk1d", bias_kind="sink_normal", seed=T)
    gpu, _ = run_spark(bsr, arrays, T, H, Nv, 0.2, 1, mode)
    assert gpu["status"] == 0
    sz = O.derive_sizes(T, H, Nv, 0.2, 1, mode)
    ref, a, o = oracle_merged(arrays, sz, list(range(H)))
    same = parity.same_list_mask(gpu["idx"], gpu["cnt"], ref)
    assert same.all()
    d = np.abs(gpu["o"] - o)
    assert d.max() <= parity.OUT_MAX_ABS and d.mean() <= parity.OUT_MEAN_ABS


def test_merged_zero_bias_is_no_bias(bsr):
    # an all-zero key bias takes the no-bias path: the same output bit for bit
    # ("Add key bias to chunked Sol-Attn producers", "Contract")
    T, H, Nv = 64 * 20 + 30, 2, 64 * 18
    base = make_inputs(T=T, H=H, video_tokens=Nv, qk_kind="walk1d", seed=77)
    none, _ = run_spark(bsr, dict(base, bias=None), T, H, Nv, 0.25, 1, "dense")
    zero, _ = run_spark(bsr, dict(base, bias=np.zeros(T, np.float32)), T, H, Nv, 0.25, 1, "dense")
    assert none["status"] == 0 and zero["status"] == 0
    assert np.array_equal(none["o"], zero["o"])
