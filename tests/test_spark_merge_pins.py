"""Pins of the merged Spark attention oracle (oracle/spark.py,
forward_merged / spark_forward): skipped video key blocks enter the softmax
as one virtual key each (summary key, logit + log-mass, summary value).

Source: "Sol-Attn and Spark for MiniMax-H3", section "Spark inference
integration" (one global representative per head from all target-video
queries; global-anchor K/V and log-mass summaries merged with exact
attention; the log-mass replaces the ordinary log(block length) mass).
"""

import math

import numpy as np

import oracle as O
from workloads import make_inputs


def _bits(x):
    return O.bf16_bits(np.asarray(x, dtype=np.float64))


def _dense(q, k, v, rows, h):
    z = q[rows, h] @ k[:, h].T / math.sqrt(128.0)
    z = z - z.max(axis=1, keepdims=True)
    p = np.exp(z)
    return (p @ v[:, h]) / p.sum(axis=1, keepdims=True)


def _sizes(T, H, Nv, r, R, mode="dense"):
    return O.derive_sizes(T, H, Nv, r, R, mode)


def test_all_blocks_exact_means_no_virtual_keys():
    arrays = make_inputs(T=64 * 6 + 20, H=2, video_tokens=64 * 6, qk_kind="walk1d", seed=31)
    sz = _sizes(64 * 6 + 20, 2, 64 * 6, 1.0, 1)
    r = O.spark_forward(arrays["q"], arrays["k"], arrays["v"], None, sz)
    for h in range(2):
        for i in range(sz.nq):
            assert O.skipped_blocks(h, i, r["idx"], r["cnt"], sz.nvk).size == 0
    o = O.forward(arrays["q"], arrays["k"], arrays["v"], None, r["idx"], r["cnt"], sz)
    assert np.array_equal(r["o"], o)


def test_queries_equal_to_the_anchor_recover_dense_attention():
    # every video query row of a head is the same vector c: the anchor (their
    # mean) is c, and each skipped block's virtual key carries exactly the
    # block's softmax mass and weighted value (unrounded summaries)
    rng = np.random.default_rng(32)
    T, H, Nv = 64 * 8 + 30, 2, 64 * 8
    base = make_inputs(T=T, H=H, video_tokens=Nv, qk_kind="walk1d", seed=33)
    c = O.round_to_bf16(rng.standard_normal((H, 128)) * 0.8)
    q = O.decode_bf16(base["q"]).copy()
    q[:Nv] = c[None]
    q_bits = _bits(q)
    sz = _sizes(T, H, Nv, 0.25, 0)
    a = O.video_query_anchor(q_bits, Nv)
    assert np.array_equal(O.decode_bf16(a[0]), c)
    s = O.spark_reweight(a, base["k"], base["v"], pre_round=True)
    ref = O.plan(q_bits, base["k"], sz)
    o = O.forward_merged(q_bits, base["k"], base["v"], None, ref["idx"], ref["cnt"], sz,
                         s["ak"][0], s["av"][0], s["lm"][0])
    k, v = O.decode_bf16(base["k"]), O.decode_bf16(base["v"])
    assert any(O.skipped_blocks(0, i, ref["idx"], ref["cnt"], sz.nvk).size for i in range(sz.nq))
    for h in range(H):
        rows = np.arange(0, Nv)
        np.testing.assert_allclose(o[rows, h], _dense(q, k, v, rows, h), rtol=0, atol=1e-11)


def test_constant_skipped_blocks_recover_dense_attention_for_any_query():
    # K and V constant inside every video block: a block's 64 equal keys and
    # its one virtual key (key c, log-mass log 64, value w) weigh the same,
    # with the stored BF16 summaries, whatever the query
    rng = np.random.default_rng(34)
    T, H, Nv = 64 * 8 + 30, 1, 64 * 8
    base = make_inputs(T=T, H=H, video_tokens=Nv, qk_kind="iid", seed=35)
    k = O.decode_bf16(base["k"]).copy()
    v = O.decode_bf16(base["v"]).copy()
    for b in range(Nv // 64):
        k[64 * b:64 * b + 64] = O.round_to_bf16(rng.standard_normal((1, H, 128)) * 0.7)
        v[64 * b:64 * b + 64] = O.round_to_bf16(rng.standard_normal((1, H, 128)))
    k_bits, v_bits = _bits(k), _bits(v)
    sz = _sizes(T, H, Nv, 0.25, 0)
    r = O.spark_forward(base["q"], k_bits, v_bits, None, sz)
    np.testing.assert_allclose(r["lm"][:, : Nv // 64], math.log(64), rtol=0, atol=1e-12)
    q = O.decode_bf16(base["q"])
    rows = np.arange(0, Nv)
    np.testing.assert_allclose(r["o"][rows, 0], _dense(q, k, v, rows, 0), rtol=0, atol=1e-11)


def test_skipped_and_listed_video_blocks_partition_the_video_blocks():
    arrays = make_inputs(T=64 * 20 + 7, H=3, video_tokens=64 * 20, qk_kind="walk1d", seed=36)
    sz = _sizes(64 * 20 + 7, 3, 64 * 20, 0.2, 1)
    ref = O.plan(arrays["q"], arrays["k"], sz)
    for h in range(3):
        for i in range(sz.nq):
            listed = [int(b) for b in ref["idx"][h, i, : ref["cnt"][h, i]] if b < sz.nvk]
            sk = O.skipped_blocks(h, i, ref["idx"], ref["cnt"], sz.nvk)
            assert sorted(listed + sk.tolist()) == list(range(sz.nvk))


def test_anchor_is_the_rounded_mean_of_the_video_queries():
    arrays = make_inputs(T=300, H=2, video_tokens=257, qk_kind="iid", seed=37)
    a = O.decode_bf16(O.video_query_anchor(arrays["q"], 257)[0])
    q = O.decode_bf16(arrays["q"])
    for h in range(2):
        for d in (0, 5, 127):
            total = 0.0
            for t in range(257):  # plain loop over the rows
                total += q[t, h, d]
            assert a[h, d] == O.round_to_bf16(np.array([total / 257]))[0]
