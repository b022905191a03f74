"""Pins of the CPU oracle against things other than itself (no GPU).

Each test states what fixes the expected value: a number printed on the
source pages (tests/golden/page_values.json), a hand-worked example
(tests/golden/hand_lists.json), a closed form, an invariant, a library
routine for a special case, or an independent brute-force formulation
(tests/brute.py).  A plausible slip in the oracle (dropped 1/sqrt(128), wrong
sign, transposed operand, off-by-one radius, wrong tie-break, wrong row
classification, mean over the wrong rows) fails at least one of them.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle as O
from tests import brute
from workloads import WORKLOADS, bf16_round_bits, make_inputs

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _bits(x):
    return bf16_round_bits(np.asarray(x, dtype=np.float32))


def _sizes(name, H=None):
    w = WORKLOADS[name]
    return O.derive_sizes(w.T, H or w.H, w.video_tokens, w.topk_ratio, w.radius, w.tail_mode)


# --------------------------------------------------------------- page values
def test_page_dense_score_bytes():
    g = _gold("page_values.json")["dense_scores_h3"]
    got = O.dense_score_bytes(g["T"], g["H"])
    assert abs(got - g["approx_bytes"]) <= g["rel_tol"] * g["approx_bytes"]


def test_page_radius_offsets():
    g = _gold("page_values.json")["forced_radius"]
    i, nvk = 10, 40
    assert O.local_video_blocks(i, 0, nvk) == [i + d for d in g["radius_0_offsets"]]
    assert O.local_video_blocks(i, 1, nvk) == [i + d for d in g["radius_1_offsets"]]
    # clipped at the ends, never wrapped
    assert O.local_video_blocks(0, 1, nvk) == [0, 1]
    assert O.local_video_blocks(nvk - 1, 1, nvk) == [nvk - 2, nvk - 1]


def test_page_block_and_head_sizes():
    g = _gold("page_values.json")
    assert O.BLOCK == g["block_tokens"]["tokens_per_block"]
    assert O.HEAD_DIM == g["head_dim"]["D"]


def test_dense_pairs_match_kept_keys_at_ratio_one():
    # At topk_ratio = 1 every row attends every key, so the kept-pair count is
    # the dense count T*T*H behind the page's 20 GB figure.
    sz = O.derive_sizes(1152, 2, 1024, 1.0, 0, "dense")
    rng = np.random.default_rng(0)
    idx, cnt = O.block_lists(rng.standard_normal((2, sz.nq, sz.nvk)), sz)
    assert int(O.kept_keys_per_row(idx, cnt, sz).sum()) * 4 == O.dense_score_bytes(1152, 2)


# --------------------------------------------------------------- sizes
@pytest.mark.parametrize(
    "name,nvk,tail,nblk,nq,K,nsink,maxl,r0",
    [
        # K = ceil(0.25*16) = 4;  maxl = min(16, 1+4) + 2
        ("tiny", 16, 0, 18, 16, 4, 2, 7, 1024),
        # K = ceil(0.1*128) = ceil(12.8) = 13; maxl = min(128, 3+13) + 8
        ("8k", 128, 0, 136, 128, 13, 8, 24, 8192),
        # 9240 = 144*64 + 24; 9505 = 148*64 + 33 -> 149 blocks; K = ceil(14.4) = 15
        ("h3", 144, 24, 149, 144, 15, 5, 23, 9216),
        # K = ceil(51.2) = 52; maxl = 55 + 16
        ("32k", 512, 0, 528, 512, 52, 16, 71, 32768),
        # 65560 = 1024*64 + 24 (pad -> 1025 query blocks); 67608 -> 1057 blocks;
        # K = ceil(0.05*1024) = ceil(51.2) = 52; dense rows start at Nv
        ("64k", 1024, 24, 1057, 1025, 52, 33, 88, 65560),
    ],
)
def test_derived_sizes(name, nvk, tail, nblk, nq, K, nsink, maxl, r0):
    sz = _sizes(name)
    assert (sz.nvk, sz.tail, sz.nblk, sz.nq, sz.K, sz.nsink, sz.maxl, sz.dense_row_start) == (
        nvk, tail, nblk, nq, K, nsink, maxl, r0)


def test_topk_count_is_decimal_ceiling():
    assert O.topk_count(0.1, 30) == 3  # binary 0.1 * 30 = 3.0000000000000004
    assert O.topk_count(0.1, 144) == 15
    assert O.topk_count(0.25, 16) == 4
    assert O.topk_count(1.0, 7) == 7
    assert O.topk_count(0.001, 7) == 1
    assert O.topk_count(0.3, 10) == 3


@pytest.mark.parametrize(
    "kw",
    [
        dict(T=1152, H=2, video_tokens=63, topk_ratio=0.1, radius=0, tail_mode="dense"),
        dict(T=1152, H=2, video_tokens=1153, topk_ratio=0.1, radius=0, tail_mode="dense"),
        dict(T=1152, H=2, video_tokens=1024, topk_ratio=0.0, radius=0, tail_mode="dense"),
        dict(T=1152, H=2, video_tokens=1024, topk_ratio=1.5, radius=0, tail_mode="dense"),
        dict(T=1152, H=2, video_tokens=1024, topk_ratio=0.1, radius=-1, tail_mode="dense"),
        dict(T=1152, H=2, video_tokens=1024, topk_ratio=0.1, radius=0, tail_mode="zig"),
        # pad mode: the tail block (16 full blocks + 24 tokens) needs T >= 17*64
        dict(T=1058, H=2, video_tokens=1048, topk_ratio=0.1, radius=0, tail_mode="pad"),
        dict(T=1087, H=2, video_tokens=1048, topk_ratio=0.1, radius=0, tail_mode="pad"),
    ],
)
def test_derive_sizes_rejects(kw):
    with pytest.raises(ValueError):
        O.derive_sizes(**kw)


def test_pad_mode_accepts_exactly_enough_slots():
    sz = O.derive_sizes(1088, 2, 1048, 0.1, 0, "pad")
    assert sz.nq == 17 and sz.dense_row_start == 1048


# --------------------------------------------------------------- centroids
def test_constant_block_centroid_is_exact():
    sz = O.derive_sizes(320, 3, 256, 0.5, 0, "dense")
    rng = np.random.default_rng(1)
    c = rng.integers(-8, 9, size=(sz.nvk, 3, 128)).astype(np.float32) / 4
    q = np.repeat(c, 64, axis=0)
    q = np.concatenate([q, np.zeros((64, 3, 128), np.float32)])
    Qc, Kc = O.centroids(_bits(q), _bits(-q), sz)
    assert np.array_equal(Qc, c.transpose(1, 0, 2).astype(np.float64))
    assert np.array_equal(Kc, -c.transpose(1, 0, 2).astype(np.float64))


def test_centroid_is_linear():
    sz = O.derive_sizes(320, 2, 256, 0.5, 0, "dense")
    rng = np.random.default_rng(2)
    a = rng.integers(-16, 17, size=(320, 2, 128)).astype(np.float32)
    b = rng.integers(-16, 17, size=(320, 2, 128)).astype(np.float32)
    Qa, _ = O.centroids(_bits(a), _bits(a), sz)
    Qb, _ = O.centroids(_bits(b), _bits(b), sz)
    Qab, _ = O.centroids(_bits(a + b), _bits(a + b), sz)
    assert np.allclose(Qab, Qa + Qb, rtol=0, atol=1e-12)


def test_pad_tail_centroid_is_mean_of_real_rows():
    # Pad mode fills the non-video slots with the mean Q of the real rows,
    # which preserves the block centroid ("H3 pipeline integration").
    sz = O.derive_sizes(448, 2, 280, 0.5, 0, "pad")  # nvk = 4, tail = 24
    assert sz.nq == 5 and sz.tail == 24
    x = make_inputs(T=448, H=2, video_tokens=280, seed=5)
    Qc, _ = O.centroids(x["q"], x["k"], sz)
    real = O.decode_bf16(x["q"][256:280])
    assert np.allclose(Qc[:, 4, :], real.mean(axis=0), rtol=0, atol=1e-14)
    filler = np.broadcast_to(Qc[:, 4, :], (40, 2, 128))
    full = np.concatenate([real, filler], axis=0)
    assert np.allclose(full.mean(axis=0), Qc[:, 4, :], rtol=0, atol=1e-14)
    # dense mode has no tail query block
    assert O.derive_sizes(448, 2, 280, 0.5, 0, "dense").nq == 4


# --------------------------------------------------------------- routing
def _hand_inputs(a, b):
    q = np.zeros((320, 1, 128), np.float32)
    k = np.zeros((320, 1, 128), np.float32)
    for i, ai in enumerate(a):
        q[64 * i:64 * i + 64, 0, 0] = ai
    for j, bj in enumerate(b):
        k[64 * j:64 * j + 64, 0, 0] = bj
    return _bits(q), _bits(k)


@pytest.mark.parametrize("case", range(2))
def test_hand_worked_lists(case):
    g = _gold("hand_lists.json")["cases"][case]
    sz = O.derive_sizes(320, 1, 256, 0.5, 0, "dense")
    q, k = _hand_inputs(g["a"], g["b"])
    p = O.plan(q, k, sz)
    expect_s = np.outer(g["a"], g["b"]) / math.sqrt(128)
    assert np.allclose(p["scores"][0], expect_s, rtol=0, atol=1e-15)
    for i, lst in enumerate(g["lists"]):
        assert list(p["idx"][0, i, : p["cnt"][0, i]]) == lst
        assert all(v == -1 for v in p["idx"][0, i, p["cnt"][0, i]:])


def test_scores_not_transposed():
    # Asymmetric centroids: s[i, j] must be Qc_i . Kc_j, not Qc_j . Kc_i.
    sz = O.derive_sizes(320, 1, 256, 0.5, 0, "dense")
    q, k = _hand_inputs([1, 2, 3, 4], [5, 7, 11, 13])
    s = O.plan(q, k, sz)["scores"][0]
    assert s[0, 3] == pytest.approx(13 / math.sqrt(128), abs=0)
    assert s[3, 0] == pytest.approx(20 / math.sqrt(128), abs=0)


@pytest.mark.parametrize("seed", range(6))
def test_topk_matches_subset_enumeration(seed):
    rng = np.random.default_rng(seed)
    nvk, K, R = 9, 3, seed % 3
    sz = O.derive_sizes(64 * nvk + 70, 1, 64 * nvk, K / nvk, R, "dense")
    assert sz.K == K
    # coarse integer scores force many exact ties
    s = rng.integers(-3, 4, size=(1, nvk, nvk)).astype(np.float64)
    idx, cnt = O.block_lists(s, sz)
    s32 = s.astype(np.float32)
    for i in range(nvk):
        lv = [j for j in range(i - R, i + R + 1) if 0 <= j < nvk]
        cand = [j for j in range(nvk) if j not in lv]
        top = brute.brute_topk(s32[0, i], cand, K)
        want = sorted(set(lv) | set(top) | set(range(nvk, sz.nblk)))
        assert list(idx[0, i, : cnt[0, i]]) == want


def test_planted_tie_takes_lower_index():
    sz = O.derive_sizes(64 * 6 + 64, 1, 64 * 6, 0.34, 0, "dense")  # K = ceil(2.04) = 3
    assert sz.K == 3
    s = np.zeros((1, 6, 6))
    s[0, 0] = [9, 5, 5, 5, 5, 1]  # candidates 1..5; 5,5,5,5 tie for 3 slots
    idx, cnt = O.block_lists(s, sz)
    assert list(idx[0, 0, : cnt[0, 0]]) == [0, 1, 2, 3, 6]


@pytest.mark.parametrize("name", ["tiny", "8k", "h3", "32k", "64k"])
def test_list_lengths_closed_form(name):
    sz = _sizes(name, H=2)
    rng = np.random.default_rng(7)
    idx, cnt = O.block_lists(rng.standard_normal((2, sz.nq, sz.nvk)), sz)
    for i in range(sz.nq):
        nlv = sum(1 for j in range(i - sz.R, i + sz.R + 1) if 0 <= j < sz.nvk)
        want = nlv + min(sz.K, sz.nvk - nlv) + sz.nsink
        assert (cnt[:, i] == want).all()
        for h in range(2):
            lst = idx[h, i, : cnt[h, i]]
            assert (np.diff(lst) > 0).all()
            assert set(range(sz.nvk, sz.nblk)) <= set(lst.tolist())  # sinks always exact
            if i < sz.nvk:
                assert i in lst  # self block forced
            assert (idx[h, i, cnt[h, i]:] == -1).all()
    assert cnt.max() <= sz.maxl


def test_kept_flops_closed_form_h3():
    sz = _sizes("h3")
    rng = np.random.default_rng(3)
    idx, cnt = O.block_lists(rng.standard_normal((sz.H, sz.nq, sz.nvk)), sz)
    sink_keys = sz.T - 64 * sz.nvk  # 289
    per_head = 0
    for i in range(sz.nq):
        nlv = sum(1 for j in range(i - 1, i + 2) if 0 <= j < sz.nvk)
        per_head += 64 * (64 * (nlv + sz.K) + sink_keys)
    per_head += (sz.T - sz.dense_row_start) * sz.T
    assert O.kept_flops(idx, cnt, sz) == per_head * sz.H * 4 * 128
    assert O.kept_flops(idx, cnt, sz) == pytest.approx(0.459e12, rel=0.01)


# --------------------------------------------------------------- attention
def _tiny_case(T=200, H=2, Nv=150, ratio=0.5, R=0, mode="dense", seed=11):
    sz = O.derive_sizes(T, H, Nv, ratio, R, mode)
    x = make_inputs(T=T, H=H, video_tokens=Nv, seed=seed)
    p = O.plan(x["q"], x["k"], sz)
    return sz, x, p


def test_ratio_one_equals_library_dense_attention():
    torch = pytest.importorskip("torch")
    T, H = 330, 2
    sz, x, p = _tiny_case(T=T, H=H, Nv=256, ratio=1.0, R=0)
    rng = np.random.default_rng(4)
    bias = np.zeros(T, np.float32)
    bias[256:] = rng.standard_normal(T - 256).astype(np.float32)
    out = O.forward(x["q"], x["k"], x["v"], bias, p["idx"], p["cnt"], sz)
    q, k, v = (torch.from_numpy(O.decode_bf16(x[n])).permute(1, 0, 2)[None] for n in "qkv")
    ref = torch.nn.functional.scaled_dot_product_attention(
        q, k, v, attn_mask=torch.from_numpy(bias.astype(np.float64))[None, None, None, :])
    ref = ref[0].permute(1, 0, 2).numpy()
    assert np.abs(out - ref).max() < 1e-12


@pytest.mark.parametrize("mode,Nv,R", [("dense", 150, 0), ("pad", 150, 1), ("dense", 192, 1),
                                       ("pad", 200, 0)])
def test_matches_token_expanded_mask(mode, Nv, R):
    T = 330
    sz, x, p = _tiny_case(T=T, H=2, Nv=Nv, ratio=0.4, R=R, mode=mode)
    rng = np.random.default_rng(9)
    bias = np.zeros(T, np.float32)
    bias[64 * sz.nvk:] = rng.standard_normal(T - 64 * sz.nvk).astype(np.float32)
    out = O.forward(x["q"], x["k"], x["v"], bias, p["idx"], p["cnt"], sz)
    mask = brute.token_mask(p["idx"], p["cnt"], T, Nv, mode)
    ref = brute.masked_dense_attention(
        O.decode_bf16(x["q"]), O.decode_bf16(x["k"]), O.decode_bf16(x["v"]),
        bias.astype(np.float64), mask)
    assert np.abs(out - ref).max() < 1e-12
    rows = [0, 63, 64, 64 * sz.nvk - 1, 64 * sz.nvk, Nv - 1, Nv, T - 1]
    got = O.forward_rows(x["q"], x["k"], x["v"], bias, p["idx"], p["cnt"], sz, rows, [0, 1])
    assert np.abs(got - O.forward(x["q"], x["k"], x["v"], bias, p["idx"], p["cnt"], sz)[rows]).max() < 1e-12


def test_zero_bias_equals_no_bias():
    sz, x, p = _tiny_case()
    a = O.forward(x["q"], x["k"], x["v"], None, p["idx"], p["cnt"], sz)
    b = O.forward(x["q"], x["k"], x["v"], np.zeros(sz.T, np.float32), p["idx"], p["cnt"], sz)
    assert np.array_equal(a, b)


def test_bias_changes_the_result_on_rows_seeing_sinks():
    sz, x, p = _tiny_case()
    bias = np.zeros(sz.T, np.float32)
    bias[64 * sz.nvk:] = 2.0
    a = O.forward(x["q"], x["k"], x["v"], None, p["idx"], p["cnt"], sz)
    b = O.forward(x["q"], x["k"], x["v"], bias, p["idx"], p["cnt"], sz)
    assert np.abs(a - b).max() > 1e-3


def test_minus_inf_bias_on_sink_block_drops_it():
    T, Nv = 330, 192
    sz, x, p = _tiny_case(T=T, Nv=Nv, ratio=0.4, R=1)
    drop = sz.nvk + 1  # second sink block, tokens [256, 320)
    bias = np.zeros(T, np.float32)
    bias[64 * drop:64 * drop + 64] = -np.inf
    out = O.forward(x["q"], x["k"], x["v"], bias, p["idx"], p["cnt"], sz)
    mask = brute.token_mask(p["idx"], p["cnt"], T, Nv, "dense")
    mask[:, :, 64 * drop:64 * drop + 64] = False
    ref = brute.masked_dense_attention(
        O.decode_bf16(x["q"]), O.decode_bf16(x["k"]), O.decode_bf16(x["v"]), np.zeros(T), mask)
    assert np.abs(out - ref).max() < 1e-12


def test_closed_forms_v_ones_and_q_zero():
    T, H, Nv = 330, 2, 192
    sz = O.derive_sizes(T, H, Nv, 0.4, 1, "dense")
    x = make_inputs(T=T, H=H, video_tokens=Nv, seed=12)
    p = O.plan(x["q"], x["k"], sz)
    ones = _bits(np.ones((T, H, 128)))
    o1 = O.forward(x["q"], x["k"], ones, None, p["idx"], p["cnt"], sz)
    assert np.abs(o1 - 1.0).max() < 1e-14
    zeros = _bits(np.zeros((T, H, 128)))
    o0 = O.forward(zeros, x["k"], x["v"], None, p["idx"], p["cnt"], sz)
    v = O.decode_bf16(x["v"])
    for t in [0, 65, 130, 191, 200, 329]:
        for h in range(H):
            keys = O.row_key_set(t, h, p["idx"], p["cnt"], sz)
            assert np.allclose(o0[t, h], v[keys, h].mean(axis=0), rtol=0, atol=1e-13)


def test_head_permutation_equivariance():
    T, H, Nv = 330, 3, 192
    sz = O.derive_sizes(T, H, Nv, 0.4, 1, "dense")
    x = make_inputs(T=T, H=H, video_tokens=Nv, qk_kind="walk1d", seed=13)
    perm = [2, 0, 1]
    p = O.plan(x["q"], x["k"], sz)
    xp = {n: np.ascontiguousarray(x[n][:, perm]) for n in "qkv"}
    pp = O.plan(xp["q"], xp["k"], sz)
    assert np.array_equal(pp["idx"], p["idx"][perm])
    a = O.forward(x["q"], x["k"], x["v"], None, p["idx"], p["cnt"], sz)
    b = O.forward(xp["q"], xp["k"], xp["v"], None, pp["idx"], pp["cnt"], sz)
    assert np.array_equal(b, a[:, perm])


# --------------------------------------------------------------- key bias contract
def test_key_bias_contract():
    sz = O.derive_sizes(330, 2, 192, 0.4, 1, "dense")
    ok = np.zeros(330, np.float32)
    ok[192:] = -np.inf  # -inf allowed on sinks
    O.check_key_bias(ok, sz)
    bad = np.zeros(330, np.float32)
    bad[100] = 0.5  # a routed video key
    with pytest.raises(ValueError):
        O.check_key_bias(bad, sz)
    for v in (np.nan, np.inf):
        b = np.zeros(330, np.float32)
        b[300] = v
        with pytest.raises(ValueError):
            O.check_key_bias(b, sz)
    with pytest.raises(ValueError):
        O.check_key_bias(np.zeros(329, np.float32), sz)
    with pytest.raises(ValueError):
        O.check_key_bias(np.zeros(330, np.float64), sz)
    negzero = np.zeros(330, np.float32)
    negzero[5] = -0.0
    O.check_key_bias(negzero, sz)


def test_bias_does_not_change_routing():
    # The plan consumes Q and K only: routing stays unweighted.
    import inspect
    assert "bias" not in inspect.signature(O.plan).parameters
