"""Pins of the virtual-summary oracle (oracle/spark.py) to facts that do not
come from the oracle itself: bit-level BF16 rounding, closed forms of the
softmax summary, the entropy identity of the log-mass, and invariances.

Source: "Sol-Attn and Spark for MiniMax-H3", section "Spark primitives"
(spark_reweight) and section "Spark inference integration" (the default
summary numerics: BF16 storage, log-mass against the stored BF16 key).
"""

import math

import numpy as np
import pytest

import oracle as O


def _bits(x):
    """float values exactly representable in BF16 -> BF16 bit patterns."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "not a BF16 value"
    return (u >> 16).astype(np.uint16)


def _rne_bits(f32):
    """Round-to-nearest-even of FP32 values to BF16, on the bit patterns."""
    u = np.asarray(f32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = (u + 0x7FFF + lsb) >> 16
    return (r.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _rand_bf16(rng, shape, scale=1.0):
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    return _rne_bits(x)


def test_round_to_bf16_matches_bit_level_rounding():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-30).astype(np.float32),
        (rng.standard_normal(2000) * 1e30).astype(np.float32),
        # exact ties: the low 16 bits are 0x8000
        ((rng.integers(0x3F00, 0x4100, 1000).astype(np.uint32) << 16) | 0x8000).view(np.float32),
        np.array([1.0, -1.0, 0.0, 1.00390625, 1.01171875, 255.5], dtype=np.float32),
    ])
    got = O.round_to_bf16(x.astype(np.float64))
    assert np.array_equal(got, _rne_bits(x))


def test_zero_anchor_gives_block_means_and_log_length():
    # a = 0: every weight is 1/n, the summaries are the block means and the
    # log-mass is log(block length) -- the ordinary mass the reweight replaces
    rng = np.random.default_rng(1)
    T, H = 64 * 3 + 17, 2
    k = _rand_bf16(rng, (T, H, 128))
    v = _rand_bf16(rng, (T, H, 128))
    a = np.zeros((1, H, 128))
    r = O.spark_reweight(_bits(a), _bits(k), _bits(v))
    for b, rows in enumerate(O.block_ranges(T)):
        n = len(rows)
        np.testing.assert_allclose(r["ak"][0, :, b], k[rows.start:rows.stop].mean(axis=0), rtol=0, atol=1e-13)
        np.testing.assert_allclose(r["av"][0, :, b], v[rows.start:rows.stop].mean(axis=0), rtol=0, atol=1e-13)
        np.testing.assert_allclose(r["lm"][0, :, b], math.log(n), rtol=0, atol=1e-13)
    assert [len(rows) for rows in O.block_ranges(T)] == [64, 64, 64, 17]


def test_identical_keys_give_that_key_and_log_length():
    rng = np.random.default_rng(2)
    T, H = 64 * 2, 1
    c = _rand_bf16(rng, (H, 128))
    k = np.broadcast_to(c, (T, H, 128)).copy()
    v = _rand_bf16(rng, (T, H, 128))
    a = _rand_bf16(rng, (3, H, 128))
    for pre in (False, True):
        r = O.spark_reweight(_bits(a), _bits(k), _bits(v), pre_round=pre)
        np.testing.assert_allclose(r["ak"], np.broadcast_to(c, r["ak"].shape), rtol=0, atol=1e-12)
        assert np.array_equal(r["ak16"], np.broadcast_to(c, r["ak"].shape))
        np.testing.assert_allclose(r["lm"], math.log(64), rtol=0, atol=1e-10)
        # values are averaged with equal weights
        np.testing.assert_allclose(r["av"][:, :, 0], np.broadcast_to(v[:64].mean(axis=0), (3, H, 128)),
                                   rtol=0, atol=1e-12)


def test_two_key_block_closed_form():
    # a partial last block of two keys: w1 = sigmoid(delta) with
    # delta = a . (k1 - k2) / sqrt(128); log-mass = binary entropy of w1
    rng = np.random.default_rng(3)
    T, H = 64 + 2, 1
    k = _rand_bf16(rng, (T, H, 128), 0.5)
    v = _rand_bf16(rng, (T, H, 128))
    a = _rand_bf16(rng, (1, H, 128), 0.5)
    r = O.spark_reweight(_bits(a), _bits(k), _bits(v), pre_round=True)
    k1, k2 = k[64, 0], k[65, 0]
    delta = float(a[0, 0] @ (k1 - k2)) / math.sqrt(128.0)
    w1 = 1.0 / (1.0 + math.exp(-delta))
    w2 = 1.0 - w1
    np.testing.assert_allclose(r["ak"][0, 0, 1], w1 * k1 + w2 * k2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["av"][0, 0, 1], w1 * v[64, 0] + w2 * v[65, 0], rtol=0, atol=1e-12)
    ent = -(w1 * math.log(w1) + w2 * math.log(w2))
    assert r["lm"][0, 0, 1] == pytest.approx(ent, abs=1e-12)
    assert abs(delta) > 0.05  # the case is not the uniform one


def test_log_mass_is_the_entropy_of_the_block_softmax():
    rng = np.random.default_rng(4)
    T, H, P = 64 * 4 + 5, 3, 2
    k = _rand_bf16(rng, (T, H, 128), 0.7)
    v = _rand_bf16(rng, (T, H, 128))
    a = _rand_bf16(rng, (P, H, 128), 0.7)
    r = O.spark_reweight(_bits(a), _bits(k), _bits(v), pre_round=True)
    for p in range(P):
        for h in range(H):
            for b, rows in enumerate(O.block_ranges(T)):
                z = np.array([a[p, h] @ k[u, h] for u in rows]) / math.sqrt(128.0)
                z = z - z.max()
                w = np.exp(z) / np.exp(z).sum()
                ent = float(-(w * np.log(w)).sum())
                assert r["lm"][p, h, b] == pytest.approx(ent, abs=1e-10)
                assert -1e-12 <= r["lm"][p, h, b] <= math.log(len(rows)) + 1e-12


def test_dominant_key_takes_all_the_weight():
    rng = np.random.default_rng(5)
    T, H = 64, 1
    k = _rand_bf16(rng, (T, H, 128), 0.01)
    k[17, 0] = _rne_bits(np.full(128, 4.0, np.float32))
    v = _rand_bf16(rng, (T, H, 128))
    a = _bits(np.full((1, H, 128), 64.0))  # s_17 - s_u > 2000
    r = O.spark_reweight(a, _bits(k), _bits(v), pre_round=True)
    np.testing.assert_allclose(r["ak"][0, 0, 0], k[17, 0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["av"][0, 0, 0], v[17, 0], rtol=0, atol=1e-12)
    assert abs(r["lm"][0, 0, 0]) < 1e-12


def test_summaries_are_per_block_and_order_free():
    rng = np.random.default_rng(6)
    T, H = 64 * 3, 2
    k = _rand_bf16(rng, (T, H, 128))
    v = _rand_bf16(rng, (T, H, 128))
    a = _rand_bf16(rng, (2, H, 128))
    r = O.spark_reweight(_bits(a), _bits(k), _bits(v))
    # permuting keys (with their values) inside block 1 changes nothing
    perm = np.arange(T)
    perm[64:128] = 64 + rng.permutation(64)
    r2 = O.spark_reweight(_bits(a), _bits(k[perm]), _bits(v[perm]))
    for key in ("ak", "av", "lm"):
        np.testing.assert_allclose(r2[key], r[key], rtol=0, atol=1e-12)
    # changing block 2 leaves blocks 0 and 1 alone; heads are independent
    k3 = k.copy()
    k3[128:, 1] = _rand_bf16(rng, (64, 128))
    r3 = O.spark_reweight(_bits(a), _bits(k3), _bits(v))
    assert np.array_equal(r3["ak"][:, :, :2], r["ak"][:, :, :2])
    assert np.array_equal(r3["ak"][:, 0], r["ak"][:, 0])
    assert not np.array_equal(r3["ak"][:, 1, 2], r["ak"][:, 1, 2])


def test_stored_key_term_uses_the_rounded_summary():
    # default log-mass subtracts a . ak16 / sqrt(128); pre_round uses ak
    rng = np.random.default_rng(7)
    T, H = 64 * 2, 2
    k = _rand_bf16(rng, (T, H, 128))
    v = _rand_bf16(rng, (T, H, 128))
    a = _rand_bf16(rng, (1, H, 128))
    r = O.spark_reweight(_bits(a), _bits(k), _bits(v))
    rp = O.spark_reweight(_bits(a), _bits(k), _bits(v), pre_round=True)
    diff = rp["lm"] - r["lm"]
    want = np.einsum("phbd,phd->phb", r["ak16"] - r["ak"], a) / math.sqrt(128.0)
    np.testing.assert_allclose(diff, want, rtol=0, atol=1e-12)
    assert np.any(np.abs(diff) > 1e-6)
    assert O.reweight_bytes(1, T, H) == 2 * T * H * 256 + H * 256 + H * 2 * (512 + 4)
