"""Parity of the CUDA reblocking (sparse_attn_spark_reblock) with the oracles:
bit for bit against the fixed-order FP32 statement (oracle/reblock.py, the
numeric contract), and under the margin rule against the float64 tree
(oracle/reblock_f64.py: ordinary dot products, no fixed order), which must
agree with the kernel on every decision whose margin exceeds the float32
error bound.

Source: "Sol-Attn and Spark for MiniMax-H3", section "Spark primitives"
(spark_reblock) and section "Spark inference integration" (power-of-two
fanout, cosine scoring on normalized FP16 vectors).

Both sides take every floating-point decision in FP32 with the same order
of operations (exact FP16 products, four terms per lane left to right, then
a 32-lane butterfly), so there is no tolerance: a single differing index is
a failure.
"""

import numpy as np
import pytest

from oracle import reblock as R
from tests.parity import oracle_pool, reblock_margin_all
from workloads import make_workload

pytestmark = pytest.mark.gpu


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


def _bits(x):
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)


def _check(bsr, xbits, fanout, L=32, heads=None):
    perm, inv = bsr.spark_reblock(_dev(xbits), fanout=fanout, landmarks=L)
    perm, inv = perm.cpu().numpy(), inv.cpu().numpy()
    T, H, _ = xbits.shape
    for h in (range(H) if heads is None else heads):
        p, iv = R.reblock_head(xbits[:, h, :], fanout, L)
        assert np.array_equal(perm[h], p), f"head {h}: first mismatch at {int(np.argmax(perm[h] != p))}"
        assert np.array_equal(inv[h], iv), f"head {h}"
    return perm, inv


@pytest.mark.parametrize("T,H,fanout", [(64 * 7 + 13, 3, 2), (64 * 7 + 13, 3, 4), (64 * 20 + 1, 2, 8),
                                        (64 * 33 + 63, 2, 16), (64 * 60, 1, 8), (128, 2, 8), (64, 2, 8),
                                        (40, 2, 8)])
def test_random_samples(bsr, T, H, fanout):
    rng = np.random.default_rng(T * 31 + fanout)
    _check(bsr, _bits(rng.standard_normal((T, H, 128))), fanout)


@pytest.mark.parametrize("L", [2, 5, 32, 64])
def test_landmark_counts(bsr, L):
    rng = np.random.default_rng(L)
    _check(bsr, _bits(rng.standard_normal((64 * 11 + 3, 2, 128))), 4, L)


def test_h3_keys_all_heads(bsr):
    # full H3 size (T = 9505, 56 heads), every head, the default fanout 8
    arrays, _ = make_workload("h3")
    _check(bsr, arrays["k"], 8)


def test_h3_queries_sampled_heads_fanout16(bsr):
    arrays, _ = make_workload("h3")
    _check(bsr, arrays["q"], 16, heads=[0, 17, 38, 55])


@pytest.mark.parametrize("name,heads", [("32k", [0, 39]), ("64k", [0, 23])])
def test_largest_configs_sampled_heads(bsr, name, heads):
    # the largest sizes (64k: a root of 1056 blocks, one CTA per head selects
    # its boundaries among 67584 keys), every head computed, two compared
    arrays, _ = make_workload(name)
    _check(bsr, arrays["k"], 8, heads=heads)


def test_8k_keys(bsr):
    arrays, _ = make_workload("8k")
    _check(bsr, arrays["k"], 8, heads=[0, 5, 11, 23])


def test_closed_forms_through_the_gpu(bsr):
    # orthogonal groups: the hand-worked permutation
    x = np.zeros((256, 1, 128), dtype=np.float32)
    for g in range(4):
        x[64 * g:64 * (g + 1), 0, g] = 1.0
    perm, _ = _check(bsr, _bits(x), 2)
    assert perm[0].tolist() == (list(range(128, 192)) + list(range(64, 128))
                                + list(range(192, 256)) + list(range(64)))
    # planar arc: blocks are runs of 64 of the angle order
    rng = np.random.default_rng(9)
    q, _ = np.linalg.qr(rng.standard_normal((128, 2)))
    n = 512
    ang = np.deg2rad(5.0 + 170.0 * np.arange(n) / n)[rng.permutation(n)]
    r = np.exp(rng.uniform(np.log(0.05), np.log(20.0), n))
    xa = _bits((r[:, None] * (np.cos(ang)[:, None] * q[:, 0] + np.sin(ang)[:, None] * q[:, 1]))[:, None, :])
    perm, _ = _check(bsr, xa, 8)
    xd = (xa[:, 0, :].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    theta = np.arctan2(xd @ q[:, 1], xd @ q[:, 0])
    want = {tuple(sorted(np.argsort(theta)[64 * b:64 * (b + 1)].tolist())) for b in range(8)}
    assert {tuple(sorted(perm[0, 64 * b:64 * (b + 1)].tolist())) for b in range(8)} == want


def test_degenerate_rows(bsr):
    T = 64 * 6 + 5
    rng = np.random.default_rng(4)
    same = np.tile(_bits(rng.standard_normal(128))[None, None], (T, 2, 1))
    perm, _ = _check(bsr, same, 8)
    assert perm[0].tolist() == list(range(T))
    zero = np.zeros((T, 2, 128), dtype=np.uint16)
    perm, _ = _check(bsr, zero, 4)
    assert perm[1].tolist() == list(range(T))
    # a few zero rows among random ones
    x = _bits(rng.standard_normal((T, 2, 128)))
    x[::7] = 0
    _check(bsr, x, 8)


def test_strided_heads_and_repeat(bsr):
    import torch

    rng = np.random.default_rng(12)
    T, Hb = 64 * 13 + 9, 6
    xb = _bits(rng.standard_normal((T, Hb, 128)))
    big = _dev(xb)
    sub = big[:, 2:5, :]  # token stride 6 * 128, head stride 128
    p1, i1 = bsr.spark_reblock(sub, fanout=8)
    p2, i2 = bsr.spark_reblock(sub, fanout=8)
    assert torch.equal(p1, p2) and torch.equal(i1, i2)
    for j, h in enumerate(range(2, 5)):
        p, iv = R.reblock_head(xb[:, h, :], 8)
        assert np.array_equal(p1[j].cpu().numpy(), p) and np.array_equal(i1[j].cpu().numpy(), iv)
    # heads-major [H, T, 128] storage seen as [T, H, 128]
    hm = _dev(np.ascontiguousarray(xb.transpose(1, 0, 2))).permute(1, 0, 2)
    p3, _ = bsr.spark_reblock(hm, fanout=8)
    assert torch.equal(p3[2:5], p1)


def test_argument_errors(bsr):
    import torch

    x = torch.zeros((256, 2, 128), dtype=torch.bfloat16, device="cuda")
    for kw in ({"fanout": 3}, {"fanout": 32}, {"fanout": 1}, {"landmarks": 1}, {"landmarks": 65}):
        with pytest.raises(bsr.SparseAttnError):
            bsr.spark_reblock(x, **kw)
    with pytest.raises(ValueError):
        bsr.spark_reblock(x.float(), fanout=8)


# ---------------------------------------------------------------- float64 tree, margin rule
@pytest.fixture(scope="module")
def pool():
    p = oracle_pool()
    yield p
    p.close()
    p.join()


def _margin(bsr, pool, name, xb, fanout, heads=None, L=32):
    """The kernel's permutation against the float64 tree, for any summation
    order (depth 127) and for the contract's depth 8; logs the coverage."""
    perm, _ = bsr.spark_reblock(_dev(xb), fanout=fanout, landmarks=L)
    perm = perm.cpu().numpy()
    for depth in (127, 8):
        res = reblock_margin_all(pool, xb, perm, fanout, L, depth, heads)
        bad = [(h, v[:2]) for h, v, _ in res if v]
        cov = [c for _, _, c in res]
        print(f"[reblock margin] {name} fanout {fanout} depth {depth}: {len(res)} heads, "
              f"leaf-certain tokens {np.mean(cov):.3f} (min {np.min(cov):.3f})")
        assert not bad, bad
    return perm


@pytest.mark.parametrize("T,H,fanout", [(64 * 7 + 13, 3, 2), (64 * 20 + 1, 2, 8), (64 * 33 + 63, 2, 16),
                                        (64 * 11 + 3, 2, 4)])
def test_margin_rule_random_samples(bsr, pool, T, H, fanout):
    rng = np.random.default_rng(T * 7 + fanout)
    _margin(bsr, pool, f"T={T}", _bits(rng.standard_normal((T, H, 128))), fanout)


def test_margin_rule_h3_keys_all_heads(bsr, pool):
    arrays, _ = make_workload("h3")
    _margin(bsr, pool, "h3 keys", arrays["k"], 8)


def test_margin_rule_h3_queries_fanout16(bsr, pool):
    arrays, _ = make_workload("h3")
    _margin(bsr, pool, "h3 queries", arrays["q"], 16, heads=range(0, 56, 4))


@pytest.mark.parametrize("name,heads", [("8k", [0, 7, 23]), ("32k", [0, 13, 39]), ("64k", [0, 23])])
def test_margin_rule_other_configs(bsr, pool, name, heads):
    arrays, _ = make_workload(name)
    _margin(bsr, pool, f"{name} keys", arrays["k"], 8, heads=heads)
