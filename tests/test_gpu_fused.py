"""The fused call (sparse_attn_fused: Top-K inside the attention kernel)
against the two-call path and the fp64 oracle.

Source: "Sol-Attn and Spark for MiniMax-H3", section "Spark inference
integration" (CTA-local fused Top-K routing with the same lists; exact FP32
boundary selection).  The fused route sums the same FP32 products in the
same order as the routing kernel, so its lists must equal sparse_attn_plan's
bit for bit, and with equal lists the attention output is bit-identical.
The oracle comparison uses the exact path's rules (near-tie list rule,
max-abs 2e-2 / mean-abs 2e-3).
"""

import os

import numpy as np
import pytest

import oracle as O
from tests import parity
from workloads import WORKLOADS, make_inputs, make_workload

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


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


def both_paths(bsr, arrays, T, H, Nv, ratio, R, mode):
    P = bsr.Params(T=T, H=H, video_tokens=Nv, topk_ratio=ratio, radius=R, tail_mode=mode)
    sz = bsr.sparse_attn_query(P)
    q, k, v = (to_dev(arrays[n], T, H) for n in "qkv")
    bias = None if arrays["bias"] is None else torch.from_numpy(arrays["bias"]).cuda()
    idx2, cnt2 = bsr.sparse_attn_plan(P, q, k)
    o2 = bsr.sparse_attn_fwd(P, q, k, v, idx2, cnt2, key_bias=bias)
    from block_sparse_routed_gb300 import _native

    ws = torch.empty(_native.sparse_attn_fused_ws_bytes(P.to_c()), dtype=torch.uint8, device="cuda")
    o1, idx1, cnt1 = bsr.sparse_attn_fused(P, q, k, v, key_bias=bias, ws=ws)
    status = bsr.sparse_attn_last_device_status(ws)
    torch.cuda.synchronize()
    f = lambda t: t.cpu().numpy().reshape(H, sz.nq, -1)
    return dict(status=status, idx1=f(idx1), cnt1=cnt1.cpu().numpy().reshape(H, sz.nq), o1=o1,
                idx2=f(idx2), cnt2=cnt2.cpu().numpy().reshape(H, sz.nq), o2=o2), sz


@pytest.mark.parametrize("name", ["tiny", "8k", "h3"])
def test_fused_equals_two_calls_and_oracle(bsr, name):
    w = WORKLOADS[name]
    arrays, prm = make_workload(name)
    r, sz = both_paths(bsr, arrays, w.T, w.H, w.video_tokens, w.topk_ratio, w.radius, w.tail_mode)
    assert r["status"] == 0
    assert np.array_equal(r["cnt1"], r["cnt2"]) and np.array_equal(r["idx1"], r["idx2"])
    assert torch.equal(r["o1"], r["o2"])
    osz = O.derive_sizes(w.T, w.H, w.video_tokens, w.topk_ratio, w.radius, w.tail_mode)
    ref = O.plan(arrays["q"], arrays["k"], osz)
    n_exact, n_tie, bad = parity.compare_lists(r["idx1"], r["cnt1"], ref, osz)
    assert not bad, bad[:5]
    rows = [0, 63, 64, osz.Nv - 1, osz.dense_row_start, osz.T - 1]
    ref_o = O.forward_rows(arrays["q"], arrays["k"], arrays["v"], arrays["bias"], ref["idx"], ref["cnt"],
                           osz, rows, [0, w.H - 1])
    got = parity.bf16_tensor_to_f64(r["o1"].reshape(w.T, w.H, 128))[rows][:, [0, w.H - 1]]
    same = parity.same_list_mask(r["idx1"], r["cnt1"], ref)
    keep = np.array([[same[h, min(t // 64, osz.nq - 1)] if t < osz.dense_row_start else True
                      for h in (0, w.H - 1)] for t in rows])
    d = np.abs(got - ref_o)[keep]
    assert d.max() <= parity.OUT_MAX_ABS and d.mean() <= parity.OUT_MEAN_ABS


@pytest.mark.parametrize("T,H,Nv,ratio,R,mode,bias", [
    (64 * 6 + 40, 2, 64 * 5 + 20, 0.25, 1, "pad", "sink_normal"),
    (64 * 40 + 9, 3, 64 * 40, 1.0, 0, "dense", "none"),
    (64 * 256 + 100, 1, 64 * 256, 0.05, 2, "dense", "zero"),
])
def test_fused_edges(bsr, T, H, Nv, ratio, R, mode, bias):
    arrays = make_inputs(T=T, H=H, video_tokens=Nv, qk_kind="walk1d", bias_kind=bias, seed=T % 97)
    r, sz = both_paths(bsr, arrays, T, H, Nv, ratio, R, mode)
    assert r["status"] == 0
    assert np.array_equal(r["cnt1"], r["cnt2"]) and np.array_equal(r["idx1"], r["idx2"])
    assert torch.equal(r["o1"], r["o2"])


def test_fused_rejects_long_rows(bsr):
    from block_sparse_routed_gb300 import _native

    P = bsr.Params(T=64 * 300, H=1, video_tokens=64 * 257, topk_ratio=0.1, radius=1)
    with pytest.raises(bsr.SparseAttnError) as e:
        _native.sparse_attn_fused_ws_bytes(P.to_c())
    assert e.value.status == _native.SA_EUNSUPPORTED


def test_fused_zero_bias_is_no_bias(bsr):
    # an all-zero key bias takes the no-bias path: the same output bit for bit
    # ("Add key bias to chunked Sol-Attn producers", "Contract")
    T, H, Nv = 64 * 20 + 30, 2, 64 * 18
    base = make_inputs(T=T, H=H, video_tokens=Nv, qk_kind="walk1d", seed=78)
    r0, _ = both_paths(bsr, dict(base, bias=None), T, H, Nv, 0.25, 1, "dense")
    r1, _ = both_paths(bsr, dict(base, bias=np.zeros(T, np.float32)), T, H, Nv, 0.25, 1, "dense")
    assert r0["status"] == 0 and r1["status"] == 0
    assert torch.equal(r0["o1"], r1["o1"]) and torch.equal(r0["o2"], r1["o2"])
