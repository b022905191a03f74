"""Failure paths of the attention kernel, made on the host (no GPU fault).

* A bounded on-device wait that gives up: the testing hook
  sparse_attn_set_single_probe_waits(1) makes every pipeline wait a single
  probe, so the launch records SA_ETIMEOUT, drains its own copies and MMAs
  (those waits keep their 1 s limit), frees its tensor memory and returns.
  The next call with the normal limit must succeed and reproduce the output
  bit for bit ("Sol-Attn and Spark for MiniMax-H3", "Spark inference
  integration": kernel failures propagate to the caller).
* Caller block lists that break the list contract (an entry past the last
  block, an unsorted pair, a count above the list width or below one) are
  rejected on the device before any of their blocks is loaded: SA_EINVAL,
  then a clean call ("Add key bias to chunked Sol-Attn producers", "Tests and
  source audit": rejection before producer execution).
"""

import numpy as np
import pytest

import oracle as O
from tests import parity
from workloads import WORKLOADS, make_workload

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def setup():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import os

    from block_sparse_routed_gb300.build import LIB_PATH, build

    if not os.path.exists(LIB_PATH):
        build()
    import block_sparse_routed_gb300 as bsr
    from block_sparse_routed_gb300 import _native

    bsr.load_library()
    w = WORKLOADS["tiny"]
    arrays, _ = make_workload("tiny")
    P = bsr.Params(T=w.T, H=w.H, video_tokens=w.video_tokens, topk_ratio=w.topk_ratio, radius=w.radius,
                   tail_mode=w.tail_mode)
    dv = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).reshape(1, w.T, w.H, 128).cuda()
    q, k, v = (dv(arrays[n]) for n in "qkv")
    idx, cnt = bsr.sparse_attn_plan(P, q, k)
    sz = bsr.sparse_attn_query(P)
    ws = torch.zeros(sz.fwd_ws_bytes, dtype=torch.uint8, device="cuda")
    o_ref = bsr.sparse_attn_fwd(P, q, k, v, idx, cnt, ws=ws)
    assert bsr.sparse_attn_last_device_status(ws) == bsr.SA_OK
    return dict(bsr=bsr, native=_native, P=P, q=q, k=k, v=v, idx=idx, cnt=cnt, ws=ws, o_ref=o_ref.clone(),
                arrays=arrays, w=w, sz=sz)


def _fwd(s, idx=None, cnt=None):
    bsr = s["bsr"]
    o = torch.full_like(s["q"], 7.0)
    bsr.sparse_attn_fwd(s["P"], s["q"], s["k"], s["v"], s["idx"] if idx is None else idx,
                        s["cnt"] if cnt is None else cnt, o=o, ws=s["ws"])
    return o, bsr.sparse_attn_last_device_status(s["ws"])


def test_wait_timeout_is_reported_and_the_next_call_is_clean(setup):
    s = setup
    native = s["native"]
    prev = native.sparse_attn_set_single_probe_waits(True)
    try:
        statuses = []
        for _ in range(5):  # a single-probe launch almost surely gives up on its first wait
            _, st = _fwd(s)
            statuses.append(st)
            if st == s["bsr"].SA_ETIMEOUT:
                break
    finally:
        native.sparse_attn_set_single_probe_waits(bool(prev))
    assert s["bsr"].SA_ETIMEOUT in statuses, statuses
    torch.cuda.synchronize()
    # normal limit again: a clean call, the same output as before bit for bit
    for _ in range(3):
        o, st = _fwd(s)
        assert st == s["bsr"].SA_OK
        assert torch.equal(o, s["o_ref"])


def test_merged_and_fused_paths_time_out_cleanly_too(setup):
    s = setup
    bsr, native = s["bsr"], s["native"]
    wsm = torch.zeros(native.sparse_attn_spark_ws_bytes(s["P"].to_c()), dtype=torch.uint8, device="cuda")
    wsf = torch.zeros(native.sparse_attn_fused_ws_bytes(s["P"].to_c()), dtype=torch.uint8, device="cuda")
    om_ref = bsr.sparse_attn_spark_fwd(s["P"], s["q"], s["k"], s["v"], s["idx"], s["cnt"], ws=wsm).clone()
    of_ref, _, _ = bsr.sparse_attn_fused(s["P"], s["q"], s["k"], s["v"], ws=wsf)
    of_ref = of_ref.clone()
    assert bsr.sparse_attn_last_device_status(wsm) == 0 and bsr.sparse_attn_last_device_status(wsf) == 0
    prev = native.sparse_attn_set_single_probe_waits(True)
    try:
        seen_m = seen_f = False
        for _ in range(5):
            bsr.sparse_attn_spark_fwd(s["P"], s["q"], s["k"], s["v"], s["idx"], s["cnt"], ws=wsm)
            seen_m |= bsr.sparse_attn_last_device_status(wsm) == bsr.SA_ETIMEOUT
            bsr.sparse_attn_fused(s["P"], s["q"], s["k"], s["v"], ws=wsf)
            seen_f |= bsr.sparse_attn_last_device_status(wsf) == bsr.SA_ETIMEOUT
            if seen_m and seen_f:
                break
    finally:
        native.sparse_attn_set_single_probe_waits(bool(prev))
    assert seen_m and seen_f
    om = bsr.sparse_attn_spark_fwd(s["P"], s["q"], s["k"], s["v"], s["idx"], s["cnt"], ws=wsm)
    assert bsr.sparse_attn_last_device_status(wsm) == 0 and torch.equal(om, om_ref)
    of, _, _ = bsr.sparse_attn_fused(s["P"], s["q"], s["k"], s["v"], ws=wsf)
    assert bsr.sparse_attn_last_device_status(wsf) == 0 and torch.equal(of, of_ref)


def _corrupt_cases(s):
    sz = s["sz"]
    idx = s["idx"].cpu().numpy().reshape(s["w"].H, sz.nq, sz.maxl)
    cnt = s["cnt"].cpu().numpy().reshape(s["w"].H, sz.nq)
    cases = {}
    a = idx.copy()
    a[1, 5, cnt[1, 5] - 1] = sz.nblk  # an entry past the last block
    cases["entry >= nblk"] = (a, cnt)
    a = idx.copy()
    a[0, 3, 0], a[0, 3, 1] = a[0, 3, 1], a[0, 3, 0]  # an unsorted pair
    cases["unsorted"] = (a, cnt)
    a = idx.copy()
    a[0, 7, 2] = a[0, 7, 1]  # a repeated block
    cases["duplicate"] = (a, cnt)
    c = cnt.copy()
    c[1, 9] = sz.maxl + 1  # count above the list width
    cases["cnt > maxl"] = (idx, c)
    c = cnt.copy()
    c[0, 0] = 0  # an empty list (first block of a pair)
    cases["cnt < 1"] = (idx, c)
    c = cnt.copy()
    c[1, 3] = 0  # an empty list (second block of a pair)
    cases["cnt < 1, second"] = (idx, c)
    a = idx.copy()
    a[0, 2, 0] = -5  # a negative entry
    cases["negative"] = (a, cnt)
    return cases


@pytest.mark.parametrize("kind", ["entry >= nblk", "unsorted", "duplicate", "cnt > maxl", "cnt < 1", "cnt < 1, second",
                                  "negative"])
def test_bad_caller_lists_are_rejected_on_the_device(setup, kind):
    s = setup
    a, c = _corrupt_cases(s)[kind]
    idx = torch.from_numpy(np.ascontiguousarray(a)).reshape(s["idx"].shape).cuda()
    cnt = torch.from_numpy(np.ascontiguousarray(c)).reshape(s["cnt"].shape).cuda()
    _, st = _fwd(s, idx, cnt)
    assert st == s["bsr"].SA_EINVAL
    # the next valid call is clean and matches the oracle
    o, st = _fwd(s)
    assert st == s["bsr"].SA_OK and torch.equal(o, s["o_ref"])
    w, sz = s["w"], O.derive_sizes(s["w"].T, s["w"].H, s["w"].video_tokens, s["w"].topk_ratio, s["w"].radius,
                                    s["w"].tail_mode)
    ref = O.plan(s["arrays"]["q"], s["arrays"]["k"], sz)
    ro = O.forward(s["arrays"]["q"], s["arrays"]["k"], s["arrays"]["v"], None, ref["idx"], ref["cnt"], sz)
    d = np.abs(parity.bf16_tensor_to_f64(o.reshape(w.T, w.H, 128)) - ro)
    assert d.max() <= parity.OUT_MAX_ABS and d.mean() <= parity.OUT_MEAN_ABS
