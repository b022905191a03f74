"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle.

Same seeded inputs on both sides.  Block lists bit-exact (near-tie rule in
tests/parity.py); centroids within the FP32 summation bound; outputs within
max-abs 2e-2 and mean-abs 2e-3.  The five workloads run at full size in the
launch configuration the benchmark times (plan + fwd on one stream), and
every output value (row, head, dim) is compared with the oracle's, which a
spawned process pool evaluates head by head; only the rows of a query block
whose list is a near-tie variant of the oracle's are left out.  Edge cases
run small and are compared on every row.
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


def run_gpu(bsr, arrays, T, H, Nv, ratio, R, mode, want_scores=True):
    P = bsr.Params(T=T, H=H, video_tokens=Nv, topk_ratio=ratio, radius=R, tail_mode=mode)
    sz = bsr.sparse_attn_query(P)
    q, k, v = (to_dev(arrays[n], T, H) for n in "qkv")
    bias = None if arrays["bias"] is None else torch.from_numpy(arrays["bias"]).cuda()
    ws_plan = torch.empty(sz.plan_ws_bytes, dtype=torch.uint8, device="cuda")
    ws_fwd = torch.empty(sz.fwd_ws_bytes, dtype=torch.uint8, device="cuda")
    rs = torch.empty(H, sz.nq, sz.nvk, dtype=torch.float32, device="cuda") if want_scores else None
    idx, cnt = bsr.sparse_attn_plan(P, q, k, route_scores=rs, ws=ws_plan)
    o = bsr.sparse_attn_fwd(P, q, k, v, idx, cnt, key_bias=bias, ws=ws_fwd)
    status = bsr.sparse_attn_last_device_status(ws_fwd)
    torch.cuda.synchronize()
    qc_bytes = H * sz.nq * 128 * 4
    off_kc = 256 + ((qc_bytes + 255) // 256) * 256
    wsb = ws_plan.cpu().numpy()
    Qc = wsb[256:256 + qc_bytes].view(np.float32).reshape(H, sz.nq, 128)
    Kc = wsb[off_kc:off_kc + H * sz.nvk * 512].view(np.float32).reshape(H, sz.nvk, 128)
    return {
        "status": status,
        "idx": idx.cpu().numpy().reshape(H, sz.nq, sz.maxl),
        "cnt": cnt.cpu().numpy().reshape(H, sz.nq),
        "scores": rs.cpu().numpy() if want_scores else None,
        "Qc": Qc,
        "Kc": Kc,
        "o": parity.bf16_tensor_to_f64(o.reshape(T, H, 128)),
        "o_dev": o,
    }


def check_centroids(gpu, ref, arrays, sz):
    # FP32 sum of n values then one division: |err| <= (n + 1) u sum|x| / n
    u = 2.0 ** -24
    for name, bits, n_of in (("Qc", arrays["q"], None), ("Kc", arrays["k"], None)):
        g, r = gpu[name], ref[name]
        assert g.shape == r.shape
        mag = np.abs(r).max() + 1.0
        assert np.abs(g - r).max() <= 66 * u * mag * 4, name


def check_lists(gpu, ref, sz):
    n_exact, n_tie, bad = parity.compare_lists(gpu["idx"], gpu["cnt"], ref, sz)
    assert not bad, bad[:5]
    return n_exact, n_tie


def check_outputs_full(gpu, ref_o, sz, same):
    # rows whose block list matched the oracle exactly (all of them, normally)
    keep = np.ones((sz.T, sz.H), dtype=bool)
    for h in range(sz.H):
        for i in range(sz.nq):
            if not same[h, i]:
                r = O.oracle.query_block_rows(i, sz)
                keep[r.start:r.stop, h] = False
    d = np.abs(gpu["o"] - ref_o)[keep]
    assert d.max() <= parity.OUT_MAX_ABS, d.max()
    assert d.mean() <= parity.OUT_MEAN_ABS, d.mean()
    return float(d.max()), float(d.mean())


@pytest.mark.parametrize("name", ["tiny", "8k", "h3", "32k", "64k"])
def test_workload_parity(bsr, pool, name):
    w = WORKLOADS[name]
    arrays, prm = make_workload(name)
    sz = O.derive_sizes(w.T, w.H, w.video_tokens, w.topk_ratio, w.radius, w.tail_mode)
    gpu = run_gpu(bsr, arrays, w.T, w.H, w.video_tokens, w.topk_ratio, w.radius, w.tail_mode)
    assert gpu["status"] == 0
    ref = O.plan(arrays["q"], arrays["k"], sz)
    check_centroids(gpu, ref, arrays, sz)
    # FP32 dot product of FP32 means: |err| <= ~(128 + 66) u |Qc| |Kc| / sqrt(128)
    qn = np.linalg.norm(ref["Qc"], axis=-1)[:, :, None]
    kn = np.linalg.norm(ref["Kc"], axis=-1)[:, None, :]
    band = 2e-5 * qn * kn / np.sqrt(128) + 1e-6
    assert (np.abs(gpu["scores"] - ref["scores"]) <= band).all()
    n_exact, n_tie = check_lists(gpu, ref, sz)
    assert n_tie <= max(2, (n_exact + n_tie) // 1000)
    same = parity.same_list_mask(gpu["idx"], gpu["cnt"], ref)
    # every output value against the oracle (all rows, all heads)
    o_ref = parity.oracle_all_heads(pool, "exact", arrays, prm, ref["idx"], ref["cnt"])
    dmax, dmean, n = parity.compare_all(gpu["o"], o_ref, same, sz)
    print(f"[parity] {name}: {n} values, max-abs {dmax:.3e}, mean-abs {dmean:.3e}, "
          f"lists exact {n_exact}, near-tie {n_tie}")
    assert n >= 0.99 * sz.T * sz.H * 128
    assert dmax <= parity.OUT_MAX_ABS, dmax
    assert dmean <= parity.OUT_MEAN_ABS, dmean


EDGE = [
    # T, H, Nv, ratio, R, mode, qk_kind, bias kind
    dict(T=1152, H=1, Nv=1024, ratio=0.25, R=0, mode="dense", kind="iid", bias="none"),
    dict(T=1000, H=3, Nv=900, ratio=0.3, R=1, mode="dense", kind="walk1d", bias="sink_normal"),
    dict(T=1000, H=3, Nv=900, ratio=0.3, R=1, mode="pad", kind="walk1d", bias="sink_normal"),
    dict(T=1350, H=2, Nv=1350, ratio=0.2, R=2, mode="dense", kind="walk1d", bias="none"),  # no context
    dict(T=1344, H=2, Nv=1344, ratio=0.2, R=0, mode="pad", kind="iid", bias="none"),  # Nv = T, no tail
    dict(T=700, H=2, Nv=100, ratio=0.5, R=1, mode="dense", kind="iid", bias="sink_normal"),  # nvk = 1
    dict(T=777, H=2, Nv=640, ratio=1.0, R=0, mode="dense", kind="walk1d", bias="zero"),  # ratio 1
    dict(T=2000, H=5, Nv=1600, ratio=0.1, R=3, mode="pad", kind="walk1d", bias="none"),  # odd nq
    dict(T=4500, H=2, Nv=4160, ratio=0.15, R=1, mode="pad", kind="walk1d", bias="sink_normal"),
]


@pytest.mark.parametrize("case", range(len(EDGE)))
def test_edge_cases_full(bsr, case):
    c = EDGE[case]
    arrays = make_inputs(T=c["T"], H=c["H"], video_tokens=c["Nv"], qk_kind=c["kind"],
                         bias_kind=c["bias"], seed=1000 + case)
    sz = O.derive_sizes(c["T"], c["H"], c["Nv"], c["ratio"], c["R"], c["mode"])
    gpu = run_gpu(bsr, arrays, c["T"], c["H"], c["Nv"], c["ratio"], c["R"], c["mode"])
    assert gpu["status"] == 0
    ref = O.plan(arrays["q"], arrays["k"], sz)
    check_lists(gpu, ref, sz)
    ref_o = O.forward(arrays["q"], arrays["k"], arrays["v"], arrays["bias"], ref["idx"],
                      ref["cnt"], sz)
    check_outputs_full(gpu, ref_o, sz, parity.same_list_mask(gpu["idx"], gpu["cnt"], ref))


def test_ratio_one_is_dense_attention(bsr):
    T, H, Nv = 777, 2, 640
    arrays = make_inputs(T=T, H=H, video_tokens=Nv, qk_kind="iid", seed=77)
    gpu = run_gpu(bsr, arrays, T, H, Nv, 1.0, 0, "dense")
    qf, kf, vf = (torch.from_numpy(O.decode_bf16(arrays[n])).permute(1, 0, 2)[None] for n in "qkv")
    ref = torch.nn.functional.scaled_dot_product_attention(qf, kf, vf)[0].permute(1, 0, 2).numpy()
    d = np.abs(gpu["o"] - ref)
    assert d.max() <= parity.OUT_MAX_ABS and d.mean() <= parity.OUT_MEAN_ABS


def test_bias_semantics_on_gpu(bsr):
    T, H, Nv = 1000, 2, 900
    base = make_inputs(T=T, H=H, video_tokens=Nv, qk_kind="walk1d", seed=31)
    sz = O.derive_sizes(T, H, Nv, 0.3, 1, "dense")
    none = run_gpu(bsr, dict(base, bias=None), T, H, Nv, 0.3, 1, "dense")
    zero = run_gpu(bsr, dict(base, bias=np.zeros(T, np.float32)), T, H, Nv, 0.3, 1, "dense")
    assert np.array_equal(none["o"], zero["o"])  # zero bias is no bias, bit for bit
    # -inf on one sink block drops it from every row's softmax
    drop = sz.nvk + 1
    b = np.zeros(T, np.float32)
    b[64 * drop:64 * drop + 64] = -np.inf
    g = run_gpu(bsr, dict(base, bias=b), T, H, Nv, 0.3, 1, "dense")
    assert g["status"] == 0
    ref = O.plan(base["q"], base["k"], sz)
    ref_o = O.forward(base["q"], base["k"], base["v"], b, ref["idx"], ref["cnt"], sz)
    check_outputs_full(g, ref_o, sz, parity.same_list_mask(g["idx"], g["cnt"], ref))
    # nonzero bias on a routed video key, NaN and +inf: device-detected errors
    bad = np.zeros(T, np.float32)
    bad[5] = 0.25
    assert run_gpu(bsr, dict(base, bias=bad), T, H, Nv, 0.3, 1, "dense")["status"] == bsr.SA_ENOSINKBIAS
    for val in (np.nan, np.inf):
        bad = np.zeros(T, np.float32)
        bad[T - 3] = val
        assert run_gpu(bsr, dict(base, bias=bad), T, H, Nv, 0.3, 1, "dense")["status"] == bsr.SA_EINVAL
    # the status clears on the next good call with the same workspace
    assert run_gpu(bsr, dict(base, bias=None), T, H, Nv, 0.3, 1, "dense")["status"] == 0


def test_bias_routing_unchanged(bsr):
    T, H, Nv = 1000, 2, 900
    base = make_inputs(T=T, H=H, video_tokens=Nv, qk_kind="walk1d", bias_kind="sink_normal", seed=41)
    a = run_gpu(bsr, base, T, H, Nv, 0.3, 1, "dense")
    b = run_gpu(bsr, dict(base, bias=None), T, H, Nv, 0.3, 1, "dense")
    assert np.array_equal(a["idx"], b["idx"])
    assert np.abs(a["o"] - b["o"]).max() > 1e-3  # the bias changes the result


def test_deterministic(bsr):
    arrays, _ = make_workload("tiny")
    w = WORKLOADS["tiny"]
    a = run_gpu(bsr, arrays, w.T, w.H, w.video_tokens, w.topk_ratio, w.radius, w.tail_mode)
    b = run_gpu(bsr, arrays, w.T, w.H, w.video_tokens, w.topk_ratio, w.radius, w.tail_mode)
    assert np.array_equal(a["idx"], b["idx"]) and np.array_equal(a["o"], b["o"])


def test_longest_lists(bsr):
    # maxl = 1 + 1023 = 1024 (the largest supported width): one video block,
    # 1023 sink blocks; plus a ragged last block.
    T, H, Nv = 64 * 1023 + 40, 1, 64
    arrays = make_inputs(T=T, H=H, video_tokens=Nv, qk_kind="iid", seed=5)
    sz = O.derive_sizes(T, H, Nv, 1.0, 0, "dense")
    assert sz.maxl == 1024
    gpu = run_gpu(bsr, arrays, T, H, Nv, 1.0, 0, "dense")
    assert gpu["status"] == 0
    ref = O.plan(arrays["q"], arrays["k"], sz)
    check_lists(gpu, ref, sz)
    rows = [0, 31, 63, 64, 5000, T - 1]
    ref_o = O.forward_rows(arrays["q"], arrays["k"], arrays["v"], None, ref["idx"], ref["cnt"],
                           sz, rows, [0])
    d = np.abs(gpu["o"][rows][:, [0]] - ref_o)
    assert d.max() <= parity.OUT_MAX_ABS and d.mean() <= parity.OUT_MEAN_ABS


def test_many_video_blocks_route(bsr):
    # nvk = 3200 takes the 4-query-blocks-per-CTA routing variant.
    T, H, Nv = 64 * 3200, 1, 64 * 3200
    arrays = make_inputs(T=T, H=H, video_tokens=Nv, qk_kind="walk1d", seed=6)
    sz = O.derive_sizes(T, H, Nv, 0.01, 1, "dense")
    gpu = run_gpu(bsr, arrays, T, H, Nv, 0.01, 1, "dense")
    assert gpu["status"] == 0
    ref = O.plan(arrays["q"], arrays["k"], sz)
    check_lists(gpu, ref, sz)
    rows = [0, 64 * 1600 + 7, T - 1]
    same = parity.same_list_mask(gpu["idx"], gpu["cnt"], ref)
    rows = [t for t in rows if same[0, t // 64]]
    ref_o = O.forward_rows(arrays["q"], arrays["k"], arrays["v"], None, ref["idx"], ref["cnt"],
                           sz, rows, [0])
    d = np.abs(gpu["o"][rows][:, [0]] - ref_o)
    assert d.max() <= parity.OUT_MAX_ABS


# Video key-block counts whose last 128-key chunk is short, one per scoring
# tile: 32 query blocks per CTA with 30, 50 and 100 keys in the last chunk;
# 16 per CTA (nvk > 1024) with 20 and 76; 8 per CTA (nvk > 2048) with 50.
@pytest.mark.parametrize("nvk", [30, 50, 100, 1044, 1100, 2098])
def test_route_short_last_chunk(bsr, nvk):
    T, H, Nv = 64 * nvk + 40, 1, 64 * nvk
    arrays = make_inputs(T=T, H=H, video_tokens=Nv, qk_kind="walk1d", seed=nvk)
    ratio = 0.1 if nvk < 1000 else 0.02
    sz = O.derive_sizes(T, H, Nv, ratio, 1, "dense")
    gpu = run_gpu(bsr, arrays, T, H, Nv, ratio, 1, "dense")
    assert gpu["status"] == 0
    ref = O.plan(arrays["q"], arrays["k"], sz)
    qn = np.linalg.norm(ref["Qc"], axis=-1)[:, :, None]
    kn = np.linalg.norm(ref["Kc"], axis=-1)[:, None, :]
    band = 2e-5 * qn * kn / np.sqrt(128) + 1e-6
    assert (np.abs(gpu["scores"] - ref["scores"]) <= band).all()
    n_exact, n_tie = check_lists(gpu, ref, sz)
    assert n_tie <= max(2, (n_exact + n_tie) // 1000)
    if nvk <= 256:
        # the fused route sums each score in the same order: identical lists
        P = bsr.Params(T=T, H=H, video_tokens=Nv, topk_ratio=ratio, radius=1, tail_mode="dense")
        q, k, v = (to_dev(arrays[n], T, H) for n in "qkv")
        _, fidx, fcnt = bsr.sparse_attn_fused(P, q, k, v)
        torch.cuda.synchronize()
        assert np.array_equal(fidx.cpu().numpy().reshape(gpu["idx"].shape), gpu["idx"])
        assert np.array_equal(fcnt.cpu().numpy().reshape(gpu["cnt"].shape), gpu["cnt"])
