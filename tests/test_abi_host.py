"""Host-side tests of the C-ABI library (no GPU needed).

The library is built in-tree when missing.  These tests load it, check that
every entry point declared in include/sparse_attn.h is exported, check the
derived sizes against the oracle's over many shapes, and check that every
argument error is reported before anything touches a device.
"""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sparse_attn.h")


@pytest.fixture(scope="module")
def native():
    from block_sparse_routed_gb300 import _native
    from block_sparse_routed_gb300.build import LIB_PATH, build

    if not os.path.exists(LIB_PATH):
        build()
    _native.load_library()
    return _native


def _declared_entry_points():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(sparse_attn_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared_entry_points()
    assert "sparse_attn_plan" in names and "sparse_attn_fwd" in names
    assert "sparse_attn_query" in names


def test_library_exports_every_declared_symbol(native):
    lib = native.load_library()
    for name in _declared_entry_points():
        assert hasattr(lib, name), name
    assert set(native.ENTRY_POINTS) >= set(_declared_entry_points())


def test_struct_layout_matches_header(native):
    # sa_params: 8 x 32-bit then a double; sa_sizes: 8 x int32 then 2 x uint64
    assert ctypes.sizeof(native.SaParams) == 40
    assert ctypes.sizeof(native.SaSizes) == 48
    txt = open(HEADER).read()
    assert "#define SA_ABI_VERSION 1u" in txt
    assert native.SA_ABI_VERSION == 1


def _params(native, T, H, Nv, r, R, mode, B=1, D=128, ver=None):
    return native.SaParams(native.SA_ABI_VERSION if ver is None else ver, B, T, H, D, Nv, R,
                           {"dense": 0, "pad": 1}.get(mode, mode), r)


def _query(native, *a, **k):
    out = native.SaSizes()
    st = native.load_library().sparse_attn_query(ctypes.byref(_params(native, *a, **k)),
                                                  ctypes.byref(out))
    return st, out


@pytest.mark.parametrize("name", ["tiny", "8k", "h3", "32k", "64k"])
def test_query_matches_oracle_on_workloads(native, name):
    from workloads import WORKLOADS

    w = WORKLOADS[name]
    st, out = _query(native, w.T, w.H, w.video_tokens, w.topk_ratio, w.radius, w.tail_mode)
    assert st == 0
    sz = O.derive_sizes(w.T, w.H, w.video_tokens, w.topk_ratio, w.radius, w.tail_mode)
    assert (out.nvk, out.tail, out.nblk, out.nq, out.topk, out.nsink, out.maxl,
            out.dense_row_start) == (sz.nvk, sz.tail, sz.nblk, sz.nq, sz.K, sz.nsink, sz.maxl,
                                     sz.dense_row_start)
    assert out.plan_ws_bytes >= 256 + 4 * w.H * 128 * (sz.nq + sz.nvk)
    assert out.fwd_ws_bytes >= 256 + 4 * w.T


def test_query_gate_parity_fuzz(native):
    """Accept/reject decisions and derived sizes agree with the oracle over
    thousands of random shapes (ratios written as short decimals)."""
    rng = np.random.default_rng(0)
    ratios = [0.01, 0.05, 0.1, 0.125, 0.2, 0.25, 0.3, 0.33, 0.5, 0.7, 0.9, 1.0, 0.0, 1.5, -0.1]
    checked = 0
    for _ in range(4000):
        T = int(rng.integers(1, 40000))
        Nv = int(rng.integers(0, T + 80))
        r = float(rng.choice(ratios))
        R = int(rng.integers(-1, 4))
        mode = "pad" if rng.random() < 0.5 else "dense"
        H = int(rng.integers(1, 8))
        st, out = _query(native, T, H, Nv, r, R, mode)
        try:
            sz = O.derive_sizes(T, H, Nv, r, R, mode)
        except ValueError:
            assert st == native.SA_EINVAL, (T, Nv, r, R, mode, st)
            continue
        if sz.maxl > 1024 or sz.nvk > 8192:
            assert st == native.SA_EUNSUPPORTED
            continue
        assert st == 0, (T, Nv, r, R, mode, st)
        assert (out.nvk, out.tail, out.nblk, out.nq, out.topk, out.nsink, out.maxl,
                out.dense_row_start) == (sz.nvk, sz.tail, sz.nblk, sz.nq, sz.K, sz.nsink,
                                         sz.maxl, sz.dense_row_start), (T, Nv, r, R, mode)
        checked += 1
    assert checked > 1000


def test_query_rejects_unsupported_and_invalid(native):
    E, U = native.SA_EINVAL, native.SA_EUNSUPPORTED
    assert _query(native, 1152, 2, 1024, 0.25, 0, "dense", B=2)[0] == U
    assert _query(native, 1152, 2, 1024, 0.25, 0, "dense", D=64)[0] == U
    assert _query(native, 1152, 2, 1024, 0.25, 0, "dense", ver=7)[0] == E
    assert _query(native, 1152, 2, 1024, float("nan"), 0, "dense")[0] == E
    assert _query(native, 1152, 2, 1024, 0.25, 0, 5)[0] == E
    assert _query(native, 1152, 0, 1024, 0.25, 0, "dense")[0] == E
    # 2^31 elements
    assert _query(native, 1 << 20, 16, 1 << 19, 0.001, 0, "dense")[0] == U
    lib = native.load_library()
    assert lib.sparse_attn_query(None, ctypes.byref(native.SaSizes())) == E
    p = _params(native, 1152, 2, 1024, 0.25, 0, "dense")
    assert lib.sparse_attn_query(ctypes.byref(p), None) == E


def test_plan_and_fwd_reject_bad_arguments_before_launch(native):
    """Every argument error returns before the device is touched (this host
    has no GPU; reaching the device would give SA_ECUDA instead)."""
    lib = native.load_library()
    p = _params(native, 1152, 2, 1024, 0.25, 0, "dense")
    sz = native.SaSizes()
    assert lib.sparse_attn_query(ctypes.byref(p), ctypes.byref(sz)) == 0
    A = 1 << 20  # a fake, aligned address: never dereferenced on these paths
    E = native.SA_EINVAL
    # null required pointers
    assert lib.sparse_attn_plan(ctypes.byref(p), None, A, A, A, None, A, sz.plan_ws_bytes, None) == E
    assert lib.sparse_attn_plan(ctypes.byref(p), A, A, A, None, None, A, sz.plan_ws_bytes, None) == E
    # misaligned q, short workspace
    assert lib.sparse_attn_plan(ctypes.byref(p), A + 2, A, A, A, None, A, sz.plan_ws_bytes, None) == E
    assert lib.sparse_attn_plan(ctypes.byref(p), A, A, A, A, None, A, sz.plan_ws_bytes - 1, None) == E
    assert lib.sparse_attn_fwd(ctypes.byref(p), A, A, A, None, A, A, None, A, sz.fwd_ws_bytes, None) == E
    assert lib.sparse_attn_fwd(ctypes.byref(p), A, A, A + 8, None, A, A, A, A, sz.fwd_ws_bytes, None) == E
    assert lib.sparse_attn_fwd(ctypes.byref(p), A, A, A, A + 2, A, A, A, A, sz.fwd_ws_bytes, None) == E
    assert lib.sparse_attn_fwd(ctypes.byref(p), A, A, A, None, A, A, A, A, 16, None) == E
    # the output is written with 32-byte stores: 16-byte alignment is not enough
    assert lib.sparse_attn_fwd(ctypes.byref(p), A, A, A, None, A, A, A + 16, A, sz.fwd_ws_bytes, None) == E
    big = 1 << 30  # past every workspace size these calls ask for
    assert lib.sparse_attn_spark_fwd(ctypes.byref(p), A, A, A, None, A, A, A + 16, A, big, None) == E
    assert lib.sparse_attn_fused(ctypes.byref(p), A, A, A, None, A, A, A + 16, A, big, None) == E
    bad = _params(native, 1152, 2, 1024, 0.25, -1, "dense")
    assert lib.sparse_attn_fwd(ctypes.byref(bad), A, A, A, None, A, A, A, A, 1 << 30, None) == E
    assert lib.sparse_attn_last_device_status(None, None, ctypes.byref(ctypes.c_int())) == E


def test_status_strings(native):
    for code in range(6):
        assert native.sparse_attn_status_string(code).startswith("SA_")
    assert "unknown" in native.sparse_attn_status_string(99)


def test_python_binding_checks_key_bias_before_the_call(native):
    torch = pytest.importorskip("torch")
    import block_sparse_routed_gb300 as bsr

    p = bsr.Params(T=1152, H=2, video_tokens=1024, topk_ratio=0.25, radius=0)
    with pytest.raises((ValueError, TypeError)):
        # CPU tensors are rejected before anything reaches the library
        bsr.sparse_attn_fwd(p, *(torch.zeros(1, 1152, 2, 128, dtype=torch.bfloat16),) * 3,
                            idx=None, cnt=None, key_bias=torch.zeros(1152))


def test_spark_reweight_rejects_bad_arguments_before_launch(native):
    """Argument errors of the virtual-summary entry point, all caught on the
    host (this host has no GPU: reaching the device would give SA_ECUDA or
    SA_EUNSUPPORTED from the device check instead)."""
    assert ctypes.sizeof(native.SaReweightParams) == 24
    lib = native.load_library()
    E, U = native.SA_EINVAL, native.SA_EUNSUPPORTED
    A = 1 << 20

    def call(p, a=A, k=A, v=A, ak=A, av=A, lm=A):
        return lib.sparse_attn_spark_reweight(ctypes.byref(p), a, k, v, ak, av, lm, None)

    def params(B=1, T=100, H=2, D=128, P=1, ver=None):
        return native.SaReweightParams(native.SA_ABI_VERSION if ver is None else ver, B, T, H, D, P)

    assert lib.sparse_attn_spark_reweight(None, A, A, A, A, A, A, None) == E
    assert call(params(ver=3)) == E
    assert call(params(B=2)) == U
    assert call(params(D=64)) == U
    assert call(params(T=0)) == E
    assert call(params(H=0)) == E
    assert call(params(P=0)) == E
    assert call(params(T=1 << 20, H=32)) == U   # 2^32 elements
    assert call(params(), a=None) == E
    assert call(params(), lm=None) == E
    assert call(params(), k=A + 8) == E
    assert call(params(), ak=A + 2) == E
    assert call(params(), lm=A + 2) == E


def test_reblock_rejects_bad_arguments_before_launch(native):
    """Argument errors of the reblocking entry point, all caught on the host."""
    assert ctypes.sizeof(native.SaReblockParams) == 40
    lib = native.load_library()
    E, U = native.SA_EINVAL, native.SA_EUNSUPPORTED
    A = 1 << 20

    def params(T=1000, H=2, D=128, f=8, L=32, ts=256, hs=128, ver=None):
        return native.SaReblockParams(native.SA_ABI_VERSION if ver is None else ver, T, H, D, f, L, ts, hs)

    def call(p, x=A, perm=A, inv=A, ws=A, nbytes=1 << 40):
        return lib.sparse_attn_spark_reblock(ctypes.byref(p), x, perm, inv, ws, nbytes, None)

    def ws_bytes(p):
        out = ctypes.c_uint64(0)
        return lib.sparse_attn_reblock_ws_bytes(ctypes.byref(p), ctypes.byref(out)), out.value

    assert lib.sparse_attn_spark_reblock(None, A, A, A, A, 1, None) == E
    assert call(params(ver=2)) == E
    assert call(params(D=64)) == U
    assert call(params(T=0)) == E
    assert call(params(H=0)) == E
    for f in (0, 1, 3, 6, 32):
        assert call(params(f=f)) == E
    for L in (0, 1, 65):
        assert call(params(L=L)) == E
    assert call(params(ts=100)) == E
    assert call(params(hs=-8)) == E
    assert call(params(H=70000)) == U
    assert call(params(T=1 << 26, H=64)) == U
    assert call(params(), x=None) == E
    assert call(params(), inv=None) == E
    assert call(params(), x=A + 8) == E
    assert call(params(), perm=A + 2) == E
    assert call(params(), ws=A + 128) == E
    st, need = ws_bytes(params())
    assert st == native.SA_OK and need > 0
    assert call(params(), nbytes=need - 1) == E
    # N = 64 floor(T / 64) = 960: FP16 rows, keys, two orders, landmark
    # pairs of the 15 blocks, each 256-byte aligned
    up = lambda b: (b + 255) // 256 * 256
    assert need == up(960 * 2 * 256) + up(960 * 2 * 8) + 2 * up(960 * 2 * 4) + up(15 * 2 * 8)
    assert ws_bytes(params(T=40)) == (native.SA_OK, 0)


def test_single_probe_hook_round_trips_on_the_host(native):
    # host-only setter: returns the previous setting, touches no device
    prev = native.sparse_attn_set_single_probe_waits(True)
    try:
        assert prev == 0  # off by default
        assert native.sparse_attn_set_single_probe_waits(False) == 1
    finally:
        native.sparse_attn_set_single_probe_waits(bool(prev))
    assert native.sparse_attn_set_single_probe_waits(False) == 0
