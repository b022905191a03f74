"""The no-allocation routing entry point, sparse_attn_plan_static.

Some callers cannot give the library device scratch memory (a plugin whose
host application owns all device memory through its own pool allocator, or
code that must not call cudaMalloc because it synchronises the device).
sparse_attn_plan_static serves them with scratch in a fixed device array
inside the library.  Here it is called through the C ABI and checked against
sparse_attn_plan on the same inputs, on two calls in a row of different
sizes (the second one runs on the array the first one left behind), and a
problem too large for the array must be rejected before any launch.

This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes alone in a fresh process.
"""

import ctypes
import os

import numpy as np
import pytest

from workloads import WORKLOADS, make_workload

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def native():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from block_sparse_routed_gb300 import _native
    from block_sparse_routed_gb300.build import LIB_PATH, build

    if not os.path.exists(LIB_PATH):
        build()
    _native.load_library()
    return _native


def _params(native, w):
    return native.SaParams(native.SA_ABI_VERSION, 1, w.T, w.H, 128, w.video_tokens, w.radius,
                           0 if w.tail_mode == "dense" else 1, w.topk_ratio)


def _dev(bits, w):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).reshape(1, w.T, w.H, 128).cuda()


def _outputs(sz, w):
    idx = torch.full((1, w.H, sz.nq, sz.maxl), 7, dtype=torch.int32, device="cuda")
    cnt = torch.full((1, w.H, sz.nq), 7, dtype=torch.int32, device="cuda")
    rs = torch.full((w.H, sz.nq, sz.nvk), 7.0, dtype=torch.float32, device="cuda")
    return idx, cnt, rs


def test_plan_static_matches_plan_on_two_calls_in_a_row(native):
    stream = torch.cuda.current_stream().cuda_stream
    for name in ("h3", "tiny"):  # large first, then small over the leftovers
        w = WORKLOADS[name]
        arrays, _ = make_workload(name)
        p = _params(native, w)
        sz = native.sparse_attn_query(p)
        assert sz.plan_ws_bytes <= 32 * 1024 * 1024
        q, k = _dev(arrays["q"], w), _dev(arrays["k"], w)

        idx_a, cnt_a, rs_a = _outputs(sz, w)
        ws = torch.empty(sz.plan_ws_bytes, dtype=torch.uint8, device="cuda")
        st = native.sparse_attn_plan(p, q.data_ptr(), k.data_ptr(), idx_a.data_ptr(),
                                     cnt_a.data_ptr(), rs_a.data_ptr(), ws.data_ptr(), ws.numel(),
                                     stream)
        assert st == native.SA_OK

        idx_b, cnt_b, rs_b = _outputs(sz, w)
        st = native.sparse_attn_plan_static(p, q.data_ptr(), k.data_ptr(), idx_b.data_ptr(),
                                            cnt_b.data_ptr(), rs_b.data_ptr(), stream)
        assert st == native.SA_OK
        torch.cuda.synchronize()
        # same kernels on the same inputs: lists bit-exact, scores identical
        assert torch.equal(idx_a, idx_b) and torch.equal(cnt_a, cnt_b)
        assert torch.equal(rs_a, rs_b)


def test_plan_static_rejects_problems_larger_than_its_array(native):
    # plan workspace 64 heads x (2969 + 2968) blocks x 512 B ~ 194 MB > 32 MiB
    p = native.SaParams(native.SA_ABI_VERSION, 1, 190000, 64, 128, 190000, 1, 0, 0.01)
    sz = native.sparse_attn_query(p)
    assert sz.plan_ws_bytes > 32 * 1024 * 1024
    A = 1 << 20  # aligned placeholder addresses: rejected before any use
    st = native.sparse_attn_plan_static(p, A, A, A, A, 0, 0)
    assert st == native.SA_EUNSUPPORTED
    lib = native.load_library()
    assert lib.sparse_attn_plan_static(ctypes.byref(p), None, None, None, None, None, None) == \
        native.SA_EUNSUPPORTED
