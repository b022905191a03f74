"""Top-K block-sparse routed attention for one GB300 (sm_103a).

Two calls, backed by hand-written CUDA kernels in a C-ABI library:

* ``sparse_attn_plan``: mean-pools Q and K over 64-token blocks, scores video
  query blocks against video key blocks, selects the Top-K key blocks per
  query block and writes sorted per-block lists (forced local blocks and
  context sink blocks included).
* ``sparse_attn_fwd``: exact softmax attention of each video query block over
  its list, dense attention for context rows (and a dense video tail), with
  an optional natural-log key bias on sink keys.
* ``spark_reweight``: Spark's per-block virtual summaries (softmax-weighted
  keys and values per anchor and 64-token block, and their log-mass).
* ``sparse_attn_spark_fwd`` / ``spark_attn``: Spark's merged attention: the
  exact lists plus one summary key per skipped video block, from a per-head
  anchor (the mean of the target-video queries).
* ``spark_reblock``: Spark's token reblocking, a per-head permutation of the
  tokens into 64-token blocks by a landmark tree, and its inverse.

This module marshals torch tensors to the C entry points of the same names.
PyTorch provides device memory and streams only; every step runs in the
library's kernels.  There is no CPU fallback.
"""

from __future__ import annotations

from dataclasses import dataclass

from . import _native
from ._native import (  # noqa: F401
    SA_EINVAL,
    SA_ENOSINKBIAS,
    SA_ETIMEOUT,
    SA_EUNSUPPORTED,
    SA_OK,
    SaParams,
    SaReblockParams,
    SaReweightParams,
    SaSizes,
    SparseAttnError,
    load_library,
    sparse_attn_status_string,
)

__all__ = [
    "Params",
    "SparseAttnError",
    "load_library",
    "sparse_attn",
    "sparse_attn_fwd",
    "sparse_attn_last_device_status",
    "sparse_attn_plan",
    "sparse_attn_query",
    "sparse_attn_status_string",
    "spark_attn",
    "sparse_attn_fused",
    "spark_reweight",
    "spark_reblock",
    "sparse_attn_spark_fwd",
]


@dataclass(frozen=True)
class Params:
    """Problem description (mirrors ``sa_params``)."""

    T: int
    H: int
    video_tokens: int
    topk_ratio: float
    radius: int = 1
    tail_mode: str = "dense"  # "dense" or "pad"
    B: int = 1
    D: int = 128

    def to_c(self) -> SaParams:
        modes = {"dense": _native.SA_TAIL_DENSE, "pad": _native.SA_TAIL_PAD}
        if self.tail_mode not in modes:
            raise ValueError("tail_mode must be 'dense' or 'pad'")
        return SaParams(
            _native.SA_ABI_VERSION,
            self.B,
            self.T,
            self.H,
            self.D,
            self.video_tokens,
            self.radius,
            modes[self.tail_mode],
            float(self.topk_ratio),
        )


def sparse_attn_query(params: Params) -> SaSizes:
    """Derived sizes and workspace bytes (host only)."""
    return _native.sparse_attn_query(params.to_c())


def _torch():
    import torch

    return torch


def _check_qkv(t, name, params):
    torch = _torch()
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    shape = tuple(t.shape)
    if shape not in ((params.B, params.T, params.H, params.D), (params.T, params.H, params.D)):
        raise ValueError(f"{name} must have shape [1, T, H, 128], got {shape}")


def _stream_handle(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _workspace(nbytes, device):
    torch = _torch()
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def sparse_attn_plan(params: Params, q, k, idx=None, cnt=None, route_scores=None, ws=None,
                     stream=None):
    """Block lists for (q, k).  Returns (idx int32 [1,H,nq,maxl], cnt int32 [1,H,nq]).

    Missing outputs and workspace are allocated with torch on q's device.
    Pass ``route_scores`` (float32 [H, nq, nvk]) to receive the scores.
    """
    torch = _torch()
    _check_qkv(q, "q", params)
    _check_qkv(k, "k", params)
    cp = params.to_c()
    sz = _native.sparse_attn_query(cp)
    dev = q.device
    if idx is None:
        idx = torch.empty((1, params.H, sz.nq, sz.maxl), dtype=torch.int32, device=dev)
    if cnt is None:
        cnt = torch.empty((1, params.H, sz.nq), dtype=torch.int32, device=dev)
    if ws is None:
        ws = _workspace(sz.plan_ws_bytes, dev)
    for t, n, want in ((idx, "idx", params.H * sz.nq * sz.maxl), (cnt, "cnt", params.H * sz.nq)):
        if t.dtype != torch.int32 or not t.is_contiguous() or t.numel() != want:
            raise ValueError(f"{n}: int32 contiguous tensor with {want} elements required")
    rs = 0
    if route_scores is not None:
        if route_scores.dtype != torch.float32 or route_scores.numel() != params.H * sz.nq * sz.nvk:
            raise ValueError("route_scores: float32 [H, nq, nvk] required")
        rs = route_scores.data_ptr()
    st = _native.sparse_attn_plan(cp, q.data_ptr(), k.data_ptr(), idx.data_ptr(), cnt.data_ptr(),
                                  rs, ws.data_ptr(), ws.numel(), _stream_handle(stream))
    if st != SA_OK:
        raise SparseAttnError(st, "sparse_attn_plan")
    return idx, cnt


def sparse_attn_fwd(params: Params, q, k, v, idx, cnt, key_bias=None, o=None, ws=None,
                    stream=None):
    """Attention output o (bf16, same shape as q).  The device status of the
    call is read with ``sparse_attn_last_device_status(ws)``."""
    torch = _torch()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check_qkv(t, n, params)
    cp = params.to_c()
    sz = _native.sparse_attn_query(cp)
    if key_bias is not None:
        # the bias carrier: packed contiguous float32 with exactly B*T elements
        if (key_bias.dtype != torch.float32 or not key_bias.is_contiguous()
                or key_bias.numel() != params.B * params.T or not key_bias.is_cuda):
            raise ValueError("key_bias must be a contiguous CUDA float32 tensor with B*T elements")
    if o is None:
        o = torch.empty_like(q)
    _check_qkv(o, "o", params)
    if ws is None:
        ws = _workspace(sz.fwd_ws_bytes, q.device)
    st = _native.sparse_attn_fwd(cp, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                 key_bias.data_ptr() if key_bias is not None else 0,
                                 idx.data_ptr(), cnt.data_ptr(), o.data_ptr(), ws.data_ptr(),
                                 ws.numel(), _stream_handle(stream))
    if st != SA_OK:
        raise SparseAttnError(st, "sparse_attn_fwd")
    return o


def sparse_attn_last_device_status(ws, stream=None) -> int:
    """Device status word of a workspace (synchronises the stream)."""
    return _native.sparse_attn_last_device_status(ws.data_ptr(), _stream_handle(stream))


def sparse_attn(params: Params, q, k, v, key_bias=None, check_status=True, stream=None):
    """plan + fwd in one call; raises on a device-detected error when
    ``check_status`` (which synchronises the stream)."""
    sz = _native.sparse_attn_query(params.to_c())
    ws = _workspace(max(sz.plan_ws_bytes, sz.fwd_ws_bytes), q.device)
    idx, cnt = sparse_attn_plan(params, q, k, ws=ws, stream=stream)
    o = sparse_attn_fwd(params, q, k, v, idx, cnt, key_bias=key_bias, ws=ws, stream=stream)
    if check_status:
        st = sparse_attn_last_device_status(ws, stream)
        if st != SA_OK:
            raise SparseAttnError(st, "sparse_attn (device)")
    return o


def spark_reweight(a, k, v, ak=None, av=None, lm=None, stream=None):
    """Spark virtual summaries of every (anchor, head, 64-token block).

    a: bf16 [1, P, H, 128] anchors; k, v: bf16 [1, T, H, 128] (CUDA,
    contiguous).  Returns (ak, av) bf16 [1, P, H, ceil(T/64), 128] and
    lm float32 [1, P, H, ceil(T/64)], written by the library's kernel.
    """
    torch = _torch()
    for t, n in ((a, "a"), (k, "k"), (v, "v")):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{n} must be a contiguous 4-D CUDA bfloat16 tensor")
    _, P, H, D = a.shape
    B, T, Hk, Dk = k.shape
    if tuple(v.shape) != tuple(k.shape) or Hk != H or Dk != D or a.shape[0] != B:
        raise ValueError("a [1, P, H, 128], k and v [1, T, H, 128] required")
    nblk = (T + 63) // 64
    dev = k.device
    if ak is None:
        ak = torch.empty((B, P, H, nblk, D), dtype=torch.bfloat16, device=dev)
    if av is None:
        av = torch.empty((B, P, H, nblk, D), dtype=torch.bfloat16, device=dev)
    if lm is None:
        lm = torch.empty((B, P, H, nblk), dtype=torch.float32, device=dev)
    for t, n, dt, want in ((ak, "ak", torch.bfloat16, B * P * H * nblk * D),
                           (av, "av", torch.bfloat16, B * P * H * nblk * D),
                           (lm, "lm", torch.float32, B * P * H * nblk)):
        if t.dtype != dt or not t.is_contiguous() or t.numel() != want or not t.is_cuda:
            raise ValueError(f"{n}: contiguous CUDA {dt} tensor with {want} elements required")
    cp = SaReweightParams(_native.SA_ABI_VERSION, B, T, H, D, P)
    st = _native.sparse_attn_spark_reweight(cp, a.data_ptr(), k.data_ptr(), v.data_ptr(),
                                            ak.data_ptr(), av.data_ptr(), lm.data_ptr(),
                                            _stream_handle(stream))
    if st != SA_OK:
        raise SparseAttnError(st, "sparse_attn_spark_reweight")
    return ak, av, lm


def spark_reblock(x, fanout=8, landmarks=32, perm=None, inv=None, ws=None, stream=None):
    """Spark token reblocking of every head's tokens.

    x: CUDA bfloat16 samples [T, H, 128] or [1, T, H, 128] (any strides that
    are multiples of 8 elements, innermost dimension contiguous).  Returns
    perm, inv: int32 [H, T] (CUDA), written by the library's kernels:
    perm[h, i] is the original token at new position i, the blocks are
    perm[h, :64 * (T // 64)].view(-1, 64) and the excluded remainder is
    perm[h, 64 * (T // 64):]; inv[h, perm[h, i]] = i.
    """
    torch = _torch()
    if x.dim() == 4:
        if x.shape[0] != 1:
            raise ValueError("batch must be 1")
        x = x[0]
    if x.dim() != 3 or x.dtype != torch.bfloat16 or not x.is_cuda or x.shape[2] != 128 or x.stride(2) != 1:
        raise ValueError("x must be a CUDA bfloat16 [T, H, 128] tensor with a contiguous last dimension")
    T, H, D = x.shape
    rp = SaReblockParams(_native.SA_ABI_VERSION, T, H, D, fanout, landmarks, x.stride(0), x.stride(1))
    need = _native.sparse_attn_reblock_ws_bytes(rp)
    dev = x.device
    if perm is None:
        perm = torch.empty((H, T), dtype=torch.int32, device=dev)
    if inv is None:
        inv = torch.empty((H, T), dtype=torch.int32, device=dev)
    for t, n in ((perm, "perm"), (inv, "inv")):
        if t.dtype != torch.int32 or not t.is_contiguous() or t.numel() != H * T or not t.is_cuda:
            raise ValueError(f"{n}: contiguous CUDA int32 tensor with {H * T} elements required")
    if ws is None:
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    st = _native.sparse_attn_spark_reblock(rp, x.data_ptr(), perm.data_ptr(), inv.data_ptr(), ws.data_ptr(),
                                           ws.numel(), _stream_handle(stream))
    if st != SA_OK:
        raise SparseAttnError(st, "sparse_attn_spark_reblock")
    return perm, inv


def sparse_attn_spark_fwd(params: Params, q, k, v, idx, cnt, key_bias=None, o=None, ws=None,
                          stream=None):
    """Merged (Spark) attention output o (bf16, same shape as q): the lists'
    exact keys plus one summary key per skipped video block.  The device
    status is read with ``sparse_attn_last_device_status(ws)``."""
    torch = _torch()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check_qkv(t, n, params)
    cp = params.to_c()
    if key_bias is not None:
        if (key_bias.dtype != torch.float32 or not key_bias.is_contiguous()
                or key_bias.numel() != params.B * params.T or not key_bias.is_cuda):
            raise ValueError("key_bias must be a contiguous CUDA float32 tensor with B*T elements")
    if o is None:
        o = torch.empty_like(q)
    _check_qkv(o, "o", params)
    nbytes = _native.sparse_attn_spark_ws_bytes(cp)
    if ws is None:
        ws = _workspace(nbytes, q.device)
    st = _native.sparse_attn_spark_fwd(cp, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                       key_bias.data_ptr() if key_bias is not None else 0,
                                       idx.data_ptr(), cnt.data_ptr(), o.data_ptr(), ws.data_ptr(),
                                       ws.numel(), _stream_handle(stream))
    if st != SA_OK:
        raise SparseAttnError(st, "sparse_attn_spark_fwd")
    return o


def spark_attn(params: Params, q, k, v, key_bias=None, check_status=True, stream=None):
    """plan + merged forward in one call; raises on a device-detected error
    when ``check_status`` (which synchronises the stream)."""
    sz = _native.sparse_attn_query(params.to_c())
    nbytes = max(sz.plan_ws_bytes, _native.sparse_attn_spark_ws_bytes(params.to_c()))
    ws = _workspace(nbytes, q.device)
    idx, cnt = sparse_attn_plan(params, q, k, ws=ws, stream=stream)
    o = sparse_attn_spark_fwd(params, q, k, v, idx, cnt, key_bias=key_bias, ws=ws, stream=stream)
    if check_status:
        st = sparse_attn_last_device_status(ws, stream)
        if st != SA_OK:
            raise SparseAttnError(st, "spark_attn (device)")
    return o


def sparse_attn_fused(params: Params, q, k, v, key_bias=None, idx=None, cnt=None, o=None, ws=None,
                      stream=None):
    """Routing and attention in one call, the Top-K taken inside the
    attention kernel.  Returns (o, idx, cnt); the lists equal
    sparse_attn_plan's.  The device status is read with
    ``sparse_attn_last_device_status(ws)`` when ``ws`` is given."""
    torch = _torch()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check_qkv(t, n, params)
    cp = params.to_c()
    sz = _native.sparse_attn_query(cp)
    dev = q.device
    if key_bias is not None:
        if (key_bias.dtype != torch.float32 or not key_bias.is_contiguous()
                or key_bias.numel() != params.B * params.T or not key_bias.is_cuda):
            raise ValueError("key_bias must be a contiguous CUDA float32 tensor with B*T elements")
    if idx is None:
        idx = torch.empty((1, params.H, sz.nq, sz.maxl), dtype=torch.int32, device=dev)
    if cnt is None:
        cnt = torch.empty((1, params.H, sz.nq), dtype=torch.int32, device=dev)
    if o is None:
        o = torch.empty_like(q)
    _check_qkv(o, "o", params)
    for t, n, want in ((idx, "idx", params.H * sz.nq * sz.maxl), (cnt, "cnt", params.H * sz.nq)):
        if t.dtype != torch.int32 or not t.is_contiguous() or t.numel() != want:
            raise ValueError(f"{n}: int32 contiguous tensor with {want} elements required")
    nbytes = _native.sparse_attn_fused_ws_bytes(cp)
    if ws is None:
        ws = _workspace(nbytes, dev)
    st = _native.sparse_attn_fused(cp, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                   key_bias.data_ptr() if key_bias is not None else 0,
                                   idx.data_ptr(), cnt.data_ptr(), o.data_ptr(), ws.data_ptr(),
                                   ws.numel(), _stream_handle(stream))
    if st != SA_OK:
        raise SparseAttnError(st, "sparse_attn_fused")
    return o, idx, cnt
