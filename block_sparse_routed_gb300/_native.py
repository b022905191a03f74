"""ctypes binding of the C ABI in include/sparse_attn.h.

Same entry-point names as the C library; this module only marshals
arguments.  Loading fails loudly when the library has not been built: there
is no other implementation to fall back on.
"""

from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

SA_ABI_VERSION = 1

SA_OK = 0
SA_EINVAL = 1
SA_EUNSUPPORTED = 2
SA_ENOSINKBIAS = 3
SA_ECUDA = 4
SA_ETIMEOUT = 5

SA_TAIL_DENSE = 0
SA_TAIL_PAD = 1

ENTRY_POINTS = (
    "sparse_attn_query",
    "sparse_attn_plan",
    "sparse_attn_plan_static",
    "sparse_attn_fwd",
    "sparse_attn_spark_reweight",
    "sparse_attn_spark_ws_bytes",
    "sparse_attn_spark_fwd",
    "sparse_attn_fused_ws_bytes",
    "sparse_attn_fused",
    "sparse_attn_reblock_ws_bytes",
    "sparse_attn_spark_reblock",
    "sparse_attn_last_device_status",
    "sparse_attn_set_single_probe_waits",
    "sparse_attn_last_cuda_error",
    "sparse_attn_status_string",
)


class SaParams(ctypes.Structure):
    _fields_ = [
        ("abi_version", ctypes.c_uint32),
        ("B", ctypes.c_int32),
        ("T", ctypes.c_int32),
        ("H", ctypes.c_int32),
        ("D", ctypes.c_int32),
        ("video_tokens", ctypes.c_int32),
        ("radius", ctypes.c_int32),
        ("tail_mode", ctypes.c_int32),
        ("topk_ratio", ctypes.c_double),
    ]


class SaSizes(ctypes.Structure):
    _fields_ = [
        ("nvk", ctypes.c_int32),
        ("tail", ctypes.c_int32),
        ("nblk", ctypes.c_int32),
        ("nq", ctypes.c_int32),
        ("topk", ctypes.c_int32),
        ("nsink", ctypes.c_int32),
        ("maxl", ctypes.c_int32),
        ("dense_row_start", ctypes.c_int32),
        ("plan_ws_bytes", ctypes.c_uint64),
        ("fwd_ws_bytes", ctypes.c_uint64),
    ]


class SaReblockParams(ctypes.Structure):
    _fields_ = [
        ("abi_version", ctypes.c_uint32),
        ("T", ctypes.c_int32),
        ("H", ctypes.c_int32),
        ("D", ctypes.c_int32),
        ("fanout", ctypes.c_int32),
        ("landmarks", ctypes.c_int32),
        ("token_stride", ctypes.c_int64),
        ("head_stride", ctypes.c_int64),
    ]


class SaReweightParams(ctypes.Structure):
    _fields_ = [
        ("abi_version", ctypes.c_uint32),
        ("B", ctypes.c_int32),
        ("T", ctypes.c_int32),
        ("H", ctypes.c_int32),
        ("D", ctypes.c_int32),
        ("P", ctypes.c_int32),
    ]


class SparseAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = int(status)
        msg = f"{what}: {status_string(status)}"
        if self.status == SA_ECUDA:
            code, text = sparse_attn_last_cuda_error()
            msg += f" (CUDA error {code}: {text})"
        super().__init__(msg)


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library (once).  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"CUDA library not built ({path} missing): run "
            "`python -c 'import __graft_entry__ as g; g.build()'`"
        )
    lib = ctypes.CDLL(path)
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    P = ctypes.POINTER
    lib.sparse_attn_query.argtypes = [P(SaParams), P(SaSizes)]
    lib.sparse_attn_query.restype = ctypes.c_int
    lib.sparse_attn_plan.argtypes = [P(SaParams), vp, vp, vp, vp, vp, vp, sz, vp]
    lib.sparse_attn_plan.restype = ctypes.c_int
    lib.sparse_attn_plan_static.argtypes = [P(SaParams), vp, vp, vp, vp, vp, vp]
    lib.sparse_attn_plan_static.restype = ctypes.c_int
    lib.sparse_attn_fwd.argtypes = [P(SaParams), vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.sparse_attn_fwd.restype = ctypes.c_int
    lib.sparse_attn_last_device_status.argtypes = [vp, vp, P(ctypes.c_int)]
    lib.sparse_attn_last_device_status.restype = ctypes.c_int
    lib.sparse_attn_set_single_probe_waits.argtypes = [ctypes.c_int]
    lib.sparse_attn_set_single_probe_waits.restype = ctypes.c_int
    lib.sparse_attn_last_cuda_error.argtypes = [P(ctypes.c_char_p)]
    lib.sparse_attn_last_cuda_error.restype = ctypes.c_int
    lib.sparse_attn_spark_reweight.argtypes = [P(SaReweightParams), vp, vp, vp, vp, vp, vp, vp]
    lib.sparse_attn_spark_reweight.restype = ctypes.c_int
    lib.sparse_attn_spark_ws_bytes.argtypes = [P(SaParams), P(ctypes.c_uint64)]
    lib.sparse_attn_spark_ws_bytes.restype = ctypes.c_int
    lib.sparse_attn_spark_fwd.argtypes = [P(SaParams), vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.sparse_attn_spark_fwd.restype = ctypes.c_int
    lib.sparse_attn_fused_ws_bytes.argtypes = [P(SaParams), P(ctypes.c_uint64)]
    lib.sparse_attn_fused_ws_bytes.restype = ctypes.c_int
    lib.sparse_attn_fused.argtypes = [P(SaParams), vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.sparse_attn_fused.restype = ctypes.c_int
    lib.sparse_attn_reblock_ws_bytes.argtypes = [P(SaReblockParams), P(ctypes.c_uint64)]
    lib.sparse_attn_reblock_ws_bytes.restype = ctypes.c_int
    lib.sparse_attn_spark_reblock.argtypes = [P(SaReblockParams), vp, vp, vp, vp, sz, vp]
    lib.sparse_attn_spark_reblock.restype = ctypes.c_int
    lib.sparse_attn_status_string.argtypes = [ctypes.c_int]
    lib.sparse_attn_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load_library().sparse_attn_status_string(int(status)).decode()
    except RuntimeError:
        return f"status {status}"


def sparse_attn_query(params: SaParams) -> SaSizes:
    out = SaSizes()
    st = load_library().sparse_attn_query(ctypes.byref(params), ctypes.byref(out))
    if st != SA_OK:
        raise SparseAttnError(st, "sparse_attn_query")
    return out


def sparse_attn_plan(params, q, k, idx, cnt, route_scores, ws, ws_bytes, stream) -> int:
    """Raw call: device pointers as ints (0 for NULL).  Returns the status."""
    return load_library().sparse_attn_plan(
        ctypes.byref(params), q, k, idx, cnt, route_scores or None, ws, ws_bytes, stream or None
    )


def sparse_attn_plan_static(params, q, k, idx, cnt, route_scores, stream) -> int:
    """Raw call of the no-allocation routing entry point (scratch in a fixed
    device array inside the library).  Returns the status."""
    return load_library().sparse_attn_plan_static(
        ctypes.byref(params), q, k, idx, cnt, route_scores or None, stream or None
    )


def sparse_attn_fwd(params, q, k, v, key_bias, idx, cnt, o, ws, ws_bytes, stream) -> int:
    """Raw call: device pointers as ints (0 for NULL).  Returns the status."""
    return load_library().sparse_attn_fwd(
        ctypes.byref(params), q, k, v, key_bias or None, idx, cnt, o, ws, ws_bytes, stream or None
    )


def sparse_attn_spark_reweight(params, a, k, v, ak, av, lm, stream) -> int:
    """Raw call of the virtual-summary entry point.  Returns the status."""
    return load_library().sparse_attn_spark_reweight(ctypes.byref(params), a, k, v, ak, av, lm,
                                                     stream or None)


def sparse_attn_spark_ws_bytes(params) -> int:
    out = ctypes.c_uint64(0)
    st = load_library().sparse_attn_spark_ws_bytes(ctypes.byref(params), ctypes.byref(out))
    if st != SA_OK:
        raise SparseAttnError(st, "sparse_attn_spark_ws_bytes")
    return int(out.value)


def sparse_attn_spark_fwd(params, q, k, v, key_bias, idx, cnt, o, ws, ws_bytes, stream) -> int:
    """Raw call of the merged (Spark) forward.  Returns the status."""
    return load_library().sparse_attn_spark_fwd(
        ctypes.byref(params), q, k, v, key_bias or None, idx, cnt, o, ws, ws_bytes, stream or None
    )


def sparse_attn_fused_ws_bytes(params) -> int:
    out = ctypes.c_uint64(0)
    st = load_library().sparse_attn_fused_ws_bytes(ctypes.byref(params), ctypes.byref(out))
    if st != SA_OK:
        raise SparseAttnError(st, "sparse_attn_fused_ws_bytes")
    return int(out.value)


def sparse_attn_fused(params, q, k, v, key_bias, idx, cnt, o, ws, ws_bytes, stream) -> int:
    """Raw call of the fused (in-kernel routing) entry point.  Returns the status."""
    return load_library().sparse_attn_fused(
        ctypes.byref(params), q, k, v, key_bias or None, idx, cnt, o, ws, ws_bytes, stream or None
    )


def sparse_attn_reblock_ws_bytes(params) -> int:
    out = ctypes.c_uint64(0)
    st = load_library().sparse_attn_reblock_ws_bytes(ctypes.byref(params), ctypes.byref(out))
    if st != SA_OK:
        raise SparseAttnError(st, "sparse_attn_reblock_ws_bytes")
    return int(out.value)


def sparse_attn_spark_reblock(params, x, perm, inv, ws, ws_bytes, stream) -> int:
    """Raw call of the reblocking entry point.  Returns the status."""
    return load_library().sparse_attn_spark_reblock(ctypes.byref(params), x, perm, inv, ws, ws_bytes,
                                                    stream or None)


def sparse_attn_last_device_status(ws, stream) -> int:
    out = ctypes.c_int(0)
    st = load_library().sparse_attn_last_device_status(ws, stream or None, ctypes.byref(out))
    if st != SA_OK:
        raise SparseAttnError(st, "sparse_attn_last_device_status")
    return out.value


def sparse_attn_set_single_probe_waits(on: bool) -> int:
    """Testing hook: later attention launches use the kernel build whose
    pipeline waits are single probes (to exercise the timeout path).  Returns
    the previous setting."""
    return int(load_library().sparse_attn_set_single_probe_waits(1 if on else 0))


def sparse_attn_last_cuda_error():
    """(code, message) of the last CUDA error behind an SA_ECUDA on this thread."""
    msg = ctypes.c_char_p()
    code = load_library().sparse_attn_last_cuda_error(ctypes.byref(msg))
    return code, (msg.value or b"").decode()


def sparse_attn_status_string(status: int) -> str:
    return status_string(status)
