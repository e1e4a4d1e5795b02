"""ctypes binding of the C ABI in include/rowsoftmax.h.

Argument marshalling only: every function forwards to ``librowsoftmax.so``
under the same name, and all arithmetic runs in the library's CUDA kernels.
There is no fallback: if the library is missing, loading fails loudly.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "librowsoftmax.so")

# rs_dtype
RS_F32, RS_F16, RS_BF16 = 0, 1, 2
# rs_status
RS_OK = 0
RS_ERR_INVALID_ARG = 1
RS_ERR_UNSUPPORTED_DTYPE = 2
RS_ERR_OVERLAP = 3
RS_ERR_CUDA = 4
RS_ERR_NOT_DEVICE_MEMORY = 5
RS_ERR_NO_PATH = 6
# rs_path
RS_PATH_AUTO, RS_PATH_ROWS, RS_PATH_CLUSTER, RS_PATH_STREAM, RS_PATH_RING = 0, 1, 2, 3, 4
RS_RING_AUTO, RS_RING_REGISTERS, RS_RING_REREAD, RS_RING_THREAD_COPIES = 0, 1, 2, 3
# rs_op
RS_OP_SOFTMAX, RS_OP_RMSNORM, RS_OP_LAYERNORM = 0, 1, 2
PATH_NAMES = {RS_PATH_AUTO: "auto", RS_PATH_ROWS: "rows", RS_PATH_CLUSTER: "cluster", RS_PATH_STREAM: "stream",
              RS_PATH_RING: "ring"}

EXPORTED = (
    "rowsoftmax_fwd",
    "rowsoftmax_fwd_ex",
    "rowsoftmax_plan",
    "rowsoftmax_device_info",
    "rowsoftmax_status_string",
    "rowsoftmax_last_cuda_error",
    "rowsoftmax_device_status",
    "rowsoftmax_layout_owner",
    "rmsnorm_fwd",
    "layernorm_fwd",
    "rownorm_fwd_ex",
    "rownorm_plan",
    "rowsoftmax_causal_fwd",
    "rowsoftmax_causal_fwd_ex",
    "rowsoftmax_causal_plan",
    "rowsoftmax_partial_fwd",
    "rowsoftmax_merge_ml",
    "rowsoftmax_finish_fwd",
    "rowsoftmax_split_workspace_size",
    "rowsoftmax_split_fwd",
    "rowsoftmax_split_fwd_noalloc",
)


class rs_options(ctypes.Structure):
    _fields_ = [
        ("path", ctypes.c_int),
        ("threads_per_row", ctypes.c_int),
        ("vec_per_thread", ctypes.c_int),
        ("block_threads", ctypes.c_int),
        ("cluster_size", ctypes.c_int),
        ("stages", ctypes.c_int),
        ("ring_values", ctypes.c_int),
        ("force_scalar", ctypes.c_int),
        ("grid_limit", ctypes.c_int64),
        ("wait_limit_us", ctypes.c_int64),
        ("withhold_copies", ctypes.c_int),
        ("strict_order", ctypes.c_int),
    ]


class rs_plan(ctypes.Structure):
    _fields_ = [
        ("path", ctypes.c_int),
        ("dtype", ctypes.c_int),
        ("vec_elems", ctypes.c_int),
        ("threads_per_row", ctypes.c_int),
        ("vec_per_thread", ctypes.c_int),
        ("rows_per_cta", ctypes.c_int),
        ("block_threads", ctypes.c_int),
        ("cluster_size", ctypes.c_int),
        ("stages", ctypes.c_int),
        ("ring_values", ctypes.c_int),
        ("chunk_elems", ctypes.c_int64),
        ("grid", ctypes.c_int64),
        ("smem_bytes", ctypes.c_size_t),
        ("wait_limit_us", ctypes.c_int64),
        ("withhold_copies", ctypes.c_int),
        ("op", ctypes.c_int),
        ("strict_order", ctypes.c_int),
        ("masked", ctypes.c_int),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class rs_device_info(ctypes.Structure):
    _fields_ = [
        ("sm_count", ctypes.c_int),
        ("max_smem_per_block_optin", ctypes.c_int),
        ("max_smem_per_sm", ctypes.c_int),
        ("max_threads_per_sm", ctypes.c_int),
        ("cc_major", ctypes.c_int),
        ("cc_minor", ctypes.c_int),
    ]


_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    """Load librowsoftmax.so (built by ``memory_bound_row_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build the CUDA library first "
                "(python -m memory_bound_row_gb300.build)"
            )
        lib = ctypes.CDLL(LIB_PATH)
        i64, vp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        lib.rowsoftmax_fwd.argtypes = [vp, vp, i64, i64, i64, i64, ci, vp]
        lib.rowsoftmax_fwd.restype = ci
        lib.rowsoftmax_fwd_ex.argtypes = [vp, vp, i64, i64, i64, i64, ci, vp, ctypes.POINTER(rs_options)]
        lib.rowsoftmax_fwd_ex.restype = ci
        lib.rowsoftmax_plan.argtypes = [vp, vp, i64, i64, i64, i64, ci, ctypes.POINTER(rs_options),
                                        ctypes.POINTER(rs_device_info), ctypes.POINTER(rs_plan)]
        lib.rowsoftmax_plan.restype = ci
        lib.rowsoftmax_device_info.argtypes = [ctypes.POINTER(rs_device_info)]
        lib.rowsoftmax_device_info.restype = ci
        lib.rowsoftmax_status_string.argtypes = [ci]
        lib.rowsoftmax_status_string.restype = ctypes.c_char_p
        lib.rowsoftmax_last_cuda_error.argtypes = []
        lib.rowsoftmax_last_cuda_error.restype = ci
        lib.rowsoftmax_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint), ci]
        lib.rowsoftmax_device_status.restype = ci
        lib.rowsoftmax_layout_owner.argtypes = [i64, ci, ci, ctypes.POINTER(ci), ctypes.POINTER(i64)]
        lib.rowsoftmax_layout_owner.restype = ci
        f64 = ctypes.c_double
        lib.rmsnorm_fwd.argtypes = [vp, vp, vp, i64, i64, i64, i64, f64, ci, vp]
        lib.rmsnorm_fwd.restype = ci
        lib.layernorm_fwd.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, f64, ci, vp]
        lib.layernorm_fwd.restype = ci
        lib.rownorm_fwd_ex.argtypes = [ci, vp, vp, vp, vp, i64, i64, i64, i64, f64, ci, vp,
                                       ctypes.POINTER(rs_options)]
        lib.rownorm_fwd_ex.restype = ci
        lib.rownorm_plan.argtypes = [ci, vp, vp, vp, vp, i64, i64, i64, i64, f64, ci, ctypes.POINTER(rs_options),
                                     ctypes.POINTER(rs_device_info), ctypes.POINTER(rs_plan)]
        lib.rownorm_plan.restype = ci
        lib.rowsoftmax_causal_fwd.argtypes = [vp, vp, i64, i64, i64, i64, i64, i64, ci, vp]
        lib.rowsoftmax_causal_fwd.restype = ci
        lib.rowsoftmax_causal_fwd_ex.argtypes = [vp, vp, i64, i64, i64, i64, i64, i64, ci, vp,
                                                 ctypes.POINTER(rs_options)]
        lib.rowsoftmax_causal_fwd_ex.restype = ci
        lib.rowsoftmax_causal_plan.argtypes = [vp, vp, i64, i64, i64, i64, i64, i64, ci, ctypes.POINTER(rs_options),
                                               ctypes.POINTER(rs_device_info), ctypes.POINTER(rs_plan)]
        lib.rowsoftmax_causal_plan.restype = ci
        lib.rowsoftmax_partial_fwd.argtypes = [vp, vp, i64, i64, i64, ci, vp]
        lib.rowsoftmax_partial_fwd.restype = ci
        lib.rowsoftmax_merge_ml.argtypes = [vp, vp, i64, i64, vp]
        lib.rowsoftmax_merge_ml.restype = ci
        lib.rowsoftmax_finish_fwd.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, ci, vp]
        lib.rowsoftmax_finish_fwd.restype = ci
        lib.rowsoftmax_split_workspace_size.argtypes = [i64, i64, ci, ctypes.POINTER(ctypes.c_size_t)]
        lib.rowsoftmax_split_workspace_size.restype = ci
        lib.rowsoftmax_split_fwd.argtypes = [vp, vp, i64, i64, i64, i64, ci, vp, ctypes.c_size_t, vp]
        lib.rowsoftmax_split_fwd.restype = ci
        lib.rowsoftmax_split_fwd_noalloc.argtypes = [vp, vp, i64, i64, i64, i64, ci, vp]
        lib.rowsoftmax_split_fwd_noalloc.restype = ci
        _lib = lib
        return lib


def _opts(options) -> "ctypes._Pointer | None":
    if options is None:
        return None
    if isinstance(options, rs_options):
        return ctypes.pointer(options)
    o = rs_options()
    for k, v in dict(options).items():
        setattr(o, k, int(v))
    return ctypes.pointer(o)


# --- the C entry points, same names and argument order ----------------------

def rowsoftmax_fwd(in_ptr: int, out_ptr: int, M: int, N: int, in_row_stride: int, out_row_stride: int,
                   dtype: int, stream: int = 0) -> int:
    return load().rowsoftmax_fwd(in_ptr, out_ptr, M, N, in_row_stride, out_row_stride, dtype, stream)


def rowsoftmax_fwd_ex(in_ptr: int, out_ptr: int, M: int, N: int, in_row_stride: int, out_row_stride: int,
                      dtype: int, stream: int = 0, options=None) -> int:
    return load().rowsoftmax_fwd_ex(in_ptr, out_ptr, M, N, in_row_stride, out_row_stride, dtype, stream,
                                    _opts(options))


def rowsoftmax_plan(in_ptr: int, out_ptr: int, M: int, N: int, in_row_stride: int, out_row_stride: int,
                    dtype: int, options=None, device: rs_device_info | None = None) -> tuple[int, dict]:
    plan = rs_plan()
    dev = ctypes.pointer(device) if device is not None else None
    rc = load().rowsoftmax_plan(in_ptr, out_ptr, M, N, in_row_stride, out_row_stride, dtype, _opts(options), dev,
                                ctypes.byref(plan))
    return rc, plan.as_dict()


def rowsoftmax_device_info() -> tuple[int, rs_device_info]:
    info = rs_device_info()
    rc = load().rowsoftmax_device_info(ctypes.byref(info))
    return rc, info


def rowsoftmax_status_string(status: int) -> str:
    return load().rowsoftmax_status_string(status).decode()


def rowsoftmax_last_cuda_error() -> int:
    return load().rowsoftmax_last_cuda_error()


def rowsoftmax_device_status(clear: bool = False) -> tuple[int, int]:
    flags = ctypes.c_uint(0)
    rc = load().rowsoftmax_device_status(ctypes.byref(flags), 1 if clear else 0)
    return rc, flags.value


def rowsoftmax_layout_owner(j: int, threads: int, vec: int) -> tuple[int, int, int]:
    t = ctypes.c_int(0)
    s = ctypes.c_int64(0)
    rc = load().rowsoftmax_layout_owner(j, threads, vec, ctypes.byref(t), ctypes.byref(s))
    return rc, t.value, s.value


def rmsnorm_fwd(in_ptr: int, out_ptr: int, weight_ptr: int | None, M: int, N: int, in_row_stride: int,
                out_row_stride: int, eps: float, dtype: int, stream: int = 0) -> int:
    return load().rmsnorm_fwd(in_ptr, out_ptr, weight_ptr, M, N, in_row_stride, out_row_stride, eps, dtype, stream)


def layernorm_fwd(in_ptr: int, out_ptr: int, weight_ptr: int | None, bias_ptr: int | None, M: int, N: int,
                  in_row_stride: int, out_row_stride: int, eps: float, dtype: int, stream: int = 0) -> int:
    return load().layernorm_fwd(in_ptr, out_ptr, weight_ptr, bias_ptr, M, N, in_row_stride, out_row_stride, eps,
                                dtype, stream)


def rownorm_fwd_ex(op: int, in_ptr: int, out_ptr: int, weight_ptr: int | None, bias_ptr: int | None, M: int,
                   N: int, in_row_stride: int, out_row_stride: int, eps: float, dtype: int, stream: int = 0,
                   options=None) -> int:
    return load().rownorm_fwd_ex(op, in_ptr, out_ptr, weight_ptr, bias_ptr, M, N, in_row_stride, out_row_stride,
                                 eps, dtype, stream, _opts(options))


def rownorm_plan(op: int, in_ptr: int, out_ptr: int, weight_ptr: int | None, bias_ptr: int | None, M: int, N: int,
                 in_row_stride: int, out_row_stride: int, eps: float, dtype: int, options=None,
                 device: rs_device_info | None = None) -> tuple[int, dict]:
    plan = rs_plan()
    dev = ctypes.pointer(device) if device is not None else None
    rc = load().rownorm_plan(op, in_ptr, out_ptr, weight_ptr, bias_ptr, M, N, in_row_stride, out_row_stride, eps,
                             dtype, _opts(options), dev, ctypes.byref(plan))
    return rc, plan.as_dict()


def rowsoftmax_causal_fwd(in_ptr: int, out_ptr: int, M: int, N: int, in_row_stride: int, out_row_stride: int,
                          period: int, diag_offset: int, dtype: int, stream: int = 0) -> int:
    return load().rowsoftmax_causal_fwd(in_ptr, out_ptr, M, N, in_row_stride, out_row_stride, period, diag_offset,
                                        dtype, stream)


def rowsoftmax_causal_fwd_ex(in_ptr: int, out_ptr: int, M: int, N: int, in_row_stride: int, out_row_stride: int,
                             period: int, diag_offset: int, dtype: int, stream: int = 0, options=None) -> int:
    return load().rowsoftmax_causal_fwd_ex(in_ptr, out_ptr, M, N, in_row_stride, out_row_stride, period,
                                           diag_offset, dtype, stream, _opts(options))


def rowsoftmax_causal_plan(in_ptr: int, out_ptr: int, M: int, N: int, in_row_stride: int, out_row_stride: int,
                           period: int, diag_offset: int, dtype: int, options=None,
                           device: rs_device_info | None = None) -> tuple[int, dict]:
    plan = rs_plan()
    dev = ctypes.pointer(device) if device is not None else None
    rc = load().rowsoftmax_causal_plan(in_ptr, out_ptr, M, N, in_row_stride, out_row_stride, period, diag_offset,
                                       dtype, _opts(options), dev, ctypes.byref(plan))
    return rc, plan.as_dict()


def rowsoftmax_partial_fwd(in_ptr: int | None, ml_ptr: int, M: int, N: int, in_row_stride: int, dtype: int,
                           stream: int = 0) -> int:
    return load().rowsoftmax_partial_fwd(in_ptr, ml_ptr, M, N, in_row_stride, dtype, stream)


def rowsoftmax_merge_ml(ml_in_ptr: int | None, ml_out_ptr: int, R: int, M: int, stream: int = 0) -> int:
    return load().rowsoftmax_merge_ml(ml_in_ptr, ml_out_ptr, R, M, stream)


def rowsoftmax_finish_fwd(in_ptr: int, out_ptr: int, ml_ptr: int, R: int, M: int, N: int, in_row_stride: int,
                          out_row_stride: int, dtype: int, stream: int = 0) -> int:
    return load().rowsoftmax_finish_fwd(in_ptr, out_ptr, ml_ptr, R, M, N, in_row_stride, out_row_stride, dtype,
                                        stream)


def rowsoftmax_split_workspace_size(M: int, N: int, dtype: int) -> tuple[int, int]:
    n = ctypes.c_size_t(0)
    rc = load().rowsoftmax_split_workspace_size(M, N, dtype, ctypes.byref(n))
    return rc, n.value


def rowsoftmax_split_fwd(in_ptr: int, out_ptr: int, M: int, N: int, in_row_stride: int, out_row_stride: int,
                         dtype: int, workspace_ptr: int | None, workspace_bytes: int, stream: int = 0) -> int:
    return load().rowsoftmax_split_fwd(in_ptr, out_ptr, M, N, in_row_stride, out_row_stride, dtype, workspace_ptr,
                                       workspace_bytes, stream)


# Largest workspace rowsoftmax_split_fwd_noalloc serves (RS_SPLIT_NOALLOC_MAX_BYTES).
RS_SPLIT_NOALLOC_MAX_BYTES = 1 << 20


def rowsoftmax_split_fwd_noalloc(in_ptr: int, out_ptr: int, M: int, N: int, in_row_stride: int,
                                 out_row_stride: int, dtype: int, stream: int = 0) -> int:
    return load().rowsoftmax_split_fwd_noalloc(in_ptr, out_ptr, M, N, in_row_stride, out_row_stride, dtype,
                                               stream)
