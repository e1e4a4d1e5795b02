"""rowsoftmax for GB300: a fused row-wise softmax behind a C ABI, and the
row normalisations (RMSNorm, LayerNorm) on the same row engine.

The product is ``librowsoftmax.so`` (CUDA, sm_103a; see include/rowsoftmax.h).
This package holds its sources (``csrc/``), its build (``build.py``), the
ctypes binding (``_abi.py``, same names as the C entry points) and tensor
front ends (``softmax``, ``softmax_causal``, ``rmsnorm``, ``layernorm``) that
only marshal torch tensors into the C calls.
"""
from __future__ import annotations

from ._abi import (  # noqa: F401
    PATH_NAMES,
    RS_BF16,
    RS_ERR_CUDA,
    RS_ERR_INVALID_ARG,
    RS_ERR_NO_PATH,
    RS_ERR_NOT_DEVICE_MEMORY,
    RS_ERR_OVERLAP,
    RS_ERR_UNSUPPORTED_DTYPE,
    RS_F16,
    RS_F32,
    RS_OK,
    RS_OP_LAYERNORM,
    RS_OP_RMSNORM,
    RS_OP_SOFTMAX,
    RS_PATH_AUTO,
    RS_PATH_CLUSTER,
    RS_PATH_RING,
    RS_PATH_ROWS,
    RS_PATH_STREAM,
    RS_RING_AUTO,
    RS_RING_REGISTERS,
    RS_RING_REREAD,
    rowsoftmax_causal_fwd,
    rowsoftmax_causal_fwd_ex,
    rowsoftmax_causal_plan,
    rowsoftmax_device_info,
    rowsoftmax_device_status,
    rowsoftmax_fwd,
    rowsoftmax_fwd_ex,
    rowsoftmax_last_cuda_error,
    rowsoftmax_layout_owner,
    rowsoftmax_plan,
    rowsoftmax_status_string,
    layernorm_fwd,
    rmsnorm_fwd,
    rownorm_fwd_ex,
    rownorm_plan,
    rs_device_info,
    rs_options,
    rs_plan,
)


class RowSoftmaxError(RuntimeError):
    def __init__(self, status: int, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        msg = rowsoftmax_status_string(status)
        if cuda_error:
            msg += f" (cudaError {cuda_error})"
        super().__init__(msg)


def dtype_code(torch_dtype) -> int:
    import torch

    codes = {torch.float32: RS_F32, torch.float16: RS_F16, torch.bfloat16: RS_BF16}
    if torch_dtype not in codes:
        raise TypeError(f"rowsoftmax supports float32, float16 and bfloat16, not {torch_dtype}")
    return codes[torch_dtype]


def _rows_args(x, out):
    """Shape checks of the 2-D row operations; returns (out, M, N, ldi, ldo)."""
    import torch

    if x.dim() != 2:
        raise ValueError("expected a 2-D tensor")
    if out is None:
        out = torch.empty_like(x)
    if out.shape != x.shape or out.dtype != x.dtype:
        raise ValueError("out must have the shape and dtype of x")
    M, N = x.shape
    if M and N and (x.stride(1) != 1 or out.stride(1) != 1):
        raise ValueError("expected a unit column stride")
    ldi = x.stride(0) if M > 1 else max(N, 1)
    ldo = out.stride(0) if M > 1 else max(N, 1)
    return out, M, N, ldi, ldo


def _stream_handle(x, stream) -> int:
    import torch

    if stream is None:
        stream = torch.cuda.current_stream(x.device) if x.is_cuda else None
    return 0 if stream is None else int(stream.cuda_stream)


def _check(rc: int):
    if rc != RS_OK:
        raise RowSoftmaxError(rc, rowsoftmax_last_cuda_error() if rc == RS_ERR_CUDA else 0)


def softmax(x, out=None, stream=None, options=None):
    """Row softmax of the 2-D CUDA tensor ``x`` (unit column stride) into
    ``out`` (allocated like ``x`` if not given; may be ``x`` itself for an
    in-place call).  Runs on ``stream`` (default: torch's current stream).
    ``options`` forces a kernel configuration (dict of rs_options fields)."""
    out, M, N, ldi, ldo = _rows_args(x, out)
    s = _stream_handle(x, stream)
    _check(rowsoftmax_fwd_ex(x.data_ptr(), out.data_ptr(), M, N, ldi, ldo, dtype_code(x.dtype), s, options))
    return out


def softmax_causal(x, period: int, diag_offset: int = 0, out=None, stream=None, options=None):
    """Row softmax under a causal mask: row r of the 2-D CUDA tensor ``x``
    keeps its first min(N, max(0, (r mod period) + 1 + diag_offset)) elements
    (the rest is never read and comes out as 0).  For attention scores
    [B, H, S_q, S_k] flattened to (B*H*S_q, S_k): period = S_q,
    diag_offset = S_k - S_q."""
    out, M, N, ldi, ldo = _rows_args(x, out)
    s = _stream_handle(x, stream)
    _check(rowsoftmax_causal_fwd_ex(x.data_ptr(), out.data_ptr(), M, N, ldi, ldo, int(period), int(diag_offset),
                                    dtype_code(x.dtype), s, options))
    return out


def _vector_ptr(v, x, what: str):
    """Device pointer of a per-column parameter vector (N values, x's dtype)."""
    if v is None:
        return None
    if v.dim() != 1 or v.shape[0] != x.shape[1] or v.dtype != x.dtype or (v.numel() > 1 and v.stride(0) != 1):
        raise ValueError(f"{what} must be a contiguous 1-D tensor of x.shape[1] values of x's dtype")
    return v.data_ptr() if v.numel() else None


def rmsnorm(x, weight=None, eps: float = 1e-6, out=None, stream=None, options=None):
    """RMSNorm of the rows of the 2-D CUDA tensor ``x``:
    y = x / sqrt(mean(x^2) + eps) * weight, computed in fp32, stored in x's
    dtype.  ``weight`` (optional) has x.shape[1] values of x's dtype."""
    out, M, N, ldi, ldo = _rows_args(x, out)
    s = _stream_handle(x, stream)
    w = _vector_ptr(weight, x, "weight")
    _check(rownorm_fwd_ex(RS_OP_RMSNORM, x.data_ptr(), out.data_ptr(), w, None, M, N, ldi, ldo, float(eps),
                          dtype_code(x.dtype), s, options))
    return out


def layernorm(x, weight=None, bias=None, eps: float = 1e-5, out=None, stream=None, options=None):
    """LayerNorm of the rows of the 2-D CUDA tensor ``x``:
    y = (x - mean) / sqrt(var + eps) * weight + bias (population variance),
    computed in fp32, stored in x's dtype."""
    out, M, N, ldi, ldo = _rows_args(x, out)
    s = _stream_handle(x, stream)
    w = _vector_ptr(weight, x, "weight")
    b = _vector_ptr(bias, x, "bias")
    _check(rownorm_fwd_ex(RS_OP_LAYERNORM, x.data_ptr(), out.data_ptr(), w, b, M, N, ldi, ldo, float(eps),
                          dtype_code(x.dtype), s, options))
    return out
