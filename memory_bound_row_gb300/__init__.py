"""rowsoftmax for GB300: a fused row-wise softmax behind a C ABI.

The product is ``librowsoftmax.so`` (CUDA, sm_103a; see include/rowsoftmax.h).
This package holds its sources (``csrc/``), its build (``build.py``), the
ctypes binding (``_abi.py``, same names as the C entry points) and a tensor
front end (``softmax``) that only marshals torch tensors into the C call.
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
    RS_PATH_AUTO,
    RS_PATH_CLUSTER,
    RS_PATH_RING,
    RS_PATH_ROWS,
    RS_PATH_STREAM,
    RS_RING_AUTO,
    RS_RING_REGISTERS,
    RS_RING_REREAD,
    rowsoftmax_device_info,
    rowsoftmax_device_status,
    rowsoftmax_fwd,
    rowsoftmax_fwd_ex,
    rowsoftmax_last_cuda_error,
    rowsoftmax_layout_owner,
    rowsoftmax_plan,
    rowsoftmax_status_string,
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


def softmax(x, out=None, stream=None, options=None):
    """Row softmax of the 2-D CUDA tensor ``x`` (unit column stride) into
    ``out`` (allocated like ``x`` if not given; may be ``x`` itself for an
    in-place call).  Runs on ``stream`` (default: torch's current stream).
    ``options`` forces a kernel configuration (dict of rs_options fields)."""
    import torch

    if x.dim() != 2:
        raise ValueError("rowsoftmax expects a 2-D tensor")
    if out is None:
        out = torch.empty_like(x)
    if out.shape != x.shape or out.dtype != x.dtype:
        raise ValueError("out must have the shape and dtype of x")
    M, N = x.shape
    if M and N and (x.stride(1) != 1 or out.stride(1) != 1):
        raise ValueError("rowsoftmax expects a unit column stride")
    if stream is None:
        stream = torch.cuda.current_stream(x.device) if x.is_cuda else None
    s = 0 if stream is None else int(stream.cuda_stream)
    ldi = x.stride(0) if M > 1 else max(N, 1)
    ldo = out.stride(0) if M > 1 else max(N, 1)
    rc = rowsoftmax_fwd_ex(x.data_ptr(), out.data_ptr(), M, N, ldi, ldo, dtype_code(x.dtype), s, options)
    if rc != RS_OK:
        raise RowSoftmaxError(rc, rowsoftmax_last_cuda_error() if rc == RS_ERR_CUDA else 0)
    return out
