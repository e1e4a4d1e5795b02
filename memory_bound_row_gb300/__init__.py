"""rowsoftmax for GB300: a fused row-wise softmax behind a C ABI, and the
row normalisations (RMSNorm, LayerNorm) on the same row engine.

The product is ``librowsoftmax.so`` (CUDA, sm_103a; see include/rowsoftmax.h).
This package holds its sources (``csrc/``), its build (``build.py``), the
ctypes binding (``_abi.py``, same names as the C entry points) and tensor
front ends (``softmax``, ``softmax_causal``, ``rmsnorm``, ``layernorm``,
``softmax_partial``, ``softmax_merge``, ``softmax_finish``, ``softmax_split``,
``softmax_vocab_parallel``) that only marshal torch tensors into the C calls
(the last one adds the exchange of the per-row pairs between the ranks of a
torch.distributed group).
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
    RS_RING_THREAD_COPIES,
    rowsoftmax_causal_fwd,
    rowsoftmax_causal_fwd_ex,
    rowsoftmax_causal_plan,
    rowsoftmax_device_info,
    rowsoftmax_finish_fwd,
    rowsoftmax_merge_ml,
    rowsoftmax_partial_fwd,
    rowsoftmax_split_fwd,
    rowsoftmax_split_workspace_size,
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


def _pairs_out(ml, M: int, device):
    import torch

    if ml is None:
        return torch.empty((M, 2), dtype=torch.float32, device=device)
    if ml.dtype != torch.float32 or ml.shape != (M, 2) or not ml.is_contiguous():
        raise ValueError("pairs must be a contiguous float32 tensor of shape (M, 2)")
    return ml


def _pairs_in(pairs, M: int) -> tuple[int, int]:
    """(pointer, R) of a contiguous float32 pair tensor of shape (R, M, 2) or (M, 2)."""
    import torch

    if pairs.dtype != torch.float32 or not pairs.is_contiguous():
        raise ValueError("pairs must be a contiguous float32 tensor")
    if pairs.dim() == 2 and pairs.shape == (M, 2):
        return pairs.data_ptr(), 1
    if pairs.dim() == 3 and pairs.shape[1:] == (M, 2):
        return pairs.data_ptr(), int(pairs.shape[0])
    raise ValueError(f"pairs must have shape (R, {M}, 2) or ({M}, 2)")


def softmax_partial(x, ml=None, stream=None):
    """The pair (m, l) of every row of the 2-D CUDA tensor ``x`` (one column
    shard of the rows): m the row max, l the sum of exp(x - m).  Returns a
    float32 tensor of shape (M, 2) (``ml`` if given)."""
    if x.dim() != 2:
        raise ValueError("expected a 2-D tensor")
    M, N = x.shape
    if M and N and x.stride(1) != 1:
        raise ValueError("expected a unit column stride")
    ml = _pairs_out(ml, M, x.device)
    ldi = x.stride(0) if M > 1 else max(N, 1)
    _check(rowsoftmax_partial_fwd(x.data_ptr() if N else None, ml.data_ptr(), M, N, ldi, dtype_code(x.dtype),
                                  _stream_handle(x, stream)))
    return ml


def softmax_merge(pairs, out=None, stream=None):
    """Merge of the (R, M, 2) pairs of R shards into (M, 2)."""
    if pairs.dim() != 3 or pairs.shape[2] != 2:
        raise ValueError("pairs must have shape (R, M, 2)")
    R, M = int(pairs.shape[0]), int(pairs.shape[1])
    out = _pairs_out(out, M, pairs.device)
    ptr, _ = _pairs_in(pairs, M)
    _check(rowsoftmax_merge_ml(ptr if R else None, out.data_ptr(), R, M, _stream_handle(pairs, stream)))
    return out


def softmax_finish(x, pairs, out=None, stream=None):
    """exp(x - m) / l over the rows of the 2-D CUDA tensor ``x`` (one column
    shard), with (m, l) the merge of each row's pairs: ``pairs`` of shape
    (R, M, 2) (all shards' pairs, shard-major) or (M, 2) (already merged)."""
    out, M, N, ldi, ldo = _rows_args(x, out)
    ptr, R = _pairs_in(pairs, M)
    _check(rowsoftmax_finish_fwd(x.data_ptr(), out.data_ptr(), ptr, R, M, N, ldi, ldo, dtype_code(x.dtype),
                                 _stream_handle(x, stream)))
    return out


def softmax_split(x, out=None, workspace=None, stream=None):
    """Row softmax of ``x`` computed by splitting each row into column blocks
    over the whole device (rowsoftmax_split_fwd): for a few very wide rows.
    ``workspace`` (a CUDA tensor of at least rowsoftmax_split_workspace_size
    bytes) is allocated by torch when not given."""
    import torch

    out, M, N, ldi, ldo = _rows_args(x, out)
    code = dtype_code(x.dtype)
    rc, need = rowsoftmax_split_workspace_size(M, N, code)
    _check(rc)
    if workspace is None:
        workspace = torch.empty(max(need, 8), dtype=torch.uint8, device=x.device)
    nbytes = workspace.numel() * workspace.element_size()
    _check(rowsoftmax_split_fwd(x.data_ptr(), out.data_ptr(), M, N, ldi, ldo, code, workspace.data_ptr(), nbytes,
                                _stream_handle(x, stream)))
    return out


def exchange_pairs(ml, group=None):
    """All-gather of every rank's (M, 2) pairs into an (R, M, 2) tensor,
    shard-major in rank order (torch.distributed; the tensor stays on its
    device, and is staged through the host for a gloo group)."""
    import torch
    import torch.distributed as dist

    R = dist.get_world_size(group)
    staged = ml
    if dist.get_backend(group) == "gloo" and ml.is_cuda:
        staged = ml.cpu()
    staged = staged.contiguous()
    gathered = torch.empty((R * staged.shape[0],) + tuple(staged.shape[1:]), dtype=staged.dtype,
                           device=staged.device)
    dist.all_gather_into_tensor(gathered, staged, group=group)  # rank order along dim 0
    return gathered.view((R,) + tuple(staged.shape)).to(ml.device)


def softmax_vocab_parallel(x_shard, group=None, out=None, stream=None):
    """Row softmax of rows whose columns are split over the ranks of
    ``group``: this rank holds ``x_shard`` (M rows, its block of columns).
    One pair per row is computed here, the pairs of all ranks are exchanged
    (an all-gather of M x 8 bytes a rank), and this rank's block of the
    result is written.  Every rank must call it with the same M."""
    ml = softmax_partial(x_shard, stream=stream)
    return softmax_finish(x_shard, exchange_pairs(ml, group), out=out, stream=stream)
