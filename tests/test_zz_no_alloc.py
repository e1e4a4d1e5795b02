"""GPU test of rowsoftmax_split_fwd_noalloc, the split-row softmax for callers
that cannot allocate device memory (a serving loop whose device memory is
owned by another allocator, or a latency-critical path where cudaMalloc is not
allowed).  It keeps its pairs in a fixed device buffer of the library instead
of a caller's workspace.  Through the C ABI, two calls in a row, each against
rowsoftmax_split_fwd (the same computation with a caller's workspace) under
the row softmax tolerances.  This file is collected last, so that a run that
stops at its first failure has run every other test first."""
import ctypes

import pytest
import torch

import memory_bound_row_gb300 as rs
from memory_bound_row_gb300 import _abi, build
from memory_bound_row_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-6, torch.float16: 4e-3, torch.bfloat16: 4e-3}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    _abi.load()


def _noalloc(x, y):
    M, N = x.shape
    ld_in = x.stride(0) if M > 1 else N
    ld_out = y.stride(0) if M > 1 else N
    return _abi.rowsoftmax_split_fwd_noalloc(x.data_ptr(), y.data_ptr(), M, N, ld_in, ld_out, rs.dtype_code(x.dtype),
                                             torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("M,N,dtype", [(1, 3000000, "f32"), (4, 500000, "f16"), (16, 100000, "bf16"),
                                       (3, 70001, "f32")])
def test_two_calls_in_a_row_match_the_workspace_entry_point(M, N, dtype):
    x = W.generate(W.custom(M, N, dtype, seed=M + N, kind="normal_spike"), "cuda")
    rc, need = rs.rowsoftmax_split_workspace_size(M, N, rs.dtype_code(x.dtype))
    assert rc == rs.RS_OK and 0 < need <= _abi.RS_SPLIT_NOALLOC_MAX_BYTES
    ref = rs.softmax_split(x)
    torch.cuda.synchronize()
    for call in range(2):
        y = torch.full_like(x, float("nan"))
        assert _noalloc(x, y) == rs.RS_OK
        torch.cuda.synchronize()
        err = float((y.double() - ref.double()).abs().max())
        assert err <= TOL[x.dtype], f"call {call}: max |difference| {err:.3e}"
        assert bool(torch.isfinite(y).all())
    rc, flags = rs.rowsoftmax_device_status(clear=False)
    assert rc == rs.RS_OK and flags == 0


def test_problems_beyond_the_fixed_buffer_are_rejected():
    # 65537 rows need 16 bytes a row more than the 1 MiB buffer holds: refused
    # before anything is launched, the output untouched
    x = torch.zeros((65537, 8), dtype=torch.float32, device="cuda")
    y = torch.full_like(x, 3.0)
    rc, need = rs.rowsoftmax_split_workspace_size(65537, 8, rs.RS_F32)
    assert rc == rs.RS_OK and need > _abi.RS_SPLIT_NOALLOC_MAX_BYTES
    assert _noalloc(x, y) == rs.RS_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert bool((y == 3.0).all())
    # the largest row count that fits is served
    x2 = W.generate(W.custom(65536, 8, "f32", seed=5), "cuda")
    y2 = torch.empty_like(x2)
    assert _noalloc(x2, y2) == rs.RS_OK
    torch.cuda.synchronize()
    assert float((y2.double() - torch.softmax(x2.double(), dim=1)).abs().max()) <= 1e-6
