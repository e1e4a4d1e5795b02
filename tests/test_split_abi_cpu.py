"""CPU checks of the split-row entry points (rowsoftmax_partial_fwd,
rowsoftmax_merge_ml, rowsoftmax_finish_fwd, rowsoftmax_split_workspace_size,
rowsoftmax_split_fwd): bad arguments are rejected before any device call, and
the workspace size follows its stated formula.  No kernel runs."""
import pytest

import memory_bound_row_gb300 as rs
from memory_bound_row_gb300 import build

A = 1 << 20   # a 16-byte aligned fake address; validation fails before it is used
FAR = 1 << 30  # far enough from A that nothing overlaps


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


@pytest.mark.parametrize(
    "args,status",
    [
        ((A, A + FAR, 4, 8, 8, 7), rs.RS_ERR_UNSUPPORTED_DTYPE),
        ((A, A + FAR, -1, 8, 8, rs.RS_F32), rs.RS_ERR_INVALID_ARG),
        ((A, A + FAR, 4, -1, 8, rs.RS_F32), rs.RS_ERR_INVALID_ARG),
        ((0, A + FAR, 4, 8, 8, rs.RS_F32), rs.RS_ERR_INVALID_ARG),       # null input with columns
        ((A, 0, 4, 8, 8, rs.RS_F32), rs.RS_ERR_INVALID_ARG),             # null pairs
        ((A, A + FAR + 4, 4, 8, 8, rs.RS_F32), rs.RS_ERR_INVALID_ARG),   # pairs not 8-byte aligned
        ((A + 2, A + FAR, 4, 8, 8, rs.RS_F32), rs.RS_ERR_INVALID_ARG),   # input not element-aligned
        ((A, A + FAR, 4, 8, 7, rs.RS_F32), rs.RS_ERR_INVALID_ARG),       # stride < N
        ((A, A + 64, 4, 8, 8, rs.RS_F32), rs.RS_ERR_OVERLAP),            # pairs inside the input
        ((A, A + FAR, 2, 1 << 31, 1 << 31, rs.RS_F16), rs.RS_ERR_INVALID_ARG),
    ],
)
def test_partial_rejects_bad_arguments(args, status):
    assert rs.rowsoftmax_partial_fwd(*args, 0) == status


def test_partial_and_merge_empty_problems():
    assert rs.rowsoftmax_partial_fwd(A, A + FAR, 0, 8, 8, rs.RS_F32, 0) == rs.RS_OK
    assert rs.rowsoftmax_merge_ml(A, A + FAR, 3, 0, 0) == rs.RS_OK


@pytest.mark.parametrize(
    "args,status",
    [
        ((A, A + FAR, -1, 4), rs.RS_ERR_INVALID_ARG),
        ((A, A + FAR, 2, -4), rs.RS_ERR_INVALID_ARG),
        ((0, A + FAR, 2, 4), rs.RS_ERR_INVALID_ARG),
        ((A, 0, 2, 4), rs.RS_ERR_INVALID_ARG),
        ((A + 4, A + FAR, 2, 4), rs.RS_ERR_INVALID_ARG),
        ((A, A + 8, 2, 4), rs.RS_ERR_OVERLAP),
        ((A, A + FAR, 1 << 40, 1 << 40), rs.RS_ERR_INVALID_ARG),
    ],
)
def test_merge_rejects_bad_arguments(args, status):
    assert rs.rowsoftmax_merge_ml(*args, 0) == status


@pytest.mark.parametrize(
    "args,status",
    [
        ((A, A + FAR, 2 * FAR, 1, 4, 8, 8, 8, 7), rs.RS_ERR_UNSUPPORTED_DTYPE),
        ((A, A + FAR, 2 * FAR, 0, 4, 8, 8, 8, rs.RS_F32), rs.RS_ERR_INVALID_ARG),      # R < 1
        ((A, A + FAR, 0, 1, 4, 8, 8, 8, rs.RS_F32), rs.RS_ERR_INVALID_ARG),            # null pairs
        ((A, A + FAR, 2 * FAR + 4, 1, 4, 8, 8, 8, rs.RS_F32), rs.RS_ERR_INVALID_ARG),  # misaligned pairs
        ((A, A + FAR, 2 * FAR, 1, 4, 8, 7, 8, rs.RS_F32), rs.RS_ERR_INVALID_ARG),
        ((A, A + 64, 2 * FAR, 1, 4, 8, 8, 8, rs.RS_F32), rs.RS_ERR_OVERLAP),           # in/out overlap
        ((A, A + FAR, A + FAR + 8, 1, 4, 8, 8, 8, rs.RS_F32), rs.RS_ERR_OVERLAP),      # pairs inside out
    ],
)
def test_finish_rejects_bad_arguments(args, status):
    assert rs.rowsoftmax_finish_fwd(*args, 0) == status


def test_finish_empty_problem_is_a_noop():
    assert rs.rowsoftmax_finish_fwd(A, A + FAR, 2 * FAR, 2, 0, 8, 8, 8, rs.RS_F32, 0) == rs.RS_OK
    assert rs.rowsoftmax_finish_fwd(A, A + FAR, 2 * FAR, 2, 4, 0, 8, 8, rs.RS_F32, 0) == rs.RS_OK


@pytest.mark.parametrize("M,N,dt", [(1, 1 << 26, rs.RS_F16), (2, 1 << 26, rs.RS_F32), (512, 131072, rs.RS_F16),
                                    (4, 1000, rs.RS_F32), (100000, 4096, rs.RS_BF16), (3, 70000, rs.RS_BF16)])
def test_workspace_size_formula(M, N, dt):
    # S blocks a row: about 4096 (row, block) items, blocks of at least 2048
    # 16-byte units, widths whole units; M * (S + 1) pairs of 8 bytes.
    vec = 4 if dt == rs.RS_F32 else 8
    units = -(-N // vec)
    s = min(-(-4096 // M), -(-units // 2048))
    s = max(s, 1)
    width = -(-(-(-N // s)) // vec) * vec
    S = -(-N // width)
    rc, n = rs.rowsoftmax_split_workspace_size(M, N, dt)
    assert rc == rs.RS_OK and n == M * (S + 1) * 8
    assert S * width >= N and (S - 1) * width < N


def test_split_rejects_bad_arguments():
    rc, need = rs.rowsoftmax_split_workspace_size(4, 100000, rs.RS_F16)
    assert rc == rs.RS_OK and need > 0
    W = 4 * FAR
    assert rs.rowsoftmax_split_workspace_size(-1, 8, rs.RS_F16)[0] == rs.RS_ERR_INVALID_ARG
    assert rs.rowsoftmax_split_workspace_size(4, 8, 9)[0] == rs.RS_ERR_UNSUPPORTED_DTYPE
    assert rs.rowsoftmax_split_workspace_size(0, 8, rs.RS_F16) == (rs.RS_OK, 0)
    ok = (A, A + FAR, 4, 100000, 100000, 100000, rs.RS_F16)
    assert rs.rowsoftmax_split_fwd(*ok, W, need - 8, 0) == rs.RS_ERR_INVALID_ARG    # too small
    assert rs.rowsoftmax_split_fwd(*ok, 0, need, 0) == rs.RS_ERR_INVALID_ARG        # null workspace
    assert rs.rowsoftmax_split_fwd(*ok, W + 4, need, 0) == rs.RS_ERR_INVALID_ARG    # misaligned
    assert rs.rowsoftmax_split_fwd(*ok, A + 64, need, 0) == rs.RS_ERR_OVERLAP       # inside the input
    assert rs.rowsoftmax_split_fwd(*ok, A + FAR + 64, need, 0) == rs.RS_ERR_OVERLAP  # inside the output
    assert rs.rowsoftmax_split_fwd(A, A + 64, 4, 100000, 100000, 100000, rs.RS_F16, W, need, 0) == rs.RS_ERR_OVERLAP
    assert rs.rowsoftmax_split_fwd(A, A + FAR, 0, 100000, 100000, 100000, rs.RS_F16, 0, 0, 0) == rs.RS_OK
