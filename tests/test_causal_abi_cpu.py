"""CPU checks of the causal-mask softmax entry points (rowsoftmax_causal_fwd,
_fwd_ex, _plan): argument validation before any device call and the kernels
the planner allows for masked rows.  No kernel runs."""
import pytest

import memory_bound_row_gb300 as rs
from memory_bound_row_gb300 import build

from test_abi_cpu import gb300

A = 1 << 20
OUT = A + (1 << 40)


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _plan(M, N, dtype, period, offset=0, opts=None, a=A, ld=None):
    rc, plan = rs.rowsoftmax_causal_plan(a, OUT, M, N, ld or N, ld or N, period, offset, dtype, opts, gb300())
    return rc, plan


@pytest.mark.parametrize("period,offset,status", [(0, 0, rs.RS_ERR_INVALID_ARG), (-3, 0, rs.RS_ERR_INVALID_ARG),
                                                  (4, 1 << 62, rs.RS_OK), (4, (1 << 62) + 1, rs.RS_ERR_INVALID_ARG),
                                                  (4, -(1 << 62) - 1, rs.RS_ERR_INVALID_ARG), (1, -5, rs.RS_OK)])
def test_period_and_offset_are_validated(period, offset, status):
    rc, plan = _plan(64, 1024, rs.RS_BF16, period, offset)
    assert rc == status
    if status == rs.RS_OK:
        assert plan["masked"] == 1
    else:
        assert rs.rowsoftmax_causal_fwd(A, OUT, 64, 1024, 1024, 1024, period, offset, rs.RS_BF16, 0) == status


def test_shape_errors_match_the_softmax():
    assert rs.rowsoftmax_causal_fwd(A, A + 64, 4, 8, 8, 8, 2, 0, rs.RS_F32, 0) == rs.RS_ERR_OVERLAP
    assert rs.rowsoftmax_causal_fwd(A, OUT, 4, 8, 7, 8, 2, 0, rs.RS_F32, 0) == rs.RS_ERR_INVALID_ARG
    assert rs.rowsoftmax_causal_fwd(A, OUT, 4, 8, 8, 8, 2, 0, 9, 0) == rs.RS_ERR_UNSUPPORTED_DTYPE
    assert rs.rowsoftmax_causal_fwd(0, 0, 0, 8, 8, 8, 2, 0, rs.RS_F32, 0) == rs.RS_OK  # empty: no-op


def test_masked_rows_use_the_same_kernels_as_the_plain_softmax():
    # (16-bit rows of 2049 to 32768 values have their own measured shape on the
    # causal copy ring: test_abi_cpu.py)
    for M, N, dt in [(1 << 20, 2048, rs.RS_BF16), (8192, 5000, rs.RS_F32), (4096, 2048, rs.RS_F16),
                     (512, 131072, rs.RS_F16)]:
        rc, plain = rs.rowsoftmax_plan(A, OUT, M, N, N, N, dt, None, gb300())
        rc2, masked = _plan(M, N, dt, period=2048)
        assert rc == rc2 == rs.RS_OK
        for k in ("path", "threads_per_row", "vec_per_thread", "block_threads", "cluster_size", "grid"):
            assert plain[k] == masked[k], (M, N, k)
        assert plain["masked"] == 0 and masked["masked"] == 1


def test_only_register_holding_kernels_serve_the_mask():
    rc, _ = _plan(64, 4096, rs.RS_BF16, 64, opts={"path": rs.RS_PATH_STREAM})
    assert rc == rs.RS_ERR_NO_PATH
    rc, _ = _plan(64, 4096, rs.RS_BF16, 64, opts={"path": rs.RS_PATH_CLUSTER, "ring_values": rs.RS_RING_REREAD})
    assert rc == rs.RS_ERR_NO_PATH
    rc, _ = _plan(64, 1 << 20, rs.RS_BF16, 64)          # wider than the clusters hold
    assert rc == rs.RS_ERR_NO_PATH
    rc, _ = _plan(64, 131072, rs.RS_F16, 64, a=A + 2)   # misaligned wide rows: only the streaming kernel
    assert rc == rs.RS_ERR_NO_PATH
    rc, p = _plan(64, 4096, rs.RS_F16, 64, a=A + 2)     # misaligned rows that fit: element-wise register rows
    assert rc == rs.RS_OK and p["path"] == rs.RS_PATH_ROWS and p["vec_elems"] == 1
    rc, _ = _plan(64, 4096, rs.RS_BF16, 64, opts={"path": rs.RS_PATH_RING, "ring_values": rs.RS_RING_REREAD})
    assert rc == rs.RS_ERR_NO_PATH  # the masked ring holds its rows in registers


def test_remainder_by_direct_computation():
    # The kernels take r mod period with the reciprocal constant of Lemire, Kaser
    # and Kurz (c = floor((2^64 - 1) / d) + 1; n mod d = high64((c n mod 2^64) d))
    # for 32-bit rows and periods; the identity, checked here on the integers.
    import random

    m64 = (1 << 64) - 1
    rng = random.Random(5)
    ds = list(range(1, 2049)) + [rng.randrange(1, 1 << 32) for _ in range(2000)] + [(1 << 32) - 1, 1 << 31]
    for d in ds:
        c = (m64 // d + 1) & m64
        for n in [0, 1, d - 1, d, d + 1, (1 << 32) - 1] + [rng.randrange(0, 1 << 32) for _ in range(50)]:
            if 0 <= n < (1 << 32):
                assert (((c * n) & m64) * d) >> 64 == n % d, (n, d)


def test_the_masked_ring_copies_only_the_kept_units_on_16bit_rows():
    # bf16 causal scores: the ring with per-thread copies of the kept units by
    # default; the bulk-copy ring (whole rows) when forced; neither elsewhere
    rc, p = _plan(1 << 20, 2048, rs.RS_BF16, 2048)
    assert rc == rs.RS_OK and p["path"] == rs.RS_PATH_RING and p["ring_values"] == rs.RS_RING_THREAD_COPIES
    assert p["stages"] == 2 and p["smem_bytes"] == 2 * p["rows_per_cta"] * 2048 * 2
    rc, p = _plan(1 << 20, 2048, rs.RS_BF16, 2048, opts={"path": rs.RS_PATH_RING, "ring_values": rs.RS_RING_REGISTERS})
    assert rc == rs.RS_OK and p["ring_values"] == rs.RS_RING_REGISTERS
    rc, p = _plan(4096, 2048, rs.RS_F16, 2048, opts={"path": rs.RS_PATH_RING, "stages": 3})
    assert rc == rs.RS_OK and p["ring_values"] == rs.RS_RING_THREAD_COPIES and p["stages"] == 3
    rc, p = _plan(4096, 2048, rs.RS_F16, 2048, opts={"path": rs.RS_PATH_RING, "stages": 4})  # copies: 2 or 3
    assert rc == rs.RS_OK and p["ring_values"] == rs.RS_RING_REGISTERS
    copies = {"ring_values": rs.RS_RING_THREAD_COPIES}
    assert _plan(4096, 2048, rs.RS_F16, 2048, opts=dict(copies, path=rs.RS_PATH_RING, stages=4))[0] == rs.RS_ERR_NO_PATH
    assert _plan(4096, 2048, rs.RS_F32, 2048, opts=dict(copies, path=rs.RS_PATH_RING))[0] == rs.RS_ERR_NO_PATH
    assert _plan(64, 131072, rs.RS_F16, 64, opts=dict(copies, path=rs.RS_PATH_CLUSTER))[0] == rs.RS_ERR_NO_PATH
    rc, _ = rs.rowsoftmax_plan(A, OUT, 4096, 2048, 2048, 2048, rs.RS_BF16, dict(copies, path=rs.RS_PATH_RING),
                               gb300())
    assert rc == rs.RS_ERR_NO_PATH  # the unmasked softmax stages whole rows
