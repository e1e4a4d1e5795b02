"""GPU parity on rows of large magnitude, through the C ABI.

The kernels that hold a row in registers take their exponentials against a
rounded base-2 offset of each warp's max while that max is below 2^23 in
magnitude, and as exp(x - m) past it; a row can mix both kinds of warps.
These rows put the max on either side of 2^23, far beyond it (1e10, 3e38,
values whose difference overflows), and mix the two kinds inside one row, on
every kernel family of the plain and the causal softmax.  Each result is
compared element by element with the oracle, and the rows whose softmax is
known in closed form (uniform over ties, zero elsewhere) are checked exactly.
"""
import math

import numpy as np
import pytest
import torch

import memory_bound_row_gb300 as rs
import oracle
from memory_bound_row_gb300 import build

from _parity import FMT, compare, oracle_rows, to_storage_numpy

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}
M = 8


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    rc, _ = rs.rowsoftmax_device_status(clear=True)
    assert rc == rs.RS_OK
    yield
    rc, flags = rs.rowsoftmax_device_status(clear=False)
    assert rc == rs.RS_OK and flags == 0, f"device status word {flags:#x}"


def large_rows(N: int, seed: int) -> np.ndarray:
    """Eight rows of N values (float64, before rounding to the storage type)."""
    g = np.random.default_rng(seed)
    j = np.arange(N)
    h = N // 2
    x = np.empty((M, N))
    x[0] = -1e10                                           # one value: uniform
    x[1] = -1e10 * (1.0 + (j % 3) * 2.0 ** -6)             # three levels far apart: uniform over the top level
    x[2] = 8388608.0 + (j % 7) - 3.0                       # around 2^23
    x[3] = 8388600.0 + (j % 7)                             # just below 2^23
    x[4, :h] = -3e9                                        # far below the rest: zeros
    x[4, h:] = g.standard_normal(N - h)
    x[5, :h] = 2e7 + np.round(g.standard_normal(h) * 4.0)  # past 2^23, with spread
    x[5, h:] = g.standard_normal(N - h)                    # negligible beside it
    x[6] = np.where(j % 2 == 0, 3.0e38, -3.0e38)           # x - m overflows to -inf: uniform over the evens
    x[7] = np.where(j % 3 == 0, 1.6e38, -1.6e38)
    return x


def _device_rows(N, dtype, seed):
    vec = 4 if dtype == "f32" else 8
    ld = -(-N // vec) * vec
    buf = torch.empty((M, ld), dtype=DT[dtype], device="cuda")
    buf[:, :N] = torch.from_numpy(large_rows(N, seed)).to(DT[dtype]).cuda()
    out = torch.empty((M, ld), dtype=DT[dtype], device="cuda")
    return buf[:, :N], out[:, :N]


def _exact_checks(y, x):
    """Rows 0, 1, 6, 7: uniform over the positions of the row's max, 0 elsewhere."""
    yd = y.double().cpu().numpy()
    xv = x.double().cpu().numpy()
    for r in (0, 1, 6, 7):
        top = xv[r] == xv[r].max()
        assert np.all(yd[r, ~top] == 0.0), f"row {r}: mass off the max"
        assert np.allclose(yd[r, top], 1.0 / top.sum(), rtol=2.0 ** -7, atol=0), f"row {r}: not uniform"


PLAIN_PATHS = {
    "rows": rs.RS_PATH_ROWS,
    "ring": rs.RS_PATH_RING,
    "cluster": rs.RS_PATH_CLUSTER,
    "stream": rs.RS_PATH_STREAM,
}


def _plain_servable(x, options):
    rc, dev = rs.rowsoftmax_device_info()
    n, k = x.shape
    rc, _ = rs.rowsoftmax_plan(x.data_ptr(), x.data_ptr() + (1 << 44), n, k, x.stride(0), x.stride(0),
                               rs.dtype_code(x.dtype), options, dev)
    assert rc in (rs.RS_OK, rs.RS_ERR_NO_PATH)
    return rc == rs.RS_OK


@pytest.mark.parametrize("path", list(PLAIN_PATHS))
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [2048, 12345, 65536])
def test_plain_softmax_large_magnitudes(path, dtype, N):
    x, out = _device_rows(N, dtype, seed=N)
    opts = {"path": PLAIN_PATHS[path]}
    if not _plain_servable(x, opts):
        pytest.skip("this kernel does not serve the shape")
    y = rs.softmax(x, out=out, options=opts)
    torch.cuda.synchronize()
    compare(y, oracle_rows(x, N), dtype, f"large magnitudes, {path} {dtype} N={N}")
    _exact_checks(y, x)


CAUSAL_PATHS = {
    "rows": {"path": rs.RS_PATH_ROWS},
    "ring": {"path": rs.RS_PATH_RING},
    "ring bulk": {"path": rs.RS_PATH_RING, "ring_values": rs.RS_RING_REGISTERS},
    "ring copies 3": {"path": rs.RS_PATH_RING, "ring_values": rs.RS_RING_THREAD_COPIES, "stages": 3},
    "ring copies, 2 warps a row": {"path": rs.RS_PATH_RING, "ring_values": rs.RS_RING_THREAD_COPIES,
                                   "threads_per_row": 64},
    "cluster": {"path": rs.RS_PATH_CLUSTER},
}


@pytest.mark.parametrize("path", list(CAUSAL_PATHS))
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [2048, 12345, 65536])
def test_causal_softmax_large_magnitudes(path, dtype, N):
    x, out = _device_rows(N, dtype, seed=N + 1)
    period, offset = M, (3 * N) // 4 - 4  # kept prefixes through three quarters of the row
    opts = CAUSAL_PATHS[path]
    rc, dev = rs.rowsoftmax_device_info()
    rc, _ = rs.rowsoftmax_causal_plan(x.data_ptr(), x.data_ptr() + (1 << 44), M, N, x.stride(0), x.stride(0),
                                      period, offset, rs.dtype_code(x.dtype), opts, dev)
    assert rc in (rs.RS_OK, rs.RS_ERR_NO_PATH)
    if rc != rs.RS_OK:
        pytest.skip("this kernel does not serve the shape")
    ref = oracle.softmax_prefix_f64(to_storage_numpy(x), FMT[x.dtype], period, offset, N)
    y = rs.softmax_causal(x, period, offset, out=out, options=opts)
    torch.cuda.synchronize()
    compare(y, ref, dtype, f"large magnitudes, causal {path} {dtype} N={N}")
    keep = [min(N, r % period + 1 + offset) for r in range(M)]
    yd = y.double().cpu().numpy()
    for r in range(M):
        assert np.all(yd[r, keep[r]:] == 0.0)
        assert math.isclose(float(yd[r, :keep[r]].sum()), 1.0, rel_tol=0, abs_tol=2e-2)
