"""The failure path of the bounded waits, exercised on the GPU without a
fault: the ring kernel (RS_PATH_RING) and the register-holding cluster kernel
(RS_PATH_CLUSTER) are told to post the expected bytes of their copies but
never issue them (withhold_copies = 1), so every copy wait runs out after a
short limit.  The call must return, the
device status word must report the timeout, the output must be left
unwritten, and the context must still compute correct results afterwards."""
import time

import numpy as np
import pytest
import torch

import memory_bound_row_gb300 as rs
from memory_bound_row_gb300 import build
from memory_bound_row_gb300 import workloads as W

from _parity import compare, oracle_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    rs.rowsoftmax_device_status(clear=True)
    yield
    rs.rowsoftmax_device_status(clear=True)


def test_a_wait_that_runs_out_is_reported_and_the_context_survives():
    w = W.custom(256, 4096, "bf16", seed=21)
    x = W.generate(w, "cuda")
    out = torch.full_like(x, 7.0)
    torch.cuda.synchronize()
    opts = {"path": rs.RS_PATH_RING, "withhold_copies": 1, "wait_limit_us": 20000}
    t0 = time.perf_counter()
    rc = rs.rowsoftmax_fwd_ex(x.data_ptr(), out.data_ptr(), w.M, w.N, w.N, w.N, rs.RS_BF16,
                              torch.cuda.current_stream().cuda_stream, opts)
    assert rc == rs.RS_OK
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 30.0
    rc, flags = rs.rowsoftmax_device_status(clear=True)
    assert rc == rs.RS_OK and flags & 1
    assert bool((out == 7.0).all())  # the abandoned rows were not written

    # The context is intact: the same call without the withheld copies is correct.
    y = rs.softmax(x)
    torch.cuda.synchronize()
    compare(y[:64], oracle_rows(x[:64], w.N), "bf16", "after the timeout")
    rc, flags = rs.rowsoftmax_device_status(clear=False)
    assert rc == rs.RS_OK and flags == 0


def test_withholding_is_only_accepted_with_a_short_limit_on_the_ring():
    x = torch.zeros(4, 64, device="cuda")
    y = torch.empty_like(x)
    for opts in [{"path": rs.RS_PATH_RING, "withhold_copies": 1},
                 {"path": rs.RS_PATH_ROWS, "withhold_copies": 1, "wait_limit_us": 1000},
                 {"path": rs.RS_PATH_RING, "withhold_copies": 1, "wait_limit_us": 10_000_000}]:
        rc = rs.rowsoftmax_fwd_ex(x.data_ptr(), y.data_ptr(), 4, 64, 64, 64, rs.RS_F32, 0, opts)
        assert rc == rs.RS_ERR_INVALID_ARG


@pytest.mark.parametrize("op", ["softmax", "layernorm"])
def test_a_cluster_wait_that_runs_out_is_reported_and_the_context_survives(op):
    # The register-holding cluster kernel (a cluster of CTAs per 131072-value
    # row) with its slot copies withheld: every CTA's first copy wait runs out,
    # the CTAs keep exchanging their (unused) pairs so that no peer waits in
    # vain, store nothing, let their copies drain and return.
    w = W.custom(48, 131072, "f16", seed=22)
    x = W.generate(w, "cuda")
    out = torch.full_like(x, 7.0)
    wt = torch.ones(w.N, dtype=torch.float16, device="cuda")
    torch.cuda.synchronize()
    opts = {"path": rs.RS_PATH_CLUSTER, "ring_values": rs.RS_RING_REGISTERS, "withhold_copies": 1,
            "wait_limit_us": 20000}
    st = torch.cuda.current_stream().cuda_stream
    t0 = time.perf_counter()
    if op == "softmax":
        rc = rs.rowsoftmax_fwd_ex(x.data_ptr(), out.data_ptr(), w.M, w.N, w.N, w.N, rs.RS_F16, st, opts)
    else:
        rc = rs.rownorm_fwd_ex(rs.RS_OP_LAYERNORM, x.data_ptr(), out.data_ptr(), wt.data_ptr(), None, w.M, w.N,
                               w.N, w.N, 1e-5, rs.RS_F16, st, opts)
    assert rc == rs.RS_OK
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 30.0
    rc, flags = rs.rowsoftmax_device_status(clear=True)
    assert rc == rs.RS_OK and flags & 1
    assert bool((out == 7.0).all())  # no row was written

    y = rs.softmax(x) if op == "softmax" else rs.layernorm(x, wt, None)
    torch.cuda.synchronize()
    if op == "softmax":
        compare(y[:8], oracle_rows(x[:8], w.N), "f16", "after the cluster timeout")
    else:
        assert bool(torch.isfinite(y).all())
        assert float(y.float().mean(dim=1).abs().max()) < 1e-2
    rc, flags = rs.rowsoftmax_device_status(clear=False)
    assert rc == rs.RS_OK and flags == 0


def test_withholding_on_a_kernel_without_it_is_no_path():
    # the shared-memory cluster variant and the streaming kernels do not implement it
    x = torch.zeros(2, 1 << 20, dtype=torch.float16, device="cuda")
    y = torch.empty_like(x)
    opts = {"path": rs.RS_PATH_CLUSTER, "ring_values": rs.RS_RING_REREAD, "withhold_copies": 1,
            "wait_limit_us": 1000}
    rc = rs.rowsoftmax_fwd_ex(x.data_ptr(), y.data_ptr(), 2, 1 << 20, 1 << 20, 1 << 20, rs.RS_F16, 0, opts)
    assert rc == rs.RS_ERR_NO_PATH
