"""Shared helpers of the GPU parity tests: run the oracle on host copies of
the inputs (several threads, one block of rows each) and compare the CUDA
library's output with it under the tolerances of the row softmax:

  fp32 output      max |y - y_ref| <= 1e-6, and |sum_j y_j - 1| <= 1e-5 per row
  fp16/bf16 output max |y - y_ref| <= 4e-3

NaN positions must agree exactly (the oracle gives NaN rows for all -inf,
NaN or +inf input rows, as the plain formula does).
"""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np
import torch

import oracle

TOL = {"f32": 1e-6, "f16": 4e-3, "bf16": 4e-3}
ROWSUM_TOL_F32 = 1e-5
FMT = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}


def to_storage_numpy(t: torch.Tensor) -> np.ndarray:
    """Host numpy view of a tensor's stored bits in the oracle's formats."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def decode(t: torch.Tensor) -> np.ndarray:
    """Exact float64 values of a tensor's elements."""
    return t.detach().cpu().to(torch.float64).numpy()


def oracle_rows(x: torch.Tensor, n_cols: int) -> np.ndarray:
    """Oracle softmax (float64) of the rows of x (2-D, possibly padded)."""
    fmt = FMT[x.dtype]
    xs = to_storage_numpy(x)
    M = xs.shape[0]
    threads = max(1, min(16, os.cpu_count() or 1, M))
    blocks = np.array_split(np.arange(M), threads)
    out = np.empty((M, n_cols), dtype=np.float64)

    def work(idx):
        if len(idx):
            out[idx[0]: idx[-1] + 1] = oracle.softmax_f64(xs[idx[0]: idx[-1] + 1], fmt, n_cols)

    with cf.ThreadPoolExecutor(threads) as ex:
        list(ex.map(work, blocks))
    return out


def compare(y: torch.Tensor, ref: np.ndarray, fmt: str, what: str = "") -> dict:
    """Element-wise comparison; raises AssertionError with the worst spot."""
    got = decode(y)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    nan_g, nan_r = np.isnan(got), np.isnan(ref)
    assert np.array_equal(nan_g, nan_r), f"{what}: NaN positions differ ({nan_g.sum()} vs {nan_r.sum()})"
    ok = ~nan_r
    err = np.abs(np.where(ok, got, 0.0) - np.where(ok, ref, 0.0))
    worst = float(err.max()) if err.size else 0.0
    if worst > TOL[fmt]:
        r, c = np.unravel_index(int(err.argmax()), err.shape)
        raise AssertionError(f"{what}: max |err| {worst:.3e} > {TOL[fmt]} at ({r}, {c}): "
                             f"got {got[r, c]!r} want {ref[r, c]!r}")
    stats = {"max_abs_err": worst}
    if fmt == "f32" and got.size:
        finite_rows = ~nan_r.any(axis=1)
        if finite_rows.any():
            dev = np.abs(got[finite_rows].sum(axis=1) - 1.0)
            stats["max_rowsum_err"] = float(dev.max())
            assert stats["max_rowsum_err"] <= ROWSUM_TOL_F32, f"{what}: row sum off by {dev.max():.3e}"
    return stats
