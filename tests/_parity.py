"""Shared helpers of the GPU parity tests: run the oracle on host copies of
the inputs (several threads, one block of rows each) and compare the CUDA
library's output with it under the tolerances of the row softmax:

  fp32 output      max |y - y_ref| <= 1e-6, and |sum_j y_j - 1| <= 1e-5 per row
  fp16/bf16 output max |y - y_ref| <= 4e-3

NaN positions must agree exactly (the oracle gives NaN rows for all -inf,
NaN or +inf input rows, as the plain formula does).

Row normalisations (RMSNorm, LayerNorm) are compared element by element
under a bound derived from the kernels' fp32 arithmetic.  Every sum a kernel
forms is a tree whose longest serial chain is c = max(64, ceil(N / 512))
additions plus at most 16 more (butterfly and per-warp merge levels, the
final scaling), so each moment carries a relative error of at most
gamma = (c + 16) * 2^-24 of the sum of the absolute values it adds.  That
gives, per element,

  |y - y_ref| <= eps_fmt * |y_ref| + sub_fmt
                 + gamma * (|y_ref| + |b_j| + |w_j| * (|mu_r| + sigma_r) * r_r)

where the last product (LayerNorm only) is the error of the row mean carried
through the scaling, mu_r and sigma_r are the row's mean and population
standard deviation, r_r = 1 / sqrt(sigma_r^2 + eps); eps_fmt is half an ulp
relative of the output format (0 for fp32, 2^-11 for fp16, 2^-8 for bf16) and
sub_fmt half the fp16 subnormal spacing (2^-25; 0 otherwise).
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


NORM_EPS_FMT = {"f32": 0.0, "f16": 2.0 ** -11, "bf16": 2.0 ** -8}
NORM_SUB_FMT = {"f32": 0.0, "f16": 2.0 ** -25, "bf16": 0.0}


def norm_gamma(N: int) -> float:
    return (max(64, -(-N // 512)) + 16) * 2.0 ** -24


def _vec_np(v):
    return None if v is None else to_storage_numpy(v.reshape(-1))


def oracle_norm_rows(op: str, x: torch.Tensor, n_cols: int, weight=None, bias=None, eps: float = 1e-5) -> np.ndarray:
    """Oracle RMSNorm ('rms') or LayerNorm ('ln') of the rows of x (float64)."""
    fmt = FMT[x.dtype]
    xs = to_storage_numpy(x)
    w, b = _vec_np(weight), _vec_np(bias)
    M = xs.shape[0]
    threads = max(1, min(16, os.cpu_count() or 1, M))
    blocks = np.array_split(np.arange(M), threads)
    out = np.empty((M, n_cols), dtype=np.float64)

    def work(idx):
        if len(idx):
            part = xs[idx[0]: idx[-1] + 1]
            if op == "rms":
                out[idx[0]: idx[-1] + 1] = oracle.rmsnorm_f64(part, fmt, w, eps, n_cols)
            else:
                out[idx[0]: idx[-1] + 1] = oracle.layernorm_f64(part, fmt, w, b, eps, n_cols)

    with cf.ThreadPoolExecutor(threads) as ex:
        list(ex.map(work, blocks))
    return out


def compare_norm(y: torch.Tensor, ref: np.ndarray, x: torch.Tensor, op: str, weight=None, bias=None,
                 eps: float = 1e-5, what: str = "") -> dict:
    """Element-wise comparison of a normalisation under the bound above."""
    fmt = FMT[y.dtype]
    got = decode(y)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    N = ref.shape[1]
    nan_g, nan_r = np.isnan(got), np.isnan(ref)
    assert np.array_equal(nan_g, nan_r), f"{what}: NaN positions differ ({nan_g.sum()} vs {nan_r.sum()})"
    ok = ~nan_r
    absref = np.abs(np.where(ok, ref, 0.0))
    w = np.ones(N) if weight is None else decode(weight.reshape(-1))
    b = np.zeros(N) if bias is None else decode(bias.reshape(-1))
    g = norm_gamma(N)
    slack = absref + np.abs(b)[None, :]
    if op == "ln":
        xv = decode(x[:, :N])
        with np.errstate(invalid="ignore", over="ignore"):
            mu = xv.mean(axis=1)
            sd = xv.std(axis=1)
            rr = 1.0 / np.sqrt(sd * sd + eps)
            carry = ((np.abs(mu) + sd) * rr)[:, None] * np.abs(w)[None, :]
        slack = slack + np.where(np.isfinite(carry), carry, 0.0)
    tol = NORM_EPS_FMT[fmt] * absref + NORM_SUB_FMT[fmt] + g * slack
    err = np.abs(np.where(ok, got, 0.0) - np.where(ok, ref, 0.0))
    over = err - tol
    worst = float(over.max()) if over.size else -1.0
    if worst > 0:
        r, c = np.unravel_index(int(over.argmax()), over.shape)
        raise AssertionError(f"{what}: |err| {err[r, c]:.3e} > tol {tol[r, c]:.3e} at ({r}, {c}): "
                             f"got {got[r, c]!r} want {ref[r, c]!r}")
    return {"max_abs_err": float(err.max()) if err.size else 0.0,
            "max_err_over_tol": float((err / np.maximum(tol, 1e-300)).max()) if err.size else 0.0}
