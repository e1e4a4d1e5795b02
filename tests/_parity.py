"""Shared helpers of the GPU parity tests: run the oracle on host copies of
the inputs (several threads, one block of rows each) and compare the CUDA
library's output with it under the tolerances of the row softmax:

  fp32 output      max |y - y_ref| <= 1e-6, and |sum_j y_j - 1| <= 1e-5 per row
  fp16/bf16 output max |y - y_ref| <= 4e-3

NaN positions must agree exactly (the oracle gives NaN rows for all -inf,
NaN or +inf input rows, as the plain formula does).

Row normalisations (RMSNorm, LayerNorm) are compared element by element
under a bound that holds for any order in which fp32 sums are formed: a sum
of n terms, each rounded once, computed by any sequence of n - 1 fp32
additions, is within gamma_n = n u / (1 - n u) (u = 2^-24) of the exact sum
relative to the sum of the absolute values of the terms (Higham, "Accuracy
and Stability of Numerical Algorithms", 2nd ed., section 4.2: the recursive
summation bound, which bounds every summation order).  The moments of a row
of N values are such sums; the square root, reciprocal, products and the
final scaling add at most 16 more roundings.  With gamma = gamma_(N + 16)
that gives, per element,

  |y - y_ref| <= eps_fmt * |y_ref| + sub_fmt
                 + gamma * (|y_ref| + |b_j| + |w_j| * (|mu_r| + sigma_r) * r_r)

where the last product (LayerNorm only) is the error of the row mean carried
through the scaling (the mean of |x| is at most sqrt(mu^2 + sigma^2) <=
|mu| + sigma), mu_r and sigma_r are the row's mean and population standard
deviation, r_r = 1 / sqrt(sigma_r^2 + eps); eps_fmt is half an ulp relative of
the output format (0 for fp32, 2^-11 for fp16, 2^-8 for bf16) and sub_fmt half
the fp16 subnormal spacing (2^-25; 0 otherwise).  Beyond 2^18 values a row's
order-independent bound says nothing useful (N u reaches 1/64): there the bound
takes the blocked order the kernels use, whose longest serial chain is
max(64, ceil(N / 512)) additions plus 16 (only the 2^26-value rows of the
maximum-size cases need it).

Full-size workloads are checked on every row by check_all_rows: the rows are
copied to the host in chunks, and 16 threads each run the oracle on a block
of a chunk and compare it with the library's rows.  The statistics of every
such check are collected in REPORT and printed in pytest's terminal summary.
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


def softmax_errors(got: np.ndarray, ref: np.ndarray, fmt: str) -> dict:
    """Errors of decoded results `got` against the oracle's `ref` (float64,
    same shape) under the softmax tolerances; asserts nothing."""
    nan_g, nan_r = np.isnan(got), np.isnan(ref)
    st = {"nan_mismatch": int(np.count_nonzero(nan_g != nan_r)), "max_abs_err": 0.0, "where": None}
    ok = ~nan_r
    err = np.abs(np.where(ok, got, 0.0) - np.where(ok, ref, 0.0))
    if err.size:
        i = int(err.argmax())
        st["max_abs_err"] = float(err.flat[i])
        r, c = np.unravel_index(i, err.shape)
        st["where"] = (int(r), int(c), float(got[r, c]), float(ref[r, c]))
    if fmt == "f32" and got.size:
        finite_rows = ~nan_r.any(axis=1)
        st["max_rowsum_err"] = float(np.abs(got[finite_rows].sum(axis=1) - 1.0).max()) if finite_rows.any() else 0.0
    return st


def _softmax_verdict(st: dict, fmt: str, what: str) -> None:
    assert st["nan_mismatch"] == 0, f"{what}: NaN positions differ at {st['nan_mismatch']} elements"
    if st["max_abs_err"] > TOL[fmt]:
        r, c, g, want = st["where"]
        raise AssertionError(f"{what}: max |err| {st['max_abs_err']:.3e} > {TOL[fmt]} at ({r}, {c}): "
                             f"got {g!r} want {want!r}")
    if "max_rowsum_err" in st:
        assert st["max_rowsum_err"] <= ROWSUM_TOL_F32, f"{what}: row sum off by {st['max_rowsum_err']:.3e}"


def compare(y: torch.Tensor, ref: np.ndarray, fmt: str, what: str = "") -> dict:
    """Element-wise comparison; raises AssertionError with the worst spot."""
    got = decode(y)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    st = softmax_errors(got, ref, fmt)
    _softmax_verdict(st, fmt, what)
    out = {"max_abs_err": st["max_abs_err"]}
    if "max_rowsum_err" in st:
        out["max_rowsum_err"] = st["max_rowsum_err"]
    return out


NORM_EPS_FMT = {"f32": 0.0, "f16": 2.0 ** -11, "bf16": 2.0 ** -8}
NORM_SUB_FMT = {"f32": 0.0, "f16": 2.0 ** -25, "bf16": 0.0}


U32 = 2.0 ** -24  # unit roundoff of fp32


def norm_gamma(N: int) -> float:
    """Relative error bound of the fp32 moments of a row of N values (see the
    module docstring): gamma_(N + 16) for any summation order, and for rows
    whose order-independent bound is uninformative, the kernels' blocked
    order's."""
    k = N + 16
    if k * U32 <= 1.0 / 64:
        return k * U32 / (1.0 - k * U32)
    k = max(64, -(-N // 512)) + 16
    return k * U32 / (1.0 - k * U32)


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


def norm_errors(got: np.ndarray, ref: np.ndarray, xv: np.ndarray, op: str, w: np.ndarray, b: np.ndarray,
                eps: float, fmt: str) -> dict:
    """Errors of decoded normalisation results against the oracle under the
    bound of the module docstring; `xv` the decoded inputs (LayerNorm's mean
    and deviation), `w` and `b` the decoded vectors.  Asserts nothing."""
    N = ref.shape[1]
    nan_g, nan_r = np.isnan(got), np.isnan(ref)
    st = {"nan_mismatch": int(np.count_nonzero(nan_g != nan_r)), "max_abs_err": 0.0, "max_err_over_tol": 0.0,
          "where": None}
    if not got.size:
        return st
    ok = ~nan_r
    absref = np.abs(np.where(ok, ref, 0.0))
    g = norm_gamma(N)
    slack = absref + np.abs(b)[None, :]
    if op == "ln":
        with np.errstate(invalid="ignore", over="ignore"):
            mu = xv.mean(axis=1)
            sd = xv.std(axis=1)
            rr = 1.0 / np.sqrt(sd * sd + eps)
            carry = ((np.abs(mu) + sd) * rr)[:, None] * np.abs(w)[None, :]
        slack = slack + np.where(np.isfinite(carry), carry, 0.0)
    tol = NORM_EPS_FMT[fmt] * absref + NORM_SUB_FMT[fmt] + g * slack
    err = np.abs(np.where(ok, got, 0.0) - np.where(ok, ref, 0.0))
    ratio = err / np.maximum(tol, 1e-300)
    i = int(ratio.argmax())
    r, c = np.unravel_index(i, ratio.shape)
    st.update(max_abs_err=float(err.max()), max_err_over_tol=float(ratio.flat[i]),
              where=(int(r), int(c), float(got[r, c]), float(ref[r, c]), float(err[r, c]), float(tol[r, c])))
    return st


def _norm_verdict(st: dict, what: str) -> None:
    assert st["nan_mismatch"] == 0, f"{what}: NaN positions differ at {st['nan_mismatch']} elements"
    if st["max_err_over_tol"] > 1.0:
        r, c, g, want, e, t = st["where"]
        raise AssertionError(f"{what}: |err| {e:.3e} > tol {t:.3e} at ({r}, {c}): got {g!r} want {want!r}")


def compare_norm(y: torch.Tensor, ref: np.ndarray, x: torch.Tensor, op: str, weight=None, bias=None,
                 eps: float = 1e-5, what: str = "") -> dict:
    """Element-wise comparison of a normalisation under the bound above."""
    got = decode(y)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    N = ref.shape[1]
    w = np.ones(N) if weight is None else decode(weight.reshape(-1))
    b = np.zeros(N) if bias is None else decode(bias.reshape(-1))
    xv = decode(x[:, :N]) if op == "ln" else None
    st = norm_errors(got, ref, xv, op, w, b, eps, FMT[y.dtype])
    _norm_verdict(st, what)
    return {"max_abs_err": st["max_abs_err"], "max_err_over_tol": st["max_err_over_tol"]}


# Statistics of every all-rows check of this session (printed by conftest.py):
# (group, line); group "workloads" (the benchmark workloads at full size) is
# printed last.
REPORT: list[tuple[str, str]] = []


def check_all_rows(kind: str, x: torch.Tensor, y: torch.Tensor, n_cols: int, *, weight=None, bias=None,
                   eps: float = 0.0, period: int = 0, offset: int = 0, what: str = "",
                   chunk_elems: int = 1 << 26, threads: int = 16, group: str = "other") -> dict:
    """Every row of y (device, M x n_cols view) against the oracle on the same
    rows of x.  kind: "softmax" (softmax tolerances), "prefix" (the softmax
    under a causal mask: row r keeps min(n_cols, max(0, r mod period + 1 +
    offset)) values), "rms" or "ln" (the normalisation bound).  Rows are
    copied to the host in chunks of about `chunk_elems` elements; `threads`
    host threads each run the oracle on one block of a chunk and compare.
    Raises AssertionError at the first violation; returns the statistics over
    all rows and appends them to REPORT."""
    fmt = FMT[x.dtype]
    M = x.shape[0]
    threads = max(1, min(threads, os.cpu_count() or 1))
    chunk_rows = max(1, chunk_elems // max(1, n_cols))
    if kind in ("rms", "ln"):
        w_np, b_np = _vec_np(weight), _vec_np(bias)
        wd = np.ones(n_cols) if weight is None else decode(weight.reshape(-1))
        bd = np.zeros(n_cols) if bias is None else decode(bias.reshape(-1))
    agg = {"rows": 0, "max_abs_err": 0.0}
    if kind in ("rms", "ln"):
        agg["max_err_over_tol"] = 0.0
    if fmt == "f32" and kind in ("softmax", "prefix"):
        agg["max_rowsum_err"] = 0.0

    def work(args):
        r0, xs, yc, lo, hi = args
        if hi <= lo:
            return None
        xb = xs[lo:hi]
        got = yc[lo:hi].to(torch.float64).numpy()
        if kind == "softmax":
            return softmax_errors(got, oracle.softmax_f64(xb, fmt, n_cols), fmt), lo
        if kind == "prefix":
            ref = oracle.softmax_prefix_f64(xb, fmt, period, offset, n_cols, row0=r0 + lo)
            return softmax_errors(got, ref, fmt), lo
        if kind == "rms":
            ref = oracle.rmsnorm_f64(xb, fmt, w_np, eps, n_cols)
            return norm_errors(got, ref, None, "rms", wd, bd, eps, fmt), lo
        ref = oracle.layernorm_f64(xb, fmt, w_np, b_np, eps, n_cols)
        xv = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy() \
            if fmt == "bf16" else xb.astype(np.float64)
        return norm_errors(got, ref, xv, "ln", wd, bd, eps, fmt), lo

    with cf.ThreadPoolExecutor(threads) as ex:
        for r0 in range(0, M, chunk_rows):
            r1 = min(M, r0 + chunk_rows)
            xs = to_storage_numpy(x[r0:r1, :n_cols])
            yc = y[r0:r1, :n_cols].detach().cpu().contiguous()
            cuts = np.linspace(0, r1 - r0, threads + 1).astype(np.int64)
            for res in ex.map(work, [(r0, xs, yc, int(cuts[i]), int(cuts[i + 1])) for i in range(threads)]):
                if res is None:
                    continue
                st, lo = res
                label = f"{what} (rows {r0 + lo}..)"
                if st.get("where") is not None:  # report the row's index in the whole tensor
                    st["where"] = (st["where"][0] + r0 + lo,) + tuple(st["where"][1:])
                if kind in ("rms", "ln"):
                    _norm_verdict(st, label)
                    agg["max_err_over_tol"] = max(agg["max_err_over_tol"], st["max_err_over_tol"])
                else:
                    _softmax_verdict(st, fmt, label)
                    if "max_rowsum_err" in agg:
                        agg["max_rowsum_err"] = max(agg["max_rowsum_err"], st["max_rowsum_err"])
                agg["max_abs_err"] = max(agg["max_abs_err"], st["max_abs_err"])
            agg["rows"] += r1 - r0
    assert agg["rows"] == M
    REPORT.append((group, f"{what}: all {M} rows x {n_cols} checked against the oracle; "
                   + ", ".join(f"{k} {v:.3e}" if isinstance(v, float) else f"{k} {v}" for k, v in agg.items()
                               if k != "rows")))
    return agg
