"""Row-softmax oracle: a plain, slow, double-precision CPU implementation.

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference arm are the only callers.  The product
(``memory_bound_row_gb300``) never imports this package; the two share no
code.

The arithmetic lives in ``softmax_ref.c`` (the plain definition of the row
softmax, see the header of that file for the passages it follows and the
readings taken where the pages are silent).  This module only compiles it
with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "softmax_ref.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_softmax.so")

# The oracle's own storage-format codes (see softmax_ref.c).
FORMATS = {"f32": 0, "f16": 1, "bf16": 2, "f64": 3}
_NP_STORAGE = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16, "f64": np.float64}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile softmax_ref.c into a shared library next to it (plain gcc)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"],
            check=True,
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            i64, vp = ctypes.c_int64, ctypes.c_void_p
            lib.orc_softmax_f64.argtypes = [vp, ctypes.c_int, i64, i64, i64, vp, i64]
            lib.orc_softmax_f64.restype = ctypes.c_int
            lib.orc_softmax_store.argtypes = [vp, vp, ctypes.c_int, i64, i64, i64, i64, ctypes.c_int]
            lib.orc_softmax_store.restype = ctypes.c_int
            lib.orc_decode_array.argtypes = [vp, ctypes.c_int, i64, vp]
            lib.orc_decode_array.restype = None
            lib.orc_encode_array.argtypes = [vp, ctypes.c_int, i64, vp]
            lib.orc_encode_array.restype = None
            lib.orc_softmax_prefix_f64.argtypes = [vp, ctypes.c_int, i64, i64, i64, i64, i64, i64, vp, i64]
            lib.orc_softmax_prefix_f64.restype = ctypes.c_int
            lib.orc_prefix_len.argtypes = [i64, i64, i64, i64]
            lib.orc_prefix_len.restype = i64
            lib.orc_rmsnorm_f64.argtypes = [vp, ctypes.c_int, i64, i64, i64, vp, ctypes.c_double, vp, i64]
            lib.orc_rmsnorm_f64.restype = ctypes.c_int
            lib.orc_layernorm_f64.argtypes = [vp, ctypes.c_int, i64, i64, i64, vp, vp, ctypes.c_double, vp, i64]
            lib.orc_layernorm_f64.restype = ctypes.c_int
            lib.orc_softmax_partial_f64.argtypes = [vp, ctypes.c_int, i64, i64, i64, vp]
            lib.orc_softmax_partial_f64.restype = ctypes.c_int
            lib.orc_merge_pairs_f64.argtypes = [vp, i64, i64, vp]
            lib.orc_merge_pairs_f64.restype = ctypes.c_int
            lib.orc_softmax_finish_f64.argtypes = [vp, ctypes.c_int, i64, i64, i64, vp, vp, i64]
            lib.orc_softmax_finish_f64.restype = ctypes.c_int
            _lib = lib
    return _lib


def _as_storage(x: np.ndarray, fmt: str) -> np.ndarray:
    want = _NP_STORAGE[fmt]
    if x.dtype != want:
        raise TypeError(f"format {fmt} expects numpy storage {np.dtype(want)}, got {x.dtype}")
    return np.ascontiguousarray(x)


def softmax_f64(x: np.ndarray, fmt: str, n_cols: int | None = None) -> np.ndarray:
    """Row softmax of the 2-D array ``x`` (rows of ``x.shape[1]`` stored
    elements; the first ``n_cols`` of each row are the data, the rest is
    padding that is never read).  ``fmt`` names the stored format ("f32",
    "f16", "bf16" as raw uint16 bits, or "f64").  Returns an (M, n_cols)
    float64 array."""
    x = _as_storage(np.atleast_2d(x), fmt)
    M, ld = x.shape
    N = ld if n_cols is None else int(n_cols)
    y = np.empty((M, N), dtype=np.float64)
    rc = _load().orc_softmax_f64(x.ctypes.data, FORMATS[fmt], M, N, ld, y.ctypes.data, N)
    if rc != 0:
        raise ValueError(f"oracle rejected the call (status {rc})")
    return y


def softmax_prefix_f64(x: np.ndarray, fmt: str, period: int, offset: int = 0, n_cols: int | None = None,
                       row0: int = 0) -> np.ndarray:
    """Row softmax under a causal mask: the rows of ``x`` are rows row0, row0 + 1,
    ... of the masked tensor; row r keeps its first
    min(N, max(0, (r mod period) + 1 + offset)) elements, the rest is 0 in the
    result and never read."""
    x = _as_storage(np.atleast_2d(x), fmt)
    M, ld = x.shape
    N = ld if n_cols is None else int(n_cols)
    y = np.empty((M, N), dtype=np.float64)
    rc = _load().orc_softmax_prefix_f64(x.ctypes.data, FORMATS[fmt], M, N, ld, int(row0), int(period), int(offset),
                                        y.ctypes.data, N)
    if rc != 0:
        raise ValueError(f"oracle rejected the call (status {rc})")
    return y


def prefix_len(r: int, n: int, period: int, offset: int = 0) -> int:
    """L_r of softmax_prefix_f64."""
    return int(_load().orc_prefix_len(int(r), int(n), int(period), int(offset)))


def softmax_store(x: np.ndarray, fmt: str, n_cols: int | None = None, nthreads: int = 1,
                  out: np.ndarray | None = None) -> np.ndarray:
    """Same definition, result encoded into the input's stored format (the
    output has the same shape and row stride as ``x``; padding columns of a
    freshly made output are zero).  ``nthreads`` POSIX threads share the rows."""
    x = _as_storage(np.atleast_2d(x), fmt)
    M, ld = x.shape
    N = ld if n_cols is None else int(n_cols)
    if out is None:
        out = np.zeros_like(x)
    rc = _load().orc_softmax_store(x.ctypes.data, out.ctypes.data, FORMATS[fmt], M, N, ld,
                                   out.shape[1], int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle rejected the call (status {rc})")
    return out


def decode(bits: np.ndarray, fmt: str) -> np.ndarray:
    """Exact decoding of stored values into float64 (the oracle's own decoder)."""
    bits = _as_storage(bits, fmt)
    out = np.empty(bits.shape, dtype=np.float64)
    _load().orc_decode_array(bits.ctypes.data, FORMATS[fmt], bits.size, out.ctypes.data)
    return out


def encode(values: np.ndarray, fmt: str) -> np.ndarray:
    """Round-to-nearest-even encoding of float64 values (the oracle's own encoder)."""
    values = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(values.shape, dtype=_NP_STORAGE[fmt])
    _load().orc_encode_array(values.ctypes.data, FORMATS[fmt], values.size, out.ctypes.data)
    return out


def _vec(v, fmt, n):
    if v is None:
        return None
    v = _as_storage(np.ascontiguousarray(v).reshape(-1), fmt)
    if v.size != n:
        raise ValueError(f"expected {n} values, got {v.size}")
    return v


def rmsnorm_f64(x: np.ndarray, fmt: str, weight=None, eps: float = 1e-6, n_cols: int | None = None) -> np.ndarray:
    """RMSNorm of the rows of x (see softmax_f64 for the layout): y = x / sqrt(mean(x^2) + eps) * w."""
    x = _as_storage(np.atleast_2d(x), fmt)
    M, ld = x.shape
    N = ld if n_cols is None else int(n_cols)
    w = _vec(weight, fmt, N)
    y = np.empty((M, N), dtype=np.float64)
    rc = _load().orc_rmsnorm_f64(x.ctypes.data, FORMATS[fmt], M, N, ld, None if w is None else w.ctypes.data,
                                 float(eps), y.ctypes.data, N)
    if rc != 0:
        raise ValueError(f"oracle rejected the call (status {rc})")
    return y


def layernorm_f64(x: np.ndarray, fmt: str, weight=None, bias=None, eps: float = 1e-5,
                  n_cols: int | None = None) -> np.ndarray:
    """LayerNorm of the rows of x: y = (x - mean) / sqrt(var + eps) * w + b (population variance)."""
    x = _as_storage(np.atleast_2d(x), fmt)
    M, ld = x.shape
    N = ld if n_cols is None else int(n_cols)
    w = _vec(weight, fmt, N)
    b = _vec(bias, fmt, N)
    y = np.empty((M, N), dtype=np.float64)
    rc = _load().orc_layernorm_f64(x.ctypes.data, FORMATS[fmt], M, N, ld, None if w is None else w.ctypes.data,
                                   None if b is None else b.ctypes.data, float(eps), y.ctypes.data, N)
    if rc != 0:
        raise ValueError(f"oracle rejected the call (status {rc})")
    return y


def softmax_partial_f64(x: np.ndarray, fmt: str, n_cols: int | None = None) -> np.ndarray:
    """The (m, l) pair of every row of ``x`` over its first ``n_cols`` columns
    (one shard of a row split by columns): m the max, l the sum of exp(x - m).
    Returns an (M, 2) float64 array."""
    x = _as_storage(np.atleast_2d(x), fmt)
    M, ld = x.shape
    N = ld if n_cols is None else int(n_cols)
    ml = np.empty((M, 2), dtype=np.float64)
    rc = _load().orc_softmax_partial_f64(x.ctypes.data, FORMATS[fmt], M, N, ld, ml.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle rejected the call (status {rc})")
    return ml


def merge_pairs_f64(pairs: np.ndarray) -> np.ndarray:
    """Merge of the (R, M, 2) pairs of R shards into (M, 2), shard 0 first."""
    pairs = np.ascontiguousarray(pairs, dtype=np.float64)
    if pairs.ndim != 3 or pairs.shape[2] != 2:
        raise ValueError("pairs must have shape (R, M, 2)")
    R, M, _ = pairs.shape
    out = np.empty((M, 2), dtype=np.float64)
    rc = _load().orc_merge_pairs_f64(pairs.ctypes.data, R, M, out.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle rejected the call (status {rc})")
    return out


def softmax_finish_f64(x: np.ndarray, fmt: str, pairs: np.ndarray, n_cols: int | None = None) -> np.ndarray:
    """y = exp(x - m) / l over the rows of ``x`` with the merged (M, 2) pairs."""
    x = _as_storage(np.atleast_2d(x), fmt)
    M, ld = x.shape
    N = ld if n_cols is None else int(n_cols)
    pairs = np.ascontiguousarray(pairs, dtype=np.float64).reshape(M, 2)
    y = np.empty((M, N), dtype=np.float64)
    rc = _load().orc_softmax_finish_f64(x.ctypes.data, FORMATS[fmt], M, N, ld, pairs.ctypes.data, y.ctypes.data, N)
    if rc != 0:
        raise ValueError(f"oracle rejected the call (status {rc})")
    return y
