"""Seeded synthetic inputs for the row softmax and the row normalisations:
the five benchmark workloads, the extra shapes used by the tests and the
normalisations' weight and bias vectors.

This module only makes input data; it contains none of the softmax or
normalisation arithmetic.  Values are a pure function of (seed, stream, flat index): a
SplitMix64 hash of the counter gives uniforms on (0, 1), and the Box-Muller
transform (cosine branch) turns two uniforms into one standard normal.  Any
subset of rows can therefore be generated on its own and equals the same rows
of the full tensor generated on the same device.  Values are formed in
float64, rounded to float32 and then to the storage type (round to nearest
even), on the device the tensor is made on.

Workloads (rows x cols, storage type, distribution):
  fp32_1024x1024      fp32 1024 x 1024, contiguous, N(0, 1), seed 0
  fp32_8192x5000_ld5120  fp32 8192 x 5000, row stride 5120, N(0, var 4);
                      82 rows (1 %) are one constant c ~ U[-5, 5]
  bf16_32768x8192     bf16 32768 x 8192, U[-20, 20]; 3277 rows (10 %) get +1e4
  fp16_512x131072     fp16 512 x 131072, N(0, var 2), one +15 spike per row
  bf16_causal_16x32x2048  bf16 [16, 32, 2048, 2048] attention scores viewed as
                      1048576 x 2048, N(0, 1)/sqrt(128), -inf where col > row mod 2048

The normalisations run on the same shapes and recipes, except that the causal
scores' -inf entries (which make every normalised row NaN) are left out: that
workload becomes N(0, 1)/sqrt(128) everywhere (norm_workload).  Weight
vectors are 1 + N(0, 1)/4 and bias vectors N(0, 1)/2 (norm_params).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

_M64 = (1 << 64) - 1


def _s64(u: int) -> int:
    """A uint64 constant as the int64 with the same bits."""
    u &= _M64
    return u - (1 << 64) if u >= (1 << 63) else u


_GOLDEN = _s64(0x9E3779B97F4A7C15)
_MIX1 = _s64(0xBF58476D1CE4E5B9)
_MIX2 = _s64(0x94D049BB133111EB)


def _shr(z: torch.Tensor, k: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns."""
    return (z >> k) & ((1 << (64 - k)) - 1)


def _splitmix64(counter: torch.Tensor, key: int) -> torch.Tensor:
    z = counter * _GOLDEN + _s64(key)
    z = (z ^ _shr(z, 30)) * _MIX1
    z = (z ^ _shr(z, 27)) * _MIX2
    return z ^ _shr(z, 31)


def _key(seed: int, stream: int) -> int:
    return _s64((seed * 0x100000001B3 + stream * 0x9E3779B1 + 0x632BE59BD9B4E019) & _M64)


def uniform(counter: torch.Tensor, seed: int, stream: int) -> torch.Tensor:
    """float64 uniforms on (0, 1) from the top 53 bits of the hash."""
    h = _shr(_splitmix64(counter, _key(seed, stream)), 11)
    return (h.to(torch.float64) + 0.5) * (2.0 ** -53)


def normal(counter: torch.Tensor, seed: int, stream: int) -> torch.Tensor:
    """float64 standard normals (Box-Muller, cosine branch; counters 2i, 2i+1)."""
    u1 = uniform(2 * counter, seed, stream)
    u2 = uniform(2 * counter + 1, seed, stream)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)


def pick_rows(M: int, count: int, seed: int, stream: int, device) -> torch.Tensor:
    """Exactly `count` distinct rows of M, chosen by ranking a per-row hash."""
    h = _splitmix64(torch.arange(M, dtype=torch.int64, device=device), _key(seed, stream))
    return torch.argsort(h)[:count].sort().values


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str      # "f32", "f16", "bf16"
    M: int
    N: int
    ld: int         # row stride of input and output, in elements
    seed: int
    kind: str       # distribution recipe, see generate()
    description: str

    @property
    def elem_size(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def algorithmic_bytes(self) -> int:
        """One read and one write of every element: M * N * (in + out size)."""
        return self.M * self.N * 2 * self.elem_size

    @property
    def torch_dtype(self) -> torch.dtype:
        return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[self.dtype]


WORKLOADS = {
    "fp32_1024x1024": Workload("fp32_1024x1024", "f32", 1024, 1024, 1024, 0, "normal1",
                               "fp32 1024 x 1024, contiguous, N(0,1), seed 0"),
    "fp32_8192x5000_ld5120": Workload("fp32_8192x5000_ld5120", "f32", 8192, 5000, 5120, 1, "normal2_const",
                                      "fp32 8192 x 5000, row stride 5120, N(0, var 4), 82 constant rows"),
    "bf16_32768x8192": Workload("bf16_32768x8192", "bf16", 32768, 8192, 8192, 2, "uniform20_offset",
                                "bf16 32768 x 8192, U[-20,20], +1e4 on 3277 rows"),
    "fp16_512x131072": Workload("fp16_512x131072", "f16", 512, 131072, 131072, 3, "normal_spike",
                                "fp16 512 x 131072, N(0, var 2), one +15 spike per row"),
    "bf16_causal_16x32x2048": Workload("bf16_causal_16x32x2048", "bf16", 16 * 32 * 2048, 2048, 2048, 4,
                                       "causal_scores",
                                       "bf16 [16,32,2048,2048] causal scores as 1048576 x 2048, "
                                       "N(0,1)/sqrt(128), -inf above the diagonal"),
}

# The benchmark workload order used by the tests and the bench.
ORDER = ["fp32_1024x1024", "fp32_8192x5000_ld5120", "bf16_32768x8192", "fp16_512x131072",
         "bf16_causal_16x32x2048"]


def custom(M: int, N: int, dtype: str = "f32", ld: int | None = None, seed: int = 0,
           kind: str = "normal1") -> Workload:
    """A workload of any shape with one of the recipes of generate()."""
    return Workload(f"{dtype}_{M}x{N}", dtype, M, N, ld or N, seed, kind, f"{dtype} {M} x {N} {kind}")


def _values(w: Workload, rows: torch.Tensor, cols: torch.Tensor) -> torch.Tensor:
    """float64 values of the given rows (1-D int64) at the given columns."""
    r = rows[:, None]
    c = cols[None, :]
    flat = r * w.N + c
    if w.kind == "normal1":
        return normal(flat, w.seed, 0)
    if w.kind == "normal2_const":
        v = 2.0 * normal(flat, w.seed, 0)
        const_rows = pick_rows(w.M, round(0.01 * w.M), w.seed, 1, rows.device)
        is_const = torch.isin(rows, const_rows)
        cval = -5.0 + 10.0 * uniform(rows, w.seed, 2)
        return torch.where(is_const[:, None], cval[:, None].expand_as(v), v)
    if w.kind == "uniform20_offset":
        v = -20.0 + 40.0 * uniform(flat, w.seed, 0)
        off_rows = pick_rows(w.M, round(0.10 * w.M), w.seed, 1, rows.device)
        return v + torch.where(torch.isin(rows, off_rows), 1e4, 0.0)[:, None]
    if w.kind == "normal_spike":
        v = math.sqrt(2.0) * normal(flat, w.seed, 0)
        spike_col = (_shr(_splitmix64(rows, _key(w.seed, 3)), 1) % w.N)[:, None]
        return v + torch.where(c == spike_col, 15.0, 0.0)
    if w.kind == "causal_scores":
        v = normal(flat, w.seed, 0) / math.sqrt(128.0)
        return torch.where(c > (r % 2048), -math.inf, v)
    if w.kind == "scores_unmasked":
        return normal(flat, w.seed, 0) / math.sqrt(128.0)
    if w.kind == "offset50":  # a large common offset: N(50, 1)
        return 50.0 + normal(flat, w.seed, 0)
    raise ValueError(f"unknown recipe {w.kind}")


def generate(w: Workload, device="cpu", row_start: int = 0, row_count: int | None = None,
             pad_value: float = float("nan"), chunk_elems: int = 1 << 25) -> torch.Tensor:
    """Rows [row_start, row_start + row_count) of workload `w` as a (rows, ld)
    tensor of its storage type on `device`; padding columns hold pad_value."""
    if row_count is None:
        row_count = w.M - row_start
    out = torch.empty((row_count, w.ld), dtype=w.torch_dtype, device=device)
    if w.ld > w.N:
        out[:, w.N:] = pad_value
    cols = torch.arange(w.N, dtype=torch.int64, device=device)
    step = max(1, chunk_elems // max(w.N, 1))
    for r0 in range(0, row_count, step):
        r1 = min(row_count, r0 + step)
        rows = torch.arange(row_start + r0, row_start + r1, dtype=torch.int64, device=device)
        out[r0:r1, : w.N] = _values(w, rows, cols).to(torch.float32).to(w.torch_dtype)
    return out


def generate_rows(w: Workload, rows: torch.Tensor, device="cpu") -> torch.Tensor:
    """Arbitrary rows (1-D int64) of workload `w`, shape (len(rows), N)."""
    rows = rows.to(device=device, dtype=torch.int64)
    cols = torch.arange(w.N, dtype=torch.int64, device=device)
    return _values(w, rows, cols).to(torch.float32).to(w.torch_dtype)


def norm_workload(name: str) -> Workload:
    """Benchmark workload `name` as the normalisations use it (the causal
    scores without their -inf mask)."""
    w = WORKLOADS[name]
    if w.kind == "causal_scores":
        return Workload(w.name, w.dtype, w.M, w.N, w.ld, w.seed, "scores_unmasked",
                        w.description.replace(", -inf above the diagonal", "").replace(
                            ", -inf where col > row mod 2048", "") + ", unmasked")
    return w


def norm_params(N: int, dtype: str, seed: int = 0, device="cpu") -> tuple[torch.Tensor, torch.Tensor]:
    """Weight (1 + N(0,1)/4) and bias (N(0,1)/2) vectors of N values in the
    storage type `dtype`, seeded."""
    td = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    idx = torch.arange(N, dtype=torch.int64, device=device)
    w = 1.0 + 0.25 * normal(idx, seed, 10)
    b = 0.5 * normal(idx, seed, 11)
    return w.to(torch.float32).to(td), b.to(torch.float32).to(td)
