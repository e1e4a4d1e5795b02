"""GPU parity of the causal-mask row softmax (rowsoftmax_causal_fwd) against the
CPU oracle's softmax_prefix_f64, through the C ABI.

Covered: every kernel that implements the mask (register rows, the bulk-copy
ring, register-holding clusters), every storage type, periods that wrap, positive and negative
diagonal offsets (rows with nothing kept give NaN rows, as the oracle), NaN
garbage in the masked part (never used), padded strides, misaligned pointers,
in-place calls, and the causal benchmark workload at full size, where the
result must equal the plain softmax of the same -inf-masked scores bit for
bit (the same kernel, the masked loads skipped).
"""
import concurrent.futures as cf
import os

import numpy as np
import pytest
import torch

import memory_bound_row_gb300 as rs
import oracle
from memory_bound_row_gb300 import build
from memory_bound_row_gb300 import workloads as W

from _parity import FMT, check_all_rows, compare, to_storage_numpy

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


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


def _oracle(x, period, offset, row0=0):
    """Oracle rows row0 .. row0 + len(x) - 1 (float64), several threads."""
    fmt = FMT[x.dtype]
    xs = to_storage_numpy(x)
    M, N = xs.shape
    threads = max(1, min(16, os.cpu_count() or 1, M))
    blocks = [b for b in np.array_split(np.arange(M), threads) if len(b)]
    out = np.empty((M, N), dtype=np.float64)

    def work(idx):
        out[idx[0]: idx[-1] + 1] = oracle.softmax_prefix_f64(xs[idx[0]: idx[-1] + 1], fmt, period, offset, N,
                                                             row0=row0 + int(idx[0]))

    with cf.ThreadPoolExecutor(len(blocks)) as ex:
        list(ex.map(work, blocks))
    return out


def _garbage(x, period, offset, row0=0):
    """Write NaN into the masked part of x (which the kernels must not use)."""
    M, N = x.shape
    r = torch.arange(row0, row0 + M, device=x.device)
    keep = (r % period + 1 + offset).clamp(0, N)
    cols = torch.arange(N, device=x.device)
    x[cols[None, :] >= keep[:, None]] = float("nan")


def _aligned(M, N, dtype, seed, kind="normal1"):
    vec = 4 if dtype == "f32" else 8
    ld = -(-N // vec) * vec
    x = W.generate(W.custom(M, N, dtype, ld=ld, seed=seed, kind=kind), "cuda")[:, :N]
    out = torch.empty((M, ld), dtype=DT[dtype], device="cuda")[:, :N]
    return x, out


def _run(x, period, offset, out=None, options=None):
    y = rs.softmax_causal(x, period, offset, out=out, options=options)
    torch.cuda.synchronize()
    return y


def _servable(x, period, offset, options):
    rc, dev = rs.rowsoftmax_device_info()
    M, N = x.shape
    ld = x.stride(0) if M > 1 else N
    rc, plan = rs.rowsoftmax_causal_plan(x.data_ptr(), x.data_ptr() + (1 << 44), M, N, ld, ld, period, offset,
                                         rs.dtype_code(x.dtype), options, dev)
    assert rc in (rs.RS_OK, rs.RS_ERR_NO_PATH)
    return rc == rs.RS_OK


PATHS = {
    "auto": None,
    "rows": {"path": rs.RS_PATH_ROWS},
    "ring": {"path": rs.RS_PATH_RING},  # 16-bit rows: per-thread copies of the kept units
    "ring bulk": {"path": rs.RS_PATH_RING, "ring_values": rs.RS_RING_REGISTERS},  # whole rows, bulk copies
    "ring copies 3": {"path": rs.RS_PATH_RING, "ring_values": rs.RS_RING_THREAD_COPIES, "stages": 3},
    "cluster": {"path": rs.RS_PATH_CLUSTER},
    "cluster3": {"path": rs.RS_PATH_CLUSTER, "cluster_size": 3},
}


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("N", [1, 7, 100, 1000, 2048, 4104, 12345])
@pytest.mark.parametrize("period,offset", [("N", 0), (64, 0), (37, -3), (5, 5)])
def test_masked_rows_against_the_oracle(path, dtype, N, period, offset):
    P = N if period == "N" else period
    M = 3 * P if P <= 64 else min(2 * P, 300)
    x, out = _aligned(M, N, dtype, seed=N + P)
    opts = PATHS[path]
    if opts and not _servable(x, P, offset, opts):
        pytest.skip("this kernel does not serve the shape")
    ref = _oracle(x, P, offset)
    _garbage(x, P, offset)
    y = _run(x, P, offset, out=out, options=opts)
    compare(y, ref, dtype, f"causal {path} {dtype} N={N} P={P} D={offset}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cs", [2, 5, 8])
@pytest.mark.parametrize("N", [65536, 100003])
def test_wide_rows_on_clusters(dtype, cs, N):
    M, P = 24, 8
    x, out = _aligned(M, N, dtype, seed=cs)
    offset = N // 3  # partial slices, whole masked CTAs and fully kept rows
    opts = {"path": rs.RS_PATH_CLUSTER, "cluster_size": cs}
    if not _servable(x, P, offset, opts):
        pytest.skip("slice does not fit a CTA's registers at this cluster size")
    ref = _oracle(x, P, offset)
    _garbage(x, P, offset)
    y = _run(x, P, offset, out=out, options=opts)
    compare(y, ref, dtype, f"causal cluster cs={cs} N={N}")


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_padded_strides_misaligned_and_in_place(dtype):
    M, N, ld = 96, 1000, 1040
    P = 32
    base = W.generate(W.custom(M, N + 8, dtype, ld=ld, seed=4), "cuda")
    x = base[:, 3: 3 + N]  # misaligned: element-wise kernels
    ref = _oracle(x, P, 2)
    _garbage(x, P, 2)
    y = _run(x, P, 2)
    compare(y, ref, dtype, "causal misaligned")
    x2 = W.generate(W.custom(M, N, dtype, ld=ld, seed=5), "cuda")[:, :N]
    ref2 = _oracle(x2, P, 0)
    _garbage(x2, P, 0)
    y2 = _run(x2, P, 0, out=x2)  # in place, padded stride
    assert y2.data_ptr() == x2.data_ptr()
    compare(y2, ref2, dtype, "causal in place")


def test_causal_workload_full_size_equals_the_plain_softmax():
    # The bf16 causal-score workload already holds -inf above the diagonal: the
    # masked call must give the plain call's result bit for bit without using
    # the masked half; with NaN written there instead, still the same.
    w = W.WORKLOADS["bf16_causal_16x32x2048"]
    x = W.generate(w, "cuda")
    plain = rs.softmax(x)
    masked = _run(x, 2048, 0)
    assert torch.equal(plain.view(torch.int16), masked.view(torch.int16))
    # every row against the prefix oracle, with the masked part made NaN first
    # (the oracle never reads it either)
    _garbage(x, 2048, 0)
    check_all_rows("prefix", x, masked, w.N, period=2048, offset=0, what="causal softmax bf16 1048576 x 2048",
                   group="workloads")
    again = _run(x, 2048, 0)
    assert torch.equal(plain.view(torch.int16), again.view(torch.int16))
    del x, plain, masked, again
    torch.cuda.empty_cache()


def test_kv_cache_offset_layout():
    # Scores [B, H, S_q, S_k] with S_k > S_q (cached keys): period S_q, offset S_k - S_q.
    B, H, Sq, Sk = 2, 4, 48, 80
    x = W.generate(W.custom(B * H * Sq, Sk, "f16", seed=9), "cuda")
    ref = _oracle(x, Sq, Sk - Sq)
    _garbage(x, Sq, Sk - Sq)
    y = _run(x, Sq, Sk - Sq)
    compare(y, ref, "f16", "kv-cache layout")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("N,tpr", [(256, 4), (300, 8), (512, 8), (768, 16), (1024, 16)])
def test_causal_narrow_16bit_rows_on_few_lanes(dtype, N, tpr):
    # The causal mask's rows of 32 to 256 units: the fewest lanes that hold the
    # row at up to 8 units a thread, 512-thread CTAs, enough rows for the rule;
    # NaN in the masked part; every row against the oracle.
    M = (512 // tpr) * 4 * 152 + 37
    x, out = _aligned(M, N, dtype, seed=N + 19)
    rc, dev = rs.rowsoftmax_device_info()
    rc, plan = rs.rowsoftmax_causal_plan(x.data_ptr(), out.data_ptr(), M, N, x.stride(0), out.stride(0), N, 0,
                                         rs.dtype_code(x.dtype), None, dev)
    assert rc == rs.RS_OK and plan["ring_values"] == rs.RS_RING_THREAD_COPIES
    assert plan["threads_per_row"] == tpr and plan["block_threads"] == 512
    xc = x.clone()
    _garbage(x, N, 0)
    y = _run(x, N, 0, out=out)
    check_all_rows("prefix", xc, y, N, period=N, offset=0, what=f"causal narrow rows {dtype} {M}x{N}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("N", [2050, 2560, 3072, 4096, 4608, 5120, 6000, 12288, 20480, 24576, 32768])
@pytest.mark.parametrize("mask", ["period N", "period 97"])
def test_causal_16bit_rows_of_2049_to_32768_values_on_the_copy_ring(dtype, N, mask):
    # The planner's measured shape for the causal mask's 16-bit rows of 257 to
    # 4096 units: its copy ring at 8 units a thread (5 or 6 where they fill
    # whole warps exactly and 8 do not, or where they fill 16 warps), one row a
    # CTA; NaN written into the masked part; every row against the oracle.
    M = 4 * 152 + 37
    period, offset = (N, 0) if mask == "period N" else (97, N // 2)
    x, out = _aligned(M, N, dtype, seed=N + 17)
    assert _servable(x, period, offset, None)
    rc, dev = rs.rowsoftmax_device_info()
    rc, plan = rs.rowsoftmax_causal_plan(x.data_ptr(), out.data_ptr(), M, N, x.stride(0), out.stride(0), period,
                                         offset, rs.dtype_code(x.dtype), None, dev)
    assert plan["path"] == rs.RS_PATH_RING and plan["ring_values"] == rs.RS_RING_THREAD_COPIES
    assert plan["vec_per_thread"] in (5, 6, 8) and plan["block_threads"] == plan["threads_per_row"]
    xc = x.clone()
    _garbage(x, period, offset)
    y = _run(x, period, offset, out=out)
    check_all_rows("prefix", xc, y, N, period=period, offset=offset,
                   what=f"causal copy ring {dtype} {M}x{N} {mask}")


@pytest.mark.parametrize("path", ["rows", "ring", "ring bulk", "cluster"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_non_finite_values_in_the_kept_prefix(path, dtype):
    # A NaN or +inf inside the kept prefix makes the kept part NaN; the masked
    # part stays exactly 0, as the definition states (the softmax of the kept
    # values, 0 past them); a row that keeps nothing is NaN throughout.
    N = 2048 if path != "cluster" else 65536
    P, offset = 16, (0 if path != "cluster" else N // 2)
    M = 2 * P
    x, out = _aligned(M, N, dtype, seed=77)
    keep = [min(N, max(0, r % P + 1 + offset)) for r in range(M)]
    x[1, 0] = float("nan")
    x[5, keep[5] - 1] = float("inf")
    x[9, keep[9] // 2] = float("nan")
    opts = PATHS[path]
    if not _servable(x, P, offset, opts):
        pytest.skip("this kernel does not serve the shape")
    ref = _oracle(x, P, offset)
    _garbage(x, P, offset)
    y = _run(x, P, offset, out=out, options=opts)
    compare(y, ref, dtype, f"non-finite kept values, {path} {dtype}")
    yd = y.double().cpu().numpy()
    for r in (1, 5, 9):
        assert np.all(np.isnan(yd[r, :keep[r]])) and np.all(yd[r, keep[r]:] == 0.0)
    # a period with an empty prefix (offset -1 on row 0 of each period)
    x2, out2 = _aligned(M, N, dtype, seed=78)
    if not _servable(x2, P, -1, opts):
        return
    ref2 = _oracle(x2, P, -1)
    y2 = _run(x2, P, -1, out=out2, options=opts)
    compare(y2, ref2, dtype, f"empty prefixes, {path} {dtype}")
    assert bool(torch.isnan(y2[0]).all()) and bool(torch.isnan(y2[P]).all())
