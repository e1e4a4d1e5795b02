"""GPU parity of the row normalisations (RMSNorm, LayerNorm) against the CPU
oracle, through the C ABI.

Each case makes seeded inputs, weight and bias vectors on the GPU, runs the
normalisation through the ctypes binding of librowsoftmax.so and compares
every output element with the oracle under the bound of tests/_parity.py.
Covered: the register-row, ring, register-holding cluster and streaming
kernels of every storage type,
forced thread shapes, persistent grids that loop over rows, ragged tails,
element-wise access (misaligned pointers, odd strides), padded rows with
guard bands, in-place calls, optional weight and bias, special values, rows
with a large common offset, eps = 0, the benchmark shapes at full size
(sampled rows) in the launch configuration the benchmark times, and the
maximum sizes.
"""
import math

import numpy as np
import pytest
import torch

import memory_bound_row_gb300 as rs
from memory_bound_row_gb300 import build
from memory_bound_row_gb300 import workloads as W

from _parity import check_all_rows, compare_norm, oracle_norm_rows

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
OPS = ["rms", "ln"]
EPS = {"rms": 1e-6, "ln": 1e-5}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    rc, flags = rs.rowsoftmax_device_status(clear=True)
    assert rc == rs.RS_OK
    yield
    rc, flags = rs.rowsoftmax_device_status(clear=False)
    assert rc == rs.RS_OK and flags == 0, f"device status word {flags:#x}"


def _params(N, dtype, seed=0, weight=True, bias=True):
    w, b = W.norm_params(N, dtype, seed, "cuda")
    return (w if weight else None), (b if bias else None)


def _run(op, x, w=None, b=None, eps=None, out=None, options=None):
    eps = EPS[op] if eps is None else eps
    if op == "rms":
        y = rs.rmsnorm(x, w, eps=eps, out=out, options=options)
    else:
        y = rs.layernorm(x, w, b, eps=eps, out=out, options=options)
    torch.cuda.synchronize()
    return y


def _check(op, x, y, w=None, b=None, eps=None, what=""):
    eps = EPS[op] if eps is None else eps
    N = x.shape[1]
    ref = oracle_norm_rows(op, x, N, w, b if op == "ln" else None, eps)
    return compare_norm(y[:, :N], ref, x, op, w, b if op == "ln" else None, eps, what)


def _servable(op, x, w, b, options):
    rc, dev = rs.rowsoftmax_device_info()
    assert rc == rs.RS_OK
    M, N = x.shape
    code = rs.RS_OP_RMSNORM if op == "rms" else rs.RS_OP_LAYERNORM
    rc, plan = rs.rownorm_plan(code, x.data_ptr(), x.data_ptr() + (1 << 44), None if w is None else w.data_ptr(),
                               None if (b is None or op == "rms") else b.data_ptr(), M, N,
                               x.stride(0) if M > 1 else N, x.stride(0) if M > 1 else N, EPS[op],
                               rs.dtype_code(x.dtype), options, dev)
    assert rc in (rs.RS_OK, rs.RS_ERR_NO_PATH)
    return rc == rs.RS_OK, plan


def _input(M, N, dtype, ld=None, kind="normal1", seed=0):
    return W.generate(W.custom(M, N, dtype, ld=ld, seed=seed, kind=kind), "cuda")


def _aligned(M, N, dtype, kind="normal1", seed=0):
    vec = 4 if dtype == "f32" else 8
    ld = -(-N // vec) * vec
    x = _input(M, N, dtype, ld=ld, kind=kind, seed=seed)[:, :N]
    out = torch.empty((M, ld), dtype=DT[dtype], device="cuda")[:, :N]
    return x, out


SHAPES = [(1, 1), (3, 2), (5, 3), (37, 7), (64, 8), (33, 33), (300, 100), (17, 255), (129, 781), (64, 1000),
          (40, 1500), (24, 4096), (16, 5000), (8, 8192), (5, 12288), (3, 16384)]


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("M,N", SHAPES)
def test_auto_path_small_shapes(op, dtype, M, N):
    x, out = _aligned(M, N, dtype, seed=M * 7 + N)
    w, b = _params(N, dtype, seed=N)
    y = _run(op, x, w, b, out=out)
    _check(op, x, y, w, b, what=f"{op} {dtype} {M}x{N}")


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("weight,bias", [(False, False), (True, False), (False, True)])
@pytest.mark.parametrize("N", [100, 4096])
def test_optional_weight_and_bias(op, dtype, weight, bias, N):
    x, out = _aligned(50, N, dtype, seed=3)
    w, b = _params(N, dtype, seed=5, weight=weight, bias=bias)
    y = _run(op, x, w, b, out=out)
    _check(op, x, y, w, b, what=f"{op} w={weight} b={bias}")


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("tpr,vpt", [(1, 1), (2, 2), (4, 3), (8, 6), (16, 8), (32, 1), (32, 5), (32, 6), (64, 4), (96, 2),
                                     (128, 8), (256, 3), (1024, 1)])
@pytest.mark.parametrize("grid_limit", [0, 3])
def test_rows_path_thread_shapes(op, dtype, tpr, vpt, grid_limit):
    vec = 4 if dtype == "f32" else 8
    N = max(1, tpr * vpt * vec - 3)  # a ragged last unit
    M = 70
    x, out = _aligned(M, N, dtype, seed=tpr + vpt)
    w, b = _params(N, dtype, seed=tpr)
    opts = {"path": rs.RS_PATH_ROWS, "threads_per_row": tpr, "vec_per_thread": vpt, "grid_limit": grid_limit}
    ok, _ = _servable(op, x, w, b, opts)
    if not ok:
        pytest.skip("register budget of this shape")
    y = _run(op, x, w, b, out=out, options=opts)
    _check(op, x, y, w, b, what=f"{op} rows tpr={tpr} vpt={vpt}")


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("N", [300, 640, 1280])
def test_fp32_rows_that_need_5_units_a_thread(op, N):
    # fp32 rows of 75, 160 and 320 units on 16, 32 and 64 lanes take 5 units a
    # thread on the register rows (a thread of 16 rows a CTA, 8 and 4 rows);
    # many rows, so that every CTA of the grid serves its rows; every row
    # against the oracle.
    M = 20011
    x, out = _aligned(M, N, "f32", seed=N + 5)
    wt, bs = _params(N, "f32", seed=N + 1)
    ok, plan = _servable(op, x, wt, bs, None)
    assert ok and plan["path"] == rs.RS_PATH_ROWS and plan["vec_per_thread"] == 5
    y = _run(op, x, wt, bs, out=out)
    check_all_rows(op, x, y, N, weight=wt, bias=bs if op == "ln" else None, eps=EPS[op],
                   what=f"{'RMSNorm' if op == 'rms' else 'LayerNorm'} fp32 {M}x{N} at 5 units a thread")


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("N", [4096, 8192, 12288, 20480, 28672, 32768, 36000])
def test_auto_path_wide_16bit_rows(op, dtype, N):
    # The planner's wide 16-bit rows: the held-parameter LayerNorm (4096,
    # 8192), the ring with 32 values a thread up to 56 KB (LayerNorm) or 64 KB
    # (RMSNorm), the clusters beyond; persistent grids loop over the rows.
    M = 700 if N <= 12288 else 260
    x, out = _aligned(M, N, dtype, kind="offset50" if op == "ln" else "normal1", seed=N)
    w, b = _params(N, dtype, seed=N)
    y = _run(op, x, w, b, out=out)
    _check(op, x, y, w, b, what=f"{op} auto wide {dtype} N={N}")


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("path", [rs.RS_PATH_ROWS, rs.RS_PATH_RING])
@pytest.mark.parametrize("tpr", [1, 2, 4, 8, 16, 32])
@pytest.mark.parametrize("short", [0, 1, 3, "unit", "half"])
def test_layernorm_rows_inside_one_warp(dtype, path, tpr, short):
    # Rows held by one warp take each lane's moments about its own mean and
    # merge them in one butterfly; ragged rows give the lanes different
    # counts (a partial unit, lanes with one unit fewer, empty lanes), and a
    # large common offset with unit variance is where a wrong merge shows.
    vec = 4 if dtype == "f32" else 8
    vpt = 2
    cap = tpr * vpt * vec
    k = {"unit": vec + 1, "half": cap // 2}.get(short, short)
    N = max(1, cap - k)
    x, out = _aligned(50, N, dtype, kind="offset50", seed=tpr + vec)
    x[7, :] = 1000.0  # a constant row (zero variance)
    w, b = _params(N, dtype, seed=tpr)
    opts = {"path": path, "threads_per_row": tpr, "vec_per_thread": vpt}
    ok, plan = _servable("ln", x, w, b, opts)
    if not ok:
        pytest.skip("no plan for this shape")
    assert plan["threads_per_row"] == tpr
    y = _run("ln", x, w, b, out=out, options=opts)
    _check("ln", x, y, w, b, what=f"ln one warp {dtype} tpr={tpr} N={N}")


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("path", [rs.RS_PATH_ROWS, rs.RS_PATH_RING])
@pytest.mark.parametrize("tpr,vpt", [(64, 1), (64, 8), (128, 4), (256, 2), (512, 1), (1024, 1), (96, 2), (160, 3)])
@pytest.mark.parametrize("grid_limit", [0, 3])
def test_layernorm_rows_that_fill_their_warps(dtype, path, tpr, vpt, grid_limit):
    # Rows that fill their threads exactly over a power-of-two number of warps
    # merge equal-count moments across the warps; 3 and 5 warps a row take
    # the two-reduction LayerNorm.  Persistent grids (grid_limit) loop over
    # rows, reusing the per-warp partials.
    vec = 4 if dtype == "f32" else 8
    N = tpr * vpt * vec
    x, out = _aligned(40, N, dtype, kind="offset50", seed=tpr * vpt)
    x[3, :] = -7.0  # a constant row
    w, b = _params(N, dtype, seed=vpt)
    opts = {"path": path, "threads_per_row": tpr, "vec_per_thread": vpt, "grid_limit": grid_limit}
    ok, plan = _servable("ln", x, w, b, opts)
    if not ok:
        pytest.skip("no plan for this shape")
    assert plan["threads_per_row"] == tpr
    y = _run("ln", x, w, b, out=out, options=opts)
    _check("ln", x, y, w, b, what=f"ln filled warps {dtype} tpr={tpr} vpt={vpt}")


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("N", [1, 5, 31, 100, 777, 4096])
def test_rows_path_element_wise(op, dtype, N):
    x = _input(45, N, dtype, seed=N)
    w, b = _params(N, dtype, seed=1)
    y = _run(op, x, w, b, options={"force_scalar": 1})
    _check(op, x, y, w, b, what=f"{op} scalar {dtype} N={N}")


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("N", [8, 100, 1001, 2048, 5000, 8192, 12345])
@pytest.mark.parametrize("stages", [2, 3, 8])
@pytest.mark.parametrize("grid_limit", [0, 2])
def test_ring_path(op, dtype, N, stages, grid_limit):
    x, out = _aligned(97, N, dtype, seed=N + stages)
    w, b = _params(N, dtype, seed=stages)
    opts = {"path": rs.RS_PATH_RING, "stages": stages, "grid_limit": grid_limit}
    ok, _ = _servable(op, x, w, b, opts)
    if not ok:
        pytest.skip("ring stages do not fit shared memory")
    y = _run(op, x, w, b, out=out, options=opts)
    _check(op, x, y, w, b, what=f"{op} ring {dtype} N={N} stages={stages}")


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("tpr,vpt", [(1, 1), (4, 2), (32, 8), (64, 4), (160, 6), (256, 4), (512, 2), (1024, 1)])
@pytest.mark.parametrize("grid_limit", [0, 3])
def test_ring_thread_shapes_and_wraparound(op, dtype, tpr, vpt, grid_limit):
    vec = 4 if dtype == "f32" else 8
    N = tpr * vpt * vec - 5 if tpr * vpt * vec > 5 else tpr * vpt * vec
    x, out = _aligned(41, N, dtype, seed=tpr * vpt)
    w, b = _params(N, dtype, seed=vpt)
    opts = {"path": rs.RS_PATH_RING, "threads_per_row": tpr, "vec_per_thread": vpt, "grid_limit": grid_limit}
    ok, _ = _servable(op, x, w, b, opts)
    if not ok:
        pytest.skip("no ring plan for this shape")
    y = _run(op, x, w, b, out=out, options=opts)
    _check(op, x, y, w, b, what=f"{op} ring tpr={tpr} vpt={vpt} grid_limit={grid_limit}")


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("scalar", [0, 1])
@pytest.mark.parametrize("N", [1, 3, 1000, 70001, 131075])
@pytest.mark.parametrize("grid_limit", [0, 2])
def test_stream_path(op, dtype, scalar, N, grid_limit):
    x, out = _aligned(9, N, dtype, seed=N, kind="normal_spike")
    w, b = _params(N, dtype, seed=2)
    opts = {"path": rs.RS_PATH_STREAM, "force_scalar": scalar, "grid_limit": grid_limit}
    y = _run(op, x, w, b, out=out, options=opts)
    _check(op, x, y, w, b, what=f"{op} stream {dtype} N={N} scalar={scalar}")


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("cs", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("N", [8, 1000, 4104, 65536, 100003])
@pytest.mark.parametrize("grid_limit", [0, 2])
def test_cluster_path(op, dtype, cs, N, grid_limit):
    # Register-holding clusters; cluster sizes that are not powers of two,
    # slices past the end of short rows (empty CTAs), persistent clusters
    # looping over rows (grid_limit).
    x, out = _aligned(7, N, dtype, seed=N + cs, kind="offset50" if op == "ln" else "normal_spike")
    w, b = _params(N, dtype, seed=cs)
    opts = {"path": rs.RS_PATH_CLUSTER, "cluster_size": cs, "grid_limit": grid_limit * cs}
    ok, plan = _servable(op, x, w, b, opts)
    if not ok:
        pytest.skip("slice does not fit a CTA's registers at this cluster size")
    assert plan["ring_values"] == rs.RS_RING_REGISTERS
    y = _run(op, x, w, b, out=out, options=opts)
    _check(op, x, y, w, b, what=f"{op} cluster {dtype} N={N} cs={cs}")


@pytest.mark.parametrize("op", OPS)
def test_paths_agree_on_the_same_input(op):
    x, _ = _aligned(64, 3000, "bf16", seed=11)
    w, b = _params(3000, "bf16", seed=11)
    ys = [_run(op, x, w, b, options={"path": p})
          for p in (rs.RS_PATH_ROWS, rs.RS_PATH_RING, rs.RS_PATH_CLUSTER, rs.RS_PATH_STREAM)]
    for y in ys:
        _check(op, x, y, w, b, what=f"{op} paths")


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_padded_strides_and_guard_bands(op, dtype):
    M, N, ld = 33, 1000, 1040
    x = _input(M, N, dtype, ld=ld, seed=4)  # padding columns hold NaN
    buf = torch.full((M + 2, ld), float("nan"), dtype=DT[dtype], device="cuda")
    before = buf.clone()
    out = buf[1: M + 1, :N]
    w, b = _params(N, dtype, seed=4)
    y = _run(op, x[:, :N], w, b, out=out)
    _check(op, x[:, :N], y, w, b, what=f"{op} padded")
    bits = torch.int32 if dtype == "f32" else torch.int16
    assert torch.equal(buf[0].view(bits), before[0].view(bits))
    assert torch.equal(buf[M + 1].view(bits), before[M + 1].view(bits))
    assert torch.equal(buf[1: M + 1, N:].view(bits), before[1: M + 1, N:].view(bits))


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("shift", [1, 3])
def test_misaligned_pointers_use_element_wise_access(op, dtype, shift):
    M, N = 20, 3001
    base = _input(M, N + 8, dtype, seed=shift)
    x = base[:, shift: shift + N]
    wbuf, bbuf = _params(N + 8, dtype, seed=shift)
    w, b = wbuf[shift: shift + N], bbuf[1: 1 + N]
    ok, plan = _servable(op, x, w, b, None)
    assert ok and plan["vec_elems"] == 1
    y = _run(op, x, w, b)
    _check(op, x, y, w, b, what=f"{op} misaligned shift={shift}")


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("N", [100, 8192, 70000])
@pytest.mark.parametrize("path", [rs.RS_PATH_AUTO, rs.RS_PATH_ROWS, rs.RS_PATH_RING, rs.RS_PATH_CLUSTER,
                                  rs.RS_PATH_STREAM])
def test_in_place(op, dtype, N, path):
    x, _ = _aligned(12, N, dtype, seed=N)
    w, b = _params(N, dtype, seed=N)
    opts = {"path": path}
    ok, _ = _servable(op, x, w, b, opts)
    if not ok:
        pytest.skip("path does not serve this shape")
    x0 = x.clone()
    y = _run(op, x, w, b, out=x, options=opts)
    assert y.data_ptr() == x.data_ptr()
    _check(op, x0, y, w, b, what=f"{op} in place")


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("path", [rs.RS_PATH_ROWS, rs.RS_PATH_RING, rs.RS_PATH_CLUSTER, rs.RS_PATH_STREAM])
def test_special_values(op, dtype, path):
    M, N = 8, 1000
    x, out = _aligned(M, N, dtype, seed=9)
    x[0, 5] = float("inf")
    x[1, 7] = float("-inf")
    x[2, 0] = float("nan")
    x[3, :] = 0.0                        # RMSNorm gives 0, LayerNorm the bias
    x[4, :] = 2.5                        # constant row: LayerNorm gives the bias
    x[5, 3] = float("inf")
    x[5, 4] = float("-inf")
    w, b = _params(N, dtype, seed=9)
    ok, _ = _servable(op, x, w, b, {"path": path})
    if not ok:
        pytest.skip("path does not serve this shape")
    y = _run(op, x, w, b, out=out, options={"path": path})
    _check(op, x, y, w, b, what=f"{op} special values")
    if op == "rms":
        assert bool((y[3] == 0).all())
    else:
        assert torch.equal(y[3], b)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("N", [1500, 8192, 100000])
def test_layernorm_of_rows_with_a_large_offset(dtype, N):
    # N(50, 1) rows: the two-pass variance keeps its accuracy where
    # E[x^2] - E[x]^2 would cancel.
    x, out = _aligned(16, N, dtype, kind="offset50", seed=N)
    w, b = _params(N, dtype, seed=1)
    y = _run("ln", x, w, b, out=out)
    _check("ln", x, y, w, b, what=f"ln offset {dtype} N={N}")


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("N", [1, 2, 1000])
def test_eps_zero(op, N):
    x, out = _aligned(30, N, "f32", seed=N)
    w, b = _params(N, "f32", seed=N)
    if N == 1 and op == "ln":
        pytest.skip("one-element rows have zero variance: 0/0 at eps = 0")
    y = _run(op, x, w, b, eps=0.0, out=out)
    _check(op, x, y, w, b, eps=0.0, what=f"{op} eps=0")


def test_rejections_on_device_memory():
    x = torch.randn(8, 64, device="cuda")
    out = torch.empty_like(x)
    w = out[0]  # the weight inside the output
    with pytest.raises(rs.RowSoftmaxError) as e:
        rs.rmsnorm(x, w, out=out)
    assert e.value.status == rs.RS_ERR_OVERLAP
    host_w = torch.ones(64)
    rc = rs.rmsnorm_fwd(x.data_ptr(), out.data_ptr(), host_w.data_ptr(), 8, 64, 64, 64, 1e-6, rs.RS_F32, 0)
    assert rc == rs.RS_ERR_NOT_DEVICE_MEMORY


def test_nonzero_stream():
    x, out = _aligned(256, 4096, "bf16", seed=1)
    w, b = _params(4096, "bf16", seed=1)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y = rs.layernorm(x, w, b, out=out)
    s.synchronize()
    _check("ln", x, y, w, b, what="side stream")


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("N", [256, 512, 768, 1024, 1280, 2560, 3072, 3584, 3840, 4608, 5120, 5632, 6144, 6400, 7680,
                               10240, 12288, 12800, 16384, 17920, 18432, 20480, 24576, 4100])
def test_16bit_norm_rows_on_the_measured_ring_shapes(op, dtype, N):
    # The planner's measured ring shapes for 16-bit norm rows take effect from
    # 64 rows an SM: LayerNorm rows of 257 to 768 units at 6 or 4 units a
    # thread (one row a CTA where they fill exactly), of 1536 and 3072 units at
    # 6 units, of 1537 to 2048 units at 8 units in 512-thread CTAs, rows that 5
    # units fill exactly at 5 units; RMSNorm rows of 5 to 7 warps with three
    # stages, of 2049 to 3072 units at 6 units a thread, rows that 5 units fill
    # and 4 do not at 5 units; a ragged width; every row against the oracle.
    M = 64 * 152 + 5
    x, out = _aligned(M, N, dtype, seed=N + 11)
    wt, bs = _params(N, dtype, seed=N)
    ok, plan = _servable(op, x, wt, bs, None)
    assert ok and plan["path"] == rs.RS_PATH_RING
    y = _run(op, x, wt, bs, out=out)
    check_all_rows(op, x, y, N, weight=wt, bias=bs if op == "ln" else None, eps=EPS[op],
                   what=f"ring shape {'RMSNorm' if op == 'rms' else 'LayerNorm'} {dtype} {M}x{N}")
    del x, y, out
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# The benchmark shapes at full size, in the launch configuration the
# benchmark times (auto plan, weight and bias present).
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("name", W.ORDER)
def test_benchmark_shapes_full_size(op, name):
    # Every row against the oracle under the normalisation bound, in the
    # launch configuration the benchmark times (auto plan, weight and bias).
    w = W.norm_workload(name)
    x = W.generate(w, "cuda")
    out = torch.full_like(x, float("nan")) if w.ld > w.N else torch.empty_like(x)
    if w.ld > w.N:
        pad_before = out[:, w.N:].clone()
    wt, bs = W.norm_params(w.N, w.dtype, w.seed, "cuda")
    eps = 1e-6 if op == "rms" else 1e-5
    y = _run(op, x[:, : w.N], wt, bs, eps=eps, out=out[:, : w.N])
    check_all_rows(op, x[:, : w.N], y, w.N, weight=wt, bias=bs if op == "ln" else None, eps=eps,
                   what=f"{'RMSNorm' if op == 'rms' else 'LayerNorm'} {name}", group="workloads")
    assert bool(torch.isfinite(y).all())
    if w.ld > w.N:
        assert torch.equal(out[:, w.N:].view(torch.int32), pad_before.view(torch.int32))
    del x, y, out
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# Maximum sizes.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("op", OPS)
def test_more_than_two_to_the_31_rows(op):
    M = (1 << 31) + 5
    x = torch.empty((M, 2), dtype=torch.bfloat16, device="cuda")
    x[:, 0] = 0.5
    x[:, 1] = -1.75
    w, b = _params(2, "bf16", seed=31)
    y = _run(op, x, w, b)
    _check(op, x[:1], y[:1], w, b, what=f"{op} 2^31+5 rows")
    last = y[-1:].clone()
    _check(op, x[:1], last, w, b, what=f"{op} 2^31+5 rows, last row")
    for col in range(2):
        assert bool((y[:, col] == y[0, col]).all())
    del x, y
    torch.cuda.empty_cache()


@pytest.mark.parametrize("op", OPS)
def test_a_row_of_two_to_the_26_elements(op):
    N = 1 << 26
    x = _input(2, N, "f32", kind="normal_spike", seed=26)
    w, b = _params(N, "f32", seed=26)
    y = _run(op, x, w, b)
    _check(op, x, y, w, b, what=f"{op} 2 x 2^26")
    del x, y
    torch.cuda.empty_cache()
