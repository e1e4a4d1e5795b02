"""GPU parity of the CUDA library against the CPU oracle, through the C ABI.

Every case generates a seeded input on the GPU, runs rowsoftmax through the
ctypes binding of librowsoftmax.so, copies input and output to the host and
compares element by element with the oracle (tests/_parity.py holds the
tolerances).  Covered: every kernel family (rows / cluster / stream), every
storage type, ragged tails, strided and padded rows, misaligned pointers,
in-place calls, guard bands around the output, special values, empty
problems, the five benchmark workloads at full size (every row against the
oracle, plus the workloads' structure) and the launch configuration the benchmark
times.
"""
import math

import numpy as np
import pytest
import torch

import memory_bound_row_gb300 as rs
from memory_bound_row_gb300 import build
from memory_bound_row_gb300 import workloads as W

from _parity import FMT, check_all_rows, compare, decode, oracle_rows, to_storage_numpy

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


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


def _run(x, out=None, options=None):
    y = rs.softmax(x, out=out, options=options)
    torch.cuda.synchronize()
    return y


def _servable(x, options):
    """False when the forced configuration cannot serve x's shape."""
    rc, dev = rs.rowsoftmax_device_info()
    assert rc == rs.RS_OK
    M, N = x.shape
    rc, _ = rs.rowsoftmax_plan(x.data_ptr(), x.data_ptr() + (1 << 44), M, N, x.stride(0), x.stride(0),
                               rs.dtype_code(x.dtype), options, dev)
    assert rc in (rs.RS_OK, rs.RS_ERR_NO_PATH)
    return rc == rs.RS_OK


def _check(x, y, N=None, what=""):
    N = x.shape[1] if N is None else N
    ref = oracle_rows(x, N)
    return compare(y[:, :N], ref, FMT[x.dtype], what)


def _input(M, N, dtype, ld=None, kind="normal1", seed=0):
    w = W.custom(M, N, dtype, ld=ld, seed=seed, kind=kind)
    return W.generate(w, "cuda")


def _aligned(M, N, dtype, kind="normal1", seed=0):
    """Input and output views whose rows start on 16-byte boundaries (row
    stride rounded up), so the 16-byte vector and bulk-copy kernels apply."""
    vec = 4 if dtype == "f32" else 8
    ld = -(-N // vec) * vec
    x = _input(M, N, dtype, ld=ld, kind=kind, seed=seed)[:, :N]
    out = torch.empty((M, ld), dtype=DT[dtype], device="cuda")[:, :N]
    return x, out


ROWS_SHAPES = [(1, 1), (3, 2), (5, 3), (37, 7), (64, 8), (33, 33), (300, 100), (17, 255), (129, 781),
               (64, 1000), (1024, 1024), (40, 2048), (20, 4097), (30, 5000), (16, 8192), (9, 12345)]


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("M,N", ROWS_SHAPES)
def test_auto_path_small_shapes(dtype, M, N):
    x = _input(M, N, dtype, kind="normal2_const" if dtype == "f32" else "normal1", seed=M + N)
    _check(x, _run(x), what=f"{dtype} {M}x{N}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("N", [16384, 20480, 24576, 28672, 32760, 40960])
def test_auto_path_wide_16bit_rows(dtype, N):
    # Where the planner sends wide 16-bit rows: the ring for rows the
    # clusters would spread thin (20480), the clusters for the others, the
    # ring's persistent CTAs looping over more rows than they are.
    M = 700 if N <= 20480 else 300
    x, out = _aligned(M, N, dtype, kind="normal_spike", seed=N)
    _check(x, _run(x, out=out), what=f"auto wide {dtype} N={N}")


# (threads a row, units a thread, threads a CTA, stages) the planner gives
# 16-bit softmax rows of 257 to 4096 units given enough rows.
RING16_SHAPES = {2560: (64, 5, 64, 2), 3584: (64, 8, 64, 2), 4096: (64, 8, 512, 3), 4608: (96, 6, 96, 2),
                 5120: (128, 5, 128, 2), 6200: (128, 8, 512, 3), 10000: (160, 8, 480, 3), 12288: (192, 8, 192, 3),
                 16384: (256, 8, 512, 3), 24576: (384, 8, 384, 3), 32768: (512, 8, 512, 3)}


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("N", list(RING16_SHAPES))
def test_16bit_softmax_rows_on_the_measured_ring_shapes(dtype, N):
    # Where the planner puts 16-bit softmax rows of 2560 to 32768 values given
    # enough rows: the ring shapes measured fastest (5, 6 or 8 units a thread);
    # a ragged last row group; every row against the oracle.
    tpr, vpt, block, stages = RING16_SHAPES[N]
    M = (block // tpr) * 4 * 152 + 37
    x, out = _aligned(M, N, dtype, kind="normal_spike", seed=N + 7)
    rc, dev = rs.rowsoftmax_device_info()
    rc, plan = rs.rowsoftmax_plan(x.data_ptr(), out.data_ptr(), M, N, x.stride(0), out.stride(0),
                                  rs.dtype_code(x.dtype), None, dev)
    assert rc == rs.RS_OK and plan["path"] == rs.RS_PATH_RING
    assert (plan["threads_per_row"], plan["vec_per_thread"], plan["block_threads"], plan["stages"]) == RING16_SHAPES[N]
    y = _run(x, out=out)
    check_all_rows("softmax", x, y, N, what=f"ring shape {dtype} {M}x{N}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("N", [512, 768, 1024])
def test_16bit_softmax_rows_of_64_to_128_units_on_16_lanes(dtype, N):
    # Rows that 16 lanes fill exactly (64, 96, 128 units) on 16 lanes, two rows
    # a warp, given enough rows; every row against the oracle.
    M = 32 * 4 * 152 + 37
    x, out = _aligned(M, N, dtype, kind="normal_spike", seed=N + 5)
    rc, dev = rs.rowsoftmax_device_info()
    rc, plan = rs.rowsoftmax_plan(x.data_ptr(), out.data_ptr(), M, N, x.stride(0), out.stride(0),
                                  rs.dtype_code(x.dtype), None, dev)
    assert rc == rs.RS_OK and plan["threads_per_row"] == 16
    y = _run(x, out=out)
    check_all_rows("softmax", x, y, N, what=f"16-lane rows {dtype} {M}x{N}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("N", [2561, 4100, 6150, 9999, 20000, 32767])
def test_16bit_softmax_ragged_rows_on_the_ring_shapes(dtype, N):
    # Ragged widths (a partial last 16-byte unit, read from global memory by
    # the ring) with enough rows for the planner's measured shapes; every row
    # against the oracle.
    M = 8 * 4 * 152 + 5
    x, out = _aligned(M, N, dtype, kind="normal_spike", seed=N + 3)
    rc, dev = rs.rowsoftmax_device_info()
    rc, plan = rs.rowsoftmax_plan(x.data_ptr(), out.data_ptr(), M, N, x.stride(0), out.stride(0),
                                  rs.dtype_code(x.dtype), None, dev)
    assert rc == rs.RS_OK and plan["path"] == rs.RS_PATH_RING and plan["vec_per_thread"] >= 5
    y = _run(x, out=out)
    check_all_rows("softmax", x, y, N, what=f"ragged ring shape {dtype} {M}x{N}")


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("tpr,vpt", [(1, 1), (2, 2), (4, 3), (8, 5), (16, 8), (32, 1), (32, 6), (64, 4), (96, 2),
                                     (256, 2), (512, 1), (1024, 1), (160, 8)])
def test_rows_path_thread_shapes(dtype, tpr, vpt):
    vec = 4 if dtype == "f32" else 8
    if vpt not in ((1, 2, 3, 4, 5, 6, 8, 10, 12, 16) if vec == 4 else (1, 2, 3, 4, 5, 6, 8)):
        pytest.skip("count not instantiated")
    if vpt * vec > 32 and tpr > 512:
        pytest.skip("instance compiled for 512 threads")
    N = max(1, tpr * vpt * vec - 3)  # a ragged last unit
    M = 37
    x, out = _aligned(M, N, dtype, seed=tpr * 100 + vpt)
    y = _run(x, out=out, options={"path": rs.RS_PATH_ROWS, "threads_per_row": tpr, "vec_per_thread": vpt})
    _check(x, y, what=f"rows tpr={tpr} vpt={vpt}")


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("N", [1, 5, 31, 100, 777, 4096])
def test_rows_path_element_wise(dtype, N):
    x = _input(23, N, dtype, seed=N)
    y = _run(x, options={"path": rs.RS_PATH_ROWS, "force_scalar": 1})
    _check(x, y, what=f"scalar rows N={N}")


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("cs", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("N", [8, 1000, 4104, 65536, 100003])
@pytest.mark.parametrize("values", [rs.RS_RING_REGISTERS, rs.RS_RING_REREAD])
@pytest.mark.parametrize("grid_limit", [0, 2])
def test_cluster_path(dtype, cs, N, values, grid_limit):
    x, out = _aligned(11, N, dtype, kind="normal_spike", seed=cs * 7 + N)
    opts = {"path": rs.RS_PATH_CLUSTER, "cluster_size": cs, "grid_limit": grid_limit * cs, "ring_values": values}
    if not _servable(x, opts):
        pytest.skip("slice larger than shared memory")
    y = _run(x, out=out, options=opts)
    _check(x, y, what=f"cluster cs={cs} N={N}")


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("cs", [1, 2, 5, 8])
@pytest.mark.parametrize("scalar", [0, 1])
@pytest.mark.parametrize("N", [3, 1000, 70001])
def test_stream_path(dtype, cs, scalar, N):
    x, out = _aligned(9, N, dtype, kind="uniform20_offset", seed=cs + N)
    y = _run(x, out=out, options={"path": rs.RS_PATH_STREAM, "cluster_size": cs, "force_scalar": scalar})
    _check(x, y, what=f"stream cs={cs} scalar={scalar} N={N}")


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("N", [8, 100, 1001, 2048, 5000, 8192, 12345])
@pytest.mark.parametrize("stages", [2, 3, 8])
@pytest.mark.parametrize("values", [rs.RS_RING_REGISTERS, rs.RS_RING_REREAD])
def test_ring_path(dtype, N, stages, values):
    x, out = _aligned(300, N, dtype, kind="uniform20_offset", seed=N + stages)
    opts = {"path": rs.RS_PATH_RING, "stages": stages, "ring_values": values}
    if not _servable(x, opts):
        pytest.skip("ring does not fit shared memory")
    y = _run(x, out=out, options=opts)
    _check(x, y, what=f"ring N={N} stages={stages}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("tpr,vpt", [(1, 1), (4, 2), (32, 8), (64, 4), (160, 8), (256, 4), (512, 2), (1024, 1)])
@pytest.mark.parametrize("grid_limit", [0, 3])
@pytest.mark.parametrize("values", [rs.RS_RING_REGISTERS, rs.RS_RING_REREAD])
def test_ring_thread_shapes_and_wraparound(dtype, tpr, vpt, grid_limit, values):
    vec = 4 if dtype == "f32" else 8
    N = max(vec + 1, tpr * vpt * vec - 5)
    x, out = _aligned(97, N, dtype, seed=tpr + vpt)
    opts = {"path": rs.RS_PATH_RING, "threads_per_row": tpr, "vec_per_thread": vpt, "grid_limit": grid_limit,
            "ring_values": values}
    if not _servable(x, opts):
        pytest.skip("ring does not fit shared memory")
    y = _run(x, out=out, options=opts)
    _check(x, y, what=f"ring tpr={tpr} vpt={vpt} grid_limit={grid_limit}")


@pytest.mark.parametrize("path", [rs.RS_PATH_ROWS, rs.RS_PATH_RING, rs.RS_PATH_CLUSTER, rs.RS_PATH_STREAM])
def test_grid_limit_makes_ctas_loop_over_rows(path):
    x = _input(1000, 512, "bf16", seed=5)
    y = _run(x, options={"path": path, "grid_limit": 16})
    _check(x, y, what=f"grid_limit path={path}")


def test_paths_agree_on_the_same_input():
    x = _input(64, 6000, "f32", kind="normal2_const", seed=9)
    ref = oracle_rows(x, 6000)
    for opts in [None, {"path": rs.RS_PATH_ROWS}, {"path": rs.RS_PATH_RING, "ring_values": rs.RS_RING_REGISTERS},
                 {"path": rs.RS_PATH_RING, "ring_values": rs.RS_RING_REREAD}, {"path": rs.RS_PATH_CLUSTER, "cluster_size": 4},
                 {"path": rs.RS_PATH_CLUSTER, "cluster_size": 2, "ring_values": rs.RS_RING_REREAD},
                 {"path": rs.RS_PATH_STREAM, "cluster_size": 2}, {"path": rs.RS_PATH_ROWS, "force_scalar": 1}]:
        compare(_run(x, options=opts), ref, "f32", f"opts={opts}")


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_padded_strides_and_guard_bands(dtype):
    M, N, ld, G = 50, 1001, 1040, 4096
    x = _input(M, N, dtype, ld=ld, seed=3)
    buf = torch.empty(M * ld + 2 * G, dtype=DT[dtype], device="cuda")
    buf.view(torch.int16 if dtype != "f32" else torch.int32).fill_(0x5A5A if dtype != "f32" else 0x5A5A5A5A)
    before = buf.clone()
    out = buf[G: G + M * ld].view(M, ld)
    _run(x[:, :N], out=out[:, :N])
    _check(x[:, :N], out[:, :N], what="padded")
    assert torch.equal(buf[:G], before[:G]) and torch.equal(buf[G + M * ld:], before[G + M * ld:])
    assert torch.equal(out[:, N:], before[G: G + M * ld].view(M, ld)[:, N:])


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("shift", [1, 3])
def test_misaligned_pointers_use_element_wise_access(dtype, shift):
    M, N = 40, 999
    base = _input(M * N + 8, 1, dtype, seed=11).view(-1)
    x = base[shift: shift + M * N].view(M, N)
    out = torch.empty(M * N + 8, dtype=DT[dtype], device="cuda")[shift + 1: shift + 1 + M * N].view(M, N)
    _run(x, out=out)
    _check(x, out, what="misaligned")


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("N", [100, 8192, 70000])
@pytest.mark.parametrize("path", [rs.RS_PATH_AUTO, rs.RS_PATH_ROWS, rs.RS_PATH_RING, rs.RS_PATH_STREAM])
def test_in_place(dtype, N, path):
    x = _input(300, N, dtype, seed=N)
    opts = {"path": path, "grid_limit": 7}
    if not _servable(x, opts):
        pytest.skip("configuration does not serve this shape")
    ref = oracle_rows(x, N)
    y = _run(x, out=x, options=opts)
    assert y.data_ptr() == x.data_ptr()
    compare(x, ref, dtype, "in-place")


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("path", [rs.RS_PATH_ROWS, rs.RS_PATH_RING, rs.RS_PATH_CLUSTER, rs.RS_PATH_STREAM])
def test_special_values(dtype, path):
    N = 300
    x, out = _aligned(8, N, dtype, seed=1)
    x[0] = -math.inf                  # all -inf: NaN row
    x[1, 17] = math.nan               # NaN: NaN row
    x[2, 200] = math.inf              # +inf: NaN row
    x[3, 1:] = -math.inf              # one finite entry: [1, 0, 0, ...]
    x[4, :150] = -math.inf            # a -inf prefix
    x[5, 150:] = -math.inf            # a -inf suffix
    x[6, ::2] = -math.inf
    x[7, 5] = 1e4 if dtype != "f16" else 6e4
    y = _run(x, out=out, options={"path": path})
    _check(x, y, what=f"special path={path}")
    yd = decode(y)
    assert yd[3, 0] == 1.0 and np.all(yd[3, 1:] == 0.0)
    assert np.all(yd[4, :150] == 0.0) and np.all(yd[5, 150:] == 0.0)


def test_empty_problems_launch_nothing():
    x = torch.empty((0, 16), device="cuda")
    assert rs.softmax(x).shape == (0, 16)
    x = torch.empty((16, 0), device="cuda")
    assert rs.softmax(x).shape == (16, 0)


def test_host_memory_is_rejected():
    x = torch.randn(4, 64)  # pageable host memory
    y = torch.empty_like(x)
    rc = rs.rowsoftmax_fwd(x.data_ptr(), y.data_ptr(), 4, 64, 64, 64, rs.RS_F32, 0)
    assert rc == rs.RS_ERR_NOT_DEVICE_MEMORY


def test_overlap_is_rejected_on_device_memory():
    buf = torch.zeros(4096, device="cuda")
    rc = rs.rowsoftmax_fwd(buf.data_ptr(), buf.data_ptr() + 64, 8, 100, 100, 100, rs.RS_F32, 0)
    assert rc == rs.RS_ERR_OVERLAP


def test_nonzero_stream():
    s = torch.cuda.Stream()
    x = _input(100, 3000, "bf16", seed=2)
    with torch.cuda.stream(s):
        y = rs.softmax(x)
    s.synchronize()
    _check(x, y, what="side stream")


@pytest.mark.parametrize("shape", [(1823, 781), (1, 1), (4096, 4096)])
def test_triton_skill_page_shapes(shape):
    # fp32 randn, seed 0: the correctness shapes of the Hugging Face
    # "triton-kernels" skill page ("Correctness Testing").
    x = _input(*shape, "f32", seed=0)
    _check(x, _run(x), what=f"skill shape {shape}")


# ---------------------------------------------------------------------------
# The five benchmark workloads at full size.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", W.ORDER)
def test_benchmark_workloads_full_size(name):
    # Every row of the workload against the oracle (1e-6 fp32, 4e-3 fp16/bf16 per
    # element, fp32 row sums within 1e-5), in the launch configuration the
    # benchmark times (rowsoftmax_fwd, no options), plus the workloads'
    # structure: untouched padding, exact zeros above the causal diagonal,
    # exactly 1/N (to fp32 rounding) on the constant rows.
    w = W.WORKLOADS[name]
    x = W.generate(w, "cuda")
    out = torch.full_like(x, float("nan")) if w.ld > w.N else torch.empty_like(x)
    if w.ld > w.N:
        pad_before = out[:, w.N:].clone()
    y = rs.softmax(x[:, : w.N], out=out[:, : w.N])
    torch.cuda.synchronize()

    check_all_rows("softmax", x[:, : w.N], y, w.N, what=f"softmax {name}", group="workloads")

    assert bool(torch.isfinite(y).all())
    assert float(y.min()) >= 0.0 and float(y.max()) <= 1.0
    if w.ld > w.N:
        assert torch.equal(out[:, w.N:].view(torch.int32), pad_before.view(torch.int32))
    if w.kind == "causal_scores":
        r = torch.arange(w.M, device="cuda") % 2048
        masked = torch.arange(w.N, device="cuda")[None, :] > r[:, None]
        assert bool((y[masked] == 0).all())
        assert bool((y[~masked] > 0).all())
        del r, masked
    if w.kind == "normal2_const":
        const_rows = W.pick_rows(w.M, 82, w.seed, 1, "cuda")
        yc = y[const_rows].double()
        assert float((yc - 1.0 / w.N).abs().max()) <= 1e-6
    del x, y, out
    torch.cuda.empty_cache()


def test_benchmark_launch_configuration_is_the_auto_plan():
    # bench.py times rowsoftmax_fwd with no options on the workload above; the
    # parity cases above ran exactly that call.
    w = W.WORKLOADS["fp32_8192x5000_ld5120"]
    rc, dev = rs.rowsoftmax_device_info()
    assert rc == rs.RS_OK
    x = W.generate(w, "cuda", 0, 4)
    rc, plan = rs.rowsoftmax_plan(x.data_ptr(), x.data_ptr() + (1 << 40), w.M, w.N, w.ld, w.ld, rs.RS_F32, None,
                                  dev)
    assert rc == rs.RS_OK and plan["path"] == rs.RS_PATH_ROWS


# ---------------------------------------------------------------------------
# Maximum sizes.
# ---------------------------------------------------------------------------

def test_more_than_two_to_the_31_rows():
    # 2^31 + 5 rows of [0, ln 3] in bf16: every row is the same, so every output
    # row must equal the oracle's result for that one row; row offsets pass 4 GB.
    M = (1 << 31) + 5
    x = torch.empty((M, 2), dtype=torch.bfloat16, device="cuda")
    x[:, 0] = 0.0
    x[:, 1] = math.log(3.0)
    y = rs.softmax(x)
    torch.cuda.synchronize()
    ref = oracle_rows(x[:1], 2)[0]
    for col in range(2):
        got = y[:, col].float()
        assert float((got.double() - ref[col]).abs().max()) <= 4e-3
        assert bool((got == got[0]).all())  # every row identical
    del x, y
    torch.cuda.empty_cache()


@pytest.mark.parametrize("dtype", ["f16", "f32"])
def test_a_row_of_two_to_the_26_elements(dtype):
    N = 1 << 26
    x = _input(2, N, dtype, kind="normal_spike", seed=26)
    y = _run(x)
    _check(x, y, what=f"2 x 2^26 {dtype}")
    del x, y
    torch.cuda.empty_cache()
