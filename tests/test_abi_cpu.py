"""CPU checks of the C-ABI library: it loads, exports every entry point that
include/rowsoftmax.h declares, rejects bad arguments before touching a
device, and plans the launches described in its header.  No kernel runs."""
import ctypes
import os
import re

import pytest

import memory_bound_row_gb300 as rs
from memory_bound_row_gb300 import _abi, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rowsoftmax.h")
GOLDEN = os.path.join(ROOT, "tests", "golden", "group_cyclic_layout.txt")


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^RS_API\s+[\w\s\*]*?\b(\w+)\s*\(", text, re.M)))


def gb300():
    d = rs.rs_device_info()
    d.sm_count = 152
    d.max_smem_per_block_optin = 232448
    d.max_smem_per_sm = 233472
    d.max_threads_per_sm = 2048
    d.cc_major, d.cc_minor = 10, 3
    return d


def test_library_exports_every_declared_entry_point():
    declared = _declared()
    assert len(declared) >= 12
    lib = ctypes.CDLL(_abi.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(_abi.EXPORTED) == declared


def test_status_strings():
    for code in range(7):
        assert rs.rowsoftmax_status_string(code) != "unknown status"
    assert rs.rowsoftmax_status_string(99) == "unknown status"


A = 1 << 20  # a 16-byte aligned fake address; validation fails before it is used


@pytest.mark.parametrize(
    "args,status",
    [
        ((A, A + (1 << 16), 4, 8, 8, 8, 7), rs.RS_ERR_UNSUPPORTED_DTYPE),
        ((A, A + (1 << 16), -1, 8, 8, 8, rs.RS_F32), rs.RS_ERR_INVALID_ARG),
        ((A, A + (1 << 16), 4, -8, 8, 8, rs.RS_F32), rs.RS_ERR_INVALID_ARG),
        ((0, A, 4, 8, 8, 8, rs.RS_F32), rs.RS_ERR_INVALID_ARG),
        ((A, 0, 4, 8, 8, 8, rs.RS_F32), rs.RS_ERR_INVALID_ARG),
        ((A, A + (1 << 16), 4, 8, 7, 8, rs.RS_F32), rs.RS_ERR_INVALID_ARG),
        ((A, A + (1 << 16), 4, 8, 8, 7, rs.RS_F32), rs.RS_ERR_INVALID_ARG),
        ((A + 1, A + (1 << 16), 4, 8, 8, 8, rs.RS_F16), rs.RS_ERR_INVALID_ARG),
        ((A + 2, A + (1 << 16), 4, 8, 8, 8, rs.RS_F32), rs.RS_ERR_INVALID_ARG),
        ((A, A + 64, 4, 8, 8, 8, rs.RS_F32), rs.RS_ERR_OVERLAP),
        ((A, A, 4, 8, 8, 16, rs.RS_F32), rs.RS_ERR_OVERLAP),
        ((A, A + 4, 1, 8, 8, 8, rs.RS_F32), rs.RS_ERR_OVERLAP),
        ((A, A + (1 << 16), 2, (1 << 31), 1 << 31, 1 << 31, rs.RS_F16), rs.RS_ERR_INVALID_ARG),
        ((A, A + (1 << 16), 1 << 62, 8, 1 << 20, 8, rs.RS_F32), rs.RS_ERR_INVALID_ARG),
    ],
)
def test_bad_arguments_are_rejected_before_any_device_call(args, status):
    assert rs.rowsoftmax_fwd(*args, 0) == status
    rc, _ = rs.rowsoftmax_plan(*args, None, gb300())
    assert rc == status


def test_empty_problems_are_a_noop():
    assert rs.rowsoftmax_fwd(0, 0, 0, 8, 8, 8, rs.RS_F32, 0) == rs.RS_OK
    assert rs.rowsoftmax_fwd(0, 0, 8, 0, 0, 0, rs.RS_BF16, 0) == rs.RS_OK
    rc, plan = rs.rowsoftmax_plan(0, 0, 0, 8, 8, 8, rs.RS_F32, None, gb300())
    assert rc == rs.RS_OK and plan["grid"] == 0


def test_exact_in_place_is_accepted_by_the_planner():
    rc, plan = rs.rowsoftmax_plan(A, A, 64, 1000, 1024, 1024, rs.RS_F32, None, gb300())
    assert rc == rs.RS_OK and plan["path"] in (rs.RS_PATH_ROWS, rs.RS_PATH_RING)


def test_disjoint_interleaved_layout_is_rejected_as_overlap():
    # Ranges are compared, not element sets: interleaved rows count as overlap.
    rc, _ = rs.rowsoftmax_plan(A, A + 32, 4, 8, 16, 16, rs.RS_F32, None, gb300())
    assert rc == rs.RS_ERR_OVERLAP


def _plan(M, N, dtype, ld=None, opts=None, a=A, b=A + (1 << 40)):
    rc, plan = rs.rowsoftmax_plan(a, b, M, N, ld or N, ld or N, dtype, opts, gb300())
    assert rc == rs.RS_OK, rs.rowsoftmax_status_string(rc)
    return plan


def _covers(plan, N):
    units = -(-N // plan["vec_elems"])
    if plan["path"] in (rs.RS_PATH_ROWS, rs.RS_PATH_RING):
        return plan["threads_per_row"] * plan["vec_per_thread"] >= units
    return plan["cluster_size"] * plan["chunk_elems"] >= N


def test_16bit_softmax_rows_take_the_measured_ring_shapes():
    # 16-bit softmax rows of 257 to 4096 units take the ring shapes measured
    # fastest; those of 769 units or more at 8 units a thread, 512-thread CTAs
    # where a row takes at most 256 threads, three stages (faster than the
    # 4-unit ring and than the clusters at every N from 8192 to 32768); given
    # 4 row groups an SM.
    for N, tpr, block in [(12288, 192, 192), (16384, 256, 512), (20480, 320, 320), (24576, 384, 384),
                          (28672, 448, 448), (32768, 512, 512)]:
        p = _plan((1 << 28) // N, N, rs.RS_BF16)
        assert p["path"] == rs.RS_PATH_RING and _covers(p, N), N
        assert (p["threads_per_row"], p["vec_per_thread"], p["block_threads"], p["stages"]) == (tpr, 8, block, 3), N
        assert p["smem_bytes"] == 3 * (block // tpr) * N * 2
    # ragged widths round the threads up to whole warps
    p = _plan(8192, 10000, rs.RS_F16, ld=10000)
    assert (p["threads_per_row"], p["vec_per_thread"], p["block_threads"]) == (160, 8, 480) and _covers(p, 10000)
    # narrower rows (257 to 768 units): 8 units a thread on a multiple of 256
    # units, else 5 units where they fill whole warps exactly, or 6 where they
    # do and 4 do not (one row a CTA, two stages), rows that 4 units fill
    # exactly their planned 4-unit shape, else 8 units on whole warps, one row
    # a CTA
    for N, shape in [(4096, (64, 8, 512, 3)), (6144, (96, 8, 480, 3)), (2560, (64, 5, 64, 2)),
                     (3072, (96, 4, 192, 2)), (4608, (96, 6, 96, 2)), (5120, (128, 5, 128, 2)),
                     (3584, (64, 8, 64, 2)), (5632, (96, 8, 96, 2))]:
        p = _plan((1 << 29) // N, N, rs.RS_BF16)
        assert p["path"] == rs.RS_PATH_RING and _covers(p, N), N
        assert (p["threads_per_row"], p["vec_per_thread"], p["block_threads"], p["stages"]) == shape, N
    assert _plan(1 << 20, 2048, rs.RS_BF16)["vec_per_thread"] == 8  # rows of one warp: their own rule
    # few rows: the clusters as before (each CTA would not loop over its stages)
    assert _plan(64, 32768, rs.RS_BF16)["path"] == rs.RS_PATH_CLUSTER
    assert _plan(4096, 40960, rs.RS_F16)["path"] == rs.RS_PATH_CLUSTER  # over 4096 units
    # the causal mask's rows of 257 to 4096 units take its copy ring at 8 units a
    # thread, one row a CTA, two stages (measured +17 to +36 % from 4096 to 32768)
    for N in (4096, 6000, 16384, 32768):
        rc, p = rs.rowsoftmax_causal_plan(A, A + (1 << 40), 8192, N, N, N, N, 0, rs.RS_BF16, None, gb300())
        tpr = -(-(-(-N // 8) // 8) // 32) * 32
        assert rc == rs.RS_OK and p["path"] == rs.RS_PATH_RING and p["ring_values"] == rs.RS_RING_THREAD_COPIES
        assert (p["threads_per_row"], p["vec_per_thread"], p["block_threads"], p["stages"]) == (tpr, 8, tpr, 2), N
    # 5 or 6 units a thread where they fill whole warps exactly and 8 do not
    # (2560 +47 %, 3072 +35 %, 4608 +34 %, 5120 +15 %)
    for N, tpr, vpt in [(2560, 64, 5), (3072, 64, 6), (4608, 96, 6), (5120, 128, 5)]:
        rc, p = rs.rowsoftmax_causal_plan(A, A + (1 << 40), 8192, N, N, N, N, 0, rs.RS_BF16, None, gb300())
        assert (p["threads_per_row"], p["vec_per_thread"], p["block_threads"]) == (tpr, vpt, tpr), N
    # and 5 or 6 where they fill 16 warps exactly, before 8 on 10 or 12 warps
    # (20480 +5.7 %, 24576 +1.9 %); 8 warps keep 8 units (10240 -18 %, 12288 -0.6 %)
    for N, tpr, vpt in [(20480, 512, 5), (24576, 512, 6), (10240, 160, 8), (12288, 192, 8)]:
        rc, p = rs.rowsoftmax_causal_plan(A, A + (1 << 40), 8192, N, N, N, N, 0, rs.RS_F16, None, gb300())
        assert (p["threads_per_row"], p["vec_per_thread"], p["block_threads"], p["stages"]) == (tpr, vpt, tpr, 2), N


def test_plans_for_the_benchmark_workloads():
    # fp32: register-resident rows; 16-bit: the bulk-copy ring; vocabulary-
    # sized rows: persistent clusters holding their slices in registers.
    p = _plan(1024, 1024, rs.RS_F32)
    assert (p["path"], p["vec_elems"], p["threads_per_row"]) == (rs.RS_PATH_ROWS, 4, 32)
    p = _plan(8192, 5000, rs.RS_F32, ld=5120)
    assert p["path"] == rs.RS_PATH_ROWS and p["vec_elems"] == 4 and _covers(p, 5000)
    p = _plan(32768, 8192, rs.RS_BF16)
    assert p["path"] == rs.RS_PATH_RING and p["vec_elems"] == 8 and _covers(p, 8192)
    assert p["ring_values"] == rs.RS_RING_REGISTERS and p["stages"] == 3
    p = _plan(512, 131072, rs.RS_F16)
    assert p["path"] == rs.RS_PATH_CLUSTER and p["ring_values"] == rs.RS_RING_REGISTERS
    assert p["cluster_size"] >= 2 and _covers(p, 131072)
    assert p["block_threads"] * p["vec_per_thread"] * 8 >= p["chunk_elems"]
    assert p["smem_bytes"] <= 232448 - 1024 and p["grid"] % p["cluster_size"] == 0
    assert p["grid"] <= 512 * p["cluster_size"]  # persistent clusters loop over rows
    p = _plan(1 << 20, 2048, rs.RS_BF16)
    assert p["path"] == rs.RS_PATH_RING and _covers(p, 2048)
    # a 2048-element bf16 row fits one warp at 64 values a thread: no CTA barrier per row
    assert (p["threads_per_row"], p["vec_per_thread"]) == (32, 8)


def test_few_rows_are_spread_over_the_sms():
    p = _plan(1024, 1024, rs.RS_F32)
    assert p["grid"] >= 2 * 152 and p["block_threads"] % 32 == 0
    assert p["rows_per_cta"] * p["grid"] >= 1024
    p = _plan(1 << 16, 1024, rs.RS_F32)  # many rows of one warp: full 128-thread CTAs
    assert p["block_threads"] == 128 and p["threads_per_row"] == 32
    p = _plan(1 << 16, 512, rs.RS_F32)   # rows narrower than a warp: 256-thread CTAs
    assert p["block_threads"] == 256


def test_fp32_rows_of_one_or_two_warps_take_128_thread_ctas():
    # the N sweep around the one-warp / two-warp switch (M = 4096): 128-thread
    # CTAs measured faster than 256 for both row widths
    for N, tpr in [(1024, 32), (1152, 64), (1536, 64), (2048, 64)]:
        p = _plan(4096, N, rs.RS_F32)
        assert p["path"] == rs.RS_PATH_ROWS and p["threads_per_row"] == tpr and p["block_threads"] == 128, (N, p)
    p = _plan(4096, 3072, rs.RS_F32)  # three warps a row: unchanged
    assert p["threads_per_row"] == 96 and p["block_threads"] == 192


def test_ring_plan_is_persistent_and_fits_shared_memory():
    for M, N, dt in [(8192, 5000, rs.RS_F32), (32768, 8192, rs.RS_BF16), (1 << 20, 2048, rs.RS_BF16),
                     (7, 300, rs.RS_F16)]:
        p = _plan(M, N, dt, ld=-(-N // 8) * 8, opts={"path": rs.RS_PATH_RING})
        assert p["path"] == rs.RS_PATH_RING
        assert 2 <= p["stages"] <= 8
        es = 4 if dt == rs.RS_F32 else 2
        stage = (N * es // 16) * 16 * p["rows_per_cta"]
        assert p["smem_bytes"] == stage * p["stages"] <= 232448 - 1024
        groups = -(-M // p["rows_per_cta"])
        assert p["grid"] <= min(groups, 152 * 32)
    p = _plan(8192, 5000, rs.RS_F32, ld=5120, opts={"path": rs.RS_PATH_RING, "stages": 3})
    assert p["stages"] == 3
    rc, _ = rs.rowsoftmax_plan(A, A + (1 << 40), 10, 1000, 1000, 1000, rs.RS_F32,
                               {"path": rs.RS_PATH_RING, "stages": 9}, gb300())
    assert rc == rs.RS_ERR_INVALID_ARG
    rc, _ = rs.rowsoftmax_plan(A + 4, A + (1 << 40), 10, 1000, 1000, 1000, rs.RS_F32,
                               {"path": rs.RS_PATH_RING}, gb300())
    assert rc == rs.RS_ERR_NO_PATH


def test_misaligned_data_gets_the_element_wise_kernels():
    p = _plan(1823, 781, rs.RS_F32)  # stride 781 * 4 bytes is not a multiple of 16
    assert p["vec_elems"] == 1 and _covers(p, 781)
    p = _plan(16, 1024, rs.RS_F32, a=A + 4)
    assert p["vec_elems"] == 1
    p = _plan(16, 1024, rs.RS_BF16, b=A + (1 << 40) + 2)
    assert p["vec_elems"] == 1
    p = _plan(1, 1000, rs.RS_F16, ld=1001)  # one row: its stride does not matter
    assert p["vec_elems"] == 8


@pytest.mark.parametrize("dtype", [rs.RS_F32, rs.RS_F16, rs.RS_BF16])
@pytest.mark.parametrize("N", [1, 2, 3, 7, 8, 9, 31, 32, 33, 255, 1000, 4096, 5000, 8192, 8193, 16384,
                               65536, 131072, 1 << 20, 1 << 24])
@pytest.mark.parametrize("aligned", [True, False])
def test_auto_plan_always_covers_the_row(dtype, N, aligned):
    a = A if aligned else A + 2 * (1 if dtype else 2)
    p = _plan(3, N, dtype, a=a)
    assert _covers(p, N)
    if N <= 4096:  # short rows stay single-pass, aligned or not
        assert p["path"] in (rs.RS_PATH_ROWS, rs.RS_PATH_RING)
    if p["path"] == rs.RS_PATH_CLUSTER:
        assert p["vec_elems"] > 1 and p["stages"] <= 16 and p["smem_bytes"] % 16 == 0
        assert (p["chunk_elems"] * (4 if dtype == rs.RS_F32 else 2)) % 16 == 0
    if p["path"] in (rs.RS_PATH_ROWS, rs.RS_PATH_RING):
        assert p["block_threads"] % p["threads_per_row"] == 0 and p["block_threads"] <= 1024
    if p["path"] == rs.RS_PATH_RING:
        assert p["vec_elems"] > 1 and p["smem_bytes"] <= 232448 - 1024


def test_forced_options():
    o = {"path": rs.RS_PATH_ROWS, "threads_per_row": 64, "vec_per_thread": 4}
    p = _plan(100, 1000, rs.RS_F32, opts=o)
    assert (p["threads_per_row"], p["vec_per_thread"]) == (64, 4)
    rc, _ = rs.rowsoftmax_plan(A, A + (1 << 40), 100, 1000, 1000, 1000, rs.RS_F32,
                               {"path": rs.RS_PATH_ROWS, "threads_per_row": 32, "vec_per_thread": 4}, gb300())
    assert rc == rs.RS_ERR_NO_PATH  # 32 threads x 4 units of 4 cannot hold 1000 elements
    rc, _ = rs.rowsoftmax_plan(A, A + (1 << 40), 100, 1000, 1000, 1000, rs.RS_F32,
                               {"path": rs.RS_PATH_ROWS, "threads_per_row": 48}, gb300())
    assert rc == rs.RS_ERR_INVALID_ARG
    rc, _ = rs.rowsoftmax_plan(A + 4, A + (1 << 40), 100, 1000, 1000, 1000, rs.RS_F32,
                               {"path": rs.RS_PATH_CLUSTER}, gb300())
    assert rc == rs.RS_ERR_NO_PATH  # bulk copies need 16-byte alignment
    p = _plan(7, 100000, rs.RS_BF16, opts={"path": rs.RS_PATH_STREAM, "cluster_size": 3})
    assert p["cluster_size"] == 3 and _covers(p, 100000)
    p = _plan(7, 1000, rs.RS_BF16, opts={"path": rs.RS_PATH_CLUSTER, "cluster_size": 16})
    assert p["cluster_size"] == 16 and p["grid"] == 7 * 16
    p = _plan(1000, 1000, rs.RS_F32, opts={"grid_limit": 5})
    assert p["grid"] == 5


def test_failure_path_options_are_validated():
    ok = {"path": rs.RS_PATH_RING, "withhold_copies": 1, "wait_limit_us": 20000}
    p = _plan(64, 4096, rs.RS_BF16, opts=ok)
    assert p["withhold_copies"] == 1 and p["wait_limit_us"] == 20000
    for bad in [{"path": rs.RS_PATH_RING, "withhold_copies": 1},
                {"path": rs.RS_PATH_ROWS, "withhold_copies": 1, "wait_limit_us": 100},
                {"withhold_copies": 2, "path": rs.RS_PATH_RING, "wait_limit_us": 100},
                {"wait_limit_us": -1}]:
        rc, _ = rs.rowsoftmax_plan(A, A + (1 << 40), 64, 4096, 4096, 4096, rs.RS_BF16, bad, gb300())
        assert rc == rs.RS_ERR_INVALID_ARG, bad


def test_strict_order_option():
    p = _plan(64, 4096, rs.RS_BF16)
    assert p["strict_order"] == 0  # programmatic dependent launch by default
    p = _plan(64, 4096, rs.RS_BF16, opts={"strict_order": 1})
    assert p["strict_order"] == 1
    for bad in (-1, 2):
        rc, _ = rs.rowsoftmax_plan(A, A + (1 << 40), 64, 4096, 4096, 4096, rs.RS_BF16, {"strict_order": bad},
                                   gb300())
        assert rc == rs.RS_ERR_INVALID_ARG


def test_layout_owner_matches_the_pages_worked_example():
    with open(GOLDEN) as f:
        lines = [ln for ln in f if ln.strip() and not ln.startswith("#")]
    for ln in lines:
        head, owners = ln.split("|")
        threads, vec = map(int, head.split())
        want = list(map(int, owners.split()))
        got = [rs.rowsoftmax_layout_owner(j, threads, vec)[1] for j in range(len(want))]
        assert got == want


def test_layout_owner_is_a_bijection():
    threads, vec, n = 32, 4, 32 * 4 * 5
    seen = set()
    for j in range(n):
        rc, t, s = rs.rowsoftmax_layout_owner(j, threads, vec)
        assert rc == rs.RS_OK
        seen.add((t, s))
        # 16-byte groups: elements of one group share a thread and fill consecutive slots
        assert t == (j // vec) % threads
    assert len(seen) == n
    assert rs.rowsoftmax_layout_owner(-1, 2, 2)[0] == rs.RS_ERR_INVALID_ARG


def _c_layout(struct: str, fields):
    """sizeof and offsetof of a struct of include/rowsoftmax.h, from a small C
    program compiled against the header (None when no C compiler or CUDA
    headers are at hand)."""
    import os
    import shutil
    import subprocess
    import tempfile

    cc = shutil.which("gcc") or shutil.which("cc")
    cuda_inc = next((d for d in ("/usr/local/cuda/include", os.path.join(os.environ.get("CUDA_HOME", "/nonexistent"),
                                                                             "include"))
                     if os.path.exists(os.path.join(d, "cuda_runtime_api.h"))), None)
    if not cc or not cuda_inc:
        return None
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    prints = "".join(f'    printf("%zu\\n", offsetof({struct}, {f}));\n' for f in fields)
    src = (f'#include <stddef.h>\n#include <stdio.h>\n#include "rowsoftmax.h"\nint main(void) {{\n'
           f'    printf("%zu\\n", sizeof({struct}));\n{prints}    return 0;\n}}\n')
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "layout.c")
        exe = os.path.join(d, "layout")
        with open(c, "w") as fh:
            fh.write(src)
        r = subprocess.run([cc, "-std=c11", "-I", os.path.join(root, "include"), "-I", cuda_inc, c, "-o", exe],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
        vals = [int(v) for v in subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split()]
    return vals[0], vals[1:]


@pytest.mark.parametrize("cls", [rs.rs_options, rs.rs_plan, rs.rs_device_info])
def test_ctypes_structs_match_the_c_header(cls):
    # The binding's structs have the C header's size and every field's offset.
    fields = [name for name, _ in cls._fields_]
    got = _c_layout(cls.__name__, fields)
    if got is None:
        pytest.skip("no C compiler or CUDA headers")
    size, offsets = got
    assert ctypes.sizeof(cls) == size
    assert [getattr(cls, f).offset for f in fields] == offsets


def test_ring_cta_sizes_for_16bit_rows():
    # Measured CTA sizes of the ring on 16-bit rows (graph-replayed, 2^18 to
    # 2^20 rows): softmax rows of one warp at 4 or 8 units a thread take
    # 512-thread CTAs (one an SM, 16 rows a stage; bf16 2048 +3.3 %), rows of
    # 64 or 128 units 16 lanes in 512-thread CTAs (bf16 512 +9 %, 1024 +6 %),
    # rows of one warp at 5 or 6 units 256 threads (1280: 512 threads measured
    # 12 % slower); LayerNorm rows of one warp 128 threads; rows of 8 warps and
    # problems of fewer than 64 rows an SM keep 256.
    for N, tpr, vpt, rows_per_cta in [(512, 16, 4, 32), (1024, 16, 8, 32), (2048, 32, 8, 16)]:
        for dt in (rs.RS_BF16, rs.RS_F16):
            p = _plan(1 << 20, N, dt)
            assert p["path"] == rs.RS_PATH_RING and (p["threads_per_row"], p["vec_per_thread"]) == (tpr, vpt)
            assert p["block_threads"] == 512 and p["rows_per_cta"] == rows_per_cta and p["grid"] % 152 == 0, (N, dt)
    for N in (1280, 1536):
        assert _plan(1 << 20, N, rs.RS_BF16)["block_threads"] == 256
    p = _plan(1 << 20, 768, rs.RS_BF16)  # 16 lanes at 6 units: 256-thread CTAs (+2.9 % over 32 lanes x 3)
    assert (p["threads_per_row"], p["vec_per_thread"], p["block_threads"]) == (16, 6, 256)
    # the causal mask's rows of 32 to 256 units: the fewest lanes that hold the
    # row at up to 8 units a thread, 512-thread CTAs (bf16 512 +27 %, 1024 +25 %)
    for N, tpr, vpt in [(256, 4, 8), (512, 8, 8), (768, 16, 6), (1024, 16, 8), (1280, 32, 5), (2048, 32, 8)]:
        rc, p = rs.rowsoftmax_causal_plan(A, A + (1 << 40), 1 << 20, N, N, N, N, 0, rs.RS_BF16, None, gb300())
        assert rc == rs.RS_OK and p["ring_values"] == rs.RS_RING_THREAD_COPIES
        assert (p["threads_per_row"], p["vec_per_thread"], p["block_threads"]) == (tpr, vpt, 512), N
    assert _plan(1 << 20, 2048, rs.RS_BF16, opts={"block_threads": 256})["block_threads"] == 256
    assert _plan(64 * 152 - 1, 2048, rs.RS_BF16)["block_threads"] == 256  # few rows: unchanged
    # rows of 769 to 1024 units: 4 warps a row at 8 units a thread, 512-thread
    # CTAs, three stages (bf16 8192 +7.8 %)
    p = _plan(32768, 8192, rs.RS_BF16)
    assert (p["threads_per_row"], p["vec_per_thread"], p["block_threads"], p["stages"]) == (128, 8, 512, 3)
    assert p["rows_per_cta"] == 4 and p["grid"] == 152 and p["smem_bytes"] == 3 * 4 * 8192 * 2
    p = _plan(32768, 6200, rs.RS_F16, ld=6208)
    assert (p["threads_per_row"], p["vec_per_thread"], p["block_threads"]) == (128, 8, 512) and _covers(p, 6200)
    p = _plan(32768, 6144, rs.RS_BF16)  # 768 units: unchanged
    assert p["block_threads"] != 512 or p["threads_per_row"] != 128
    rc, p = rs.rownorm_plan(rs.RS_OP_LAYERNORM, A, A + (1 << 40), A, A, 1 << 20, 2048, 2048, 2048, 1e-5,
                            rs.RS_BF16, None, gb300())
    assert rc == rs.RS_OK and p["path"] == rs.RS_PATH_RING and p["threads_per_row"] == 32
    assert p["block_threads"] == 128


@pytest.mark.parametrize("dtype", [rs.RS_F16, rs.RS_BF16])
@pytest.mark.parametrize("masked", [False, True])
def test_measured_shapes_are_valid_plans_at_every_16bit_width(dtype, masked):
    # Every multiple of 64 values from 256 to 32768 with enough rows for the
    # measured shapes, plain and under a causal mask of period N: the plan
    # covers the row with an instantiated unit count, its CTA holds whole rows
    # within the block limit of that count, and its stages fit the opt-in
    # shared memory.
    instantiated = {1, 2, 3, 4, 5, 6, 8}
    for N in range(256, 32768 + 1, 64):
        M = max(64 * 152, (1 << 27) // N)
        if masked:
            rc, p = rs.rowsoftmax_causal_plan(A, A + (1 << 40), M, N, N, N, N, 0, dtype, None, gb300())
            assert rc == rs.RS_OK, N
        else:
            p = _plan(M, N, dtype)
        assert _covers(p, N), N
        if p["path"] in (rs.RS_PATH_ROWS, rs.RS_PATH_RING):
            assert p["vec_per_thread"] in instantiated, N
            assert p["block_threads"] % p["threads_per_row"] == 0, N
            limit = 1024 if p["vec_per_thread"] * p["vec_elems"] <= 32 else 512
            assert p["block_threads"] <= limit, N
            assert p["smem_bytes"] <= 232448 - 1024, N
