"""CPU checks of the row normalisations' C entry points (rmsnorm_fwd,
layernorm_fwd, rownorm_fwd_ex, rownorm_plan): argument validation before any
device call, and the launches the planner picks.  No kernel runs."""
import pytest

import memory_bound_row_gb300 as rs
from memory_bound_row_gb300 import build

from test_abi_cpu import gb300

A = 1 << 20            # 16-byte aligned fake addresses; validation fails before they are used
OUT = A + (1 << 40)
W = A + (1 << 41)
B = A + (1 << 42)
NORM_VPT_VEC = {1, 2, 3, 4, 5, 6, 8}
NORM_VPT_SCALAR = {1, 2, 4, 8, 16}


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _plan(op, M, N, dtype, ld=None, opts=None, a=A, o=OUT, w=W, b=None, eps=1e-5):
    rc, plan = rs.rownorm_plan(op, a, o, w, b, M, N, ld or N, ld or N, eps, dtype, opts, gb300())
    assert rc == rs.RS_OK, rs.rowsoftmax_status_string(rc)
    return plan


def _covers(plan, N):
    units = -(-N // plan["vec_elems"])
    if plan["path"] in (rs.RS_PATH_ROWS, rs.RS_PATH_RING):
        return plan["threads_per_row"] * plan["vec_per_thread"] >= units
    if plan["path"] == rs.RS_PATH_CLUSTER:  # register-holding clusters: every slice fits its CTA
        return (plan["ring_values"] == rs.RS_RING_REGISTERS and plan["cluster_size"] * plan["chunk_elems"] >= N
                and plan["block_threads"] * plan["vec_per_thread"] * plan["vec_elems"] >= plan["chunk_elems"])
    return plan["path"] == rs.RS_PATH_STREAM and plan["cluster_size"] == 1


@pytest.mark.parametrize(
    "op,b,eps,status",
    [
        (rs.RS_OP_SOFTMAX, None, 1e-5, rs.RS_ERR_INVALID_ARG),      # not a normalisation
        (7, None, 1e-5, rs.RS_ERR_INVALID_ARG),
        (rs.RS_OP_RMSNORM, B, 1e-5, rs.RS_ERR_INVALID_ARG),         # RMSNorm has no bias
        (rs.RS_OP_RMSNORM, None, -1e-6, rs.RS_ERR_INVALID_ARG),
        (rs.RS_OP_LAYERNORM, None, float("nan"), rs.RS_ERR_INVALID_ARG),
        (rs.RS_OP_LAYERNORM, B, float("inf"), rs.RS_ERR_INVALID_ARG),
        (rs.RS_OP_LAYERNORM, B, 1e39, rs.RS_ERR_INVALID_ARG),       # not a finite float
        (rs.RS_OP_LAYERNORM, B, 0.0, rs.RS_OK),
        (rs.RS_OP_RMSNORM, None, 1e-6, rs.RS_OK),
    ],
)
def test_op_bias_and_eps_are_validated(op, b, eps, status):
    rc, plan = rs.rownorm_plan(op, A, OUT, W, b, 64, 1024, 1024, 1024, eps, rs.RS_F32, None, gb300())
    assert rc == status
    assert rs.rownorm_fwd_ex(op, A, OUT, W, b, 64, 1024, 1024, 1024, eps, rs.RS_F32, 0, None) == (
        status if status != rs.RS_OK else rs.rownorm_fwd_ex(op, A, OUT, W, b, 64, 1024, 1024, 1024, eps,
                                                            rs.RS_F32, 0, None))
    if status == rs.RS_OK:
        assert plan["op"] == op


@pytest.mark.parametrize(
    "w,b,status",
    [
        (OUT + 64, None, rs.RS_ERR_OVERLAP),          # weight inside the output
        (None, OUT + 4096 * 4 - 8, rs.RS_ERR_OVERLAP),  # bias straddles the output's end
        (OUT - 1024 * 4 + 4, None, rs.RS_ERR_OVERLAP),  # weight's last value is the output's first
        (OUT - 1024 * 4, None, rs.RS_OK),             # ends where the output starts
        (A + 64, None, rs.RS_OK),                     # inside the input: read-only, allowed
        (W + 2, None, rs.RS_ERR_INVALID_ARG),         # not element-aligned
        (None, B + 1, rs.RS_ERR_INVALID_ARG),
    ],
)
def test_weight_and_bias_pointers_are_validated(w, b, status):
    rc, _ = rs.rownorm_plan(rs.RS_OP_LAYERNORM, A, OUT, w, b, 4, 1024, 1024, 1024, 1e-5, rs.RS_F32, None,
                            gb300())
    assert rc == status
    if status != rs.RS_OK:  # rejected before any device call
        assert rs.layernorm_fwd(A, OUT, w, b, 4, 1024, 1024, 1024, 1e-5, rs.RS_F32, 0) == status


def test_shape_errors_match_the_softmax():
    for args, status in [((A, OUT, -1, 8, 8, 8), rs.RS_ERR_INVALID_ARG),
                         ((A, OUT, 4, 8, 7, 8), rs.RS_ERR_INVALID_ARG),
                         ((A, A + 64, 4, 8, 8, 8), rs.RS_ERR_OVERLAP),
                         ((0, OUT, 4, 8, 8, 8), rs.RS_ERR_INVALID_ARG)]:
        assert rs.rmsnorm_fwd(args[0], args[1], None, *args[2:], 1e-6, rs.RS_F32, 0) == status
        assert rs.rmsnorm_fwd(args[0], args[1], None, *args[2:], 1e-6, 9, 0) == rs.RS_ERR_UNSUPPORTED_DTYPE
    assert rs.rmsnorm_fwd(0, 0, None, 0, 8, 8, 8, 1e-6, rs.RS_F32, 0) == rs.RS_OK  # empty: no-op
    assert rs.layernorm_fwd(0, 0, None, None, 8, 0, 0, 0, 1e-5, rs.RS_BF16, 0) == rs.RS_OK


def test_plans_for_typical_hidden_sizes():
    # 16-bit rows between 512 B and 32 KB: the bulk-copy ring, holding the row in registers
    for op in (rs.RS_OP_RMSNORM, rs.RS_OP_LAYERNORM):
        p = _plan(op, 32768, 8192, rs.RS_BF16)
        assert p["path"] == rs.RS_PATH_RING and p["ring_values"] == rs.RS_RING_REGISTERS and _covers(p, 8192)
        assert p["vec_per_thread"] in NORM_VPT_VEC
        p = _plan(op, 8192, 5000, rs.RS_F32, ld=5120)   # fp32: register rows (LayerNorm: the held ring)
        assert p["path"] == (rs.RS_PATH_ROWS if op == rs.RS_OP_RMSNORM else rs.RS_PATH_RING)
        assert p["vec_elems"] == 4 and _covers(p, 5000)
        p = _plan(op, 512, 131072, rs.RS_F16)          # wide rows: a cluster per row, slices in registers
        assert p["path"] == rs.RS_PATH_CLUSTER and p["ring_values"] == rs.RS_RING_REGISTERS
        assert p["cluster_size"] >= 2 and p["grid"] % p["cluster_size"] == 0 and _covers(p, 131072)
        p = _plan(op, 512, 131072, rs.RS_F16, a=A + 2)  # misaligned wide rows: one streaming CTA per row
        assert p["path"] == rs.RS_PATH_STREAM and p["grid"] == 2 * 152 and p["vec_elems"] == 1
        p = _plan(op, 100, 1 << 22, rs.RS_F32)          # beyond the clusters' registers
        assert p["path"] == rs.RS_PATH_STREAM and p["grid"] == 100


def test_layernorm_ring_stages_its_vectors_in_shared_memory():
    # LayerNorm's ring CTAs copy weight and bias into shared memory once, after
    # the ring stages (padded to whole 16-byte units); RMSNorm's do not.
    N = 2047
    p = _plan(rs.RS_OP_LAYERNORM, 1 << 20, N, rs.RS_BF16, ld=2048, b=B)
    stage = (N // 8) * 16 * p["rows_per_cta"]
    assert p["path"] == rs.RS_PATH_RING and p["smem_bytes"] == stage * p["stages"] + 2 * 2048 * 2
    p = _plan(rs.RS_OP_LAYERNORM, 1 << 20, N, rs.RS_BF16, ld=2048, w=None, b=B)
    assert p["smem_bytes"] == stage * p["stages"] + 2048 * 2
    p = _plan(rs.RS_OP_RMSNORM, 1 << 20, N, rs.RS_BF16, ld=2048)
    assert p["smem_bytes"] == (N // 8) * 16 * p["rows_per_cta"] * p["stages"]


@pytest.mark.parametrize("dtype", [rs.RS_F16, rs.RS_BF16])
def test_layernorm_rows_of_4_or_8_warps_hold_their_vectors_in_registers(dtype):
    # 16-bit LayerNorm rows that fill 4 or 8 warps at 4 units a thread run the
    # instance with weight and bias in registers: 256-thread CTAs, 128
    # registers a thread, so the persistent grid is 2 CTAs an SM, and nothing
    # is staged in shared memory beside the ring stages.
    # (4096-value rows: one row a 128-thread CTA, 4 CTAs an SM, measured 8 % faster)
    for N, tpr, block, grid in [(4096, 128, 128, 4 * 152), (8192, 256, 256, 2 * 152)]:
        p = _plan(rs.RS_OP_LAYERNORM, 32768, N, dtype, b=B)
        assert p["path"] == rs.RS_PATH_RING and p["vec_per_thread"] == 4 and p["threads_per_row"] == tpr
        assert p["block_threads"] == block and p["grid"] == grid
        assert p["smem_bytes"] == (N // 8) * 16 * p["rows_per_cta"] * p["stages"]
    # rows of 2 warps keep one warp a row (measured faster), RMSNorm keeps its plan,
    # and a ragged row of the same size keeps the staged vectors
    p = _plan(rs.RS_OP_LAYERNORM, 32768, 2048, dtype, b=B)
    assert p["threads_per_row"] <= 32
    # RMSNorm rows of 8 warps at 4 units a thread hold their weight too (2 CTAs
    # an SM); the 12288-value rows' 384-thread CTAs read it from L1
    p = _plan(rs.RS_OP_RMSNORM, 32768, 8192, dtype)
    assert p["path"] == rs.RS_PATH_RING and p["smem_bytes"] == 8192 * 2 * p["rows_per_cta"] * p["stages"]
    assert p["threads_per_row"] == 256 and p["block_threads"] == 256 and p["grid"] == 2 * 152
    # RMSNorm rows of 4 warps hold their weight in 128-thread CTAs, one row a CTA and 4
    # CTAs an SM (measured 6.1 % faster than 2 rows a 256-thread CTA on bf16 4096)
    p = _plan(rs.RS_OP_RMSNORM, 32768, 4096, dtype)
    assert p["threads_per_row"] == 128 and p["block_threads"] == 128 and p["grid"] == 4 * 152
    p = _plan(rs.RS_OP_RMSNORM, 32768, 12288, dtype)
    assert p["threads_per_row"] == 384 and p["grid"] == 2 * 152  # 64 registers, 384 threads: 2 CTAs by threads
    p = _plan(rs.RS_OP_LAYERNORM, 32768, 8184, dtype, ld=8192, b=B)
    assert p["path"] == rs.RS_PATH_RING and p["vec_per_thread"] != 4


def test_ragged_fp32_layernorm_rows_of_4_to_8_warps_take_the_held_ring():
    # fp32 LayerNorm rows that would take two reductions on the register rows
    # and span 4-8 warps at 8 units a thread go to the ring with weight and
    # bias in registers, where at least 14 warps of it fit an SM; filled rows,
    # rows of 2-3 warps and 192-thread rows (2 CTAs, 12 warps an SM) stay.
    for N, tpr, grid in [(4100, 160, 3 * 152), (5000, 160, 3 * 152), (7000, 224, 2 * 152)]:
        ld = -(-N // 4) * 4
        p = _plan(rs.RS_OP_LAYERNORM, 8192, N, rs.RS_F32, ld=ld, b=B)
        assert p["path"] == rs.RS_PATH_RING and p["vec_per_thread"] == 8 and p["threads_per_row"] == tpr, N
        assert p["block_threads"] == tpr and p["grid"] == grid
        assert p["smem_bytes"] == (N // 4) * 16 * p["stages"]  # no staged vectors
    for N in (2048, 3000, 4096, 6000, 8192):
        assert _plan(rs.RS_OP_LAYERNORM, 8192, N, rs.RS_F32, b=B)["path"] == rs.RS_PATH_ROWS, N
    assert _plan(rs.RS_OP_RMSNORM, 8192, 5000, rs.RS_F32, ld=5120)["path"] == rs.RS_PATH_ROWS


def test_wide_16bit_rows_take_the_ring_where_it_fits():
    # Normalisations: the ring wherever its stages fit, 32 values a thread for
    # LayerNorm rows over 8192 values; beyond, the clusters.
    for N in (12288, 20480, 28672):
        for op in (rs.RS_OP_RMSNORM, rs.RS_OP_LAYERNORM):
            p = _plan(op, 8192, N, rs.RS_BF16, b=B if op == rs.RS_OP_LAYERNORM else None)
            assert p["path"] == rs.RS_PATH_RING and p["vec_per_thread"] == 4 and _covers(p, N), (op, N)
    assert _plan(rs.RS_OP_RMSNORM, 8192, 32768, rs.RS_BF16)["path"] == rs.RS_PATH_RING
    p = _plan(rs.RS_OP_LAYERNORM, 8192, 32768, rs.RS_BF16, b=B)  # two 64 KB stages + two 64 KB vectors
    assert p["path"] == rs.RS_PATH_CLUSTER
    p = _plan(rs.RS_OP_RMSNORM, 8192, 40960, rs.RS_BF16)  # 1280 threads at 4 units: beyond a CTA
    assert p["path"] == rs.RS_PATH_CLUSTER and _covers(p, 40960)


def test_misaligned_parameter_vectors_select_element_wise_kernels():
    p = _plan(rs.RS_OP_RMSNORM, 64, 4096, rs.RS_BF16, w=W + 2)
    assert p["vec_elems"] == 1 and p["path"] == rs.RS_PATH_ROWS and p["vec_per_thread"] in NORM_VPT_SCALAR
    p = _plan(rs.RS_OP_LAYERNORM, 64, 4096, rs.RS_F32, w=W, b=B + 4)
    assert p["vec_elems"] == 1
    p = _plan(rs.RS_OP_LAYERNORM, 64, 4096, rs.RS_F32, w=None, b=None)
    assert p["vec_elems"] == 4


def test_paths_without_a_normalisation_kernel():
    for opts in [{"path": rs.RS_PATH_CLUSTER, "ring_values": rs.RS_RING_REREAD},
                 {"path": rs.RS_PATH_CLUSTER, "force_scalar": 1},
                 {"path": rs.RS_PATH_RING, "ring_values": rs.RS_RING_REREAD},
                 {"path": rs.RS_PATH_STREAM, "cluster_size": 2}]:
        rc, _ = rs.rownorm_plan(rs.RS_OP_RMSNORM, A, OUT, W, None, 64, 4096, 4096, 4096, 1e-6, rs.RS_BF16,
                                opts, gb300())
        assert rc == rs.RS_ERR_NO_PATH, opts
    p = _plan(rs.RS_OP_RMSNORM, 64, 4096, rs.RS_BF16, opts={"path": rs.RS_PATH_STREAM})
    assert p["path"] == rs.RS_PATH_STREAM
    p = _plan(rs.RS_OP_LAYERNORM, 64, 4096, rs.RS_BF16, opts={"path": rs.RS_PATH_CLUSTER, "cluster_size": 4})
    assert p["path"] == rs.RS_PATH_CLUSTER and p["cluster_size"] == 4 and _covers(p, 4096)
    p = _plan(rs.RS_OP_LAYERNORM, 64, 4096, rs.RS_F32, opts={"path": rs.RS_PATH_ROWS, "threads_per_row": 128,
                                                              "vec_per_thread": 8})
    assert (p["threads_per_row"], p["vec_per_thread"]) == (128, 8)
    rc, _ = rs.rownorm_plan(rs.RS_OP_LAYERNORM, A, OUT, W, None, 64, 4096, 4096, 4096, 1e-6, rs.RS_F32,
                            {"path": rs.RS_PATH_ROWS, "threads_per_row": 128, "vec_per_thread": 10}, gb300())
    assert rc == rs.RS_ERR_NO_PATH  # 10 units a thread is a softmax-only instance


@pytest.mark.parametrize("op", [rs.RS_OP_RMSNORM, rs.RS_OP_LAYERNORM])
@pytest.mark.parametrize("dtype", [rs.RS_F32, rs.RS_F16, rs.RS_BF16])
@pytest.mark.parametrize("N", [1, 2, 7, 8, 9, 33, 255, 1000, 1500, 4096, 5000, 8192, 8193, 16384, 65536,
                               1 << 20])
@pytest.mark.parametrize("aligned", [True, False])
def test_auto_plan_uses_instantiated_kernels_and_covers_the_row(op, dtype, N, aligned):
    a = A if aligned else A + 2 * (1 if dtype else 2)
    p = _plan(op, 3, N, dtype, a=a)
    assert _covers(p, N)
    if p["path"] in (rs.RS_PATH_ROWS, rs.RS_PATH_RING):
        table = NORM_VPT_VEC if p["vec_elems"] > 1 else NORM_VPT_SCALAR
        assert p["vec_per_thread"] in table
        assert p["block_threads"] % p["threads_per_row"] == 0 and p["block_threads"] <= 1024
    if N <= 4096 or (p["vec_elems"] > 1 and N * (4 if dtype == rs.RS_F32 else 2) <= 32 * 1024):
        assert p["path"] in (rs.RS_PATH_ROWS, rs.RS_PATH_RING)  # single pass over HBM


def test_layernorm_16bit_rows_of_2048_units_take_8_units_a_thread():
    # LayerNorm rows of 1537 to 2048 units: 8 units a thread, two rows a
    # 512-thread CTA (measured on bf16 16384: 274.5 -> 220.7 us against 4
    # units a thread in 512-thread CTAs); fewer rows than 64 an SM keep the plan.
    p = _plan(rs.RS_OP_LAYERNORM, 16384, 16384, rs.RS_BF16, b=B)
    assert p["path"] == rs.RS_PATH_RING
    assert (p["threads_per_row"], p["vec_per_thread"], p["block_threads"]) == (256, 8, 512)
    assert _plan(rs.RS_OP_LAYERNORM, 1024, 16384, rs.RS_BF16, b=B)["vec_per_thread"] == 4


def test_16bit_norm_rows_of_257_to_768_units():
    # LayerNorm rows that 6 (else 5, else 4) units a thread fill on whole warps
    # exactly take that shape, one row a CTA (at 5 units at least 128 threads a
    # CTA); RMSNorm rows of 5 to 7 warps at 4 units a thread take three stages
    # (bf16, measured against the previous plans).
    for N, shape in [(2560, (64, 5, 128)), (3072, (64, 6, 64)), (4096, (128, 4, 128)), (4608, (96, 6, 96)),
                     (5120, (128, 5, 128)), (6144, (128, 6, 128))]:
        p = _plan(rs.RS_OP_LAYERNORM, (1 << 29) // N, N, rs.RS_BF16, b=B)
        assert p["path"] == rs.RS_PATH_RING and (p["threads_per_row"], p["vec_per_thread"], p["block_threads"]) == shape
    for N in (4608, 5120, 6144):
        p = _plan(rs.RS_OP_RMSNORM, (1 << 29) // N, N, rs.RS_BF16)
        assert p["vec_per_thread"] == 4 and 128 < p["threads_per_row"] < 256 and p["stages"] == 3, N
    # LayerNorm rows that none fills exactly: 4 units a thread, the planned CTA size
    for N, tpr in [(3584, 128), (5632, 192)]:
        p = _plan(rs.RS_OP_LAYERNORM, (1 << 29) // N, N, rs.RS_BF16, b=B)
        assert (p["threads_per_row"], p["vec_per_thread"]) == (tpr, 4), N


def test_16bit_norm_rows_that_5_units_fill_exactly():
    # 5 units a thread where they fill whole warps exactly (bf16, against the
    # previous plans): LayerNorm from 257 units, one row a CTA (5120 +12 %,
    # 10240 +13 %, 20480 +12 %; 2560 two rows a 128-thread CTA, +40 %);
    # RMSNorm where 4 units do not fill whole warps within 512 threads (1280
    # in 128-thread CTAs +31 %, 2560 +21 %, 20480 +12 %; at 5120 and 10240,
    # where 4 units fill 5 and 10 warps, 5 units measured 8 and 2.5 % slower).
    for dt in (rs.RS_F16, rs.RS_BF16):
        for N, shape in [(10240, (256, 5, 256)), (20480, (512, 5, 512))]:
            p = _plan(rs.RS_OP_LAYERNORM, (1 << 28) // N, N, dt, b=B)
            assert p["path"] == rs.RS_PATH_RING and (p["threads_per_row"], p["vec_per_thread"], p["block_threads"]) == shape
        for N, shape in [(1280, (32, 5, 128)), (2560, (64, 5, 64)), (20480, (512, 5, 512)), (5120, (160, 4, 160)),
                         (10240, (320, 4, 320))]:
            p = _plan(rs.RS_OP_RMSNORM, (1 << 28) // N, N, dt)
            assert p["path"] == rs.RS_PATH_RING and (p["threads_per_row"], p["vec_per_thread"], p["block_threads"]) == shape
    # rows that need exactly 5 units a thread at the first-guess lane count take
    # 5 (the instance list has no gap there): fp32 register rows of 1280 values
    p = _plan(rs.RS_OP_RMSNORM, 100000, 1280, rs.RS_F32)
    assert p["path"] == rs.RS_PATH_ROWS and (p["threads_per_row"], p["vec_per_thread"]) == (64, 5)


def test_16bit_norm_rows_that_6_units_fill_exactly_on_wide_rows():
    # LayerNorm rows of 1536 and 3072 units: 6 units a thread on 8 or 16 warps,
    # one row a CTA (bf16 12288 +9.1 %, 24576 +8.6 %); RMSNorm rows of 2049 to
    # 3072 units that 6 units fill on whole warps: 6 units, one row a CTA
    # (18432 +6.9 %, 21504 +9.9 %, 24576 +11.1 %); rows of other widths, and
    # fewer rows than 64 an SM, keep the plan.
    for op, N, tpr in [(rs.RS_OP_LAYERNORM, 12288, 256), (rs.RS_OP_LAYERNORM, 24576, 512),
                       (rs.RS_OP_RMSNORM, 18432, 384), (rs.RS_OP_RMSNORM, 21504, 448), (rs.RS_OP_RMSNORM, 24576, 512)]:
        for dt in (rs.RS_F16, rs.RS_BF16):
            p = _plan(op, (1 << 28) // N, N, dt, b=B if op == rs.RS_OP_LAYERNORM else None)
            assert p["path"] == rs.RS_PATH_RING and p["stages"] == 2, (op, N)
            assert (p["threads_per_row"], p["vec_per_thread"], p["block_threads"]) == (tpr, 6, tpr), (op, N)
    for op, N, shape in [(rs.RS_OP_LAYERNORM, 18432, (576, 4)), (rs.RS_OP_LAYERNORM, 9216, (288, 4)),
                         (rs.RS_OP_RMSNORM, 12288, (384, 4)), (rs.RS_OP_RMSNORM, 15360, (480, 4))]:
        p = _plan(op, (1 << 28) // N, N, rs.RS_BF16, b=B if op == rs.RS_OP_LAYERNORM else None)
        assert (p["threads_per_row"], p["vec_per_thread"]) == shape, (op, N)
    assert _plan(rs.RS_OP_RMSNORM, 1024, 24576, rs.RS_BF16)["vec_per_thread"] == 4


def test_16bit_layernorm_rows_of_32_to_128_units_hold_about_4_units_a_thread():
    # the fewest lanes (8 to 32) that hold the row at about 4 units a thread
    # (bf16 256 +24 %, 512 +11 %, 768 +12 %, 1024 +2.8 % over 8 units a thread)
    for N, tpr, vpt in [(256, 8, 4), (512, 16, 4), (768, 32, 3), (1024, 32, 4)]:
        p = _plan(rs.RS_OP_LAYERNORM, (1 << 28) // N, N, rs.RS_BF16, b=B)
        assert p["path"] == rs.RS_PATH_RING and (p["threads_per_row"], p["vec_per_thread"]) == (tpr, vpt), N


@pytest.mark.parametrize("op", [rs.RS_OP_RMSNORM, rs.RS_OP_LAYERNORM])
@pytest.mark.parametrize("dtype", [rs.RS_F16, rs.RS_BF16])
def test_measured_shapes_are_valid_plans_at_every_16bit_width(op, dtype):
    # Every multiple of 64 values from 256 to 32768 with enough rows for the
    # measured shapes: the plan covers the row with an instantiated unit count,
    # its CTA holds whole rows within the block limit of that count, and its
    # stages fit the opt-in shared memory.
    for N in range(256, 32768 + 1, 64):
        M = max(64 * 152, (1 << 27) // N)
        p = _plan(op, M, N, dtype, b=B if op == rs.RS_OP_LAYERNORM else None)
        assert _covers(p, N), N
        if p["path"] in (rs.RS_PATH_ROWS, rs.RS_PATH_RING):
            assert p["vec_per_thread"] in NORM_VPT_VEC, N
            assert p["block_threads"] % p["threads_per_row"] == 0, N
            limit = 1024 if p["vec_per_thread"] * p["vec_elems"] <= 32 else 512
            assert p["block_threads"] <= limit, N
            assert p["smem_bytes"] <= 232448 - 1024, N
