"""GPU parity of the split-row softmax (rowsoftmax_partial_fwd,
rowsoftmax_merge_ml, rowsoftmax_finish_fwd, rowsoftmax_split_fwd) against the
CPU oracle, through the C ABI.

Rows are cut into R column shards on one device (the shards of the
vocabulary-parallel softmax, cut at aligned and unaligned columns, empty
shards included): each shard's pairs are compared with the oracle's (the max
exactly, the sum under the recursive-summation bound), the merged pairs with
the oracle's merge, and the finished rows, assembled from the shards, with
the oracle's softmax of the whole rows under the row softmax tolerances.
The one-device split of few wide rows is compared the same way, and the two
largest benchmark workloads are split into shards and checked on every row."""
import math

import numpy as np
import pytest
import torch
import torch.distributed as dist

import memory_bound_row_gb300 as rs
import oracle
from memory_bound_row_gb300 import build
from memory_bound_row_gb300 import workloads as W

from _parity import FMT, check_all_rows, compare, norm_gamma, oracle_rows, to_storage_numpy

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


def _input(M, N, dtype, ld=None, kind="normal1", seed=0):
    return W.generate(W.custom(M, N, dtype, ld=ld, seed=seed, kind=kind), "cuda")


def _cuts(N, R, seed, aligned):
    """R + 1 column cuts 0 = c_0 <= ... <= c_R = N (16-byte multiples when aligned)."""
    rng = np.random.default_rng(seed)
    inner = sorted(rng.integers(0, N + 1, size=R - 1).tolist())
    if aligned:
        inner = [c - c % 8 for c in inner]
    return [0] + inner + [N]


def _pairs_ref(x, a, b):
    xs = to_storage_numpy(x[:, a:b])
    return oracle.softmax_partial_f64(xs, FMT[x.dtype], b - a)


def _check_pairs(got, ref, n, what):
    """m bit for bit (the max of stored values is exact in fp32); l within the
    summation bound of n terms plus the exponential's own error."""
    g = got.double().cpu().numpy()
    assert np.array_equal(g[:, 0], ref[:, 0].astype(np.float32).astype(np.float64), equal_nan=True), what
    nan_g, nan_r = np.isnan(g[:, 1]), np.isnan(ref[:, 1])
    assert np.array_equal(nan_g, nan_r), what
    ok = ~nan_r
    tol = (norm_gamma(max(n, 1)) + 2.0 ** -20) * np.abs(ref[ok, 1])
    err = np.abs(g[ok, 1] - ref[ok, 1])
    assert np.all(err <= tol), f"{what}: l off by {float((err / np.maximum(tol, 1e-300)).max()):.3g} of its bound"


def _split_and_finish(x, cuts, out=None):
    """partial on every shard, finish of every shard with all R pairs."""
    M, N = x.shape
    R = len(cuts) - 1
    pairs = torch.empty((R, M, 2), dtype=torch.float32, device="cuda")
    for s in range(R):
        rs.softmax_partial(x[:, cuts[s]:cuts[s + 1]], ml=pairs[s])
    y = torch.empty_like(x) if out is None else out
    for s in range(R):
        a, b = cuts[s], cuts[s + 1]
        if b > a:
            rs.softmax_finish(x[:, a:b], pairs, out=y[:, a:b])
    torch.cuda.synchronize()
    return pairs, y


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("M,N", [(1, 1), (5, 3), (37, 100), (64, 1000), (300, 2048), (20, 5000), (7, 40000),
                                 (3, 131072)])
@pytest.mark.parametrize("R", [1, 2, 3, 8])
@pytest.mark.parametrize("aligned", [True, False])
def test_shards_partial_merge_finish(dtype, M, N, R, aligned):
    vec = 4 if dtype == "f32" else 8
    ld = -(-N // vec) * vec
    x = _input(M, N, dtype, ld=ld, kind="normal_spike", seed=M * 31 + N + R)[:, :N]
    cuts = _cuts(N, R, seed=N + R, aligned=aligned)
    pairs, y = _split_and_finish(x, cuts)
    for s in range(R):
        _check_pairs(pairs[s], _pairs_ref(x, cuts[s], cuts[s + 1]), cuts[s + 1] - cuts[s], f"pairs of shard {s}")
    merged = rs.softmax_merge(pairs)
    torch.cuda.synchronize()
    ref_merged = oracle.merge_pairs_f64(pairs.double().cpu().numpy())
    g = merged.double().cpu().numpy()
    assert np.array_equal(g[:, 0], ref_merged[:, 0].astype(np.float32).astype(np.float64))
    assert np.allclose(g[:, 1], ref_merged[:, 1], rtol=R * 2.0 ** -20, atol=0)
    compare(y, oracle_rows(x, N), dtype, f"{R} shards {dtype} {M}x{N} aligned={aligned}")
    # the finish from the already merged pairs gives the same rows
    y1 = torch.empty_like(y)
    for s in range(R):
        a, b = cuts[s], cuts[s + 1]
        if b > a:
            rs.softmax_finish(x[:, a:b], merged, out=y1[:, a:b])
    torch.cuda.synchronize()
    compare(y1, oracle_rows(x, N), dtype, f"{R} shards, merged first")


def test_special_values_across_shards():
    # an all -inf row (NaN), a row whose first shard is all -inf, NaN and +inf
    # in one shard (NaN rows), a single finite value, a huge common offset
    M, N = 6, 64
    x = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    x[0] = -math.inf
    x[1, :32] = -math.inf
    x[1, 40] = 3.0
    x[2, 5] = math.nan
    x[3, 50] = math.inf
    x[4] = -math.inf
    x[4, 63] = 7.0
    x[5] = 1e4 + torch.arange(N, device="cuda") * 1e-2
    cuts = [0, 32, 64]
    pairs, y = _split_and_finish(x, cuts)
    for s in range(2):
        _check_pairs(pairs[s], _pairs_ref(x, cuts[s], cuts[s + 1]), 32, f"special pairs {s}")
    assert float(pairs[0, 1, 0]) == -math.inf and float(pairs[0, 1, 1]) == 0.0  # no mass: the starting pair
    compare(y, oracle_rows(x, N), "f32", "special values across shards")
    yd = y.cpu().numpy()
    assert np.all(np.isnan(yd[0])) and np.all(np.isnan(yd[2])) and np.all(np.isnan(yd[3]))
    assert yd[4, 63] == 1.0 and np.all(yd[4, :63] == 0.0)


def test_empty_shard_and_zero_pairs():
    x = _input(9, 300, "bf16", seed=5)
    cuts = [0, 0, 150, 150, 300]  # two shards with no column
    pairs, y = _split_and_finish(x, cuts)
    for s in (0, 2):
        assert bool((pairs[s, :, 0] == -math.inf).all()) and bool((pairs[s, :, 1] == 0).all())
    compare(y, oracle_rows(x, 300), "bf16", "empty shards")
    empty = torch.empty((0, 9, 2), dtype=torch.float32, device="cuda")
    merged = rs.softmax_merge(empty)
    torch.cuda.synchronize()
    assert bool((merged[:, 0] == -math.inf).all()) and bool((merged[:, 1] == 0).all())


def test_merge_of_given_pairs_against_the_oracle():
    rng = np.random.default_rng(3)
    R, M = 37, 500
    p = np.empty((R, M, 2), dtype=np.float32)
    p[..., 0] = rng.normal(scale=30.0, size=(R, M))
    p[..., 1] = rng.uniform(0.5, 1000.0, size=(R, M))
    p[3, :100] = (-np.inf, 0.0)   # empty shards
    p[:, 200] = (-np.inf, 0.0)    # a row with no mass anywhere
    p[5, 300, 1] = np.nan         # a NaN sum
    t = torch.from_numpy(p).cuda()
    got = rs.softmax_merge(t).double().cpu().numpy()
    ref = oracle.merge_pairs_f64(p.astype(np.float64))
    assert np.array_equal(got[:, 0], ref[:, 0].astype(np.float32).astype(np.float64))
    assert np.array_equal(np.isnan(got[:, 1]), np.isnan(ref[:, 1]))
    ok = ~np.isnan(ref[:, 1])
    assert np.allclose(got[ok, 1], ref[ok, 1], rtol=R * 2.0 ** -20, atol=0)
    assert got[200, 0] == -np.inf and got[200, 1] == 0.0 and np.isnan(got[300, 1])


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("M,N", [(1, 1), (1, 1000), (2, 70001), (3, 1 << 20), (1, 3000000), (16, 300000),
                                 (64, 65536), (600, 5000)])
def test_split_fwd(dtype, M, N):
    x = _input(M, N, dtype, kind="normal_spike", seed=M + N)
    y = rs.softmax_split(x)
    torch.cuda.synchronize()
    check_all_rows("softmax", x, y, N, what=f"split {dtype} {M}x{N}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_split_fwd_strides_misalignment_in_place(dtype):
    M, N, ld = 5, 200001, 200016
    base = _input(M, N + 8, dtype, ld=ld, seed=7)
    x = base[:, 3: 3 + N]  # misaligned: element-wise kernels
    ref = oracle_rows(x, N)
    out = torch.full((M, ld), 5.0, dtype=DT[dtype], device="cuda")
    y = rs.softmax_split(x, out=out[:, :N])
    torch.cuda.synchronize()
    compare(y, ref, dtype, "split misaligned, padded")
    assert bool((out[:, N:] == 5.0).all())  # padding untouched
    x2 = _input(M, N, dtype, ld=ld, seed=8)[:, :N]
    ref2 = oracle_rows(x2, N)
    y2 = rs.softmax_split(x2, out=x2)
    torch.cuda.synchronize()
    compare(y2, ref2, dtype, "split in place")


def test_split_fwd_reuses_a_dirty_workspace():
    x = _input(4, 500000, "f16", kind="normal_spike", seed=11)
    rc, need = rs.rowsoftmax_split_workspace_size(4, 500000, rs.RS_F16)
    assert rc == rs.RS_OK
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")  # NaN patterns everywhere
    ref = oracle_rows(x, 500000)
    for _ in range(2):
        y = rs.softmax_split(x, workspace=ws)
        torch.cuda.synchronize()
        compare(y, ref, "f16", "split with a reused workspace")


def test_two_to_the_26_elements_split():
    x = _input(2, 1 << 26, "f16", kind="normal_spike", seed=26)
    y = rs.softmax_split(x)
    torch.cuda.synchronize()
    check_all_rows("softmax", x, y, 1 << 26, what="split f16 2 x 2^26")
    del x, y
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,R", [("bf16_causal_16x32x2048", 2), ("fp16_512x131072", 8)])
def test_benchmark_workloads_split_into_shards(name, R):
    # every row of the full-size workload, split into R aligned column shards
    w = W.WORKLOADS[name]
    x = W.generate(w, "cuda")
    cuts = [w.N * s // R for s in range(R + 1)]
    _, y = _split_and_finish(x, cuts)
    check_all_rows("softmax", x, y, w.N, what=f"{R} shards of softmax {name}")
    del x, y
    torch.cuda.empty_cache()


def test_vocab_parallel_front_end_on_one_rank():
    # the whole path of softmax_vocab_parallel (partial, exchange, finish) in a
    # one-rank group: the result is the row softmax
    store = dist.HashStore()
    dist.init_process_group("gloo", store=store, rank=0, world_size=1)
    try:
        x = _input(333, 3000, "bf16", kind="normal_spike", seed=12)
        y = rs.softmax_vocab_parallel(x)
        torch.cuda.synchronize()
        compare(y, oracle_rows(x, 3000), "bf16", "vocab parallel, one rank")
    finally:
        dist.destroy_process_group()
