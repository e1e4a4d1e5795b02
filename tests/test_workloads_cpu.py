"""CPU checks of the seeded input generator (memory_bound_row_gb300.workloads):
the SplitMix64 hash against its published definition and test vectors, the
uniform and normal transforms, determinism (any subset of rows equals the same
rows of the whole tensor), and each benchmark recipe's stated structure."""
import math

import numpy as np
import pytest
import torch

from memory_bound_row_gb300 import workloads as W

M64 = (1 << 64) - 1


def splitmix64_stream(state: int, n: int):
    """Vigna's SplitMix64 as published: state += 0x9e3779b97f4a7c15, then
    z ^= z >> 30, z *= 0xbf58476d1ce4e5b9, z ^= z >> 27, z *= 0x94d049bb133111eb,
    z ^= z >> 31 (all mod 2^64)."""
    out = []
    for _ in range(n):
        state = (state + 0x9E3779B97F4A7C15) & M64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
        out.append(z ^ (z >> 31))
    return out


def test_splitmix64_published_test_vectors():
    # the first outputs of SplitMix64 seeded with 1234567
    assert splitmix64_stream(1234567, 3) == [6457827717110365317, 3203168211198807973, 9817491932198370423]


@pytest.mark.parametrize("key", [0, 1234567, (1 << 63) + 12345, M64])
def test_counter_hash_is_the_splitmix64_stream(key):
    # hash(counter i, key) is output i of the stream seeded with key (i >= 1),
    # for small and huge counters alike
    ref = splitmix64_stream(key, 40)
    got = W._splitmix64(torch.arange(1, 41, dtype=torch.int64), W._s64(key))
    assert [int(v) & M64 for v in got] == ref
    big = (1 << 62) + 7
    z = (key + big * 0x9E3779B97F4A7C15) & M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    assert int(W._splitmix64(torch.tensor([big]), W._s64(key))[0]) & M64 == z ^ (z >> 31)


def test_uniforms_are_the_top_53_bits_on_the_open_interval():
    c = torch.arange(0, 5000, dtype=torch.int64)
    u = W.uniform(c, 7, 3)
    h = [int(v) & M64 for v in W._splitmix64(c, W._key(7, 3))]
    want = torch.tensor([((x >> 11) + 0.5) * 2.0 ** -53 for x in h], dtype=torch.float64)
    assert torch.equal(u, want)
    assert float(u.min()) > 0.0 and float(u.max()) < 1.0


def test_normals_are_box_muller_of_consecutive_uniforms():
    c = torch.arange(0, 3000, dtype=torch.int64)
    z = W.normal(c, 2, 0)
    u1, u2 = W.uniform(2 * c, 2, 0), W.uniform(2 * c + 1, 2, 0)
    want = torch.sqrt(-2.0 * torch.log(u1)) * torch.cos(2.0 * math.pi * u2)
    assert torch.equal(z, want)
    big = W.normal(torch.arange(200000, dtype=torch.int64), 11, 0).numpy()
    assert abs(big.mean()) < 0.01 and abs(big.var() - 1.0) < 0.02


@pytest.mark.parametrize("kind", ["normal1", "normal2_const", "uniform20_offset", "normal_spike", "causal_scores",
                                  "scores_unmasked", "offset50"])
def test_any_rows_equal_the_same_rows_of_the_whole_tensor(kind):
    w = W.custom(300, 97, "f32", ld=100, seed=5, kind=kind)
    full = W.generate(w, "cpu")
    again = W.generate(w, "cpu")
    assert torch.equal(full[:, :97].view(torch.int32), again[:, :97].view(torch.int32))
    part = W.generate(w, "cpu", row_start=123, row_count=40)
    assert torch.equal(part[:, :97].view(torch.int32), full[123:163, :97].view(torch.int32))
    rows = torch.tensor([299, 0, 7, 150])
    picked = W.generate_rows(w, rows)
    assert torch.equal(picked.view(torch.int32), full[rows, :97].view(torch.int32))
    assert bool(torch.isnan(full[:, 97:]).all())  # padding columns


def test_default_workload_has_exactly_one_percent_constant_rows():
    w = W.WORKLOADS["fp32_8192x5000_ld5120"]
    x = W.generate(w, "cpu", row_start=0, row_count=w.M)[:, : w.N]
    const = (x == x[:, :1]).all(dim=1)
    assert int(const.sum()) == round(0.01 * w.M)
    c = x[const, 0]
    assert float(c.min()) >= -5.0 and float(c.max()) <= 5.0
    rest = x[~const].double()
    assert abs(float(rest.std()) - 2.0) < 0.01  # N(0, var 4)


def test_bf16_offset_rows_and_range():
    w = W.custom(2000, 64, "bf16", seed=2, kind="uniform20_offset")
    x = W.generate(w, "cpu").float()
    off = x.mean(dim=1) > 5000
    assert int(off.sum()) == 200
    assert float(x[~off].abs().max()) <= 20.0
    assert float((x[off] - 1e4).abs().max()) <= 20.0 + 64.0  # bf16 spacing at 1e4 is 64


def test_spike_rows_have_one_plus_15_column():
    w = W.custom(64, 4096, "f16", seed=3, kind="normal_spike")
    x = W.generate(w, "cpu").float()
    spike = (x > 10.0).sum(dim=1)
    assert bool((spike >= 1).all())
    cols = (W._shr(W._splitmix64(torch.arange(64), W._key(3, 3)), 1) % 4096)
    assert bool((x[torch.arange(64), cols] > 8.0).all())


def test_causal_scores_keep_the_prefix_of_each_row():
    w = W.WORKLOADS["bf16_causal_16x32x2048"]
    for r0 in (0, 2040, 2048 * 37 + 5):
        x = W.generate(w, "cpu", row_start=r0, row_count=6).float()
        for i in range(6):
            keep = (r0 + i) % 2048 + 1
            assert bool(torch.isfinite(x[i, :keep]).all())
            assert bool((x[i, keep:] == -math.inf).all())
    xs = W.generate(W.norm_workload("bf16_causal_16x32x2048"), "cpu", row_start=5, row_count=2)
    assert bool(torch.isfinite(xs.float()).all())  # the normalisations' version has no mask


def test_norm_parameters():
    w, b = W.norm_params(100000, "f32", seed=9)
    wn, bn = w.double().numpy(), b.double().numpy()
    assert abs(wn.mean() - 1.0) < 0.005 and abs(wn.std() - 0.25) < 0.005
    assert abs(bn.mean()) < 0.01 and abs(bn.std() - 0.5) < 0.01
    w16, _ = W.norm_params(100, "bf16", seed=9)
    assert torch.equal(w16, w[:100].to(torch.bfloat16))
    assert not np.allclose(W.norm_params(100, "f32", seed=10)[0].numpy(), w[:100].numpy())
