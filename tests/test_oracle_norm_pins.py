"""Pins for the oracle's RMSNorm and LayerNorm, independent of the oracle:
hand-derived closed forms (tests/golden/norm_closed_forms.txt), a 40-digit
mpmath brute force, and invariants fixed by the mathematics (LayerNorm output
has mean 0 and variance var/(var+eps); shift and scale invariance; RMSNorm
output has mean square ms/(ms+eps); RMSNorm is odd and scale invariant)."""
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "norm_closed_forms.txt")


def _cases():
    out = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            op, name, xin, w, b, eps, want, tol, _why = [p.strip() for p in line.split("|")]
            vec = lambda s: None if s == "-" else np.array([float(t) for t in s.split()])
            want = np.array([eval(t, {"sqrt": math.sqrt}) for t in want.split()])
            out.append((op, name, vec(xin), vec(w), vec(b), float(eps), want, float(tol)))
    return out


@pytest.mark.parametrize("case", _cases(), ids=lambda c: f"{c[0]}-{c[1]}")
def test_closed_forms(case):
    op, _name, x, w, b, eps, want, tol = case
    if op == "rms":
        got = oracle.rmsnorm_f64(x[None, :], "f64", weight=w, eps=eps)[0]
    else:
        got = oracle.layernorm_f64(x[None, :], "f64", weight=w, bias=b, eps=eps)[0]
    assert np.all(np.abs(got - want) <= tol), (got, want)


def test_brute_force_mpmath():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    rng = np.random.default_rng(77)
    for n in range(1, 9):
        for _ in range(10):
            x = rng.normal(0, 3, size=n)
            w = rng.normal(1, 0.5, size=n)
            b = rng.normal(0, 1, size=n)
            eps = float(rng.choice([0.0, 1e-5, 0.5])) if n > 1 else 0.5
            X = [mpmath.mpf(float(v)) for v in x]
            ms = mpmath.fsum(v * v for v in X) / n
            want_r = np.array([float(X[j] / mpmath.sqrt(ms + eps) * w[j]) for j in range(n)])
            mu = mpmath.fsum(X) / n
            var = mpmath.fsum((v - mu) ** 2 for v in X) / n
            want_l = np.array([float((X[j] - mu) / mpmath.sqrt(var + eps) * w[j] + b[j]) for j in range(n)])
            got_r = oracle.rmsnorm_f64(x[None, :], "f64", weight=w, eps=eps)[0]
            got_l = oracle.layernorm_f64(x[None, :], "f64", weight=w, bias=b, eps=eps)[0]
            assert np.allclose(got_r, want_r, rtol=1e-12, atol=1e-12)
            assert np.allclose(got_l, want_l, rtol=1e-10, atol=1e-10)


def test_layernorm_output_moments():
    rng = np.random.default_rng(5)
    x = rng.normal(3.0, 2.0, size=(20, 513))
    for eps in (0.0, 1e-5, 0.7):
        y = oracle.layernorm_f64(x, "f64", eps=eps)
        var = x.var(axis=1)
        assert np.max(np.abs(y.mean(axis=1))) <= 1e-12
        assert np.max(np.abs(y.var(axis=1) - var / (var + eps))) <= 1e-12


def test_layernorm_shift_and_scale_invariance():
    rng = np.random.default_rng(6)
    x = rng.normal(0.0, 1.0, size=(8, 300))
    y0 = oracle.layernorm_f64(x, "f64", eps=0.0)
    assert np.max(np.abs(oracle.layernorm_f64(x + 1e3, "f64", eps=0.0) - y0)) <= 1e-9
    assert np.max(np.abs(oracle.layernorm_f64(x * 7.5, "f64", eps=0.0) - y0)) <= 1e-12


def test_rmsnorm_moments_oddness_and_scale():
    rng = np.random.default_rng(7)
    x = rng.normal(0.5, 2.0, size=(16, 257))
    for eps in (0.0, 1e-6, 2.0):
        y = oracle.rmsnorm_f64(x, "f64", eps=eps)
        ms = (x * x).mean(axis=1)
        assert np.max(np.abs((y * y).mean(axis=1) - ms / (ms + eps))) <= 1e-12
    y0 = oracle.rmsnorm_f64(x, "f64", eps=0.0)
    assert np.array_equal(oracle.rmsnorm_f64(-x, "f64", eps=0.0), -y0)
    assert np.max(np.abs(oracle.rmsnorm_f64(x * 0.125, "f64", eps=0.0) - y0)) <= 1e-15


def test_weight_and_bias_are_per_column():
    x = np.array([[1.0, 2.0, 3.0], [3.0, 2.0, 1.0]])
    w = np.array([1.0, 10.0, 100.0])
    y = oracle.rmsnorm_f64(x, "f64", weight=w, eps=0.0)
    y1 = oracle.rmsnorm_f64(x, "f64", eps=0.0)
    assert np.allclose(y, y1 * w[None, :], rtol=1e-15, atol=0)
    b = np.array([-1.0, 0.0, 1.0])
    z = oracle.layernorm_f64(x, "f64", weight=w, bias=b, eps=0.0)
    z1 = oracle.layernorm_f64(x, "f64", eps=0.0)
    assert np.allclose(z, z1 * w[None, :] + b[None, :], rtol=1e-15, atol=1e-15)


@pytest.mark.parametrize("fmt", ["f32", "f16", "bf16"])
def test_stored_formats_decode_input_and_weights(fmt):
    rng = np.random.default_rng(8)
    x64 = rng.normal(0, 2, size=(5, 70))
    w64 = rng.normal(1, 0.3, size=70)
    b64 = rng.normal(0, 0.3, size=70)
    xs, ws, bs = oracle.encode(x64, fmt), oracle.encode(w64, fmt), oracle.encode(b64, fmt)
    xd, wd, bd = oracle.decode(xs, fmt), oracle.decode(ws, fmt), oracle.decode(bs, fmt)
    assert np.array_equal(oracle.rmsnorm_f64(xs, fmt, weight=ws, eps=1e-6),
                          oracle.rmsnorm_f64(xd, "f64", weight=wd, eps=1e-6))
    assert np.array_equal(oracle.layernorm_f64(xs, fmt, weight=ws, bias=bs, eps=1e-5),
                          oracle.layernorm_f64(xd, "f64", weight=wd, bias=bd, eps=1e-5))


def test_padding_is_never_read():
    rng = np.random.default_rng(9)
    x = rng.normal(size=(4, 11))
    padded = np.full((4, 16), np.nan)
    padded[:, :11] = x
    assert np.array_equal(oracle.rmsnorm_f64(padded, "f64", n_cols=11), oracle.rmsnorm_f64(x, "f64"))
    assert np.array_equal(oracle.layernorm_f64(padded, "f64", n_cols=11), oracle.layernorm_f64(x, "f64"))


def test_zero_variance_with_zero_eps_is_nan():
    y = oracle.layernorm_f64(np.array([[2.0, 2.0]]), "f64", eps=0.0)
    assert np.all(np.isnan(y))  # 0 / 0
    y = oracle.rmsnorm_f64(np.array([[0.0, 0.0]]), "f64", eps=0.0)
    assert np.all(np.isnan(y))
