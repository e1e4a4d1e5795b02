"""Pins for the CPU oracle, independent of the oracle itself.

Each check ties the oracle to something it does not compute: hand-derived
closed forms (tests/golden/softmax_closed_forms.txt), a high-precision
brute-force evaluation of the unshifted formula (mpmath), exact library
conversions (numpy float16, torch bfloat16), and invariants that the
mathematics fixes (rows sum to one, shift invariance, all-equal rows give
1/N, order preservation, the spike closed form).  The definition pinned is
the row softmax of "stanleyjacob.dev: Triton", Part II, "Worked example:
fused softmax", with -inf padding from the "Safe Softmax Pattern" of the
Hugging Face "triton-kernels" skill page.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "softmax_closed_forms.txt")


def _parse_in(tok):
    if tok == "-inf":
        return -math.inf
    if tok.startswith("ln(") and tok.endswith(")"):
        return math.log(int(tok[3:-1]))
    return float(tok)


def _golden_cases():
    cases = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, xin, yout, tol, _why = [p.strip() for p in line.split("|")]
            x = np.array([_parse_in(t) for t in xin.split()], dtype=np.float64)
            y = [Fraction(t) for t in yout.split()]
            cases.append((name, x, y, float(tol)))
    return cases


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c[0])
def test_closed_forms(case):
    _name, x, y, tol = case
    got = oracle.softmax_f64(x[None, :], "f64")[0]
    want = np.array([float(v) for v in y])
    assert np.all(np.abs(got - want) <= tol), (got, want)


def test_golden_two_by_four_batch():
    # The 2x4 hand case as one batch: row 0 zeros, row 1 ln(1..4).
    x = np.array([[0, 0, 0, 0], [math.log(k) for k in (1, 2, 3, 4)]], dtype=np.float64)
    y = oracle.softmax_f64(x, "f64")
    assert np.array_equal(y[0], np.full(4, 0.25))
    assert np.max(np.abs(y[1] - np.array([0.1, 0.2, 0.3, 0.4]))) <= 1e-15


def test_brute_force_mpmath_unshifted():
    """For |x| < 50 the unshifted quotient exp(x_j)/sum exp(x_k) does not
    overflow; evaluated at 40 digits it is the exact value the oracle must
    reach to within double rounding."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    rng = np.random.default_rng(12345)
    for n in range(1, 9):
        for _ in range(25):
            x = rng.uniform(-49.0, 49.0, size=n)
            got = oracle.softmax_f64(x[None, :], "f64")[0]
            den = mpmath.fsum(mpmath.exp(mpmath.mpf(float(v))) for v in x)
            want = np.array([float(mpmath.exp(mpmath.mpf(float(v))) / den) for v in x])
            assert np.allclose(got, want, rtol=1e-13, atol=1e-300), (x, got, want)


def test_hand_case_one_to_four():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    e = [mpmath.e ** k for k in (1, 2, 3, 4)]
    want = np.array([float(v / sum(e)) for v in e])
    got = oracle.softmax_f64(np.array([[1.0, 2.0, 3.0, 4.0]]), "f64")[0]
    assert np.max(np.abs(got - want)) <= 1e-15


def test_spike_closed_form():
    """One entry of +15 over a row of zeros: y_spike = e^15/(e^15 + N - 1),
    every other entry 1/(e^15 + N - 1).  The oracle sums the row in plain
    recursive order, whose rounding error is bounded by (N-1) * 2^-53 times
    the sum of the terms (the textbook bound for recursive summation); the
    tolerance is that bound plus a few roundings for exp and the divide."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    for n, pos in [(2, 0), (7, 3), (1000, 999), (4096, 17)]:
        x = np.zeros((1, n))
        x[0, pos] = 15.0
        got = oracle.softmax_f64(x, "f64")[0]
        den = mpmath.e ** 15 + (n - 1)
        rel = (n + 3) * 2.0 ** -53
        want_spike = float(mpmath.e ** 15 / den)
        want_other = float(1 / den)
        assert abs(got[pos] - want_spike) <= rel * want_spike
        others = np.delete(got, pos)
        assert np.max(np.abs(others - want_other)) <= rel * want_other


def test_rows_sum_to_one_and_order_preserved():
    rng = np.random.default_rng(7)
    x = rng.normal(0.0, 3.0, size=(64, 257))
    y = oracle.softmax_f64(x, "f64")
    assert np.max(np.abs(y.sum(axis=1) - 1.0)) <= 1e-12
    assert np.all(y > 0)
    for r in range(8):
        order = np.argsort(x[r], kind="stable")
        ys = y[r][order]
        assert np.all(np.diff(ys) >= 0)
        # strictly larger input -> strictly larger output
        strict = np.diff(x[r][order]) > 1e-12
        assert np.all(np.diff(ys)[strict] > 0)


@pytest.mark.parametrize("c", [-1e4, -5.0, 3.7, 1e4])
def test_shift_invariance(c):
    rng = np.random.default_rng(11)
    x = rng.normal(0.0, 1.0, size=(16, 300))
    y0 = oracle.softmax_f64(x, "f64")
    y1 = oracle.softmax_f64(x + c, "f64")
    # x + c is rounded to the spacing of doubles near |c| (< 2e-12 at 1e4),
    # which moves each output by a relative amount of that order.
    assert np.max(np.abs(y0 - y1)) <= 1e-11
    assert np.all(np.isfinite(y1))


@pytest.mark.parametrize("n", [1, 3, 4, 1000, 5000, 8192])
def test_all_equal_rows_give_one_over_n(n):
    for c in (-4.75, 0.0, 2.5, 9984.0):
        y = oracle.softmax_f64(np.full((1, n), c), "f64")[0]
        assert np.all(y == 1.0 / n)


def test_padding_is_never_read():
    rng = np.random.default_rng(3)
    x = rng.normal(size=(5, 13))
    padded = np.full((5, 20), np.nan)
    padded[:, 13:] = np.inf
    padded[:, :13] = x
    assert np.array_equal(oracle.softmax_f64(padded, "f64", n_cols=13), oracle.softmax_f64(x, "f64"))


def test_rows_are_rows_not_columns():
    x = np.array([[0.0, 1.0, 2.0], [5.0, 5.0, 5.0]])
    y = oracle.softmax_f64(x, "f64")
    assert np.allclose(y[1], 1 / 3, atol=0, rtol=1e-15)
    assert y[0, 2] > y[0, 1] > y[0, 0]


def test_special_values_follow_the_formula():
    y = oracle.softmax_f64(np.array([[-np.inf, -np.inf, -np.inf]]), "f64")
    assert np.all(np.isnan(y))                      # (-inf) - (-inf) is NaN
    y = oracle.softmax_f64(np.array([[0.0, np.nan, 1.0]]), "f64")
    assert np.all(np.isnan(y))                      # NaN reaches the sum
    y = oracle.softmax_f64(np.array([[0.0, np.inf, 1.0]]), "f64")
    assert np.all(np.isnan(y))                      # inf - inf is NaN
    y = oracle.softmax_f64(np.array([[-np.inf, 2.0, -np.inf, -np.inf]]), "f64")
    assert np.array_equal(y, np.array([[0.0, 1.0, 0.0, 0.0]]))


def test_empty_shapes():
    assert oracle.softmax_f64(np.zeros((0, 4)), "f64").shape == (0, 4)
    assert oracle.softmax_f64(np.zeros((3, 4)), "f64", n_cols=0).shape == (3, 0)


# ---------------------------------------------------------------------------
# Stored formats: the oracle decodes, computes in double, and encodes with
# round-to-nearest-even.  Pinned against numpy float16 and torch bfloat16.
# ---------------------------------------------------------------------------

def test_decode_f16_all_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode(bits.view(np.float16), "f16")
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_decode_bf16_all_patterns_match_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode(bits, "bf16")
    want = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def _random_doubles(rng, n):
    mant = rng.uniform(1.0, 2.0, size=n)
    expo = rng.integers(-30, 20, size=n)
    sign = rng.choice([-1.0, 1.0], size=n)
    return sign * np.ldexp(mant, expo)


def test_encode_f16_matches_numpy():
    rng = np.random.default_rng(5)
    v = np.concatenate([
        _random_doubles(rng, 200000),
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0 ** -24, 2.0 ** -25,
                  2.0 ** -25 * 1.0000001, 2.0 ** -14, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11,
                  np.inf, -np.inf]),
    ])
    got = oracle.encode(v, "f16").view(np.uint16)
    with np.errstate(over="ignore"):
        want = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)


def test_encode_bf16_matches_torch_on_float32_values():
    rng = np.random.default_rng(6)
    v = _random_doubles(rng, 200000).astype(np.float32).astype(np.float64)
    v = np.concatenate([v, [0.0, -0.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 3.3895313892515355e38,
                            1e-40, -1e-40, np.inf, -np.inf]])
    got = oracle.encode(v, "bf16")
    want = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_encode_bf16_is_nearest_even_for_any_double():
    """Property check through the pinned decoder: the encoding is one of the
    two neighbours of v, the nearer one, and on a tie the one with an even
    last fraction bit."""
    rng = np.random.default_rng(8)
    v = np.abs(_random_doubles(rng, 50000))
    b = oracle.encode(v, "bf16").astype(np.int64)
    here = oracle.decode(b.astype(np.uint16), "bf16")
    lo = oracle.decode(np.where(here > v, b - 1, b).astype(np.uint16), "bf16")
    hi = oracle.decode(np.where(here > v, b, b + 1).astype(np.uint16), "bf16")
    assert np.all((lo <= v) & (v <= hi))
    d_here = np.abs(here - v)
    assert np.all(d_here <= np.minimum(np.abs(lo - v), np.abs(hi - v)))
    tie = np.abs(lo - v) == np.abs(hi - v)
    assert np.all((b[tie] & 1) == 0)


@pytest.mark.parametrize("fmt", ["f32", "f16", "bf16"])
def test_stored_formats_are_decoded_exactly(fmt):
    rng = np.random.default_rng(9)
    x64 = rng.normal(0.0, 2.0, size=(6, 77))
    if fmt == "f32":
        xs = x64.astype(np.float32)
        dec = xs.astype(np.float64)
    elif fmt == "f16":
        xs = x64.astype(np.float16)
        dec = xs.astype(np.float64)
    else:
        t = torch.from_numpy(x64.astype(np.float32)).to(torch.bfloat16)
        xs = t.view(torch.int16).numpy().view(np.uint16)
        dec = t.double().numpy()
    assert np.array_equal(oracle.softmax_f64(xs, fmt), oracle.softmax_f64(dec, "f64"))


@pytest.mark.parametrize("fmt", ["f32", "f16", "bf16", "f64"])
@pytest.mark.parametrize("nthreads", [1, 3])
def test_store_variant_encodes_the_f64_result(fmt, nthreads):
    rng = np.random.default_rng(10)
    x64 = rng.normal(0.0, 1.0, size=(11, 40))
    xs = oracle.encode(x64, fmt)
    y = oracle.softmax_store(xs, fmt, n_cols=33, nthreads=nthreads)
    ref = oracle.encode(oracle.softmax_f64(xs, fmt, n_cols=33), fmt)
    assert np.array_equal(y[:, :33].view(np.uint8), ref.view(np.uint8))
    assert np.all(y[:, 33:].view(np.uint8) == 0)


def test_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.softmax_f64(np.zeros((2, 4)), "f64", n_cols=5)
