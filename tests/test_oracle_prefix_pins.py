"""Pins for the oracle's row softmax under a causal mask (softmax_prefix_f64),
independent of the oracle: hand-derived closed forms
(tests/golden/softmax_prefix_closed_forms.txt), a 40-digit mpmath brute force
over the kept prefix, the masked part never read, the prefix-length formula
of the attention layout, and the special case L = N that is the plain
(separately pinned) softmax."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "softmax_prefix_closed_forms.txt")


def _num(tok):
    if tok.startswith("ln("):
        return math.log(int(tok[3:-1]))
    return float(tok)


def _want(tok):
    return float("nan") if tok == "nan" else float(Fraction(tok))


def _cases():
    out = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, r, period, offset, xin, want, tol, _why = [p.strip() for p in line.split("|")]
            out.append((name, int(r), int(period), int(offset), np.array([_num(t) for t in xin.split()]),
                        np.array([_want(t) for t in want.split()]), float(tol)))
    return out


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c[0])
def test_closed_forms(case):
    _name, r, period, offset, x, want, tol = case
    got = oracle.softmax_prefix_f64(x[None, :], "f64", period, offset, row0=r)[0]
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.all(np.abs(got[ok] - want[ok]) <= tol), (got, want)


def test_prefix_length_of_the_attention_layout():
    # [B, H, S_q, S_k] scores as (B*H*S_q) x S_k rows: row r is query q = r mod S_q,
    # which sees keys 0 .. q + (S_k - S_q).
    B, H, Sq, Sk = 2, 3, 5, 7
    for r in range(B * H * Sq):
        q = r % Sq
        assert oracle.prefix_len(r, Sk, Sq, Sk - Sq) == min(Sk, q + 1 + Sk - Sq)
        assert oracle.prefix_len(r, Sq, Sq, 0) == q + 1


def test_brute_force_mpmath_over_the_kept_prefix():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    rng = np.random.default_rng(7)
    for n in range(1, 9):
        for period in (1, 3, n):
            for offset in (-1, 0, 2):
                x = rng.uniform(-40.0, 40.0, size=(2 * period, n))
                got = oracle.softmax_prefix_f64(x, "f64", period, offset)
                for r in range(x.shape[0]):
                    L = min(n, max(0, r % period + 1 + offset))
                    if L == 0:
                        assert np.all(np.isnan(got[r]))
                        continue
                    den = mpmath.fsum(mpmath.exp(mpmath.mpf(float(v))) for v in x[r, :L])
                    want = [float(mpmath.exp(mpmath.mpf(float(v))) / den) for v in x[r, :L]]
                    assert np.allclose(got[r, :L], want, rtol=1e-13, atol=1e-300)
                    assert np.all(got[r, L:] == 0.0)


def test_masked_part_is_never_read():
    rng = np.random.default_rng(3)
    x = rng.normal(size=(64, 40))
    a = x.copy()
    b = x.copy()
    for r in range(64):
        L = oracle.prefix_len(r, 40, 16, 3)
        a[r, L:] = np.nan
        b[r, L:] = np.inf
    ya = oracle.softmax_prefix_f64(a, "f64", 16, 3)
    yb = oracle.softmax_prefix_f64(b, "f64", 16, 3)
    assert np.all(np.isfinite(ya)) and np.array_equal(ya, yb)
    assert np.allclose(ya.sum(axis=1), 1.0, rtol=0, atol=1e-14)


def test_full_prefix_is_the_plain_softmax():
    rng = np.random.default_rng(5)
    x = rng.normal(size=(10, 33)).astype(np.float32)
    got = oracle.softmax_prefix_f64(x, "f32", period=1, offset=100)
    assert np.array_equal(got, oracle.softmax_f64(x, "f32"))


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_stored_formats_are_decoded_before_the_mask(fmt):
    rng = np.random.default_rng(9)
    vals = rng.normal(size=(6, 12))
    bits = oracle.encode(vals, fmt)
    dec = oracle.decode(bits, fmt).reshape(6, 12)
    got = oracle.softmax_prefix_f64(bits.reshape(6, 12), fmt, 6, 2)
    assert np.array_equal(got, oracle.softmax_prefix_f64(dec, "f64", 6, 2))


def test_rows_offset_by_row0():
    rng = np.random.default_rng(11)
    x = rng.normal(size=(12, 8))
    whole = oracle.softmax_prefix_f64(x, "f64", 5, 1)
    for r0 in range(12):
        part = oracle.softmax_prefix_f64(x[r0:], "f64", 5, 1, row0=r0)
        assert np.array_equal(part, whole[r0:])
