"""Pins for the oracle's softmax of a row split by columns into shards
(softmax_partial_f64, merge_pairs_f64, softmax_finish_f64), independent of
the oracle: hand-derived closed forms (tests/golden/softmax_split_closed_forms.txt),
a 40-digit mpmath brute force of the merged pair's log-sum-exp and of the
finished row, the merge's order independence and identity element, and the
split-then-finish result equal to the (separately pinned) plain softmax of
the whole row."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "softmax_split_closed_forms.txt")


def _num(tok):
    if tok.startswith("ln("):
        return math.log(int(tok[3:-1]))
    return float(tok)


def _want(tok):
    if tok.startswith("ln("):
        return math.log(int(tok[3:-1]))
    if tok in ("nan", "-inf", "inf"):
        return float(tok)
    return float(Fraction(tok))


def _cases():
    out = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, shards, pairs, merged, row, tol, _why = [p.strip() for p in line.split("|")]
            shards = [np.array([_num(t) for t in s.split()], dtype=np.float64) for s in shards.split(";")]
            pairs = [tuple(_want(t) for t in p.split()) for p in pairs.split(";")]
            merged = tuple(_want(t) for t in merged.split())
            out.append((name, shards, pairs, merged, np.array([_want(t) for t in row.split()]), float(tol)))
    return out


def _same(got, want, tol):
    if math.isnan(want):
        return math.isnan(got)
    if math.isinf(want):
        return got == want
    return abs(got - want) <= tol


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c[0])
def test_closed_forms(case):
    _name, shards, pairs, merged, row, tol = case
    got_pairs = [oracle.softmax_partial_f64(s.reshape(1, -1), "f64", s.size)[0] for s in shards]
    for (m, l), g in zip(pairs, got_pairs):
        assert _same(g[0], m, tol) and _same(g[1], l, tol), (g, m, l)
    mm = oracle.merge_pairs_f64(np.stack([g.reshape(1, 2) for g in got_pairs]))[0]
    assert _same(mm[0], merged[0], tol) and _same(mm[1], merged[1], tol), (mm, merged)
    y = np.concatenate([oracle.softmax_finish_f64(s.reshape(1, -1), "f64", mm.reshape(1, 2), s.size)[0]
                        for s in shards])
    assert y.shape == row.shape
    for g, w in zip(y, row):
        assert _same(g, w, tol), (y, row)


def _splits(n, rng, k):
    cuts = sorted(rng.choice(np.arange(0, n + 1), size=k - 1, replace=True).tolist())
    return [0] + cuts + [n]


def test_brute_force_mpmath_log_sum_exp_and_finish():
    # For random rows and random column splits (empty shards included): the
    # merged max is the row's max exactly, m + ln l is ln sum exp(x) to 40
    # digits, and the finished row is exp(x) / sum exp(x).
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    rng = np.random.default_rng(17)
    for n in range(1, 12):
        for k in (1, 2, 3, 5):
            x = rng.uniform(-60.0, 60.0, size=(3, n))
            cuts = _splits(n, rng, k)
            parts = [oracle.softmax_partial_f64(np.ascontiguousarray(x[:, a:b]), "f64", b - a)
                     for a, b in zip(cuts[:-1], cuts[1:])]
            mm = oracle.merge_pairs_f64(np.stack(parts))
            for r in range(3):
                assert mm[r, 0] == x[r].max()
                lse = mpmath.log(mpmath.fsum(mpmath.exp(mpmath.mpf(float(v))) for v in x[r]))
                assert abs(float(lse) - (mm[r, 0] + math.log(mm[r, 1]))) <= 1e-13 * max(1.0, abs(float(lse)))
                den = mpmath.fsum(mpmath.exp(mpmath.mpf(float(v))) for v in x[r])
                want = [float(mpmath.exp(mpmath.mpf(float(v))) / den) for v in x[r]]
                y = np.concatenate([oracle.softmax_finish_f64(np.ascontiguousarray(x[r:r + 1, a:b]), "f64",
                                                              mm[r:r + 1], b - a)[0]
                                    for a, b in zip(cuts[:-1], cuts[1:])])
                assert np.allclose(y, want, rtol=1e-13, atol=1e-300)


def test_merge_is_order_independent_and_has_an_identity():
    rng = np.random.default_rng(23)
    x = rng.normal(scale=6.0, size=(40, 96))
    cuts = [0, 7, 30, 31, 64, 96]
    parts = np.stack([oracle.softmax_partial_f64(np.ascontiguousarray(x[:, a:b]), "f64", b - a)
                      for a, b in zip(cuts[:-1], cuts[1:])])
    ref = oracle.merge_pairs_f64(parts)
    for perm in ([4, 3, 2, 1, 0], [2, 0, 4, 1, 3]):
        got = oracle.merge_pairs_f64(parts[perm])
        assert np.array_equal(got[:, 0], ref[:, 0])
        assert np.allclose(got[:, 1], ref[:, 1], rtol=1e-14, atol=0)
    # grouping: merge of merges
    left = oracle.merge_pairs_f64(parts[:2])
    right = oracle.merge_pairs_f64(parts[2:])
    assert np.allclose(oracle.merge_pairs_f64(np.stack([left, right])), ref, rtol=1e-14, atol=0)
    # the starting pair (-inf, 0) changes nothing, bit for bit
    ident = np.tile(np.array([-np.inf, 0.0]), (40, 1))
    assert np.array_equal(oracle.merge_pairs_f64(np.stack([ident, ref])), ref)
    assert np.array_equal(oracle.merge_pairs_f64(np.stack([ref, ident])), ref)
    assert np.array_equal(oracle.merge_pairs_f64(parts[:1]), parts[0])


@pytest.mark.parametrize("fmt", ["f32", "f16", "bf16"])
def test_split_then_finish_is_the_plain_softmax(fmt):
    rng = np.random.default_rng(29)
    vals = rng.normal(scale=3.0, size=(24, 200))
    bits = oracle.encode(vals, fmt) if fmt != "f32" else vals.astype(np.float32)
    bits = bits.reshape(24, 200)
    whole = oracle.softmax_f64(bits, fmt)
    for cuts in ([0, 200], [0, 100, 200], [0, 1, 64, 199, 200], [0, 0, 37, 200, 200]):
        parts = np.stack([oracle.softmax_partial_f64(np.ascontiguousarray(bits[:, a:b]), fmt, b - a)
                          for a, b in zip(cuts[:-1], cuts[1:])])
        mm = oracle.merge_pairs_f64(parts)
        y = np.concatenate([oracle.softmax_finish_f64(np.ascontiguousarray(bits[:, a:b]), fmt, mm, b - a)
                            for a, b in zip(cuts[:-1], cuts[1:])], axis=1)
        assert np.allclose(y, whole, rtol=1e-14, atol=1e-300)
        assert np.allclose(y.sum(axis=1), 1.0, rtol=0, atol=1e-14)


def test_pairs_read_stored_formats_and_strides():
    rng = np.random.default_rng(31)
    vals = rng.normal(size=(5, 40))
    bits = oracle.encode(vals, "bf16").reshape(5, 40)
    dec = oracle.decode(bits, "bf16").reshape(5, 40)
    assert np.array_equal(oracle.softmax_partial_f64(bits, "bf16", 33), oracle.softmax_partial_f64(dec, "f64", 33))
    # columns past n_cols (padding) are never read
    padded = dec.copy()
    padded[:, 33:] = np.nan
    assert np.array_equal(oracle.softmax_partial_f64(padded, "f64", 33), oracle.softmax_partial_f64(dec, "f64", 33))
