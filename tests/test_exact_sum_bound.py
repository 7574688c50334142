"""The exactness argument behind the persistent BatchNorm forward's per-stage
channel sums, checked on the host.

For bf16 input, a thread adds the differences d = x - shift of its values in
a stage in plain fp32 and only then adds the result in double-fp32.  That is
exact when the biased exponent fields of all those values and of shift lie
in E_min .. E_max with E_min > 0 and E_max - E_min <= 15 - ceil(log2 n), n the
number of terms one fp32 accumulator lane sees: every value is then a
multiple of Q = 2^(E_min - 134) below 2^(E_max - 126), each d a multiple of Q
below 2^(E_max - 125), and every partial sum of at most n of them a multiple
of Q below 2^24 Q, so each fp32 addition is exact in any order.

These tests sample bf16 values, apply the same predicate, and compare fp32
sums taken in several orders with the exact sum; they also show the bound is
not vacuous (one binade past it, fp32 sums do round).
"""
import math

import numpy as np
import pytest


def _bf16_round(v):
    """Round fp32 values to bf16 (round to nearest even), returned as fp32."""
    u = np.asarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def _exp_field(v):
    return ((np.asarray(v, dtype=np.float32).view(np.uint32) >> 23) & 0xFF).astype(np.int64)


def _span_limit(n):
    return 15 - math.ceil(math.log2(n))


def _predicate(vals, shift, n):
    e = np.concatenate([_exp_field(vals), _exp_field(np.float32([shift]))])
    return e.min() > 0 and e.max() - e.min() <= _span_limit(n)


def _fp32_sums(d):
    """fp32 sums of d in three orders: sequential, two interleaved chains (as
    the kernel's two accumulators), pairwise."""
    f = np.float32
    seq = f(0)
    for v in d:
        seq = f(seq + v)
    a, b = f(0), f(0)
    for i, v in enumerate(d):
        if i % 2 == 0:
            a = f(a + v)
        else:
            b = f(b + v)
    two = f(a + b)
    w = list(d)
    while len(w) > 1:
        w = [f(w[i] + w[i + 1]) if i + 1 < len(w) else w[i] for i in range(0, len(w), 2)]
    return [seq, two, w[0]]


@pytest.mark.parametrize("n", [4, 8, 24, 48])
def test_sums_exact_when_the_span_predicate_holds(n):
    rng = np.random.default_rng(1234 + n)
    checked = 0
    for trial in range(3000):
        # magnitudes over a window of binades around a random centre, both signs
        centre = rng.uniform(-20, 20)
        width = rng.integers(0, _span_limit(n) + 3)
        mags = np.exp2(centre + rng.uniform(0, width, size=n))
        vals = _bf16_round(mags * rng.choice([-1.0, 1.0], size=n))
        shift = vals[rng.integers(0, n)] if trial % 3 else _bf16_round(np.float32([2.0 ** centre]))[0]
        if not _predicate(vals, shift, n):
            continue
        d = (vals - np.float32(shift)).astype(np.float32)
        exact_d = vals.astype(np.float64) - np.float64(shift)
        assert np.array_equal(d.astype(np.float64), exact_d), "x - shift not exact"
        exact = math.fsum(exact_d.tolist())
        for s in _fp32_sums(d):
            assert float(s) == exact
        checked += 1
    assert checked > 300


def test_bound_is_not_vacuous():
    """One binade past the limit, an fp32 sum of n terms does round: large
    positive values against a large negative shift (every d near the bound)
    and one value 2^(lim + 1) times smaller setting the granularity."""
    n = 24
    lim = _span_limit(n)
    rng = np.random.default_rng(99)
    rounded = 0
    for _ in range(500):
        big = _bf16_round(np.float32(rng.uniform(1.5, 1.96, size=n - 1)) * np.float32(2.0 ** lim))
        small = _bf16_round(np.float32([rng.uniform(1.0, 1.96) * 0.5]))
        vals = np.concatenate([big, small]).astype(np.float32)
        shift = _bf16_round(np.float32([-1.9 * 2.0 ** lim]))[0]
        e = np.concatenate([_exp_field(vals), _exp_field(np.float32([shift]))])
        assert e.max() - e.min() == lim + 1 and not _predicate(vals, shift, n)
        d = (vals - shift).astype(np.float32)
        exact = math.fsum((vals.astype(np.float64) - np.float64(shift)).tolist())
        if any(float(s) != exact for s in _fp32_sums(d)):
            rounded += 1
    assert rounded > 100


def test_zero_and_subnormal_fail_the_predicate():
    vals = np.float32([1.0, 0.0, 2.0, 3.0])
    assert not _predicate(vals, np.float32(1.0), 4)
    sub = np.float32([1e-40, 1e-40, 1e-40, 1e-40])
    assert not _predicate(sub, np.float32(1e-40), 4)
    assert _predicate(np.float32([1.0, 2.0, 3.0, 1.5]), np.float32(1.0), 24)
