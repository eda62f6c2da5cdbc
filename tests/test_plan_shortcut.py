"""The plan kernel's shortcut, checked on CPU against the oracle's plan.

The oracle's bisection counts, at every probe theta, the depths
sum_j t_j(theta) = #{(j, m) : g_j >= theta * 2^(2m+1)} and keeps theta if the
count fits the budget.  The GPU plan instead finds once the critical
breakpoint b*, the (B + 1)-th largest of the 4 D breakpoints g_j * 2^-(2m+1)
(with multiplicity), and keeps theta iff theta > b*.  Both scalings by powers
of two are exact in fp64, so the two tests agree at every theta, and the two
bisections (the same fp64 sqrt(lo * hi) chain) end on the same theta bit for
bit.  This test runs the shortcut in numpy against the oracle on random and
tie-heavy channel importances."""
import numpy as np
import pytest

from oracle import oracle as O


def breakpoints(g):
    return np.concatenate([g[g > 0] * 2.0 ** -(2 * m + 1) for m in range(4)])


def total(g, theta):
    return sum(int(np.sum(g >= theta * 2.0 ** (2 * m + 1))) for m in range(4))


def shortcut_plan(q, var, B):
    g = O.importance(q, var)
    gmax = g.max()
    if gmax == 0.0:
        return np.zeros_like(g, dtype=np.uint8), 0.0
    hi, lo = gmax, g[g > 0].min() / 512.0
    if total(g, lo) <= B:
        return np.array([O.depth_of(x, lo) for x in g], np.uint8), lo
    bstar = np.sort(breakpoints(g))[::-1][B]          # the (B + 1)-th largest
    for _ in range(30):
        mid = np.sqrt(lo * hi)
        if mid > bstar:
            hi = mid
        else:
            lo = mid
    return np.array([O.depth_of(x, hi) for x in g], np.uint8), hi


def _cases(rng):
    G, D = 4, 128
    for trial in range(60):
        sigma = np.exp(rng.standard_normal(D) * (0.5 + trial % 3))
        q = (rng.standard_normal((G, D)) * np.sqrt(sigma)).astype(np.float32)
        var = (sigma ** 2).astype(np.float32)
        if trial % 4 == 1:                    # many equal importances
            q[:, ::3] = q[:, :1]
            var[::3] = var[0]
        if trial % 4 == 2:                    # importances a power of 4 apart: coinciding breakpoints
            q[:, 1::2] = 0.5 * q[:, 0::2]
            var[1::2] = var[0::2]
        if trial % 4 == 3:                    # some dead channels
            q[:, rng.random(D) < 0.3] = 0.0
        yield q, var


def test_threshold_fits_iff_above_the_critical_breakpoint():
    rng = np.random.default_rng(31)
    for q, var in _cases(rng):
        g = O.importance(q, var)
        bp = np.sort(breakpoints(g))[::-1]
        for B in (0, 1, 7, 48, 100, len(bp) - 1):
            bstar = bp[B]
            for theta in (bstar, np.nextafter(bstar, np.inf), np.nextafter(bstar, 0.0),
                          bstar * 1.5, bstar / 1.5, *bp[max(0, B - 2):B + 3]):
                assert (total(g, theta) <= B) == (theta > bstar), (B, theta, bstar)


@pytest.mark.parametrize("B", [8, 24, 48, 64, 128, 200])
def test_shortcut_bisection_equals_the_oracle_plan(B):
    rng = np.random.default_rng(100 + B)
    for q, var in _cases(rng):
        depth, theta = shortcut_plan(q, var, B)
        od, oth, _ = O.plan(q, var, B)
        assert theta == oth                     # bit for bit
        np.testing.assert_array_equal(depth, od)
        assert int(od.sum()) <= B


def _exponent(x):
    return int(np.frexp(np.float64(x))[1])


def thetaless_plan(q, var, B):
    """The plan kernel without a theta output: after b*, the depths at the next
    breakpoint above b* whenever that breakpoint lies beyond b* (1 + 4x), where
    the bisection's final hi provably lies below b* (1 + 2x); the bisection
    otherwise.  Returns (depths, took_shortcut)."""
    g = O.importance(q, var)
    if g.max() == 0.0:
        return np.zeros_like(g, dtype=np.uint8), False
    hi, lo = g.max(), g[g > 0].min() / 512.0
    if total(g, lo) <= B:
        return np.array([O.depth_of(x, lo) for x in g], np.uint8), False
    bp = breakpoints(g)
    bstar = np.sort(bp)[::-1][B]
    above = bp[bp > bstar]
    bnext = above.min() if above.size else np.inf
    x = (_exponent(hi) - _exponent(lo) + 1) * 0.6931471805599453 * 2.0 ** -30 + 2.0 ** -51
    if bnext > bstar * (1.0 + 4.0 * x):
        return np.array([O.depth_of(v, bnext) for v in g], np.uint8), True
    return shortcut_plan(q, var, B)[0], False


def _close_breakpoint_cases(rng):
    """Importances whose breakpoints nearly coincide around every rank: the
    shortcut must fall back to the bisection wherever the gap is below 4x."""
    G, D = 4, 128
    for trial in range(12):
        q = rng.standard_normal((G, D)).astype(np.float32)
        var = np.exp(rng.standard_normal(D)).astype(np.float32)
        # pairs of channels whose importances differ in the last few float bits
        q[:, 1::2] = q[:, 0::2]
        var[1::2] = np.nextafter(var[0::2], np.float32(np.inf)) if trial % 2 else var[0::2]
        yield q, var


@pytest.mark.parametrize("B", [1, 8, 48, 64, 200])
def test_thetaless_shortcut_gives_the_bisection_depths(B):
    rng = np.random.default_rng(700 + B)
    took = 0
    for q, var in list(_cases(rng)) + list(_close_breakpoint_cases(rng)):
        depth, short = thetaless_plan(q, var, B)
        od, oth, _ = O.plan(q, var, B)
        np.testing.assert_array_equal(depth, od)
        took += short
        # the bound the shortcut rests on: the bisection's final theta is within
        # b* (1 + 2x) whenever the budget binds
        g = O.importance(q, var)
        lo = g[g > 0].min() / 512.0
        if g.max() > 0 and total(g, lo) > B:
            bstar = np.sort(breakpoints(g))[::-1][B]
            x = (_exponent(g.max()) - _exponent(lo) + 1) * 0.6931471805599453 * 2.0 ** -30 + 2.0 ** -51
            assert bstar < oth <= bstar * (1.0 + 2.0 * x)
    assert took > 0


def test_thetaless_shortcut_falls_back_when_breakpoints_nearly_coincide():
    # channels 0 and 1 have importances 4e-14 apart (q one fp32 ulp above 1, var
    # 2^-22 below 1): with B = 1, b* is channel 1's first breakpoint and the
    # next one up is channel 0's, far closer than 4x, so the shortcut must not be
    # taken and the bisection's depths are returned
    G, D = 4, 8
    q = np.ones((G, D), np.float32)
    q[:, 1] = np.nextafter(np.float32(1.0), np.float32(2.0))
    var = np.array([1.0, 1.0 - 2.0 ** -22, 0.5, 0.25, 0.125, 0.0625, 0.03125, 0.015625], np.float32)
    g = O.importance(q, var)
    bp = np.sort(breakpoints(g))[::-1]
    B = 1
    assert 0.0 < bp[0] / bp[1] - 1.0 < 1e-12
    depth, short = thetaless_plan(q, var, B)
    od, _, _ = O.plan(q, var, B)
    np.testing.assert_array_equal(depth, od)
    assert not short
