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
