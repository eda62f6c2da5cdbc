"""The plan's integer square root against IEEE sqrt (CPU).

The plan kernel's bisection takes sqrt(lo * hi) through
bit_plane_kv_gb300/csrc/exact_sqrt.cuh, which must return exactly the bits of
the correctly rounded fp64 square root.  Its last step makes the result exact
for any seed within the Newton steps' convergence range, so the host build
(seeded with 1 / sqrtf instead of the device's rsqrt.approx) is checked here
against numpy's float64 sqrt, with the seed also scaled by +-1e-6 (several
times the device seed's error) and on perfect squares and their neighbours.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "bit_plane_kv_gb300", "csrc")


@pytest.fixture(scope="module")
def xsqrt(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("xsqrt") / "libxsqrt.so")
    subprocess.run(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-shared", "-fPIC", "-I", CSRC,
                    os.path.join(HERE, "exact_sqrt_harness.cpp"), "-o", out], check=True)
    L = ctypes.CDLL(out)
    L.xsqrt_many.argtypes = [ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p]

    def run(x, scale=1.0):
        x = np.ascontiguousarray(x, dtype=np.float64)
        out = np.empty(x.size, dtype=np.uint64)
        L.xsqrt_many(x.size, ctypes.c_void_p(x.ctypes.data), scale, ctypes.c_void_p(out.ctypes.data))
        return out
    return run


def _doubles(rng, n, keep_bits):
    frac = rng.integers(0, 1 << 52, n, dtype=np.uint64)
    frac &= np.uint64(((1 << keep_bits) - 1) << (52 - keep_bits)) if keep_bits < 52 else np.uint64((1 << 52) - 1)
    e = rng.integers(1, 2047, n).astype(np.uint64)
    return ((e << np.uint64(52)) | frac).view(np.float64)


@pytest.mark.parametrize("scale", [1.0, 1.0 + 1e-6, 1.0 - 1e-6])
def test_random_operands(xsqrt, scale):
    rng = np.random.default_rng(21)
    for keep in (52, 30, 8, 0):
        x = _doubles(rng, 300000, keep)
        assert np.array_equal(xsqrt(x, scale), np.sqrt(x).view(np.uint64)), f"keep={keep}"


def test_squares_and_neighbours(xsqrt):
    a = np.arange(1 << 26, (1 << 26) + 300000, dtype=np.float64)
    q = a * a                                     # exact: < 2^54
    for x in (q, np.nextafter(q, np.inf), np.nextafter(q, 0.0), q * 2.0 ** -600, q * 2.0 ** 501):
        assert np.array_equal(xsqrt(x), np.sqrt(x).view(np.uint64))
    # mantissas at the ends of [1, 4)
    ends = np.array([1.0, np.nextafter(1.0, 2.0), np.nextafter(2.0, 0.0), 2.0, np.nextafter(4.0, 0.0)])
    assert np.array_equal(xsqrt(ends * 2.0 ** 100), np.sqrt(ends * 2.0 ** 100).view(np.uint64))


def test_results_are_rounded_not_truncated(xsqrt):
    """The comparison can tell a truncated root from the rounded one."""
    rng = np.random.default_rng(22)
    x = _doubles(rng, 10000, 52)
    got = xsqrt(x)
    trunc = np.sqrt(x)
    below = np.nextafter(trunc, 0.0)
    assert np.array_equal(got, trunc.view(np.uint64)) and not np.array_equal(got, below.view(np.uint64))
