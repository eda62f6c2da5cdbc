"""Pins of the CPU oracle against what the Fathom review page and plain
mathematics fix (no GPU).  Each test names the passage it checks:

* Appx. A toy example (6 keys x 4 channels, heads A and B): printed values.
* §3.2 prefix identity: reading t planes is the t-bit mid-rise quantiser.
* §3.3 error law a^2 / (3 * 4^t) and reverse water-filling optimality
  (brute force over tiny channel counts).
* §2 selection rule (forced sink/recent tokens + top k-|forced|) against a
  library sort.
* attention special cases and a library softmax.
* fp16 rounding against numpy's float16, exact floor against fractions.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import oracle as O

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "toy_appx_a.json")))


def toy_qv():
    q = np.array([GOLD["q_A"], GOLD["q_B"]], np.float32)
    var = np.array(GOLD["var"], np.float32)
    return q, var


# ------------------------------------------------------------------ Appx. A
def test_toy_importance_matches_printed_g():
    q, var = toy_qv()
    g = O.importance(q, var)
    # printed to 2 decimals (g3 printed as "≈ 0")
    for gj, pj in zip(g[:3], GOLD["g_printed"][:3]):
        assert abs(gj - pj) <= 0.0051, (gj, pj)
    assert g[3] < 1e-4
    # the page's own arithmetic: g0 = (9+1)*1.222, g1 = (1+4)*0.755, g2 = (4+1)*0.127
    assert g[0] == pytest.approx(10 * 1.222, rel=1e-6)
    assert g[1] == pytest.approx(5 * 0.755, rel=1e-6)
    assert g[2] == pytest.approx(5 * 0.127, rel=1e-6)
    assert g[3] == pytest.approx((0.01 + 0.04) * 0.001, rel=1e-5)


def test_toy_bisection_first_two_probes():
    q, var = toy_qv()
    depth, theta, steps, probes, sums = O.plan(q, var, 8, bracket=GOLD["bracket"], trace=True)
    assert steps == 30
    p1, p2 = GOLD["probe_1"], GOLD["probe_2"]
    assert probes[0] == pytest.approx(p1["theta"], rel=1e-12)
    assert sums[0] == p1["sum"]
    assert probes[1] == pytest.approx(p2["theta"], rel=1e-12)
    assert sums[1] == p2["sum"]
    g = O.importance(q, var)
    assert [O.depth_of(x, probes[0]) for x in g] == p1["depth"]
    assert [O.depth_of(x, probes[1]) for x in g] == p2["depth"]


def test_toy_depths_and_theta_B8():
    q, var = toy_qv()
    depth, theta, _ = O.plan(q, var, 8, bracket=GOLD["bracket"])
    assert depth.tolist() == GOLD["B8"]["depth"]
    assert abs(theta - GOLD["B8"]["theta_printed"]) < 5e-4
    # closed form: theta approaches the breakpoint g2 / 2^3 from above
    g = O.importance(q, var)
    bp = g[2] / 8.0
    assert bp <= theta <= bp * (1 + 1e-7)
    # the automatic bracket lands on the same plan
    d2, th2, _ = O.plan(q, var, 8)
    assert d2.tolist() == GOLD["B8"]["depth"]
    assert bp <= th2 <= bp * (1 + 1e-7)


def test_toy_depths_B6():
    q, var = toy_qv()
    depth, theta, _ = O.plan(q, var, 6, bracket=GOLD["bracket"])
    assert depth.tolist() == GOLD["B6"]["depth"]
    g = O.importance(q, var)
    bp = g[1] / 32.0          # the breakpoint that B = 6 stops at
    assert bp <= theta <= bp * (1 + 1e-7)


def toy_channel2_keys():
    k = np.zeros((6, 4), np.float32)
    k[:, 2] = GOLD["channel2"]["values"]
    return k


def test_toy_channel2_codes_scale_planes():
    ch = GOLD["channel2"]
    planes, scales, codes = O.quantize_pack(toy_channel2_keys())
    assert codes[:, 2].tolist() == ch["codes"]
    assert O.fp16_value(int(scales[2, 0])) == ch["a"]
    assert O.fp16_value(int(scales[2, 0])) / 8 == ch["s"]
    assert [int(w) for w in planes[2, :, 0]] == GOLD["channel2_plane_words_derived"]["words"]


def test_toy_channel2_one_plane_values():
    ch = GOLD["channel2"]
    planes, scales, _ = O.quantize_pack(toy_channel2_keys())
    # score of a unit query on channel 2 at depth 1 is the 1-plane value itself
    depth = np.array([[0, 0, 1, 0]], np.uint8)
    q = np.array([[[0, 0, 1, 0]]], np.float32)
    s = O.scores(planes[None], scales[None], depth, q, 6)[0, 0]
    assert s.tolist() == ch["one_plane_values"]
    # 1 bit already orders t3 above t0 (the decision head B hinges on)
    assert s[3] > s[0]


def test_toy_channel2_variance_ddof1():
    mean, var = O.calibrate(toy_channel2_keys())
    assert abs(var[2] - GOLD["channel2"]["var_printed"]) < 5e-4


# ------------------------------------------------------------------ §3.2
def midrise(x, a, t):
    """t-bit mid-rise quantiser on [-a, a): 2^t cells of width 2a/2^t."""
    delta = 2 * a / 2 ** t
    m = math.floor((x + a) / delta)
    m = min(max(m, 0), 2 ** t - 1)
    return -a + (m + 0.5) * delta


@pytest.mark.parametrize("a", [1.0, 0.5, 0.37109375, 3.0])
def test_prefix_identity_exhaustive(a):
    s = a / 8
    for c in range(16):
        centre = -a + (c + 0.5) * s          # centre of the 4-bit cell of code c
        for t in range(1, 5):
            got = O.dequant(c >> (4 - t), t, a)
            assert got == pytest.approx(midrise(centre, a, t), abs=1e-15), (c, t)
        assert O.dequant(c, 4, a) == (c - 8 + 0.5) * s
    assert O.dequant(5, 0, a) == 0.0


@pytest.mark.parametrize("a", [1.0, 0.5, 0.37109375, 3.0])
def test_prefix_value_is_a_signed_binary_expansion(a):
    # Each plane read halves the cell: the t-plane value is the sum over the read
    # planes p = 0..t-1 (0 = MSB) of +a/2^(p+1) where the plane's bit is 1 and
    # -a/2^(p+1) where it is 0 (a bisection of [-a, a) that starts at 0).
    for c in range(16):
        for t in range(0, 5):
            bits = [(c >> (3 - p)) & 1 for p in range(t)]
            x = sum((1 if b else -1) * a / 2 ** (p + 1) for p, b in enumerate(bits))
            assert O.dequant(c >> (4 - t), t, a) == x, (c, t)


def test_error_law_a2_over_3_4t():
    rng = np.random.default_rng(7)
    nblk = 16384
    a = 1.0
    k = rng.uniform(-a, a, size=(nblk, 64)).astype(np.float32)
    k[:, 0] = a                                  # pin the block maximum to a
    keys = k.reshape(-1, 1)
    planes, scales, _ = O.quantize_pack(keys)
    n = keys.shape[0]
    for t in range(1, 5):
        depth = np.array([[t]], np.uint8)
        q = np.ones((1, 1, 1), np.float32)
        khat = O.scores(planes[None], scales[None], depth, q, n)[0, 0]
        err = (khat - keys[:, 0])[k.reshape(-1) != a]
        mse = float(np.mean(err ** 2))
        law = a * a / (3 * 4 ** t)
        assert abs(mse / law - 1) < 0.02, (t, mse, law)


def test_fp16_rounding_matches_numpy():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.lognormal(0, 4, 20000),
        np.ldexp(np.arange(1, 2048, dtype=np.float64), -24),       # subnormal grid
        np.ldexp(np.arange(1, 4096, dtype=np.float64) + 0.5, -24),  # subnormal ties
        1 + (np.arange(1, 2048) + 0.5) / 1024.0,                    # normal ties
        np.array([65504.0, 65519.0, 65520.0, 1e6, 6.1e-5, 5.96e-8, 2.98e-8]),
    ]).astype(np.float32).astype(np.float64)
    for v in vals:
        with np.errstate(over="ignore"):
            h = float(np.float16(v))
        ref = min(h, 65504.0) if math.isfinite(h) else 65504.0
        assert O.round_fp16(v) == ref, v
        assert O.fp16_value(O.fp16_bits(ref)) == ref
        assert O.fp16_bits(ref) == int(np.array(ref, np.float16).view(np.uint16))


def test_code_is_exact_floor():
    rng = np.random.default_rng(3)
    for _ in range(4000):
        a16 = float(np.float16(abs(rng.normal()) * 4 + 1e-3))
        s = Fraction(a16) / 8
        if rng.random() < 0.3:
            # values on or next to cell edges
            m = int(rng.integers(-9, 9))
            k = np.float32(float(m * s))
            k = np.nextafter(k, np.float32(rng.choice([-1, 1]) * 10)) if rng.random() < 0.5 else k
        else:
            k = np.float32(rng.normal() * a16 / 2)
        f = math.floor(Fraction(float(k)) / s)
        ref = min(max(f, -8), 7) + 8
        assert O.code(float(k), a16) == ref, (float(k), a16)
    assert O.code(0.3, 0.0) == 8


def test_quantize_codes_and_planes_definition():
    rng = np.random.default_rng(5)
    n, D = 200, 8                       # ragged tail: 200 = 3*64 + 8
    keys = (rng.normal(size=(n, D)) * np.exp(rng.normal(size=D))).astype(np.float32)
    planes, scales, codes = O.quantize_pack(keys)
    nb = 4
    assert planes.shape == (D, 4, nb)
    for j in range(D):
        for b in range(nb):
            blk = keys[64 * b:min(64 * b + 64, n), j]
            a16 = float(np.float16(np.abs(blk).max()))
            assert O.fp16_value(int(scales[j, b])) == a16
            s = a16 / 8
            c = codes[64 * b:64 * b + len(blk), j].astype(int)
            inside = (blk >= -a16) & (blk < a16)
            # cell membership: (c-8)*s <= k < (c-7)*s for unclipped values
            assert np.all((c[inside] - 8) * s <= blk[inside])
            assert np.all(blk[inside] < (c[inside] - 7) * s)
            for p in range(4):
                w = int(planes[j, p, b])
                bits = [(w >> i) & 1 for i in range(64)]
                assert bits[:len(blk)] == [(int(x) >> (3 - p)) & 1 for x in c]
                assert all(v == 0 for v in bits[len(blk):])   # tail is zero


# ------------------------------------------------------------------ §3.3
def all_depths(D):
    return np.array(list(itertools.product(range(5), repeat=D)), np.int64)


@pytest.mark.parametrize("D", [3, 4, 5, 6])
def test_water_filling_is_brute_force_optimal(D):
    rng = np.random.default_rng(100 + D)
    T = all_depths(D)
    tot = T.sum(1)
    for trial in range(6):
        q = (rng.normal(size=(2, D)) * np.exp(rng.normal(size=D))).astype(np.float32)
        var = np.exp(rng.normal(size=D) * 1.5).astype(np.float32)
        g = O.importance(q, var)
        obj_all = (g[None, :] * np.power(4.0, -T)).sum(1)
        for B in range(0, 4 * D + 2):
            depth, theta, steps = O.plan(q, var, B)
            t = depth.astype(np.int64)
            assert t.sum() <= B
            # optimal among all integer allocations using at most the same bits
            best = obj_all[tot <= t.sum()].min()
            obj = float((g * np.power(4.0, -t)).sum())
            assert obj <= best * (1 + 1e-12), (B, t, obj, best)
            if steps:
                # theta is (within the bisection's resolution) the smallest that fits
                assert sum(O.depth_of(x, theta * (1 - 1e-6)) for x in g) > B
                # the closed form clip(round(log4(g/theta)), 0, 4) away from ties
                for gj, tj in zip(g, t):
                    if gj <= 0:
                        continue
                    x = math.log(gj / theta, 4)
                    if min(abs(x - (m + 0.5)) for m in range(4)) > 1e-9:
                        assert tj == min(max(math.floor(x + 0.5), 0), 4)
            else:
                assert t.sum() == 4 * np.count_nonzero(g)


def test_plan_degenerate_cases():
    q = np.zeros((2, 4), np.float32)
    var = np.ones(4, np.float32)
    depth, theta, steps = O.plan(q, var, 8)
    assert depth.tolist() == [0, 0, 0, 0] and theta == 0.0
    q[0, 1] = 1.0
    depth, theta, steps = O.plan(q, var, 0)          # no budget at all
    assert depth.tolist() == [0, 0, 0, 0]
    depth, theta, steps = O.plan(q, var, 3)          # one live channel, capped by B
    assert depth.tolist() == [0, 3, 0, 0]
    depth, theta, steps = O.plan(q, var, 100)        # not binding: depth 4
    assert depth.tolist() == [0, 4, 0, 0] and steps == 0


def test_depth_rounds_half_up_at_exact_breakpoints():
    # t = clip(round(log4(g / theta)), 0, 4): at g / theta = 2^(2m+1), log4 is m + 1/2 and the
    # depth is m + 1 (round half up, the depth reading); just below it, m.  Exact in fp64.
    for theta in (1.0, 0.0625, 3.0, 1e-7):
        for m in range(4):
            g = theta * 2.0 ** (2 * m + 1)
            assert O.depth_of(g, theta) == m + 1, (theta, m)
            assert O.depth_of(float(np.nextafter(g, 0.0)), theta) == m, (theta, m)
            away = theta * 4.0 ** (m + 0.25)                # log4 = m + 1/4: rounds to m
            assert O.depth_of(away, theta) == m, (theta, m)
        assert O.depth_of(theta * 2.0 ** 20, theta) == 4     # clipped at 4
        assert O.depth_of(0.0, theta) == 0


def test_plan_fixed_is_top_channels_by_g():
    rng = np.random.default_rng(9)
    q = rng.normal(size=(4, 16)).astype(np.float32)
    var = np.exp(rng.normal(size=16)).astype(np.float32)
    var[3] = var[5]
    q[:, 3] = q[:, 5]                                   # an exact tie
    g = O.importance(q, var)
    order = np.lexsort((np.arange(16), -g))             # g desc, index asc
    for n_sel, t in ((5, 4), (7, 2), (16, 1)):
        depth = O.plan_fixed(q, var, n_sel, t)
        ref = np.zeros(16, np.uint8)
        ref[order[:n_sel]] = t
        assert depth.tolist() == ref.tolist()


def test_dense_reduction_B_equals_4D():
    rng = np.random.default_rng(11)
    n, D, G = 300, 16, 4
    keys = (rng.normal(size=(n, D)) * np.exp(rng.normal(size=D))).astype(np.float32)
    q = rng.normal(size=(G, D)).astype(np.float32)
    var = keys.var(0, ddof=1).astype(np.float32)
    depth, theta, steps = O.plan(q, var, 4 * D)
    assert np.all(depth == 4)
    planes, scales, codes = O.quantize_pack(keys)
    s = O.scores(planes[None], scales[None], depth[None], q[None], n)[0]
    # independent dense 4-bit dequantisation: (c - 8 + 0.5) * a16 / 8
    a16 = np.array([[O.fp16_value(int(scales[j, i // 64])) for j in range(D)] for i in range(n)])
    khat = (codes.astype(np.float64) - 7.5) * a16 / 8
    ref = khat @ q.astype(np.float64).T
    np.testing.assert_allclose(s.T, ref, rtol=1e-12, atol=1e-12)


def test_runs_gather_and_staged_scores():
    rng = np.random.default_rng(13)
    n, D, G = 448, 12, 2
    keys = (rng.normal(size=(n, D)) * np.exp(rng.normal(size=D))).astype(np.float32)
    planes, scales, _ = O.quantize_pack(keys)
    nb = 7
    depth = rng.integers(0, 5, size=D).astype(np.uint8)
    depth[3] = 0
    r = O.runs(depth, n)
    # fixed size: one slot per channel; inactive channels have zero length
    assert r.shape == (D, 6)
    assert np.all(r[:, 1] == depth.astype(np.uint32) * nb)
    assert np.all(r[:, 4] == (depth > 0) * nb)
    assert np.all(r[:, 0] == np.arange(D) * 4 * nb) and np.all(r[:, 3] == np.arange(D) * nb)
    # destinations are contiguous, channels ascending
    assert np.all(r[1:, 2] == r[:-1, 2] + r[:-1, 1]) and r[0, 2] == 0
    assert np.all(r[1:, 5] == r[:-1, 5] + r[:-1, 4]) and r[0, 5] == 0
    # each run is the channel's first t_j planes, contiguous over the sequence
    sp, ss = O.gather(r, planes, scales, int(depth.sum()) * nb, int((depth > 0).sum()) * nb)
    for j in range(D):
        t = int(depth[j])
        np.testing.assert_array_equal(sp[r[j, 2]:r[j, 2] + t * nb], planes[j, :t].reshape(-1))
    q = rng.normal(size=(G, D)).astype(np.float32)
    a = O.scores(planes[None], scales[None], depth[None], q[None], n)[0]
    b = O.scores_staged(r, sp, ss, depth, q, n)
    np.testing.assert_array_equal(a, b)


# ------------------------------------------------------------------ §2 selection
def ref_select(s, k, n_sink, n_recent):
    G, n = s.shape
    out = []
    for h in range(G):
        forced = [i for i in range(n) if i < n_sink or i >= n - n_recent]
        rest = np.array([i for i in range(n) if i not in set(forced)], np.int64)
        order = rest[np.lexsort((rest, -s[h, rest]))] if len(rest) else rest
        out.append(sorted(forced + order[:k - len(forced)].tolist()))
    return np.array(out)


@pytest.mark.parametrize("n,k,ns,nr", [(300, 64, 4, 32), (100, 36, 4, 32), (100, 100, 4, 32),
                                       (20, 20, 16, 16), (50, 7, 0, 0), (6, 2, 0, 0)])
def test_select_matches_library_sort(n, k, ns, nr):
    rng = np.random.default_rng(n + k)
    s = rng.integers(-5, 5, size=(3, n)).astype(np.float64)   # many exact ties
    idx, sel = O.select(s, k, ns, nr)
    np.testing.assert_array_equal(idx, ref_select(s, k, ns, nr))
    for h in range(3):
        np.testing.assert_array_equal(sel[h], s[h, idx[h]])


def test_select_rejects_bad_k():
    s = np.zeros((1, 10))
    with pytest.raises(ValueError):
        O.select(s, 11, 0, 0)
    with pytest.raises(ValueError):
        O.select(s, 5, 4, 4)


# ------------------------------------------------------------------ attention
def to_bf16_bits(x):
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_to_f64(b):
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_attention_special_cases_and_softmax():
    rng = np.random.default_rng(17)
    n, D, G = 64, 16, 2
    K = to_bf16_bits(rng.normal(size=(n, D)))
    V = to_bf16_bits(rng.normal(size=(n, D)))
    q = rng.normal(size=(G, D)).astype(np.float32)
    # one selected row: output is that row's value vector
    idx = np.array([[5], [40]], np.int32)
    out = O.attention(K, V, q, idx)
    np.testing.assert_array_equal(out[0], bf16_to_f64(V[5]))
    np.testing.assert_array_equal(out[1], bf16_to_f64(V[40]))
    # identical keys: uniform weights, output is the mean of the value rows
    K2 = np.repeat(K[:1], n, axis=0)
    idx = np.array([[1, 2, 3, 9], [0, 10, 20, 30]], np.int32)
    out = O.attention(K2, V, q, idx)
    for h in range(G):
        np.testing.assert_allclose(out[h], bf16_to_f64(V[idx[h]]).mean(0), rtol=1e-12, atol=1e-15)
    # general case against scipy's softmax
    from scipy.special import softmax
    idx = np.sort(rng.choice(n, size=(G, 12), replace=True), axis=1).astype(np.int32)
    out = O.attention(K, V, q, idx)
    for h in range(G):
        lg = bf16_to_f64(K[idx[h]]) @ q[h].astype(np.float64) / math.sqrt(D)
        ref = softmax(lg) @ bf16_to_f64(V[idx[h]])
        np.testing.assert_allclose(out[h], ref, rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------------ calibration / KLT
def test_calibrate_matches_numpy():
    rng = np.random.default_rng(19)
    keys = (rng.normal(size=(1024, 32)) * 3 + 1).astype(np.float32)
    mean, var, cov = O.calibrate(keys, with_cov=True)
    k64 = keys.astype(np.float64)
    np.testing.assert_allclose(mean, k64.mean(0), rtol=1e-12)
    np.testing.assert_allclose(var, k64.var(0, ddof=1), rtol=1e-12)
    np.testing.assert_allclose(cov, np.cov(k64, rowvar=False, ddof=1), rtol=1e-10, atol=1e-12)


def test_eigh_matches_numpy():
    rng = np.random.default_rng(23)
    D = 24
    A = rng.normal(size=(D, D))
    A = A @ A.T
    lam, V = O.eigh(A)
    ref = np.linalg.eigvalsh(A)[::-1]
    np.testing.assert_allclose(lam, ref, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(V @ np.diag(lam) @ V.T, A, rtol=1e-9, atol=1e-9)
    np.testing.assert_allclose(V.T @ V, np.eye(D), atol=1e-12)
    for c in range(D):
        assert V[np.argmax(np.abs(V[:, c])), c] > 0


def test_rotation_preserves_dot_products_and_norms():
    # V from the oracle's own eigh is orthogonal, so the rotated keys keep the
    # norms of the centred keys and q' . k' = q . (k - mu): the ranking of the
    # tokens by the rotated scores is their ranking by q . k
    rng = np.random.default_rng(29)
    D, n = 16, 200
    R, _ = np.linalg.qr(rng.normal(size=(D, D)))
    sig = np.exp(rng.normal(size=D))
    calib = ((rng.normal(size=(512, D)) * sig) @ R.T + 0.5).astype(np.float32)
    keys = ((rng.normal(size=(n, D)) * sig) @ R.T + 0.5).astype(np.float32)
    q = rng.normal(size=(3, D)).astype(np.float32)
    mean, _, cov = O.calibrate(calib, with_cov=True)
    lam, V = O.eigh(cov)
    kr = O.rotate(keys, mean, V).astype(np.float64)
    qr = O.rotate_query(q, V)
    kc = keys.astype(np.float64) - mean
    np.testing.assert_allclose(np.linalg.norm(kr, axis=1), np.linalg.norm(kc, axis=1), rtol=1e-6)
    np.testing.assert_allclose(qr @ kr.T, q.astype(np.float64) @ kc.T, rtol=1e-5, atol=1e-5 * np.abs(q).sum())
    # the rotated channels are uncorrelated on the calibration keys, with variances lambda
    cr = O.rotate(calib, mean, V).astype(np.float64)
    np.testing.assert_allclose(np.cov(cr, rowvar=False), np.diag(lam), atol=1e-5 * lam[0])
    # identity basis: rotation is centring only
    np.testing.assert_allclose(O.rotate(keys, mean, np.eye(D)), (keys - mean).astype(np.float32), rtol=1e-6)


# ------------------------------------------------------------------ §4/§5 fidelity references
def test_exact_scores_one_hot_keys_and_hand_example():
    # key i is c_i times the unit vector of channel i mod D: its score for head h
    # is q[h, i mod D] * c_i exactly, so a transposed operand, a wrong head or
    # channel index, or a dropped sign fails
    rng = np.random.default_rng(31)
    D, n, G = 8, 40, 3
    c = rng.choice([-2.0, -0.5, 0.25, 1.0, 3.0], size=n)
    keys = np.zeros((n, D), np.float32)
    keys[np.arange(n), np.arange(n) % D] = c
    q = rng.normal(size=(G, D)).astype(np.float32)
    s = O.exact_scores(keys, q)
    assert s.shape == (G, n)
    for h in range(G):
        for i in range(n):
            assert s[h, i] == float(q[h, i % D]) * c[i]
    # a hand example: (2, 0.25, -4) . (1, -2, 0.5) = 2 - 0.5 - 2
    assert O.exact_scores([[1.0, -2.0, 0.5]], [[2.0, 0.25, -4.0]])[0, 0] == -0.5


def test_dense_attention_two_token_closed_form():
    # keys 0 and a e_0, query x e_0: weights 1 / (1 + e^z) and e^z / (1 + e^z)
    # with z = a x / sqrt(D)
    D, a, x = 4, 1.5, 2.0
    K = to_bf16_bits(np.array([[0, 0, 0, 0], [a, 0, 0, 0]], np.float32))
    V = to_bf16_bits(np.array([[1, 2, 3, 4], [-1, 0.5, 0, 8]], np.float32))
    q = np.array([[x, 0, 0, 0], [0, 1, 0, 0]], np.float32)
    out = O.dense_attention(K, V, q)
    z = a * x / math.sqrt(D)
    w1 = math.exp(z) / (1 + math.exp(z))
    v0, v1 = bf16_to_f64(V[0]), bf16_to_f64(V[1])
    np.testing.assert_allclose(out[0], (1 - w1) * v0 + w1 * v1, rtol=1e-14)
    np.testing.assert_allclose(out[1], 0.5 * (v0 + v1), rtol=1e-14)   # head 2 is orthogonal to both keys


def test_rel_l2_definition():
    assert O.rel_l2([3.0, 4.0, 0.0], [0.0, 0.0, 5.0]) == pytest.approx(math.sqrt(2.0), rel=1e-15)
    assert O.rel_l2([3.0, 4.0], [0.0, 0.0]) == 5.0              # zero reference: the norm of a
    np.testing.assert_array_equal(O.rel_l2(np.ones((2, 3)), np.ones((2, 3))), [0.0, 0.0])


# ------------------------------------------------------------------ §3.4 greedy per-layer budgets
def _convex_table(rng, layers, levels):
    # strictly decreasing errors with strictly shrinking drops, distinct across layers
    drops = np.sort(rng.uniform(0.01, 1.0, size=(layers, levels - 1)), axis=1)[:, ::-1]
    err = np.zeros((layers, levels))
    err[:, 0] = rng.uniform(5.0, 6.0, size=layers)
    err[:, 1:] = err[:, :1] - np.cumsum(drops, axis=1)
    return err


@pytest.mark.parametrize("layers,levels", [(2, 4), (3, 5), (4, 4)])
def test_greedy_budgets_are_brute_force_optimal_on_convex_errors(layers, levels):
    # with decreasing drops, adding the largest next drop each time minimises the
    # total error among all allocations of the same total
    rng = np.random.default_rng(37 + layers)
    b_min, step = 24, 8
    for _ in range(5):
        err = _convex_table(rng, layers, levels)
        for m in range(levels):
            b_mean = b_min + step * m
            got = O.greedy_budgets(err, b_min, step, b_mean)
            assert got.sum() == layers * b_mean
            best, best_lev = None, None
            for lev in itertools.product(range(levels), repeat=layers):
                if sum(lev) != layers * m:
                    continue
                tot = sum(err[l, lev[l]] for l in range(layers))
                if best is None or tot < best - 1e-12:
                    best, best_lev = tot, lev
            np.testing.assert_array_equal(got, b_min + step * np.array(best_lev))


def test_greedy_budgets_hand_examples():
    # non-convex layer 0: one step goes to layer 1 (drop 0.5 > 0.1), the next to
    # layer 0 (0.1 > 0.05); the brute-force optimum (40, 24) is not what greedy picks
    err = [[1.0, 0.9, 0.0], [1.0, 0.5, 0.45]]
    np.testing.assert_array_equal(O.greedy_budgets(err, 24, 8, 32), [32, 32])
    # equal drops: the lower layer first
    np.testing.assert_array_equal(O.greedy_budgets([[2.0, 1.0], [2.0, 1.0]], 24, 8, 28), [32, 24])
    # layers at the top level take no more: the target mean at the top puts all at the top
    np.testing.assert_array_equal(O.greedy_budgets([[3.0, 2.0], [3.0, 0.0]], 24, 104, 128), [128, 128])
    # flat target at the floor
    np.testing.assert_array_equal(O.greedy_budgets([[3.0, 2.0], [3.0, 0.0]], 24, 8, 24), [24, 24])


# ------------------------------------------------------------------ §7 keys rebuilt from the store
def test_reconstruct_reads_the_codes_back_from_the_planes():
    # the rebuilt key is the 4-bit mid-rise value of the code the quantiser chose:
    # (c - 7.5) a16 / 8 with c from the codes array (not from the plane bits), and
    # within half a step of the key; a16 may round a down by up to 2^-11 relative,
    # and then the largest key (clipped to code 15) is off by a - 7.5 a16 / 8,
    # at most (1 + 16 * 2^-11) half steps
    rng = np.random.default_rng(43)
    n, D = 200, 12                        # a ragged last block
    keys = (rng.normal(size=(n, D)) * np.exp(rng.normal(size=D))).astype(np.float32)
    P, S, C = O.quantize_pack(keys)
    got = O.reconstruct(P, S, n)
    a16 = S.view(np.float16).astype(np.float64)          # [D][nb]
    blk = np.arange(n) // 64
    expect = (C.astype(np.float64) - 7.5) * a16[:, blk].T / 8.0
    np.testing.assert_array_equal(got, expect)
    step = a16[:, blk].T / 8.0
    assert np.all(np.abs(got - keys) <= 0.5 * step * (1 + 16 * 2.0 ** -11) + 1e-30)
    # a capacity layout (cb > nb) reads the same words
    Pc = np.zeros((D, 4, 7), np.uint64)
    Sc = np.zeros((D, 7), np.uint16)
    Pc[:, :, :P.shape[2]] = P
    Sc[:, :S.shape[1]] = S
    np.testing.assert_array_equal(O.reconstruct(Pc, Sc, n), got)


def test_attention_with_fp64_keys_equals_bf16_row_attention():
    # keys that are bf16 values give exactly the attention over the bf16 rows
    rng = np.random.default_rng(47)
    n, D, G = 50, 16, 2
    K = to_bf16_bits(rng.normal(size=(n, D)))
    V = to_bf16_bits(rng.normal(size=(n, D)))
    q = rng.normal(size=(G, D)).astype(np.float32)
    idx = np.sort(rng.choice(n, size=(G, 9), replace=False), axis=1).astype(np.int32)
    np.testing.assert_array_equal(O.attention_keys(bf16_to_f64(K), V, q, idx), O.attention(K, V, q, idx))


# ------------------------------------------------------------------ Appx. A toy, reconstructed K
def test_toy_reconstruction_reproduces_every_printed_statement():
    # The page prints only channel 2 of the toy's K.  toy_k_reconstruction.json
    # holds channels 0, 1 and 3 fitted by tests/golden/fit_toy_k.py (oracle only)
    # and is labelled a reconstruction: this pins that one K consistent with all
    # of the page's statements exists under the oracle's quantiser, planner and
    # scorer, and that on it the oracle's scan ranks as the page says.
    rec = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "toy_k_reconstruction.json")))
    assert "RECONSTRUCTION" in rec["what"]
    K = np.array(rec["K"], np.float32)
    np.testing.assert_array_equal(K[:, 2], np.array(GOLD["channel2"]["values"], np.float32))
    v = np.var(K.astype(np.float64), axis=0, ddof=1)
    assert np.all(np.abs(v - np.array(GOLD["var"])) <= 0.0005)                # printed to 3 decimals
    q = np.array([GOLD["q_A"], GOLD["q_B"]], np.float32)
    P, S, C = O.quantize_pack(K)
    np.testing.assert_array_equal(C[:, 2], GOLD["channel2"]["codes"])          # printed codes of channel 2
    exact = q.astype(np.float64) @ K.astype(np.float64).T
    np.testing.assert_allclose(exact[1], GOLD["head_B_scores"]["exact"], rtol=0, atol=0.005)

    def top2(s):
        return set(sorted(range(6), key=lambda i: (-s[i], i))[:2])

    assert top2(exact[0]) == set(GOLD["top2"]["A"]) and top2(exact[1]) == set(GOLD["top2"]["B"])
    var = np.array(GOLD["var"], np.float32)
    d8, _, _ = O.plan(q, var, 8, bracket=GOLD["bracket"])
    d6, _, _ = O.plan(q, var, 6, bracket=GOLD["bracket"])
    a8 = O.scores(P[None], S[None], d8[None], q[None], 6)[0]
    a6 = O.scores(P[None], S[None], d6[None], q[None], 6)[0]
    np.testing.assert_allclose(a8[1], GOLD["head_B_scores"]["approx"], rtol=0, atol=0.005)
    assert top2(a8[0]) == set(GOLD["top2"]["A"]) and top2(a8[1]) == set(GOLD["top2"]["B"])   # B = 8 gets both
    assert top2(a6[1]) != set(GOLD["top2"]["B"])                                             # B = 6 misses B
    # reading channels 0 and 1 only (the fixed 2-channel rules at 8 bits) ranks {t5, t3} for head B
    assert top2(q[1, 0] * K[:, 0].astype(np.float64) + q[1, 1] * K[:, 1].astype(np.float64)) == {5, 3}
