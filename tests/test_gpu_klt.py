"""Rotated basis (Fathom §3.5) on the GPU against the oracle: calibration
(mean, eigenvalues, eigenvectors), rotated keys and queries, then the whole
path on the rotated store with per-layer budgets.

Tolerances:
* mean: bit-exact (fp64 sums in row order on both sides);
* eigenvalues: within 1e-9 of the largest (fp64 Jacobi on both sides, the
  covariance summed in a different order);
* eigenvectors: within 1e-6 per component (eigenvalue gaps of the synthetic
  keys are far above the 1e-9 perturbation);
* rotated keys and queries: |gpu - oracle| <= 8e-6 * sum_j |x_j V_jc| with
  the oracle fed the GPU's mean and V, i.e. the fp32 arithmetic alone:
  (k - mu) and V rounded to fp32 (2 u) and a fp32 sum of 128 products
  (<= 128 u), u = 2^-24, bound 130 u < 8e-6;
* the store, plan, scores, selection and attention given the GPU's rotated
  keys, rotated queries and eigenvalues: the tolerances of the unrotated path.
"""
import numpy as np
import pytest
import torch

from bit_plane_kv_gb300 import binding as B
from bit_plane_kv_gb300 import synth
from oracle import oracle as O

from fathom_cases import ATTN_RTOL, SCORE_RTOL, khat_magnitude, u16, u32, u64

pytestmark = pytest.mark.gpu
ROT_RTOL = 8e-6


def _klt_workload():
    # the 32-session rotated-basis batch shrunk to 2 sequences x 2 layers x 2 heads
    w = synth.WORKLOADS["klt_32x64k"]
    return synth.shrink(w, seqs=2, layers=2, kv_heads=2, budgets=(24, 128))


def _calib(w):
    groups = w.layers * w.kv_heads
    return groups, torch.stack([synth.unit_calib(w, g, "cuda") for g in range(groups)]).contiguous()


def test_klt_calibration_matches_oracle():
    w = _klt_workload()
    groups, calib = _calib(w)
    mean, V, lam = B.fathom_calibrate_klt(calib)
    torch.cuda.synchronize()
    for g in range(groups):
        om, _, cov = O.calibrate(calib[g].cpu().numpy(), with_cov=True)
        ol, oV = O.eigh(cov)
        np.testing.assert_array_equal(mean[g].cpu().numpy(), om)
        gl = lam[g].cpu().numpy().astype(np.float64)
        np.testing.assert_allclose(gl, ol.astype(np.float32), rtol=0, atol=1e-9 * ol[0] + 1e-30 + np.spacing(np.float32(ol[0])))
        np.testing.assert_allclose(V[g].cpu().numpy(), oV, rtol=0, atol=1e-6)


def _rotation_bound(x, Vg):
    # sum_j |x_j| |V_jc| per output
    return np.abs(x) @ np.abs(Vg)


def test_klt_rotations_match_oracle():
    w = _klt_workload()
    groups, calib = _calib(w)
    mean, V, _ = B.fathom_calibrate_klt(calib)
    n = 1000   # a ragged last tile of 64 tokens
    units = list(range(w.units))
    shape = B.make_shape(len(units), n, w.D, w.G, 64, 4, 32)
    keys = torch.stack([synth.unit_keys(w, u, "cuda", n=n) for u in units]).to(torch.bfloat16)
    q = torch.stack([synth.unit_query(w, u, "cuda") for u in units]).contiguous()
    kr = B.fathom_rotate_keys(shape, keys, groups, mean, V)
    k32 = B.fathom_rotate_keys(shape, keys.float().contiguous(), groups, mean, V)
    qr = B.fathom_rotate_query(shape, q, groups, V)
    torch.cuda.synchronize()
    assert torch.equal(kr, k32)     # bf16 input widened exactly
    for ui, u in enumerate(units):
        g = u % groups
        Vg, mu = V[g].cpu().numpy(), mean[g].cpu().numpy()
        kk = keys[ui].float().cpu().numpy()
        ref = O.rotate(kk, mu, Vg).astype(np.float64)
        bound = _rotation_bound(kk.astype(np.float64) - mu, Vg)
        err = np.abs(kr[ui].cpu().numpy().astype(np.float64) - ref)
        assert np.all(err <= ROT_RTOL * bound + 1e-30), float(np.max(err / np.maximum(bound, 1e-30)))
        qq = q[ui].cpu().numpy()
        qref = O.rotate_query(qq, Vg)
        qerr = np.abs(qr[ui].cpu().numpy().astype(np.float64) - qref)
        assert np.all(qerr <= ROT_RTOL * _rotation_bound(qq.astype(np.float64), Vg) + 1e-30)


def test_klt_full_path_with_per_layer_budgets():
    w = _klt_workload()
    groups, calib = _calib(w)
    mean, V, lam = B.fathom_calibrate_klt(calib)
    n, k = 6000, 300
    units = list(range(w.units))
    U = len(units)
    shape = B.make_shape(U, n, w.D, w.G, k, w.n_sink, w.n_recent)
    keys = torch.stack([synth.unit_keys(w, u, "cuda", n=n) for u in units])
    krows = keys.to(torch.bfloat16)
    vrows = torch.stack([synth.unit_values(w, u, "cuda", n=n) for u in units]).to(torch.bfloat16)
    q = torch.stack([synth.unit_query(w, u, "cuda") for u in units]).contiguous()
    layer_of = [(u // w.kv_heads) % w.layers for u in units]
    budget = torch.tensor([w.budgets[l] for l in layer_of], dtype=torch.int32, device="cuda")
    lam_u = lam[torch.tensor([u % groups for u in units], device="cuda")].contiguous()
    kr = B.fathom_rotate_keys(shape, krows, groups, mean, V)
    qr = B.fathom_rotate_query(shape, q, groups, V)
    planes, scales = B.fathom_quantize_pack(shape, kr)
    depth, theta, runs = B.fathom_plan(shape, qr, lam_u, budget)
    scores = torch.full((U, w.G, n), float("nan"), device="cuda")
    idx, sel = B.fathom_scan_topk(shape, planes, scales, runs, qr, B.alloc_workspace(shape, B.WS_SCAN_TOPK),
                                  scores=scores)
    out = B.fathom_sparse_attn(shape, krows, vrows, q, idx, B.alloc_workspace(shape, B.WS_SPARSE_ATTN))
    torch.cuda.synchronize()
    for ui in range(U):
        keys_r = kr[ui].cpu().numpy()
        qq = qr[ui].cpu().numpy()
        P, S, C = O.quantize_pack(keys_r)                    # the oracle quantises the GPU's rotated keys
        np.testing.assert_array_equal(u64(planes[ui]), P)
        np.testing.assert_array_equal(u16(scales[ui]), S)
        b = int(budget[ui].item())
        od, oth, _ = O.plan(qq, lam_u[ui].cpu().numpy(), b)
        np.testing.assert_array_equal(depth[ui].cpu().numpy(), od)
        assert theta[ui].item() == oth
        assert od.sum() <= b
        np.testing.assert_array_equal(u32(runs[ui]), O.runs(od, n))
        ref = O.scores(P[None], S[None], od[None], qq[None], n)[0]
        got = scores[ui].cpu().numpy().astype(np.float64)
        mag = khat_magnitude(C, S, od, qq, n)
        assert np.all(np.abs(got - ref) <= SCORE_RTOL * mag + 1e-30)
        oi, _ = O.select(got, k, w.n_sink, w.n_recent)
        np.testing.assert_array_equal(idx[ui].cpu().numpy(), oi)
        o = O.attention(u16(krows[ui]), u16(vrows[ui]), q[ui].cpu().numpy(), oi)
        rel = np.linalg.norm(out[ui].cpu().numpy().astype(np.float64) - o, axis=1) / np.linalg.norm(o, axis=1)
        assert np.all(rel <= ATTN_RTOL), rel
    # the rotated scores rank tokens as q . k does, up to the quantisation: at
    # the 128-bit layer the kept sets overlap the exact top-k of q . k widely
    qk = torch.einsum("ugd,und->ugn", q.double(), krows.double())
    exact = qk.topk(k, dim=-1).indices.cpu().numpy()
    for ui in range(U):
        if layer_of[ui] != 1:
            continue
        for h in range(w.G):
            inter = len(set(idx[ui, h].cpu().numpy().tolist()) & set(exact[ui, h].tolist()))
            assert inter >= 0.5 * k, inter


# ---------------------------------------------------------------- online basis (Appx. D)
# Tolerances of the fp32 online basis against the oracle's fp64 calibration of
# the same bf16 rows, each derived from the arithmetic:
# * mean: fp32 sums of 64-token runs folded in fp64, |err| <= 64 u mean|k_j|
#   (u = 2^-24), tested at 4e-6 mean|k_j|;
# * covariance: per slice of T <= 2048 tokens fp32 sums of 32-token stages, so
#   each entry is within c u sum_i |x_ia x_ib| / (n - 1), c = 32 + T/32 + 1 = 97:
#   |dC| <= E entrywise for the matrix E computed from the data, and
#   ||dC||_2 <= ||E||_2;
# * the fp32 Jacobi: a backward error of order sweeps * D * u ||C||, allowed
#   1024 u lambda_max (8 sweeps at D = 128);
# so eps = ||E||_2 + 1024 u lambda_max bounds the backward error
# ||V diag(lambda) V^T - C||_2 of the GPU's decomposition against the oracle's
# covariance C, every eigenvalue (Weyl: |lambda_i - lambda_i(C)| <= eps), and,
# for an eigenvalue separated from the others by gap_i > 10 eps, its
# eigenvector (Davis-Kahan: ||v - v(C)|| <= 2 eps / gap_i, signs fixed by the
# same rule).  Orthonormality of V is tested at 1e-5.
ONLINE_C = 97
ONLINE_JACOBI = 1024


def _online_eps(kk, om, ol):
    xc = kk.astype(np.float64) - om
    E = ONLINE_C * 2.0 ** -24 * (np.abs(xc).T @ np.abs(xc)) / max(len(kk) - 1, 1)
    return float(np.linalg.norm(E, 2) + ONLINE_JACOBI * 2.0 ** -24 * ol[0])


def _online_case(n, cap=0, units=None):
    w = _klt_workload()
    units = list(range(w.units)) if units is None else units
    cap = cap or n
    krows = torch.full((len(units), cap, w.D), 9e3, dtype=torch.bfloat16, device="cuda")   # never read past n
    for i, u in enumerate(units):
        krows[i, :n] = synth.unit_keys(w, u, "cuda", n=n).to(torch.bfloat16)
    shape = B.make_shape(len(units), n, w.D, w.G, 1, 0, 0, n_cap=cap if cap != n else 0)   # k is not used
    return w, units, shape, krows


def _check_online_unit(keys_bf16, mean, V, lam, q=None):
    """q ([G][D], optional): also compare the plans the two bases give."""
    kk = keys_bf16.float().cpu().numpy()
    om, _, cov = O.calibrate(kk, with_cov=True)
    ol, oV = O.eigh(cov)
    m = mean.cpu().numpy()
    assert np.all(np.abs(m - om) <= 4e-6 * np.abs(kk.astype(np.float64)).mean(0) + 1e-30)
    gl = lam.cpu().numpy().astype(np.float64)
    Vg = V.cpu().numpy()
    eps = _online_eps(kk, om, ol)
    assert np.all(np.diff(gl) <= 0)                                      # descending
    back = np.linalg.norm(Vg @ np.diag(gl) @ Vg.T - cov, 2)
    assert back <= eps, (back / ol[0], eps / ol[0])
    np.testing.assert_allclose(gl, ol, rtol=0, atol=eps)
    np.testing.assert_allclose(Vg.T @ Vg, np.eye(Vg.shape[0]), rtol=0, atol=1e-5)
    arg = np.argmax(np.abs(Vg), axis=0)
    assert np.all(Vg[arg, np.arange(Vg.shape[1])] > 0)
    D = len(ol)
    gaps = np.array([np.min(np.abs(np.delete(ol, i) - ol[i])) if D > 1 else np.inf for i in range(D)])
    sep = gaps > 10 * eps
    eta = np.where(sep, 2 * eps / np.maximum(gaps, 1e-300), np.inf)
    dv = np.linalg.norm(Vg - oV, axis=0)
    assert np.all(dv[sep] <= eta[sep]), float(np.max(dv[sep] / eta[sep]))
    if q is not None:
        # The planner on the GPU's basis against the planner on the oracle's: a
        # channel's depth may differ only if one of its breakpoints lies within the
        # importance error bound of the oracle plan's critical breakpoint (the
        # channels of near-degenerate eigenvalues, whose vectors are not pinned,
        # are exempt).
        q64 = q.astype(np.float64)
        qn = np.linalg.norm(q64, axis=1)                               # ||q_h||
        qo = q64 @ oV                                                  # [G][D]
        go = ol * np.sum(qo ** 2, axis=0)
        dq = qn[:, None] * np.where(sep, eta, 0.0)[None, :]
        dg = eps * np.sum(qo ** 2, axis=0) + ol * np.sum(2 * np.abs(qo) * dq + dq ** 2, axis=0)
        rel = np.where(sep & (go > 0), dg / np.maximum(go, 1e-300), np.inf)
        rmax = float(np.max(rel[np.isfinite(rel)])) if np.any(np.isfinite(rel)) else 0.0
        for budget in (24, 48, 128):
            dg_, _, _ = O.plan((q64 @ Vg).astype(np.float32), gl.astype(np.float32), budget)
            do_, _, _ = O.plan(qo.astype(np.float32), ol.astype(np.float32), budget)
            bp = np.sort(np.concatenate([go[go > 0] * 2.0 ** -(2 * mm + 1) for mm in range(4)]))[::-1]
            bstar = bp[budget] if budget < len(bp) else 0.0
            for j in np.nonzero(dg_ != do_)[0]:
                if not np.isfinite(rel[j]):
                    continue
                near = [abs(go[j] * 2.0 ** -(2 * mm + 1) / bstar - 1.0) <= rel[j] + 2 * rmax for mm in range(4)]
                assert any(near), (budget, j, rel[j], rmax)


@pytest.mark.parametrize("n,cap", [(5000, 0), (777, 1024), (64, 0), (2, 0)])
def test_online_basis_matches_oracle(n, cap):
    w, units, shape, krows = _online_case(n, cap)
    mean, V, lam = B.fathom_klt_online(shape, krows)
    torch.cuda.synchronize()
    for ui in range(len(units)):
        _check_online_unit(krows[ui, :n], mean[ui], V[ui], lam[ui],
                           q=synth.unit_query(w, units[ui], "cpu").numpy())


def test_online_basis_at_100k_tokens():
    # the size the pages quote: 100k tokens of one layer's 8 KV heads, two units checked
    w = synth.WORKLOADS["klt_32x64k"]
    n = 100000
    units = w.layer_units(0)[:8]
    krows = torch.stack([synth.unit_keys(w, u, "cuda", n=n) for u in units]).to(torch.bfloat16)
    shape = B.make_shape(len(units), n, w.D, w.G, 64, 4, 32)
    mean, V, lam = B.fathom_klt_online(shape, krows)
    torch.cuda.synchronize()
    for ui in (0, 5):
        _check_online_unit(krows[ui], mean[ui], V[ui], lam[ui], q=synth.unit_query(w, units[ui], "cpu").numpy())


def test_online_basis_full_path():
    # the whole path on a store built in each unit's own basis (groups = units)
    w, units, shape0, krows = _online_case(6000)
    U, n, k = len(units), 6000, 300
    shape = B.make_shape(U, n, w.D, w.G, k, w.n_sink, w.n_recent)
    vrows = torch.stack([synth.unit_values(w, u, "cuda", n=n) for u in units]).to(torch.bfloat16)
    q = torch.stack([synth.unit_query(w, u, "cuda") for u in units]).contiguous()
    mean, V, lam = B.fathom_klt_online(shape, krows)
    kr = B.fathom_rotate_keys(shape, krows, U, mean, V)
    qr = B.fathom_rotate_query(shape, q, U, V)
    planes, scales = B.fathom_quantize_pack(shape, kr)
    budget = torch.full((U,), 48, dtype=torch.int32, device="cuda")
    depth, theta, runs = B.fathom_plan(shape, qr, lam, budget)
    scores = torch.full((U, w.G, n), float("nan"), device="cuda")
    idx, _ = B.fathom_scan_topk(shape, planes, scales, runs, qr, B.alloc_workspace(shape, B.WS_SCAN_TOPK),
                                scores=scores)
    out = B.fathom_sparse_attn(shape, krows, vrows, q, idx, B.alloc_workspace(shape, B.WS_SPARSE_ATTN))
    torch.cuda.synchronize()
    for ui in range(U):
        Vg, mu = V[ui].cpu().numpy(), mean[ui].cpu().numpy()
        kk = krows[ui].float().cpu().numpy()
        ref = O.rotate(kk, mu, Vg).astype(np.float64)
        err = np.abs(kr[ui].cpu().numpy().astype(np.float64) - ref)
        assert np.all(err <= ROT_RTOL * _rotation_bound(kk.astype(np.float64) - mu, Vg) + 1e-30)
        keys_r = kr[ui].cpu().numpy()
        qq = qr[ui].cpu().numpy()
        P, S, C = O.quantize_pack(keys_r)
        np.testing.assert_array_equal(u64(planes[ui]), P)
        od, oth, _ = O.plan(qq, lam[ui].cpu().numpy(), 48)
        np.testing.assert_array_equal(depth[ui].cpu().numpy(), od)
        assert theta[ui].item() == oth
        ref_s = O.scores(P[None], S[None], od[None], qq[None], n)[0]
        got = scores[ui].cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - ref_s) <= SCORE_RTOL * khat_magnitude(C, S, od, qq, n) + 1e-30)
        oi, _ = O.select(got, k, w.n_sink, w.n_recent)
        np.testing.assert_array_equal(idx[ui].cpu().numpy(), oi)
        o = O.attention(u16(krows[ui]), u16(vrows[ui]), q[ui].cpu().numpy(), oi)
        rel = np.linalg.norm(out[ui].cpu().numpy().astype(np.float64) - o, axis=1) / np.linalg.norm(o, axis=1)
        assert np.all(rel <= ATTN_RTOL), rel
