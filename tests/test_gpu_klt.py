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
