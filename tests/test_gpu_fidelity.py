"""Fidelity references on the GPU against the oracle (Fathom §4, §5): the
exact top-k with every token scored from its bf16 key row, dense attention,
the relative-error and kept-set overlap reductions, and the greedy per-layer
budgets (§3.4) driven by errors measured on the GPU.

Tolerances:
* exact scores: |s_gpu - s_ref| <= 1e-5 * sum_j |q_hj k_ij| (a fp32 sum of at
  most 128 exact products of a fp32 query and a bf16 key, <= 128 u with
  u = 2^-24, against fp64);
* kept sets: the oracle's selection on the GPU's own scores equals the GPU's
  sets bit for bit (the decision taken in the kernel's precision);
* dense attention: relative L2 error per head <= 2e-3 against fp64;
* relative error: within 1e-12 relative of the fp64 definition on the same
  fp32 inputs; overlap counts: exact;
* the per-level errors of the greedy plan: within 5e-3 absolute of the
  oracle's on the same kept sets (each output within 2e-3 of fp64, so the
  quotient moves by at most about twice that).
"""
import numpy as np
import pytest
import torch

from bit_plane_kv_gb300 import binding as B
from bit_plane_kv_gb300 import fidelity as F
from bit_plane_kv_gb300 import synth
from oracle import oracle as O

from fathom_cases import ATTN_RTOL, Inputs, u16, u64

pytestmark = pytest.mark.gpu
EXACT_RTOL = 1e-5


def _generic(D, G, seed=20261000):
    return synth.Workload("fidelity_case", seed, n=4096, kv_heads=3, G=G, D=D, outliers=1)


@pytest.mark.parametrize("D,G,n,k,ns,nr,host", [
    (128, 4, 3000, 300, 4, 32, False),     # ragged last block, 128-bit vector loads
    (128, 4, 4096, 512, 4, 32, True),      # rows in pinned host memory
    (64, 1, 4096, 64, 4, 32, False),
    (128, 8, 1500, 100, 0, 0, False),      # no forced tokens
    (98, 2, 777, 50, 4, 32, False),        # D % 4 != 0: scalar row loads
])
def test_exact_topk_matches_oracle(D, G, n, k, ns, nr, host):
    w = _generic(D, G)
    inp = Inputs(w, range(3), n)
    U = 3
    shape = B.make_shape(U, n, D, G, k, ns, nr)
    kr = inp.krows.cpu().pin_memory() if host else inp.krows
    scores = torch.full((U, G, n), float("nan"), device="cuda")
    idx, sel = B.fathom_exact_topk(shape, kr, inp.q, B.alloc_workspace(shape, B.WS_SCAN_TOPK), scores=scores)
    torch.cuda.synchronize()
    for ui in range(U):
        keys = inp.krows[ui].float().cpu().numpy()
        q = inp.q[ui].cpu().numpy()
        ref = O.exact_scores(keys, q)
        got = scores[ui].cpu().numpy().astype(np.float64)
        mag = np.abs(q.astype(np.float64)) @ np.abs(keys.astype(np.float64)).T
        assert np.all(np.abs(got - ref) <= EXACT_RTOL * mag + 1e-30)
        oi, osel = O.select(got, k, ns, nr)
        np.testing.assert_array_equal(idx[ui].cpu().numpy(), oi)
        np.testing.assert_array_equal(sel[ui].cpu().numpy().astype(np.float64), osel)


def test_exact_topk_on_a_capacity_layout():
    w = _generic(128, 4)
    n, cap, k = 2000, 2560, 128
    inp = Inputs(w, range(2), n)
    krows = torch.full((2, cap, 128), 7e3, dtype=torch.bfloat16, device="cuda")   # never read past n
    krows[:, :n] = inp.krows
    shape = B.make_shape(2, n, 128, 4, k, 4, 32, n_cap=cap)
    idx, _ = B.fathom_exact_topk(shape, krows, inp.q, B.alloc_workspace(shape, B.WS_SCAN_TOPK))
    ref_shape = B.make_shape(2, n, 128, 4, k, 4, 32)
    ridx, _ = B.fathom_exact_topk(ref_shape, inp.krows, inp.q, B.alloc_workspace(ref_shape, B.WS_SCAN_TOPK))
    torch.cuda.synchronize()
    assert torch.equal(idx, ridx)


@pytest.mark.parametrize("D,G,n,host", [(128, 4, 3000, False), (128, 8, 70000, True), (64, 2, 100, False),
                                        (98, 1, 1025, False)])
def test_dense_attention_matches_oracle(D, G, n, host):
    w = _generic(D, G)
    inp = Inputs(w, range(2), n)
    shape = B.make_shape(2, n, D, G, 1, 0, 0)
    kr, vr = (inp.krows.cpu().pin_memory(), inp.vrows.cpu().pin_memory()) if host else (inp.krows, inp.vrows)
    ws = B.alloc_workspace(shape, B.WS_DENSE_ATTN)
    out = B.fathom_dense_attn(shape, kr, vr, inp.q, ws)
    out2 = B.fathom_dense_attn(shape, kr, vr, inp.q, ws)     # the workspace is left ready for the next call
    torch.cuda.synchronize()
    assert torch.equal(out, out2)
    for ui in range(2):
        o = O.dense_attention(u16(inp.krows[ui]), u16(inp.vrows[ui]), inp.q[ui].cpu().numpy())
        rel = O.rel_l2(out[ui].cpu().numpy(), o)
        assert np.all(rel <= ATTN_RTOL), rel


def test_rel_err_and_overlap_kernels():
    g = torch.Generator(device="cpu").manual_seed(5)
    a = torch.randn(37, 5, 128, generator=g)
    ref = torch.randn(37, 5, 128, generator=g)
    ref[3, 2] = 0.0
    err = B.fathom_rel_err(a.cuda(), ref.cuda())
    np.testing.assert_allclose(err.cpu().numpy(), O.rel_l2(a.numpy(), ref.numpy()), rtol=1e-12, atol=0)
    rows, k = 50, 300
    A = np.zeros((rows, k), np.int32)
    Bb = np.zeros((rows, k), np.int32)
    rng = np.random.default_rng(3)
    for r in range(rows):
        pool = rng.choice(900, size=2 * k, replace=False)
        shared = int(rng.integers(0, k + 1))
        A[r] = np.sort(pool[:k])
        Bb[r] = np.sort(np.concatenate([pool[:shared], pool[k:2 * k - shared]]))
    cnt = B.fathom_set_overlap(torch.from_numpy(A).cuda(), torch.from_numpy(Bb).cuda())
    expect = [len(set(A[r]) & set(Bb[r])) for r in range(rows)]
    np.testing.assert_array_equal(cnt.cpu().numpy(), expect)


def test_compare_reports_fidelity_of_the_sparse_path():
    w = synth.shrink(synth.WORKLOADS["qwen3_32k"], layers=1, kv_heads=2)
    n, k = 8192, 512
    inp = Inputs(w, range(2), n)
    shape = B.make_shape(2, n, 128, 4, k, 4, 32)
    _, var = B.fathom_calibrate(inp.calib)
    planes, scales = B.fathom_quantize_pack(shape, inp.keys_in)
    res = {}
    for b in (24, 48, 512):
        _, _, runs = B.fathom_plan(shape, inp.q, var, torch.full((2,), b, dtype=torch.int32, device="cuda"))
        idx, _ = B.fathom_scan_topk(shape, planes, scales, runs, inp.q, B.alloc_workspace(shape, B.WS_SCAN_TOPK))
        out = B.fathom_sparse_attn(shape, inp.krows, inp.vrows, inp.q, idx, B.alloc_workspace(shape, B.WS_SPARSE_ATTN))
        res[b] = F.compare(shape, inp.krows, inp.vrows, inp.q, idx, out)
    for ui in range(2):
        q = inp.q[ui].cpu().numpy()
        dense = O.dense_attention(u16(inp.krows[ui]), u16(inp.vrows[ui]), q)
        ex, _ = O.select(O.exact_scores(inp.krows[ui].float().cpu().numpy(), q), k, 4, 32)
        oex = O.attention(u16(inp.krows[ui]), u16(inp.vrows[ui]), q, ex)
        np.testing.assert_allclose(res[48]["exact_vs_dense"][ui], O.rel_l2(oex, dense), rtol=0, atol=5e-3)
    # more bits read, closer to the exact top-k: the full 4-plane scan keeps nearly all of it
    assert res[512]["overlap"].mean() >= res[48]["overlap"].mean() >= res[24]["overlap"].mean() - 0.02
    assert res[512]["overlap"].mean() > 0.9
    for b in res:
        assert np.all(res[b]["overlap"] <= 1.0) and np.all(res[b]["rel_dense"] >= 0)


def test_greedy_budgets_from_errors_measured_on_the_gpu():
    # the rotated-basis batch shrunk to 2 layers x 2 heads of one sequence; the
    # per-level error table from the GPU's sparse and dense attention matches the
    # oracle's on the same kept sets, and the greedy plan on it averages the target
    w = synth.shrink(synth.WORKLOADS["klt_32x64k"], seqs=1, layers=2, kv_heads=2, rotated=False)
    n, k = 2048, 128
    levels = list(range(24, 129, 8))
    table = np.zeros((w.layers, len(levels)))
    for layer in range(w.layers):
        units = w.layer_units(layer)
        inp = Inputs(w, units, n)
        U = len(units)
        shape = B.make_shape(U, n, w.D, w.G, k, 4, 32)
        _, var = B.fathom_calibrate(inp.calib)
        planes, scales = B.fathom_quantize_pack(shape, inp.keys_in)
        table[layer] = F.level_errors(shape, planes, scales, inp.krows, inp.vrows, [inp.q], var, levels)
        # the oracle on the GPU's kept sets at three of the levels
        ws = B.alloc_workspace(shape, B.WS_SCAN_TOPK)
        for li in (0, 3, len(levels) - 1):
            bud = torch.full((U,), levels[li], dtype=torch.int32, device="cuda")
            _, _, runs = B.fathom_plan(shape, inp.q, var, bud)
            sc = torch.empty(U, w.G, n, device="cuda")
            B.fathom_scan_topk(shape, planes, scales, runs, inp.q, ws, scores=sc)
            errs = []
            for ui in range(U):
                q = inp.q[ui].cpu().numpy()
                oi, _ = O.select(sc[ui].cpu().numpy().astype(np.float64), k, 4, 32)
                kk, vv = u16(inp.krows[ui]), u16(inp.vrows[ui])
                errs.append(O.rel_l2(O.attention(kk, vv, q, oi), O.dense_attention(kk, vv, q)))
            assert abs(table[layer, li] - float(np.mean(errs))) <= 5e-3, (layer, li)
    budgets = F.greedy_layer_budgets(table, 24, 8, 48)
    np.testing.assert_array_equal(budgets, O.greedy_budgets(table, 24, 8, 48))
    assert budgets.sum() == 48 * w.layers and np.all((budgets >= 24) & (budgets <= 128))


# ------------------------------------------------------------------ keys rebuilt from the store
@pytest.mark.parametrize("D,G,n,k,where,cap", [
    (128, 4, 3000, 300, "hbm", 0),
    (128, 4, 4096, 512, "host", 0),        # store in pinned host memory
    (128, 4, 2000, 256, "hbm", 2560),      # capacity layout
    (98, 2, 777, 60, "hbm", 0),            # D % 4 != 0
    (128, 8, 1500, 100, "hbm", 0),
])
def test_attention_with_keys_rebuilt_from_planes_matches_oracle(D, G, n, k, where, cap):
    w = _generic(D, G)
    U = 2
    inp = Inputs(w, range(U), n)
    c = cap or n
    keys = torch.zeros(U, c, D, dtype=torch.bfloat16, device="cuda")
    vals = torch.zeros(U, c, D, dtype=torch.bfloat16, device="cuda")
    keys[:, :n], vals[:, :n] = inp.krows, inp.vrows
    shape = B.make_shape(U, n, D, G, k, 4, 32, n_cap=cap)
    planes, scales = B.fathom_quantize_pack(shape, keys)
    # any valid kept sets: the exact top-k
    idx, _ = B.fathom_exact_topk(shape, keys, inp.q, B.alloc_workspace(shape, B.WS_SCAN_TOPK))
    if where == "host":
        planes, scales = planes.cpu().pin_memory(), scales.cpu().pin_memory()
    out = B.fathom_sparse_attn_planes(shape, planes, scales, vals, inp.q, idx, B.alloc_workspace(shape, B.WS_SPARSE_ATTN))
    torch.cuda.synchronize()
    for ui in range(U):
        kk = O.reconstruct(u64(planes[ui].cpu()), u16(scales[ui].cpu()), n)
        o = O.attention_keys(kk, u16(inp.vrows[ui]), inp.q[ui].cpu().numpy(), idx[ui].cpu().numpy())
        rel = O.rel_l2(out[ui].cpu().numpy(), o)
        assert np.all(rel <= ATTN_RTOL), rel
