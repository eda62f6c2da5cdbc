"""Parity at the benchmarked sizes, in the launch configuration bench.py times:
one layer of each workload (all of the layer's units in one launch of every
call), the same paths (fused host-resident store for the 1M and 256k
workloads, HBM for the others, the rotated basis with its per-layer budget).
The oracle checks sampled units in full (store, plan, every token's score,
the kept sets, attention), which it finishes in seconds per unit."""
import numpy as np
import pytest
import torch

from bit_plane_kv_gb300 import binding as B
from bit_plane_kv_gb300 import synth
from oracle import oracle as O

from fathom_cases import (ATTN_RTOL, SCORE_RTOL, Inputs, check_unit, khat_magnitude, run_gpu, u16, u32,
                          u64)

pytestmark = pytest.mark.gpu


def _layer0(w):
    return w.layer_units(0)


@pytest.mark.parametrize("name,regime,sample", [
    ("host_1m", "fused", (0, 7)),          # 8 units x 1,048,576 tokens, store and rows in pinned host memory
    ("host_256k", "fused", (3,)),          # 8 units x 262,144 tokens
    ("qwen3_32k", "hbm", range(8)),        # 8 units x 32,768 tokens
])
def test_full_size_layer(name, regime, sample):
    w = synth.WORKLOADS[name]
    inp = Inputs(w, _layer0(w), w.n)
    r = run_gpu(inp, k=w.k, budget=48, n_sink=w.n_sink, n_recent=w.n_recent, regime=regime)
    for ui in sample:
        check_unit(inp, r, ui, w.k, 48, w.n_sink, w.n_recent, check_attn=True)


def test_full_size_rotated_layer():
    # one layer of the 32-session rotated-basis batch: 256 units x 65,536 tokens, B_0 = 24
    w = synth.WORKLOADS["klt_32x64k"]
    H = w.kv_heads
    units = _layer0(w)
    U, n, k = len(units), w.n, w.k
    calib = torch.stack([synth.unit_calib(w, g, "cuda") for g in range(H)]).contiguous()   # layer 0's heads
    mean, V, lam = B.fathom_calibrate_klt(calib)
    shape = B.make_shape(U, n, w.D, w.G, k, w.n_sink, w.n_recent)
    krows = torch.empty(U, n, w.D, dtype=torch.bfloat16, device="cuda")
    vrows = torch.empty(U, n, w.D, dtype=torch.bfloat16, device="cuda")
    for i, u in enumerate(units):
        krows[i] = synth.unit_keys(w, u, "cuda").to(torch.bfloat16)
        vrows[i] = synth.unit_values(w, u, "cuda").to(torch.bfloat16)
    q = torch.stack([synth.unit_query(w, u, "cuda", step=1) for u in units]).contiguous()
    b0 = w.budgets[0]
    budget = torch.full((U,), b0, dtype=torch.int32, device="cuda")
    lam_u = lam.repeat(U // H, 1).contiguous()            # unit i of the layer: head i % H
    kr = B.fathom_rotate_keys(shape, krows, H, mean, V)
    qr = B.fathom_rotate_query(shape, q, H, V)
    planes, scales = B.fathom_quantize_pack(shape, kr)
    depth, theta, runs = B.fathom_plan(shape, qr, lam_u, budget)
    scores = torch.full((U, w.G, n), float("nan"), device="cuda")
    idx, _ = B.fathom_scan_topk(shape, planes, scales, runs, qr, B.alloc_workspace(shape, B.WS_SCAN_TOPK),
                                scores=scores)
    out = B.fathom_sparse_attn(shape, krows, vrows, q, idx, B.alloc_workspace(shape, B.WS_SPARSE_ATTN))
    torch.cuda.synchronize()
    for ui in (0, U - 1):
        qq = qr[ui].cpu().numpy()
        P, S, C = O.quantize_pack(kr[ui].cpu().numpy())
        np.testing.assert_array_equal(u64(planes[ui]), P)
        np.testing.assert_array_equal(u16(scales[ui]), S)
        od, oth, _ = O.plan(qq, lam_u[ui].cpu().numpy(), b0)
        np.testing.assert_array_equal(depth[ui].cpu().numpy(), od)
        assert theta[ui].item() == oth
        np.testing.assert_array_equal(u32(runs[ui]), O.runs(od, n))
        ref = O.scores(P[None], S[None], od[None], qq[None], n)[0]
        got = scores[ui].cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - ref) <= SCORE_RTOL * khat_magnitude(C, S, od, qq, n) + 1e-30)
        oi, _ = O.select(got, k, w.n_sink, w.n_recent)
        np.testing.assert_array_equal(idx[ui].cpu().numpy(), oi)
        o = O.attention(u16(krows[ui]), u16(vrows[ui]), q[ui].cpu().numpy(), oi)
        rel = np.linalg.norm(out[ui].cpu().numpy().astype(np.float64) - o, axis=1) / np.linalg.norm(o, axis=1)
        assert np.all(rel <= ATTN_RTOL), rel
