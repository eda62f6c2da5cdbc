"""Fidelity measurements and the greedy per-layer plan, over the C ABI.

The Fathom review page ("Fathom: 쿼리마다 깊이를 바꾸는 스캔으로 1M 토큰 디코딩을
1.67배 빠르게 하다") judges the sparse path by the relative L2 error of its
attention output against dense attention and against attention over the exact
top-k (§4, §5), and gives a greedy per-layer plan that moves bits to the layers
whose error falls the most per bit (§3.4).  Every number here comes from the
library's kernels (exact top-k, dense attention, the error and overlap
reductions); Python only orders the calls and averages the per-row results.
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding as B


def compare(shape, k_rows, v_rows, q, topk_idx, sparse_out, q_scan=None, workspaces=None):
    """Fidelity of one step's sparse output against the two references.

    k_rows, v_rows [U][cap][D] bf16 (device or pinned host), q [U][G][D] fp32 (the
    attention queries), topk_idx [U][G][k] the kept sets, sparse_out [U][G][D]
    fp32 their attention output.  q_scan: the queries the exact top-k ranks by
    (default q; the rotated basis keeps q . k, so the unrotated queries serve).
    Returns per-(unit, head) numpy arrays: rel_dense (sparse vs dense),
    rel_exact (sparse vs exact top-k attention), exact_vs_dense (exact top-k
    attention vs dense) and overlap (fraction of the exact top-k kept)."""
    ws = workspaces or {}
    ws_scan = ws.get("scan") if ws.get("scan") is not None else B.alloc_workspace(shape, B.WS_SCAN_TOPK)
    ws_attn = ws.get("attn") if ws.get("attn") is not None else B.alloc_workspace(shape, B.WS_SPARSE_ATTN)
    ws_dense = ws.get("dense") if ws.get("dense") is not None else B.alloc_workspace(shape, B.WS_DENSE_ATTN)
    ex_idx, _ = B.fathom_exact_topk(shape, k_rows, q if q_scan is None else q_scan, ws_scan)
    ex_out = B.fathom_sparse_attn(shape, k_rows, v_rows, q, ex_idx, ws_attn)
    dense = B.fathom_dense_attn(shape, k_rows, v_rows, q, ws_dense)
    rel_dense = B.fathom_rel_err(sparse_out, dense)
    rel_exact = B.fathom_rel_err(sparse_out, ex_out)
    exact_vs_dense = B.fathom_rel_err(ex_out, dense)
    overlap = B.fathom_set_overlap(topk_idx, ex_idx)
    return {
        "rel_dense": rel_dense.cpu().numpy(),
        "rel_exact": rel_exact.cpu().numpy(),
        "exact_vs_dense": exact_vs_dense.cpu().numpy(),
        "overlap": overlap.cpu().numpy().astype(np.float64) / shape.k,
    }


def level_errors(shape, planes, scales, k_rows, v_rows, q_steps, var, levels, q_plan_steps=None):
    """Mean relative L2 error against dense attention of one layer's sparse path
    at each budget level.

    planes/scales: the layer's store; k_rows/v_rows its rows; q_steps a list of
    [U][G][D] query tensors (the calibration steps); var [U][D] the plan's
    channel statistics; q_plan_steps the plan and scan queries per step (the
    rotated queries in the rotated basis; default q_steps).  Returns
    err [len(levels)] fp64: the mean over steps, units and heads."""
    U = shape.units
    ws_scan = B.alloc_workspace(shape, B.WS_SCAN_TOPK)
    ws_attn = B.alloc_workspace(shape, B.WS_SPARSE_ATTN)
    ws_dense = B.alloc_workspace(shape, B.WS_DENSE_ATTN)
    dense = [B.fathom_dense_attn(shape, k_rows, v_rows, q, ws_dense) for q in q_steps]
    out = np.zeros(len(levels), np.float64)
    qp = q_steps if q_plan_steps is None else q_plan_steps
    for li, b in enumerate(levels):
        budget = torch.full((U,), int(b), dtype=torch.int32, device=q_steps[0].device)
        errs = []
        for q, qs, d in zip(q_steps, qp, dense):
            _, _, runs = B.fathom_plan(shape, qs, var, budget)
            idx, _ = B.fathom_scan_topk(shape, planes, scales, runs, qs, ws_scan)
            o = B.fathom_sparse_attn(shape, k_rows, v_rows, q, idx, ws_attn)
            errs.append(B.fathom_rel_err(o, d).cpu().numpy())
        out[li] = float(np.mean(errs))
    return out


def greedy_layer_budgets(err_table, b_min=24, step=8, b_mean=48):
    """err_table [layers][levels] -> per-layer budgets (the library's greedy plan)."""
    return B.fathom_greedy_budgets(err_table, b_min, step, b_mean)
