"""fathom_sparse_attn_noalloc: the sparse-attention call for callers that may
not allocate device memory for the library (a host framework that owns all
device memory and forbids plug-ins to call cudaMalloc, or a decode loop that
must never allocate).  It uses the library's fixed 8 MiB scratch array instead
of a caller workspace.  Called here through the C ABI, twice in a row, and
compared with fathom_sparse_attn on the same inputs.

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from bit_plane_kv_gb300 import binding as B
from bit_plane_kv_gb300 import synth

pytestmark = pytest.mark.gpu

ATTN_RTOL = 2e-3   # the attention tolerance of the parity tests


def _kept_sets(w, units, n, k, step):
    """Queries of one decode step and the kept sets the scan selects for them."""
    keys = torch.stack([synth.unit_keys(w, u, "cuda", n=n) for u in units]).to(torch.bfloat16)
    vals = torch.stack([synth.unit_values(w, u, "cuda", n=n) for u in units]).to(torch.bfloat16)
    q = torch.stack([synth.unit_query(w, u, "cuda", step=step) for u in units]).contiguous()
    calib = torch.stack([synth.unit_calib(w, u, "cuda") for u in units]).contiguous()
    shape = B.make_shape(len(units), n, w.D, w.G, k, w.n_sink, w.n_recent)
    _, var = B.fathom_calibrate(calib)
    planes, scales = B.fathom_quantize_pack(shape, keys)
    budget = torch.full((len(units),), 48, dtype=torch.int32, device="cuda")
    _, _, runs = B.fathom_plan(shape, q, var, budget)
    idx, _ = B.fathom_scan_topk(shape, planes, scales, runs, q, B.alloc_workspace(shape, B.WS_SCAN_TOPK))
    return shape, keys, vals, q, idx


def _noalloc(shape, keys, vals, q, idx):
    out = torch.full((shape.units, shape.G, shape.D), float("nan"), device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = B.lib().fathom_sparse_attn_noalloc(ctypes.byref(shape), ctypes.c_void_p(keys.data_ptr()),
                                            ctypes.c_void_p(vals.data_ptr()), ctypes.c_void_p(q.data_ptr()),
                                            ctypes.c_void_p(idx.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                            ctypes.c_void_p(stream))
    assert rc == 0, B.lib().fathom_last_error().decode()
    return out


def _rel_l2(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return np.linalg.norm(a - b, axis=-1) / np.linalg.norm(b, axis=-1)


def test_noalloc_matches_workspace_call_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = synth.WORKLOADS["qwen3_32k"]
    units, n, k = list(range(8)), 32768, 512
    outs = []
    for step in (1, 2):   # two calls in a row, each with its own kept sets
        shape, keys, vals, q, idx = _kept_sets(w, units, n, k, step)
        ref = B.fathom_sparse_attn(shape, keys, vals, q, idx, B.alloc_workspace(shape, B.WS_SPARSE_ATTN))
        got = _noalloc(shape, keys, vals, q, idx)
        torch.cuda.synchronize()
        assert torch.isfinite(got).all()
        assert np.all(_rel_l2(got, ref) <= ATTN_RTOL)
        outs.append(got)
    assert not torch.equal(outs[0], outs[1])      # the second call did its own work


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # 2048 units with k = 2048 need far more than 8 MiB of scratch: rejected up front
    shape = B.make_shape(2048, 1 << 16, 128, 4, 2048)
    assert B.workspace_size(shape, B.WS_SPARSE_ATTN) > (8 << 20)
    d = ctypes.c_void_p(256)   # never dereferenced: the size check comes first
    rc = B.lib().fathom_sparse_attn_noalloc(ctypes.byref(shape), d, d, d, d, d, None)
    assert rc == 1
    assert "scratch" in B.lib().fathom_last_error().decode()
