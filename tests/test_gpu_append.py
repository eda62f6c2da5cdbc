"""Decode-time append and capacity layouts on the GPU against the oracle.

A store allocated for C tokens grows as a decode loop appends tokens:
fathom_append_block codes the block each new token falls in (a block that is
still filling is coded again as it fills), and every call reads the arrays at
their capacity strides while using only the live n tokens.  The store must
equal, bit for bit, what fathom_quantize_pack and the oracle give for the
live prefix, the blocks past the live length must stay untouched, and the
whole path on a capacity layout must match the oracle on the live prefix.
"""
import numpy as np
import pytest
import torch

from bit_plane_kv_gb300 import binding as B
from bit_plane_kv_gb300 import synth
from oracle import oracle as O

from fathom_cases import ATTN_RTOL, SCORE_RTOL, khat_magnitude, u16, u32, u64

pytestmark = pytest.mark.gpu
SENTINEL = 0x5A5A5A5A5A5A5A5A


def _rows(w, units, n, cap, fill):
    """bf16 key/value rows laid out for `cap` tokens; tokens past n hold `fill`."""
    k = torch.full((len(units), cap, w.D), fill, dtype=torch.float32, device="cuda")
    v = torch.full((len(units), cap, w.D), fill, dtype=torch.float32, device="cuda")
    for i, u in enumerate(units):
        k[i, :n] = synth.unit_keys(w, u, "cuda", n=n)
        v[i, :n] = synth.unit_values(w, u, "cuda", n=n)
    return k.to(torch.bfloat16), v.to(torch.bfloat16)


def _store_equals_prefix(planes, scales, keys, n, units_idx):
    nb = B.nblocks(n)
    for ui in units_idx:
        P, S, _ = O.quantize_pack(keys[ui, :n].float().cpu().numpy())
        np.testing.assert_array_equal(u64(planes[ui])[:, :, :nb], P)
        np.testing.assert_array_equal(u16(scales[ui])[:, :nb], S)


def test_append_grows_the_store_like_a_prefix_quantisation():
    w = synth.WORKLOADS["qwen3_32k"]
    units = [0, 1, 2]
    n_final, cap = 4000, 4160            # 62 full blocks + 32 tokens, capacity 65 blocks
    keys, _ = _rows(w, units, n_final, cap, fill=1e4)   # garbage past n_final must never be read
    shape = B.make_shape(len(units), 2048, w.D, w.G, 64, n_cap=cap)
    cb = B.nblocks(cap)
    planes = torch.full((len(units), w.D, 4, cb), SENTINEL, dtype=torch.int64, device="cuda")
    scales = torch.full((len(units), w.D, cb), 0x1234, dtype=torch.int16, device="cuda")
    B.fathom_quantize_pack(shape, keys, planes=planes, scales=scales)      # prefill: 2048 tokens
    torch.cuda.synchronize()
    _store_equals_prefix(planes, scales, keys, 2048, [0])
    checkpoints = {2049, 2100, 3000, 3968, 3969, n_final}
    for t in range(2048, n_final):
        n = t + 1
        # a decode loop codes the block of every new token; here every token of the
        # last two blocks and the others only at block ends and at the checkpoints
        if t >= 3904 or n % 64 == 0 or n in checkpoints:
            B.fathom_append_block(shape, keys, t // 64, t % 64 + 1, planes, scales)
        if n in checkpoints:
            torch.cuda.synchronize()
            _store_equals_prefix(planes, scales, keys, n, [0, 2])
    torch.cuda.synchronize()
    # the live prefix equals fathom_quantize_pack of the prefix; blocks past it are untouched
    ref_shape = B.make_shape(len(units), n_final, w.D, w.G, 64)
    rp, rs = B.fathom_quantize_pack(ref_shape, keys[:, :n_final].contiguous())
    torch.cuda.synchronize()
    nb = B.nblocks(n_final)
    assert torch.equal(planes[..., :nb], rp) and torch.equal(scales[..., :nb], rs)
    assert np.all(u64(planes)[:, :, :, nb:] == SENTINEL)
    assert np.all(u16(scales)[:, :, nb:] == 0x1234)


@pytest.mark.parametrize("regime", ["hbm", "staged", "fused"])
@pytest.mark.parametrize("n", [3000, 3072])   # a ragged live length; one whose 16-byte staging path runs
def test_whole_path_on_a_capacity_layout(regime, n):
    w = synth.WORKLOADS["qwen3_32k"]
    units = [3, 4]
    cap, k = 4608, 300                   # arrays laid out for 4608 tokens
    keys, vals = _rows(w, units, n, cap, fill=3e3)
    U = len(units)
    shape = B.make_shape(U, n, w.D, w.G, k, w.n_sink, w.n_recent, n_cap=cap)
    q = torch.stack([synth.unit_query(w, u, "cuda") for u in units]).contiguous()
    _, var = B.fathom_calibrate(torch.stack([synth.unit_calib(w, u, "cuda") for u in units]).contiguous())
    planes, scales = B.fathom_quantize_pack(shape, keys)
    budget = torch.full((U,), 48, dtype=torch.int32, device="cuda")
    depth, theta, runs = B.fathom_plan(shape, q, var, budget)
    scores = torch.full((U, w.G, n), float("nan"), device="cuda")
    ws = B.alloc_workspace(shape, B.WS_SCAN_TOPK)
    kr, vr = keys, vals
    if regime == "hbm":
        idx, _ = B.fathom_scan_topk(shape, planes, scales, runs, q, ws, scores=scores)
    else:
        hp, hs = planes.cpu().pin_memory(), scales.cpu().pin_memory()
        kr, vr = keys.cpu().pin_memory(), vals.cpu().pin_memory()
        if regime == "fused":
            idx, _ = B.fathom_scan_topk(shape, hp, hs, runs, q, ws, scores=scores)
        else:
            nb = B.nblocks(n)
            sp = torch.zeros(U, 48 * nb, dtype=torch.int64, device="cuda")
            ss = torch.zeros(U, 48 * nb, dtype=torch.int16, device="cuda")
            B.fathom_gather(shape, hp, hs, runs, sp, ss)
            idx, _ = B.fathom_scan_topk(shape, sp, ss, runs, q, ws, source=B.SRC_STAGING, scores=scores)
    out = B.fathom_sparse_attn(shape, kr, vr, q, idx, B.alloc_workspace(shape, B.WS_SPARSE_ATTN))
    torch.cuda.synchronize()
    cb = B.nblocks(cap)
    for ui in range(U):
        qq = q[ui].cpu().numpy()
        P, S, C = O.quantize_pack(keys[ui, :n].float().cpu().numpy())
        nb = B.nblocks(n)
        np.testing.assert_array_equal(u64(planes[ui])[:, :, :nb], P)
        od, oth, _ = O.plan(qq, var[ui].cpu().numpy(), 48)
        np.testing.assert_array_equal(depth[ui].cpu().numpy(), od)
        assert theta[ui].item() == oth
        oruns = O.runs(od, n).astype(np.int64)
        oruns[:, 0] = np.arange(w.D) * 4 * cb          # the store keeps planes cb words apart
        oruns[:, 3] = np.arange(w.D) * cb
        np.testing.assert_array_equal(u32(runs[ui]).astype(np.int64), oruns)
        ref = O.scores(P[None], S[None], od[None], qq[None], n)[0]
        got = scores[ui].cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - ref) <= SCORE_RTOL * khat_magnitude(C, S, od, qq, n) + 1e-30)
        oi, _ = O.select(got, k, w.n_sink, w.n_recent)
        np.testing.assert_array_equal(idx[ui].cpu().numpy(), oi)
        o = O.attention(u16(keys[ui, :n]), u16(vals[ui, :n]), qq, oi)
        rel = np.linalg.norm(out[ui].cpu().numpy().astype(np.float64) - o, axis=1) / np.linalg.norm(o, axis=1)
        assert np.all(rel <= ATTN_RTOL), rel
