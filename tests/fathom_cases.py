"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
and the CPU oracle on the same seeded inputs and compare them.

Tolerances (each derived in the design notes):
* plane words, codes, scales, calibration statistics, depths, theta, run
  lists, staging contents, kept index sets: bit-exact;
* scores: |s_gpu - s_ref| <= 1e-5 * sum_j |q_hj * khat_ij| (fp32 accumulation
  of at most 128 exact products against fp64);
* top-k against the oracle's fp64 scores: equal sets except swaps between
  tokens whose oracle scores lie within 1e-6 of the k-th score plus the score
  tolerance; against the GPU's own fp32 scores: identical;
* attention: relative L2 error per head <= 2e-3.
"""
from __future__ import annotations

import numpy as np
import torch

from bit_plane_kv_gb300 import binding as B
from bit_plane_kv_gb300 import synth
from oracle import oracle as O

SCORE_RTOL = 1e-5
TIE_RTOL = 1e-6
ATTN_RTOL = 2e-3


def u64(t):
    return t.detach().cpu().contiguous().numpy().view(np.uint64)


def u16(t):
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return t.numpy().view(np.uint16)


def u32(t):
    return t.detach().cpu().contiguous().numpy().view(np.uint32)


class Inputs:
    """Seeded inputs of `units` units (indices into the workload), on `device`."""

    def __init__(self, w: synth.Workload, units, n, device="cuda"):
        self.w, self.units, self.n = w, list(units), n
        keys = torch.stack([synth.unit_keys(w, u, device, n=n) for u in self.units])
        if w.keys_dtype == "bf16":
            self.keys_in = keys.to(torch.bfloat16)          # what the quantiser reads
            self.keys32 = self.keys_in.float()               # exact widening
        else:
            self.keys_in = keys
            self.keys32 = keys
        self.krows = keys.to(torch.bfloat16)                 # full-precision rows for attention
        self.vrows = torch.stack([synth.unit_values(w, u, device, n=n) for u in self.units]).to(torch.bfloat16)
        self.q = torch.stack([synth.unit_query(w, u, device) for u in self.units]).contiguous()
        self.calib = torch.stack([synth.unit_calib(w, u, device) for u in self.units]).contiguous()


class Canaries:
    """Device buffers with guard bytes on both sides (the stand-in for a memory
    checker, which is closed on this machine): every buffer a call writes is the
    middle of a larger allocation whose first and last 256 bytes hold a fixed
    pattern, and check() asserts after the calls that no guard byte changed."""

    PAD = 256
    PATTERN = 0xA5

    def __init__(self):
        self.bufs = []

    def alloc(self, name, shape, dtype, fill=None):
        shape = tuple(int(x) for x in shape)
        numel = int(np.prod(shape)) if shape else 1
        es = torch.empty((), dtype=dtype).element_size()
        pad = self.PAD // es
        raw = torch.empty(numel + 2 * pad, dtype=dtype, device="cuda")
        raw.view(torch.uint8).fill_(self.PATTERN)
        body = raw[pad:pad + numel].view(shape)
        if fill is not None:
            body.fill_(fill)
        self.bufs.append((name, raw, pad * es, numel * es))
        return body

    def check(self):
        torch.cuda.synchronize()
        for name, raw, pad, nbytes in self.bufs:
            b = raw.view(torch.uint8)
            head, tail = b[:pad], b[pad + nbytes:]
            assert bool((head == self.PATTERN).all()), f"{name}: bytes before the buffer were written"
            assert bool((tail == self.PATTERN).all()), f"{name}: bytes after the buffer were written"
        return len(self.bufs)


def run_gpu(inp: Inputs, k, budget, n_sink=4, n_recent=32, regime="hbm", bracket=None,
            fixed=None, want_scores=True):
    w = inp.w
    U = len(inp.units)
    shape = B.make_shape(U, inp.n, w.D, w.G, k, n_sink, n_recent)
    cz = Canaries()
    r = {"shape": shape, "canaries": cz}
    nb = B.nblocks(inp.n)
    r["mean"], r["var"] = B.fathom_calibrate(inp.calib, mean=cz.alloc("mean", (U, w.D), torch.float32),
                                             var=cz.alloc("var", (U, w.D), torch.float32))
    r["planes"], r["scales"] = B.fathom_quantize_pack(
        shape, inp.keys_in, planes=cz.alloc("planes", (U, w.D, 4, nb), torch.int64),
        scales=cz.alloc("scales", (U, w.D, nb), torch.int16))
    bud = torch.as_tensor(np.broadcast_to(np.asarray(budget, np.int32), (U,)).copy(), device="cuda")
    depth_b = cz.alloc("depth", (U, w.D), torch.uint8)
    runs_b = cz.alloc("runs", (U, w.D, 6), torch.int32)
    if fixed is not None:
        r["depth"], r["runs"] = B.fathom_plan_fixed(shape, inp.q, r["var"], fixed[0], fixed[1],
                                                    depth=depth_b, runs=runs_b)
        r["theta"] = None
    else:
        br = None if bracket is None else torch.as_tensor(np.tile(np.asarray(bracket, np.float64), (U, 1)), device="cuda")
        r["depth"], r["theta"], r["runs"] = B.fathom_plan(shape, inp.q, r["var"], bud, bracket=br, depth=depth_b,
                                                          theta=cz.alloc("theta", (U,), torch.float64),
                                                          runs=runs_b)
    ws = cz.alloc("scan workspace", (B.workspace_size(shape, B.WS_SCAN_TOPK),), torch.uint8, fill=0)
    scores = cz.alloc("scores", (U, w.G, inp.n), torch.float32, fill=float("nan")) if want_scores else None
    if regime == "fused":
        # host-resident store read by the scan straight from pinned memory (the bench's default path)
        hp = r["planes"].cpu().pin_memory()
        hs = r["scales"].cpu().pin_memory()
        src_p, src_s, source = hp, hs, B.SRC_STORE
    elif regime == "host":
        hp = r["planes"].cpu().pin_memory()
        hs = r["scales"].cpu().pin_memory()
        bmax = int(np.max(budget)) if fixed is None else fixed[0] * fixed[1]
        W = min(bmax, 4 * w.D) * nb
        W += W % 2
        S = min(bmax, w.D) * nb
        S = (S + 7) // 8 * 8
        r["stage_planes"] = cz.alloc("staging planes", (U, W), torch.int64, fill=0)
        r["stage_scales"] = cz.alloc("staging scales", (U, S), torch.int16, fill=0)
        B.fathom_gather(shape, hp, hs, r["runs"], r["stage_planes"], r["stage_scales"])
        src_p, src_s, source = r["stage_planes"], r["stage_scales"], B.SRC_STAGING
    else:
        src_p, src_s, source = r["planes"], r["scales"], B.SRC_STORE
    r["idx"], r["sel"] = B.fathom_scan_topk(shape, src_p, src_s, r["runs"], inp.q, ws, source=source,
                                            scores=scores,
                                            topk_idx=cz.alloc("topk_idx", (U, w.G, k), torch.int32),
                                            topk_score=cz.alloc("topk_score", (U, w.G, k), torch.float32))
    r["scores"] = scores
    aws = cz.alloc("attention workspace", (B.workspace_size(shape, B.WS_SPARSE_ATTN),), torch.uint8, fill=0)
    kr, vr = inp.krows, inp.vrows
    if regime in ("host", "fused"):
        kr, vr = kr.cpu().pin_memory(), vr.cpu().pin_memory()
    r["out"] = B.fathom_sparse_attn(shape, kr, vr, inp.q, r["idx"], aws,
                                    out=cz.alloc("out", (U, w.G, w.D), torch.float32))
    torch.cuda.synchronize()
    assert cz.check() >= 10
    return r


def khat_magnitude(codes, scales_u, depth_u, q_u, n):
    """sum_j |q_hj| |khat_ij| over active channels ([G][n]), the score tolerance scale."""
    G = q_u.shape[0]
    mag = np.zeros((G, n))
    act = np.nonzero(depth_u)[0]
    for j in act:
        t = int(depth_u[j])
        a16 = scales_u[j].view(np.float16).astype(np.float64)[np.arange(n) // 64]
        ct = codes[:n, j].astype(np.int64) >> (4 - t)
        kh = np.abs((ct + 0.5 - 2 ** (t - 1)) * a16 / 2 ** (t - 1))
        mag += np.abs(q_u[:, j:j + 1].astype(np.float64)) * kh[None, :]
    return mag


def check_unit(inp: Inputs, r, ui, k, budget, n_sink=4, n_recent=32, bracket=None, fixed=None,
               check_attn=True):
    """Full oracle comparison of unit `ui` (index into inp.units)."""
    n, w = inp.n, inp.w
    keys = inp.keys32[ui].cpu().numpy()
    q = inp.q[ui].cpu().numpy()
    # calibration statistics: bit-exact fp32 rounding of the fp64 oracle
    mean64, var64 = O.calibrate(inp.calib[ui].cpu().numpy())
    np.testing.assert_array_equal(r["var"][ui].cpu().numpy(), var64.astype(np.float32))
    np.testing.assert_array_equal(r["mean"][ui].cpu().numpy(), mean64.astype(np.float32))
    var32 = var64.astype(np.float32)
    # store: bit-exact
    P, S, C = O.quantize_pack(keys)
    np.testing.assert_array_equal(u64(r["planes"][ui]), P)
    np.testing.assert_array_equal(u16(r["scales"][ui]), S)
    # plan: bit-exact
    b = int(np.broadcast_to(np.asarray(budget), (len(inp.units),))[ui])
    if fixed is not None:
        depth = O.plan_fixed(q, var32, fixed[0], fixed[1])
    else:
        depth, theta, _ = O.plan(q, var32, b, bracket=bracket)
        assert r["theta"][ui].item() == theta
    np.testing.assert_array_equal(r["depth"][ui].cpu().numpy(), depth)
    runs = O.runs(depth, n)
    np.testing.assert_array_equal(u32(r["runs"][ui]), runs)
    if "stage_planes" in r:
        sp, ss = O.gather(runs, P, S, r["stage_planes"].shape[1], r["stage_scales"].shape[1])
        np.testing.assert_array_equal(u64(r["stage_planes"][ui]), sp)
        np.testing.assert_array_equal(u16(r["stage_scales"][ui]), ss)
    # scores within tolerance
    ref = O.scores(P[None], S[None], depth[None], q[None], n)[0]
    got = r["scores"][ui].cpu().numpy().astype(np.float64)
    mag = khat_magnitude(C, S, depth, q, n)
    err = np.abs(got - ref)
    assert np.all(err <= SCORE_RTOL * mag + 1e-30), float(np.max(err / np.maximum(mag, 1e-30)))
    # selection: identical to the oracle's selector run on the GPU's own scores
    idx = r["idx"][ui].cpu().numpy()
    sel = r["sel"][ui].cpu().numpy()
    oi, _ = O.select(got, k, n_sink, n_recent)
    np.testing.assert_array_equal(idx, oi)
    np.testing.assert_array_equal(sel, r["scores"][ui].cpu().numpy()[np.arange(w.G)[:, None], idx])
    # against the oracle's fp64 scores: only near-tie swaps
    ri, _ = O.select(ref, k, n_sink, n_recent)
    ns = min(n_sink, n)
    r0 = max(ns, n - n_recent)
    for h in range(w.G):
        a, bset = set(idx[h].tolist()), set(ri[h].tolist())
        if a == bset:
            continue
        free = [i for i in ri[h].tolist() if ns <= i < r0]
        kth = float(np.min(ref[h, free]))
        for i in a ^ bset:
            tol = TIE_RTOL * abs(kth) + 2 * SCORE_RTOL * max(mag[h, i], 1e-30)
            assert abs(ref[h, i] - kth) <= tol, (h, i, ref[h, i], kth)
    # attention over the GPU's kept sets
    if check_attn:
        out = O.attention(u16(inp.krows[ui]), u16(inp.vrows[ui]), q, idx)
        got_o = r["out"][ui].cpu().numpy().astype(np.float64)
        rel = np.linalg.norm(got_o - out, axis=1) / np.linalg.norm(out, axis=1)
        assert np.all(rel <= ATTN_RTOL), rel
    return {"depth": depth, "ref": ref, "mag": mag}
