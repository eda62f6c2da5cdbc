"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.  Needs an sm_103a GPU and the built library."""
import dataclasses
import json
import os

import numpy as np
import pytest
import torch

from bit_plane_kv_gb300 import binding as B
from bit_plane_kv_gb300 import synth
from oracle import oracle as O

import fathom_cases
from fathom_cases import Inputs, check_unit, run_gpu, u16, u32, u64

pytestmark = pytest.mark.gpu

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "toy_appx_a.json")))


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.lib()


def W(name, **kw):
    return synth.shrink(synth.WORKLOADS[name], **kw)


# ------------------------------------------------------------------ toy (Appx. A)
class ToyInputs:
    """The page's 6 x 4 toy: channel 2 as printed, the other channels seeded."""

    def __init__(self):
        rng = np.random.default_rng(20260000)
        keys = rng.normal(size=(6, 4)).astype(np.float32)
        keys[:, 2] = GOLD["channel2"]["values"]
        self.w = synth.Workload("toy", 0, n=6, G=2, D=4, k=2, n_sink=0, n_recent=0, keys_dtype="f32")
        self.units, self.n = [0], 6
        self.keys_in = torch.tensor(keys[None], device="cuda")
        self.keys32 = self.keys_in
        self.krows = self.keys_in.to(torch.bfloat16)
        self.vrows = torch.tensor(rng.normal(size=(1, 6, 4)), dtype=torch.bfloat16, device="cuda")
        self.q = torch.tensor([[GOLD["q_A"], GOLD["q_B"]]], dtype=torch.float32, device="cuda")
        # calibration rows whose unbiased variance is close to the printed Var
        cal = rng.normal(size=(1024, 4)) * np.sqrt(GOLD["var"])
        self.calib = torch.tensor(cal[None], dtype=torch.float32, device="cuda")


def test_toy_plan_with_printed_bracket_and_var():
    toy = ToyInputs()
    shape = B.make_shape(1, 6, 4, 2, 2, 0, 0)
    var = torch.tensor([GOLD["var"]], dtype=torch.float32, device="cuda")
    for Bud, ref in ((8, GOLD["B8"]["depth"]), (6, GOLD["B6"]["depth"])):
        bud = torch.tensor([Bud], dtype=torch.int32, device="cuda")
        br = torch.tensor([GOLD["bracket"]], dtype=torch.float64, device="cuda")
        depth, theta, runs = B.fathom_plan(shape, toy.q, var, bud, bracket=br)
        assert depth[0].tolist() == ref
        od, oth, _ = O.plan(toy.q[0].cpu().numpy(), np.array(GOLD["var"], np.float32), Bud,
                            bracket=GOLD["bracket"])
        assert theta[0].item() == oth
        np.testing.assert_array_equal(u32(runs[0]), O.runs(od, 6))
    assert abs(theta[0].item() - 0.11796875) < 1e-7   # B = 6 stops at g1 / 32


def test_toy_channel2_codes_and_full_path():
    toy = ToyInputs()
    r = run_gpu(toy, k=2, budget=8, n_sink=0, n_recent=0)
    # printed codes of channel 2 via the plane words (token i at bit i)
    words = u64(r["planes"][0, 2, :, 0])
    codes = [sum(((int(words[p]) >> i) & 1) << (3 - p) for p in range(4)) for i in range(6)]
    assert codes == GOLD["channel2"]["codes"]
    assert u16(r["scales"][0, 2])[0] == np.float16(0.5).view(np.uint16)
    check_unit(toy, r, 0, 2, 8, n_sink=0, n_recent=0)


def test_toy_reconstructed_k_printed_top2_on_the_gpu():
    # The toy's full K is not printed (only channel 2); tests/golden holds a K
    # reconstructed under the oracle so that every printed statement holds.  On
    # it the CUDA path must reproduce the printed outcomes: with the printed Var
    # and bracket, B = 8 keeps {t0, t3} for head A and {t5, t0} for head B, head
    # B's approximate scores match the printed ones to their 2 decimals, and
    # B = 6 misses head B's pair.
    rec = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "toy_k_reconstruction.json")))
    K = np.array(rec["K"], np.float32)
    keys = torch.tensor(K[None], device="cuda")
    q = torch.tensor([[GOLD["q_A"], GOLD["q_B"]]], dtype=torch.float32, device="cuda")
    var = torch.tensor([GOLD["var"]], dtype=torch.float32, device="cuda")
    br = torch.tensor([GOLD["bracket"]], dtype=torch.float64, device="cuda")
    shape = B.make_shape(1, 6, 4, 2, 2, 0, 0)
    planes, scales = B.fathom_quantize_pack(shape, keys)
    ws = B.alloc_workspace(shape, B.WS_SCAN_TOPK)
    P, S, C = O.quantize_pack(K)
    qn = q[0].cpu().numpy()
    for Bud in (8, 6):
        bud = torch.tensor([Bud], dtype=torch.int32, device="cuda")
        depth, theta, runs = B.fathom_plan(shape, q, var, bud, bracket=br)
        scores = torch.full((1, 2, 6), float("nan"), device="cuda")
        idx, sel = B.fathom_scan_topk(shape, planes, scales, runs, q, ws, scores=scores)
        torch.cuda.synchronize()
        od, _, _ = O.plan(qn, np.array(GOLD["var"], np.float32), Bud, bracket=GOLD["bracket"])
        np.testing.assert_array_equal(depth[0].cpu().numpy(), od)
        got = scores[0].cpu().numpy().astype(np.float64)
        ref = O.scores(P[None], S[None], od[None], qn[None], 6)[0]
        mag = fathom_cases.khat_magnitude(C, S, od, qn, 6)
        assert np.all(np.abs(got - ref) <= fathom_cases.SCORE_RTOL * mag + 1e-30)
        kept = [set(idx[0, h].tolist()) for h in range(2)]
        if Bud == 8:
            assert depth[0].tolist() == GOLD["B8"]["depth"]
            assert kept[0] == set(GOLD["top2"]["A"]) and kept[1] == set(GOLD["top2"]["B"])
            np.testing.assert_allclose(got[1], GOLD["head_B_scores"]["approx"], rtol=0, atol=0.005)
        else:
            assert depth[0].tolist() == GOLD["B6"]["depth"]
            assert kept[1] != set(GOLD["top2"]["B"])


# ------------------------------------------------------------------ store / calibration
@pytest.mark.parametrize("n,dtype", [(4096, "f32"), (4096 + 37, "bf16"), (64, "bf16"), (1, "f32")])
def test_quantize_bit_exact(n, dtype):
    w = W("qwen3_32k", keys_dtype=dtype)
    inp = Inputs(w, [0, 5, 17], n)
    shape = B.make_shape(3, n, 128, 4, 1, 0, 0)
    planes, scales = B.fathom_quantize_pack(shape, inp.keys_in)
    torch.cuda.synchronize()
    for ui in range(3):
        P, S, _ = O.quantize_pack(inp.keys32[ui].cpu().numpy())
        np.testing.assert_array_equal(u64(planes[ui]), P)
        np.testing.assert_array_equal(u16(scales[ui]), S)


def test_quantize_edge_values():
    # zeros, exact cell edges, values above the fp16-rounded maximum, huge and tiny blocks
    rng = np.random.default_rng(3)
    n, D = 256, 16
    k = rng.normal(size=(n, D)).astype(np.float32)
    k[:64, 0] = 0.0                                  # a == 0 block
    k[64:128, 1] = np.float32(0.5) * np.arange(-32, 32) / 4   # exact multiples of s
    k[128:192, 2] = 1e-9                             # subnormal-range fp16 scale
    k[192:, 3] = 7e4                                 # saturating scale
    k[192, 3] = -7.1e4
    k[:, 4] = np.float32(1.00048828125)              # rounds down in fp16: |k| > a16
    keys = torch.tensor(k[None], device="cuda")
    shape = B.make_shape(1, n, D, 4, 1, 0, 0)
    planes, scales = B.fathom_quantize_pack(shape, keys)
    torch.cuda.synchronize()
    P, S, _ = O.quantize_pack(k)
    np.testing.assert_array_equal(u64(planes[0]), P)
    np.testing.assert_array_equal(u16(scales[0]), S)


def test_calibrate_bit_exact():
    w = W("qwen3_32k")
    calib = torch.stack([synth.unit_calib(w, u, "cuda") for u in range(5)])
    mean, var = B.fathom_calibrate(calib)
    torch.cuda.synchronize()
    for u in range(5):
        m64, v64 = O.calibrate(calib[u].cpu().numpy())
        np.testing.assert_array_equal(var[u].cpu().numpy(), v64.astype(np.float32))
        np.testing.assert_array_equal(mean[u].cpu().numpy(), m64.astype(np.float32))


# ------------------------------------------------------------------ plan
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_plan_bit_exact_over_budgets(G):
    w = W("qwen3_32k", G=G)
    U = 64
    q = torch.stack([synth.unit_query(w, u, "cuda") for u in range(U)])
    calib = torch.stack([synth.unit_calib(w, u, "cuda") for u in range(U)])
    _, var = B.fathom_calibrate(calib)
    q[3] = 0.0                       # no live channel
    q[4, :, 5:] = 0.0                # few live channels
    budgets = np.array([0, 1, 7, 24, 32, 40, 48, 56, 64, 96, 128, 300, 512, 600] * 5, np.int32)[:U]
    shape = B.make_shape(U, 32768, 128, G, 1, 0, 0)
    depth, theta, runs = B.fathom_plan(shape, q, var, torch.tensor(budgets, device="cuda"))
    torch.cuda.synchronize()
    qn, vn = q.cpu().numpy(), var.cpu().numpy()
    for u in range(U):
        od, oth, _ = O.plan(qn[u], vn[u], int(budgets[u]))
        np.testing.assert_array_equal(depth[u].cpu().numpy(), od)
        assert theta[u].item() == oth
        np.testing.assert_array_equal(u32(runs[u]), O.runs(od, 32768))
        assert od.sum() <= max(budgets[u], 0)


def test_plan_bit_exact_across_magnitudes():
    # queries and variances scaled by powers of ten from 1e-30 to 1e30: the
    # bisection's geometric midpoints then cover most of the double exponent
    # range (including the ends, where the plan falls back to fp64 operations)
    # and must still give the oracle's theta bit for bit
    w = W("qwen3_32k")
    U = 512
    gen = torch.Generator(device="cpu").manual_seed(20260123)
    q = torch.stack([synth.unit_query(w, u % 64, "cuda") for u in range(U)])
    _, var = B.fathom_calibrate(torch.stack([synth.unit_calib(w, u % 64, "cuda") for u in range(U)]))
    sq = 10.0 ** torch.randint(-15, 16, (U, 1, 1), generator=gen).double()
    sv = 10.0 ** torch.randint(-30, 31, (U, 1), generator=gen).double()
    q = (q.double().cpu() * sq).float().cuda().contiguous()
    var = (var.double().cpu() * sv).float().cuda().contiguous()
    budgets = np.array([8, 24, 48, 64, 100, 200, 400], np.int32)[np.arange(U) % 7]
    shape = B.make_shape(U, 65536, 128, 4, 1, 0, 0)
    depth, theta, runs = B.fathom_plan(shape, q, var, torch.tensor(budgets, device="cuda"))
    torch.cuda.synchronize()
    qn, vn = q.cpu().numpy(), var.cpu().numpy()
    th = theta.cpu().numpy()
    dn = depth.cpu().numpy()
    for u in range(U):
        od, oth, _ = O.plan(qn[u], vn[u], int(budgets[u]))
        np.testing.assert_array_equal(dn[u], od)
        assert th[u] == oth, (u, th[u], oth)


def test_plan_without_theta_gives_the_same_depths_and_runs():
    # theta not requested: the kernel may take the depths straight from the
    # breakpoint above b*; over budgets, magnitudes and near-coincident
    # breakpoints the depths and runs must equal the oracle's (and the call with
    # theta), bit for bit
    w = W("qwen3_32k")
    U = 448
    gen = torch.Generator(device="cpu").manual_seed(20260311)
    q = torch.stack([synth.unit_query(w, u % 64, "cuda") for u in range(U)])
    _, var = B.fathom_calibrate(torch.stack([synth.unit_calib(w, u % 64, "cuda") for u in range(U)]))
    sq = 10.0 ** torch.randint(-15, 16, (U, 1, 1), generator=gen).double()
    sv = 10.0 ** torch.randint(-30, 31, (U, 1), generator=gen).double()
    sq[:64] = 1.0
    sv[:64] = 1.0
    q = (q.double().cpu() * sq).float()
    var = (var.double().cpu() * sv).float()
    # units 64..127: pairs of channels with importances a few ulps apart
    # (q one fp32 ulp up, var 2^-22 down), so breakpoints nearly coincide
    q[64:128, :, 1::2] = torch.nextafter(q[64:128, :, 0::2], torch.full_like(q[64:128, :, 0::2], 1e30))
    var[64:128, 1::2] = var[64:128, 0::2] * (1.0 - 2.0 ** -22)
    q[5] = 0.0
    q, var = q.cuda().contiguous(), var.cuda().contiguous()
    budgets = np.array([0, 1, 7, 8, 24, 48, 64, 100, 200, 400, 512, 600], np.int32)[np.arange(U) % 12]
    bt = torch.tensor(budgets, device="cuda")
    shape = B.make_shape(U, 65536, 128, 4, 1, 0, 0)
    d1, t1, r1 = B.fathom_plan(shape, q, var, bt)
    d0, t0, r0 = B.fathom_plan(shape, q, var, bt, want_theta=False)
    torch.cuda.synchronize()
    assert t0 is None
    torch.testing.assert_close(d0, d1, rtol=0, atol=0)
    torch.testing.assert_close(r0, r1, rtol=0, atol=0)
    qn, vn, dn = q.cpu().numpy(), var.cpu().numpy(), d0.cpu().numpy()
    for u in range(U):
        od, _, _ = O.plan(qn[u], vn[u], int(budgets[u]))
        np.testing.assert_array_equal(dn[u], od)
        np.testing.assert_array_equal(u32(r0[u]), O.runs(od, 65536))


def test_plan_explicit_bracket_and_fixed():
    w = W("qwen3_32k")
    U = 16
    q = torch.stack([synth.unit_query(w, u, "cuda") for u in range(U)])
    _, var = B.fathom_calibrate(torch.stack([synth.unit_calib(w, u, "cuda") for u in range(U)]))
    shape = B.make_shape(U, 1 << 20, 128, 4, 1, 0, 0)
    br = torch.tensor([[1e-3, 1e3]] * U, dtype=torch.float64, device="cuda")
    bud = torch.full((U,), 48, dtype=torch.int32, device="cuda")
    depth, theta, runs = B.fathom_plan(shape, q, var, bud, bracket=br)
    fdepth, fruns = B.fathom_plan_fixed(shape, q, var, 32, 4)
    torch.cuda.synchronize()
    for u in range(U):
        qn, vn = q[u].cpu().numpy(), var[u].cpu().numpy()
        od, oth, _ = O.plan(qn, vn, 48, bracket=[1e-3, 1e3])
        np.testing.assert_array_equal(depth[u].cpu().numpy(), od)
        assert theta[u].item() == oth
        fd = O.plan_fixed(qn, vn, 32, 4)
        np.testing.assert_array_equal(fdepth[u].cpu().numpy(), fd)
        np.testing.assert_array_equal(u32(fruns[u]), O.runs(fd, 1 << 20))


def test_gather_copies_nothing_for_a_corrupted_run():
    # a run whose source fields are not the ones the plan writes for its channel
    # (another channel's planes, more than four planes, a partial plane, another
    # channel's scales, more scales than blocks) would read outside the channel's
    # part of the store: the gather copies nothing for it, and every other
    # channel exactly as the oracle does
    w = W("qwen3_32k", n=4096)
    inp = Inputs(w, [0], 4096)
    shape = B.make_shape(1, 4096, 128, 4, 1, 0, 0)
    planes, scales = B.fathom_quantize_pack(shape, inp.keys_in)
    _, var = B.fathom_calibrate(inp.calib)
    depth, _, runs = B.fathom_plan(shape, inp.q, var, torch.tensor([48], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    nb = B.nblocks(4096)
    r = u32(runs[0]).copy()
    act = np.nonzero(depth[0].cpu().numpy())[0]
    assert len(act) >= 5
    bad = act[:5]
    r[bad[0], 0] = (bad[0] + 1) * 4 * nb          # src_word of the next channel
    r[bad[1], 1] = 5 * nb                          # five planes
    r[bad[2], 1] = r[bad[2], 1] + 1                # not whole planes
    r[bad[3], 3] = (bad[3] + 1) * nb               # src_scale of the next channel
    r[bad[4], 4] = nb + 1                          # more scales than blocks
    runs_bad = torch.tensor(r.view(np.int32)[None], device="cuda").contiguous()
    W_, S_ = 48 * nb, 48 * nb
    sp = torch.zeros(1, W_, dtype=torch.int64, device="cuda")
    ss = torch.zeros(1, S_, dtype=torch.int16, device="cuda")
    B.fathom_gather(shape, planes.cpu().pin_memory(), scales.cpu().pin_memory(), runs_bad, sp, ss)
    torch.cuda.synchronize()
    ref_runs = u32(runs[0]).copy()
    ref_runs[bad, 1] = 0                           # nothing copied for the corrupted channels
    ref_runs[bad, 4] = 0
    rp, rs = O.gather(ref_runs, u64(planes[0]), u16(scales[0]), W_, S_)
    np.testing.assert_array_equal(u64(sp[0]), rp)
    np.testing.assert_array_equal(u16(ss[0]), rs)


# ------------------------------------------------------------------ whole path, small
@pytest.mark.parametrize("regime", ["hbm", "host"])
def test_single_layer_4k_full_parity(regime):
    w = synth.WORKLOADS["single_4k"]
    inp = Inputs(w, [0], w.n)
    r = run_gpu(inp, k=w.k, budget=48, regime=regime)
    check_unit(inp, r, 0, w.k, 48)


def test_ragged_multi_tile_multi_unit():
    # several sub-chunks and chunks per unit, a ragged tail block, bf16 keys
    w = W("qwen3_32k", n=6481)
    inp = Inputs(w, [0, 1, 2], 6481)
    r = run_gpu(inp, k=300, budget=[40, 48, 56])
    for ui in range(3):
        check_unit(inp, r, ui, 300, [40, 48, 56])


@pytest.mark.parametrize("regime", ["hbm", "host", "fused"])
def test_scan_and_select_halves_equal_scan_topk(regime):
    # fathom_scan then fathom_select (here on two streams, ordered by an event)
    # give exactly fathom_scan_topk's kept sets and scores, for grids that fill
    # every SM and for grids limited to 1 or 2 scan CTAs per SM
    w = W("qwen3_32k", n=40000)
    inp = Inputs(w, [0, 1, 2, 3], 40000)
    r = run_gpu(inp, k=512, budget=48, regime=regime)
    if regime == "host":
        src_p, src_s, source = r["stage_planes"], r["stage_scales"], B.SRC_STAGING
    elif regime == "fused":
        src_p, src_s, source = r["planes"].cpu().pin_memory(), r["scales"].cpu().pin_memory(), B.SRC_STORE
    else:
        src_p, src_s, source = r["planes"], r["scales"], B.SRC_STORE
    side = torch.cuda.Stream()
    for per_sm in (0, 1, 2):
        shape = B.make_shape(4, 40000, 128, 4, 512, 4, 32, 0, per_sm)
        ws = B.alloc_workspace(shape, B.WS_SCAN_TOPK)
        scores = torch.full((4, 4, 40000), float("nan"), device="cuda")
        B.fathom_scan(shape, src_p, src_s, r["runs"], inp.q, ws, source=source, scores=scores)
        ev = torch.cuda.Event()
        ev.record()
        side.wait_event(ev)
        with torch.cuda.stream(side):
            idx, sel = B.fathom_select(shape, src_p, src_s, r["runs"], inp.q, ws, source=source)
        torch.cuda.synchronize()
        torch.testing.assert_close(idx, r["idx"], rtol=0, atol=0)
        torch.testing.assert_close(sel, r["sel"], rtol=0, atol=0)
        torch.testing.assert_close(scores, r["scores"], rtol=0, atol=0)
        # and the one-call form with the limited grid
        idx2, sel2 = B.fathom_scan_topk(shape, src_p, src_s, r["runs"], inp.q, ws, source=source)
        torch.cuda.synchronize()
        torch.testing.assert_close(idx2, r["idx"], rtol=0, atol=0)


def test_long_chunks_exercise_pruning():
    # 152 units x 64k tokens: a few chunks per unit (one full wave of CTAs over
    # 152 units), each of 8 or more sub-chunks -> in-CTA prunes
    w = W("qwen3_32k", n=65536)
    U = 152
    inp = Inputs(w, range(U), 65536)
    r = run_gpu(inp, k=512, budget=48, want_scores=True)
    for ui in (0, 77, 151):
        check_unit(inp, r, ui, 512, 48, check_attn=(ui == 0))


@pytest.mark.parametrize("G", [1, 2, 8])
def test_other_group_sizes(G):
    w = W("qwen3_32k", G=G, n=5000)
    inp = Inputs(w, [3, 4], 5000)
    r = run_gpu(inp, k=128, budget=64)
    for ui in range(2):
        check_unit(inp, r, ui, 128, 64)


def test_dense_budget_and_small_D():
    w = W("qwen3_32k", D=24, n=3000)
    inp = Inputs(w, [1], 3000)
    r = run_gpu(inp, k=100, budget=4 * 24)        # every channel at depth 4
    assert int(r["depth"].min()) == 4
    check_unit(inp, r, 0, 100, 4 * 24)


@pytest.mark.parametrize("k,ns,nr", [(36, 4, 32), (2000, 4, 32), (2000, 0, 0), (7, 0, 0), (40, 20, 20),
                                     (2048, 0, 0)])
def test_selection_edges(k, ns, nr):
    n = 2000 if k <= 2000 else 2600
    w = W("qwen3_32k", n=n)
    inp = Inputs(w, [2], n)
    r = run_gpu(inp, k=k, budget=48, n_sink=ns, n_recent=nr)
    check_unit(inp, r, 0, k, 48, n_sink=ns, n_recent=nr)


def test_tiny_sequences():
    for n, k, ns, nr in ((1, 1, 0, 0), (5, 5, 4, 32), (40, 36, 4, 32), (70, 40, 4, 32)):
        w = W("qwen3_32k", n=n)
        inp = Inputs(w, [0], n)
        r = run_gpu(inp, k=k, budget=48, n_sink=ns, n_recent=nr)
        check_unit(inp, r, 0, k, 48, n_sink=ns, n_recent=nr)


def test_all_ties_break_by_index():
    w = W("qwen3_32k", n=4096)
    inp = Inputs(w, [0], 4096)
    inp.q.zero_()                      # every score is 0: lowest free indices win
    r = run_gpu(inp, k=64, budget=48)
    assert int(r["depth"].sum()) == 0
    idx = r["idx"][0].cpu().numpy()
    for h in range(4):
        assert idx[h].tolist() == list(range(4)) + list(range(4, 32)) + list(range(4064, 4096))


def test_staged_equals_in_place_and_fixed_plan():
    w = W("host_256k", n=20000)
    inp = Inputs(w, [0, 1], 20000)
    a = run_gpu(inp, k=256, budget=64, regime="hbm")
    b = run_gpu(inp, k=256, budget=64, regime="host")
    assert torch.equal(a["idx"], b["idx"]) and torch.equal(a["scores"], b["scores"])
    c = run_gpu(inp, k=256, budget=0, regime="host", fixed=(32, 4))
    check_unit(inp, c, 1, 256, 0, fixed=(32, 4))


def test_workspace_reuse_across_calls():
    w = W("qwen3_32k", n=8192)
    inp = Inputs(w, [0, 1, 2, 3], 8192)
    shape = B.make_shape(4, 8192, 128, 4, 256)
    r = run_gpu(inp, k=256, budget=48)
    ws = B.alloc_workspace(shape, B.WS_SCAN_TOPK)
    aws = B.alloc_workspace(shape, B.WS_SPARSE_ATTN)
    outs = []
    for _ in range(3):
        idx, _ = B.fathom_scan_topk(shape, r["planes"], r["scales"], r["runs"], inp.q, ws)
        outs.append((idx.clone(), B.fathom_sparse_attn(shape, inp.krows, inp.vrows, inp.q, idx, aws).clone()))
    torch.cuda.synchronize()
    for idx, out in outs[1:]:
        assert torch.equal(idx, outs[0][0]) and torch.equal(out, outs[0][1])
    assert torch.equal(outs[0][0], r["idx"])


def test_concentrated_winners_force_the_exact_second_pass():
    # one unit of 64k tokens is split into 32 chunks that each keep only about
    # their top-60 in the first pass; amplifying the keys of one 2048-token stretch
    # puts all k' = 476 winners in one chunk, which the merge must flag and the
    # second pass must rescan exactly
    w = W("qwen3_32k", n=65536)
    inp = Inputs(w, [0, 1], 65536)
    for t in (inp.keys_in, inp.keys32, inp.krows):
        t[:, 40960:43008] *= 4
    r = run_gpu(inp, k=512, budget=48)
    for ui in range(2):
        check_unit(inp, r, ui, 512, 48)
    idx = r["idx"][0].cpu().numpy()
    free = idx[:, 4:-32]
    assert np.mean((free >= 40960) & (free < 43008)) > 0.9


@pytest.mark.parametrize("where", ["device", "host"])
@pytest.mark.parametrize("rows", [128, 256, 512])
def test_attention_for_each_rows_per_cta_choice(rows, where):
    # The attention takes 128, 256 or 512 kept-list entries per CTA depending on how
    # many (unit, head) pairs the call has (more pairs: fewer, longer CTAs).  Unit
    # counts that select each choice on this device, rows in device and in pinned
    # host memory; random strictly ascending kept lists (one entry out of range per
    # head: skipped) checked on every unit.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    G, k, n, D = 4, 512, 2048, 128
    per_unit128, per_unit512 = G * (k // 128), G * (k // 512)
    units = {128: 8,
             256: 4 * sms // per_unit128 + 1,
             512: -(-4 * sms // per_unit512)}[rows]
    shape = B.make_shape(units, n, D, G, k, 4, 32)
    rng = np.random.default_rng(900 + rows)
    kr = torch.from_numpy(rng.standard_normal((units, n, D)).astype(np.float32)).to(torch.bfloat16).cuda()
    vr = torch.from_numpy(rng.standard_normal((units, n, D)).astype(np.float32)).to(torch.bfloat16).cuda()
    q = torch.from_numpy(rng.standard_normal((units, G, D)).astype(np.float32)).cuda()
    idx = np.empty((units, G, k), np.int32)
    for u in range(units):
        for h in range(G):
            sel = np.sort(rng.choice(n, size=k - 1, replace=False)).astype(np.int32)
            idx[u, h] = np.concatenate([sel, [n + 5]])       # the last entry lies outside [0, n)
    if where == "host":
        kr, vr = kr.cpu().pin_memory(), vr.cpu().pin_memory()
    out = B.fathom_sparse_attn(shape, kr, vr, q, torch.from_numpy(idx).cuda(),
                               B.alloc_workspace(shape, B.WS_SPARSE_ATTN))
    torch.cuda.synchronize()
    for u in range(units):
        # the oracle over the in-range entries (it reads every entry it is given)
        ref = O.attention(u16(kr[u]), u16(vr[u]), q[u].cpu().numpy(), np.ascontiguousarray(idx[u][:, :k - 1]))
        got = out[u].cpu().numpy().astype(np.float64)
        rel = np.linalg.norm(got - ref, axis=1) / np.linalg.norm(ref, axis=1)
        assert np.all(rel <= fathom_cases.ATTN_RTOL), (u, rel)


@pytest.mark.parametrize("k", [512, 36])
def test_many_units_use_the_small_merge(k):
    # enough (unit, head) pairs for the 256-thread merge build (four CTAs per SM):
    # every unit's store, plan, scores, kept set and attention against the oracle
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    units = -(-2 * sms // 4)                     # 2 x SMs pairs at G = 4
    w = W("qwen3_32k", n=4096)
    inp = Inputs(w, range(units), 4096)
    r = run_gpu(inp, k=k, budget=48)
    for ui in range(units):
        check_unit(inp, r, ui, k, 48)


def test_attention_union_form_beyond_the_grid_limit():
    # more than 65535 (unit, head) pairs: the attention falls back to one grid row
    # per unit (the union of its heads' kept rows, fetched once for all G heads)
    G, k, n, D = 4, 40, 64, 128
    units = 65536 // G + 3
    shape = B.make_shape(units, n, D, G, k, 4, 4)
    g = torch.Generator(device="cuda").manual_seed(31)
    kr = torch.randn(units, n, D, device="cuda", generator=g).to(torch.bfloat16)
    vr = torch.randn(units, n, D, device="cuda", generator=g).to(torch.bfloat16)
    q = torch.randn(units, G, D, device="cuda", generator=g)
    idx = torch.stack([torch.stack([torch.randperm(n, device="cuda", generator=g)[:k].sort().values
                                    for _ in range(G)]) for _ in range(8)]).int()
    idx = idx.repeat((units + 7) // 8, 1, 1)[:units].contiguous()
    out = B.fathom_sparse_attn(shape, kr, vr, q, idx, B.alloc_workspace(shape, B.WS_SPARSE_ATTN))
    torch.cuda.synchronize()
    for u in (0, 1, units // 2, units - 1):
        ref = O.attention(u16(kr[u]), u16(vr[u]), q[u].cpu().numpy(), idx[u].cpu().numpy())
        got = out[u].cpu().numpy().astype(np.float64)
        rel = np.linalg.norm(got - ref, axis=1) / np.linalg.norm(ref, axis=1)
        assert np.all(rel <= fathom_cases.ATTN_RTOL), (u, rel)
